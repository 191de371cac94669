"""GPU parity of ctx_attn_lq_gkv against the fp64 oracle.

Tolerance (bf16 N(0,1) inputs): O within max-abs 2e-2 and mean-abs 2e-3 of
the oracle, LSE within 1e-3 (absolute, natural log). Small shapes are
compared in full; the workload shapes at full size in the launch
configuration the benchmark uses are compared on a seeded sample of query
rows that always holds the first tile and the ragged tail.
"""
import math

import numpy as np
import pytest
import torch

import workloads
from gpu_util import Guarded, u16

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def ctx():
    import diffusion_transformer_context_gb300 as m
    m.build()
    return m


def _run(ctx, q, k, v, mask=None, scale=None, guard=False, split=False):
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if guard:
        out = Guarded((B, Sq, H, D), q.dtype)
        lse = Guarded((B, H, Sq), torch.float32)
        o_t, l_t = out.t, lse.t
    else:
        o_t = torch.empty((B, Sq, H, D), dtype=q.dtype, device="cuda")
        l_t = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    ws = ctx.attn_workspace(B, Sq, Sk, H, D) if split else None
    m = None if mask is None else torch.from_numpy(mask).cuda()
    ctx.ctx_attn_lq_gkv(q.cuda(), k.cuda(), v.cuda(), o_t, l_t, key_mask=m, scale=scale, workspace=ws)
    st = ctx.ctx_device_status()
    assert st == 0, ctx.ctx_status_string(st)
    if guard:
        assert out.intact() and lse.intact()
    if split:
        # the arrival counters at the head of the workspace are zero again
        n_units = ((Sq + 255) // 256) * H * B
        assert int(ws[:n_units * 2 * 2 * 4].count_nonzero()) == 0  # arrived / written per tile
    return o_t.float().cpu().numpy(), l_t.cpu().numpy()


def _check_full(orc, q, k, v, O, L, mask=None, scale=None, dtype="bf16"):
    eO, eL = orc.attention(u16(q), u16(k), u16(v), mask, scale, dtype)
    err = np.abs(O - eO)
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    fin = np.isfinite(eL)
    assert np.array_equal(np.isfinite(L), fin)
    assert (L[~fin] == -np.inf).all()
    if fin.any():
        assert np.abs(L[fin] - eL[fin]).max() <= LSE_TOL
    return err


SMALL = [  # B, Sq, Sk, H, D
    (1, 128, 128, 1, 128),
    (1, 512, 512, 2, 128),
    (2, 300, 700, 3, 128),
    (1, 1, 1, 1, 128),
    (1, 200, 129, 2, 64),
    (1, 257, 1000, 2, 128),
    (3, 64, 130, 1, 64),
]


@pytest.mark.parametrize("split", [False, True], ids=["per_unit", "balanced"])
@pytest.mark.parametrize("B,Sq,Sk,H,D", SMALL)
def test_small_shapes_full(ctx, orc, B, Sq, Sk, H, D, split):
    gen = torch.Generator().manual_seed(1234)
    q, k, v = (workloads.randn(s, gen) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    O, L = _run(ctx, q, k, v, guard=True, split=split)
    _check_full(orc, q, k, v, O, L)


def test_fp16(ctx, orc):
    gen = torch.Generator().manual_seed(3)
    B, Sq, Sk, H, D = 2, 190, 333, 2, 128
    q, k, v = (workloads.randn(s, gen, "fp16") for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    O, L = _run(ctx, q, k, v)
    _check_full(orc, q, k, v, O, L, dtype="fp16")


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("split", [False, True], ids=["per_unit", "balanced"])
@pytest.mark.parametrize("kind", ["random", "rear_text", "front_text", "first_block_empty", "first_half_empty",
                                  "row_empty"])
def test_key_mask(ctx, orc, kind, split, D):
    gen = torch.Generator().manual_seed(11)
    B, Sq, Sk, H = 2, 200, 600, 2
    q, k, v = (workloads.randn(s, gen) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    mask = np.ones((B, Sk), np.uint8)
    rng = np.random.default_rng(0)
    if kind == "random":
        mask = (rng.random((B, Sk)) > 0.3).astype(np.uint8) * rng.integers(1, 255, (B, Sk)).astype(np.uint8)
    elif kind == "rear_text":       # 344 image keys then 256 text keys, padded suffix
        mask[0, 344 + 40:] = 0
        mask[1, 344 + 200:] = 0
    elif kind == "front_text":      # 256 text keys (padded) then image keys
        mask[0, 33:256] = 0
        mask[1, 180:256] = 0
    elif kind == "first_block_empty":
        mask[:, :300] = 0
    elif kind == "first_half_empty":  # 5 key blocks: without a workspace the first 3 (one slot's half) are all masked
        mask[:, :384] = 0
    elif kind == "row_empty":
        mask[1, :] = 0
    O, L = _run(ctx, q, k, v, mask=mask, guard=True, split=split)
    _check_full(orc, q, k, v, O, L, mask=mask)
    if kind == "row_empty":
        assert (O[1] == 0).all() and np.isneginf(L[1]).all()


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("scale", [1.0, 0.01, 0.35])
def test_scale_and_rescaling(ctx, orc, scale, D):
    """scale 1.0 makes the scores ~N(0, D): row maxima keep growing across
    key blocks, which exercises the conditional O rescaling (D = 128 and 64)."""
    gen = torch.Generator().manual_seed(12)
    B, Sq, Sk, H = 1, 256, 1024, 2
    q, k, v = (workloads.randn(s, gen) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    O, L = _run(ctx, q, k, v, scale=scale)
    _check_full(orc, q, k, v, O, L, scale=scale)


def test_growing_maximum_sorted_keys(ctx, orc):
    """Keys ordered so that later blocks hold larger scores: every block
    raises the row maximum by more than the rescale threshold."""
    gen = torch.Generator().manual_seed(13)
    B, Sq, Sk, H, D = 1, 128, 1024, 1, 128
    q = workloads.randn((B, Sq, H, D), gen)
    k = workloads.randn((B, Sk, H, D), gen).float()
    v = workloads.randn((B, Sk, H, D), gen)
    k = (k * torch.linspace(0.1, 4.0, Sk).view(1, Sk, 1, 1)).to(torch.bfloat16)
    O, L = _run(ctx, q, k, v, scale=0.5)
    _check_full(orc, q, k, v, O, L, scale=0.5)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("split", [False, True], ids=["per_unit", "balanced"])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_running_maximum_jumps(ctx, orc, dtype, split, D):
    """After a segment's first key block the kernel takes the exps against
    the running maximum and checks the block's probability sum (at most 2^15)
    instead of computing the block maximum. Query rows close to one direction
    u and small random keys keep the early maxima near 0; in key block 5 one
    key is a multiple of u whose score jumps by about 11.4 log2 units on head
    0 (p ~ 2^11: accepted, no rescale) and by about 17.3 on head 1 (p ~ 2^17:
    the block is redone with its exact maximum and O rescaled). At D = 128
    and D = 64."""
    gen = torch.Generator().manual_seed(21)
    B, Sq, Sk, H = 1, 256, 1024, 2
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    u = torch.where(torch.rand(D, generator=gen) < 0.5, -1.0, 1.0)
    q = (u.view(1, 1, 1, D) + 0.05 * torch.randn((B, Sq, H, D), generator=gen)).to(tdt)
    k = (0.1 * torch.randn((B, Sk, H, D), generator=gen))
    v = torch.randn((B, Sk, H, D), generator=gen).to(tdt)
    j = 5 * 128 + 37
    for h, s_nat in ((0, 8.0), (1, 12.0)):  # natural-log score of the special key
        k[0, j, h] = u * (s_nat / math.sqrt(D))
    k = k.to(tdt)
    O, L = _run(ctx, q, k, v, split=split)
    _check_full(orc, q, k, v, O, L, dtype=dtype)


@pytest.mark.parametrize("D", [128, 64])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("split", [False, True], ids=["per_unit", "balanced"])
def test_running_maximum_jumps_late_in_block(ctx, orc, dtype, split, D):
    """Jumps of the running maximum late in a key block (key 100 of block 5,
    past the first 64 keys): about 17.3 log2 units on head 0 (the block sum
    check fails and the block is redone with its exact maximum, O rescaled),
    about 11.4 on head 1 (accepted), and on head 2 two jumps in a row, early
    in block 5 and late in block 6, the second far above the first."""
    gen = torch.Generator().manual_seed(24)
    B, Sq, Sk, H = 1, 256, 1024, 3
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    u = torch.where(torch.rand(D, generator=gen) < 0.5, -1.0, 1.0)
    q = (u.view(1, 1, 1, D) + 0.05 * torch.randn((B, Sq, H, D), generator=gen)).to(tdt)
    k = (0.1 * torch.randn((B, Sk, H, D), generator=gen))
    v = torch.randn((B, Sk, H, D), generator=gen).to(tdt)
    for h, j, s_nat in ((0, 5 * 128 + 100, 12.0), (1, 5 * 128 + 100, 8.0),
                        (2, 5 * 128 + 20, 12.0), (2, 6 * 128 + 90, 20.0)):
        k[0, j, h] = u * (s_nat / math.sqrt(D))  # natural-log score of the special key
    k = k.to(tdt)
    O, L = _run(ctx, q, k, v, split=split)
    _check_full(orc, q, k, v, O, L, dtype=dtype)


@pytest.mark.parametrize("masked", [False, True])
def test_one_unit_cut_over_every_sm(ctx, orc, masked):
    """One work unit (256 query rows of one head) against 304 key blocks: the
    balanced schedule gives every SM two of its key blocks, so the unit's
    last piece merges one partial result per SM by log-sum-exp."""
    gen = torch.Generator().manual_seed(22)
    B, Sq, Sk, H, D = 1, 256, 304 * 128, 1, 128
    q, k, v = (workloads.randn(s, gen) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    mask = None
    if masked:  # whole pieces and single keys masked out
        mask = (np.random.default_rng(22).random((B, Sk)) > 0.3).astype(np.uint8)
        mask[:, 5000:9000] = 0
    O, L = _run(ctx, q, k, v, mask=mask, split=True)
    _check_full(orc, q, k, v, O, L, mask=mask)


@pytest.mark.parametrize("shape", [(1, 2048, 4352, 12), (1, 300, 4096, 1)], ids=["two_three_pieces", "many_pieces"])
def test_split_merge_reproducible(ctx, shape):
    """A short call's split units are merged by whichever piece arrives last;
    the result must not depend on which one that is. One Qwen-like rank (96
    units of 34 key blocks over the SMs' even shares: units cut into two and
    into three pieces) and one unit cut over every SM, each called repeatedly
    on one workspace: outputs and LSE bit-identical every time."""
    B, Sq, Sk, H = shape
    gen = torch.Generator().manual_seed(23)
    q, k, v = (workloads.randn(s, gen).cuda() for s in ((B, Sq, H, 128), (B, Sk, H, 128), (B, Sk, H, 128)))
    ws = ctx.attn_workspace(B, Sq, Sk, H, 128)
    o0, l0 = torch.empty_like(q), torch.empty((B, H, Sq), device="cuda")
    ctx.ctx_attn_lq_gkv(q, k, v, o0, l0, workspace=ws)
    for _ in range(6):
        o, l = torch.empty_like(q), torch.empty((B, H, Sq), device="cuda")
        ctx.ctx_attn_lq_gkv(q, k, v, o, l, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(o.view(torch.int16), o0.view(torch.int16))
        assert torch.equal(l.view(torch.int32), l0.view(torch.int32))
    assert ctx.ctx_device_status() == 0


def test_deterministic(ctx):
    gen = torch.Generator().manual_seed(14)
    B, Sq, Sk, H, D = 1, 512, 2048, 4, 128
    q, k, v = (workloads.randn(s, gen).cuda() for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    o1, l1 = torch.empty_like(q), torch.empty((B, H, Sq), device="cuda")
    o2, l2 = torch.empty_like(q), torch.empty((B, H, Sq), device="cuda")
    ctx.ctx_attn_lq_gkv(q, k, v, o1, l1)
    ctx.ctx_attn_lq_gkv(q, k, v, o2, l2)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_lse_optional(ctx, orc):
    gen = torch.Generator().manual_seed(15)
    q, k, v = (workloads.randn(s, gen) for s in ((1, 130, 2, 128), (1, 260, 2, 128), (1, 260, 2, 128)))
    out = torch.empty((1, 130, 2, 128), dtype=torch.bfloat16, device="cuda")
    ctx.ctx_attn_lq_gkv(q.cuda(), k.cuda(), v.cuda(), out)
    torch.cuda.synchronize()
    eO, _ = orc.attention(u16(q), u16(k), u16(v))
    assert np.abs(out.float().cpu().numpy() - eO).max() <= O_MAX


# ---------------------------------------------------------------- full sizes

def full_size_rows(B, H, Sq, n_random, seed=1234):
    """(b, h, i) rows checked at full size: n_random seeded random rows spread
    evenly over every (b, h) pair, the first 128-row tile of the first and
    last (b, h), and, for EVERY (b, h), the last 256-row work unit (the
    ragged tail included) and the last 256 rows (so the last full 128-row
    tile too when the last unit is short)."""
    rng = np.random.default_rng(seed)
    rows = set()
    pairs = [(b, h) for b in range(B) for h in range(H)]
    for k in range(n_random):
        b, h = pairs[k % len(pairs)]
        rows.add((b, h, int(rng.integers(0, Sq))))
    for b, h in (pairs[0], pairs[-1]):
        rows.update((b, h, i) for i in range(min(128, Sq)))
    unit0 = min(((Sq - 1) // 256) * 256, max(0, Sq - 256))
    for b, h in pairs:
        rows.update((b, h, i) for i in range(unit0, Sq))
    return np.array(sorted(rows), dtype=np.int64)


def _sampled(ctx, orc, B, Sq, Sk, H, D, n_rows, mask=None, seed=1234, split=True, all_heads_tail=False):
    gen = torch.Generator().manual_seed(seed)
    q, k, v = (workloads.randn(s, gen) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    O, L = _run(ctx, q, k, v, mask=mask, split=split)
    if all_heads_tail:
        bhi = full_size_rows(B, H, Sq, n_rows, seed)
    else:
        rows_i = workloads.sample_rows(Sq, n_rows)
        rng = np.random.default_rng(seed)
        bhi = np.stack([rng.integers(0, B, rows_i.size), rng.integers(0, H, rows_i.size), rows_i], axis=1)
    eo, el = orc.attention_rows(u16(q), u16(k), u16(v), bhi, mask)
    got_o = O[bhi[:, 0], bhi[:, 2], bhi[:, 1]]
    got_l = L[bhi[:, 0], bhi[:, 1], bhi[:, 2]]
    err = np.abs(got_o - eo)
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    assert np.abs(got_l - el).max() <= LSE_TOL
    return len(bhi)


def test_full_size_row_sample_covers_the_tails():
    """The sampler itself: >= 512 random rows over all heads plus every
    (b, h)'s last unit (the 480p call: 4095 query rows, a ragged last tile)."""
    bhi = full_size_rows(1, 12, 4095, 512)
    assert len(bhi) >= 512 + 12 * 255
    for h in range(12):
        sel = bhi[bhi[:, 1] == h, 2]
        assert set(range(3840, 4095)) <= set(sel.tolist())


def test_qwen_full_size_sampled(ctx, orc):
    """U=2 x A=2 Qwen-Image-like: both head groups batched, local-Q of both
    A ranks stacked: Q [2,4096,12,128] vs K/V [2,4352,12,128] with the
    text-padding mask (valid text length uniform in [32,256]), merged by the
    oracle from the raw joint mask (joint keys after the image keys)."""
    wl = workloads.WORKLOADS["qwen"]
    inp = workloads.make_inputs(wl)
    m = orc.merge_joint_attn_mask(inp.image_mask, inp.joint_mask, wl.B, wl.S, wl.joint, wl.joint_front)
    mask = np.tile(m, (wl.U, 1))
    _sampled(ctx, orc, wl.U * wl.B, wl.S, wl.Sk, wl.h_l, wl.D, 512, mask=mask, all_heads_tail=True)


def test_wan480_full_size_sampled(ctx, orc):
    """The 480p call as the benchmark runs it (8 ranks' local-Q stacked: Q
    [1,32760,12,128] vs K/V [1,32760,12,128], balanced schedule): 512 random
    rows over all 12 heads plus every head's last 256 rows."""
    wl = workloads.WORKLOADS["wan480"]
    n = _sampled(ctx, orc, wl.U * wl.B, wl.S, wl.Sk, wl.h_l, wl.D, 512, all_heads_tail=True)
    assert n >= 512 + 12 * 256


def test_wan480_one_rank_full_size_sampled(ctx, orc):
    """One rank of the 480p layer alone (Q [1,4095,12,128], the ragged last
    tile of 127 rows) against the whole gathered K/V."""
    _sampled(ctx, orc, 1, 4095, 32760, 12, 128, 512, all_heads_tail=True)


@pytest.mark.parametrize("shape,masked", [((1, 4095, 32760, 12), True), ((1, 9450, 75600, 10), False)],
                         ids=["wan480_rank_masked", "wan14b_rank_odd_blocks"])
def test_no_workspace_full_size_sampled(ctx, orc, shape, masked):
    """Calls without a workspace whose 256-row units would leave a partial
    last wave take the halves mode (128-row units, the two halves of the key
    range side by side in one CTA). One 480p rank (256 key blocks, a ragged
    last tile of 127 rows; 20 % of the keys masked), and one rank of Q 9450
    rows against 75600 keys (591 key blocks: the halves differ by one, the
    last block holds 80 keys; a ragged tail of 106 rows)."""
    B, Sq, Sk, H = shape
    mask = None
    if masked:
        mask = (np.random.default_rng(7).random((B, Sk)) > 0.2).astype(np.uint8)
    n = _sampled(ctx, orc, B, Sq, Sk, H, 128, 512, mask=mask, split=False, all_heads_tail=True)
    assert n >= 512 + H * 255


def test_wan14b_full_size_sampled(ctx, orc):
    """The Wan-14B-like call as the layer runs it (4 head groups batched, the
    local-Q of both A ranks stacked: Q [4,75600,10,128] vs K/V
    [4,75600,10,128]): 512 random rows over all 40 (b, h) pairs plus every
    pair's last 256 rows (the last unit holds 80)."""
    wl = workloads.WORKLOADS["wan14b"]
    n = _sampled(ctx, orc, wl.U * wl.B, wl.S, wl.Sk, wl.h_l, wl.D, 512, all_heads_tail=True)
    assert n >= 512 + 40 * 256


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_masked_long_call_takes_the_write_then_count_merge(ctx, orc, dtype):
    """A call whose CTAs run more than 160 key blocks (64 units of 512 key
    blocks on 152 SMs: ~215 each) merges its split units with the
    write-then-count protocol; here with a random key mask with masked
    stretches, in both 16-bit types, against the oracle at full size."""
    B, Sq, Sk, H, D = 1, 4096, 65536, 4, 128
    gen = torch.Generator().manual_seed(41)
    q, k, v = (workloads.randn(s, gen, dtype) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    rng = np.random.default_rng(41)
    mask = (rng.random((B, Sk)) > 0.2).astype(np.uint8)
    mask[:, 10000:30000] = 0
    O, L = _run(ctx, q, k, v, mask=mask, split=True)
    bhi = full_size_rows(B, H, Sq, 512, seed=41)
    eo, el = orc.attention_rows(u16(q), u16(k), u16(v), bhi, mask, dtype=dtype)
    err = np.abs(O[bhi[:, 0], bhi[:, 2], bhi[:, 1]] - eo)
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, (err.max(), err.mean())
    assert np.abs(L[bhi[:, 0], bhi[:, 1], bhi[:, 2]] - el).max() <= LSE_TOL


@pytest.mark.parametrize("B,Sq,Sk,H", [(1, 4095, 32760, 12), (1, 300, 4096, 1), (2, 2000, 3000, 5),
                                       (1, 40000, 700, 16)])
def test_balanced_schedule_matches_per_unit(ctx, B, Sq, Sk, H):
    """The key-split schedule (units cut between SMs, merged by log-sum-exp)
    agrees with one CTA per unit to fp32 rounding of the merge: same bf16
    output up to one ulp, LSE to 1e-5. Shapes: one rank of the Wan-like 480p
    layer (192 units: one whole wave, the 40 left over each cut into ~4
    pieces), a single unit split over many SMs, and uneven wave remainders
    where the last whole wave is split too (fewer than 32 key blocks per SM
    in the leftover units alone)."""
    gen = torch.Generator().manual_seed(21)
    q, k, v = (workloads.randn(s, gen).cuda() for s in ((B, Sq, H, 128), (B, Sk, H, 128), (B, Sk, H, 128)))
    o1, l1 = torch.empty_like(q), torch.empty((B, H, Sq), device="cuda")
    o2, l2 = torch.empty_like(q), torch.empty((B, H, Sq), device="cuda")
    ws = ctx.attn_workspace(B, Sq, Sk, H, 128)
    ctx.ctx_attn_lq_gkv(q, k, v, o1, l1)
    ctx.ctx_attn_lq_gkv(q, k, v, o2, l2, workspace=ws)
    ctx.ctx_attn_lq_gkv(q, k, v, o2, l2, workspace=ws)  # reuse: counters were left at zero
    assert ctx.ctx_device_status() == 0
    d = (o1.float() - o2.float()).abs()
    assert float(d.max()) <= 2.0 ** -7 * max(1.0, float(o1.float().abs().max()))
    assert float((l1 - l2).abs().max()) <= 1e-5


@pytest.mark.parametrize("B_rank,U,S_l,A,split", [(2, 4, 300, 1, False), (1, 2, 512, 2, True), (2, 2, 96, 3, True)])
def test_pack_out_fused_epilogue_equals_attention_then_pack_out(ctx, B_rank, U, S_l, A, split):
    """ctx_attn_lq_gkv_pack_out == ctx_attn_lq_gkv followed by ctx_pack_out,
    bit for bit, for one rank (A = 1, one batch block) and for stacked ranks."""
    gen = torch.Generator().manual_seed(17)
    H, D, Sk = 2, 128, 777
    Ub = U if A > 1 else 1          # batch blocks (head groups) stacked in the call
    B, Sq = Ub * B_rank, A * U * S_l
    q, k, v = (workloads.randn(s, gen).cuda() for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    ws = ctx.attn_workspace(B, Sq, Sk, H, D) if split else None
    out = torch.empty_like(q)
    lse1 = torch.empty((B, H, Sq), device="cuda")
    ctx.ctx_attn_lq_gkv(q, k, v, out, lse1, workspace=ws)
    send_ref = torch.empty((A, Ub, U, B_rank, S_l, H, D), dtype=q.dtype, device="cuda")
    ov = out.view(Ub, B_rank, Sq, H, D)
    for a in range(A):
        for u in range(Ub):
            ctx.ctx_pack_out(ov[u, :, a * U * S_l:], send_ref[a, u], U, o_batch_stride_rows=Sq)
    send = torch.full_like(send_ref, float("nan"))
    lse2 = torch.empty_like(lse1)
    ctx.ctx_attn_lq_gkv_pack_out(q, k, v, send, U, B_rank, S_l, lse=lse2, workspace=ws)
    assert ctx.ctx_device_status() == 0
    assert torch.equal(send, send_ref) and torch.equal(lse1, lse2)


# ---------------------------------------------------------------- failure path

def test_bounded_wait_times_out_and_context_survives(ctx, orc):
    st = ctx.ctx_selftest_wait_timeout(2_000_000)  # 2 ms
    assert st == 6, ctx.ctx_status_string(st)
    assert ctx.ctx_device_status() == 0  # cleared by the read
    gen = torch.Generator().manual_seed(16)
    q, k, v = (workloads.randn(s, gen) for s in ((1, 64, 1, 128), (1, 64, 1, 128), (1, 64, 1, 128)))
    O, L = _run(ctx, q, k, v)
    _check_full(orc, q, k, v, O, L)


def test_beyond_2pow31_elements(ctx, orc):
    """Q and O of more than 2^31 elements (64-bit output, LSE and TMA row
    arithmetic): Q [1, 524365, 32, 128] (ragged last tile) against 130 keys.
    Q is a seeded [1, 4096, 32, 128] block repeated along the rows on the
    device, so the oracle computes any sampled row from the block."""
    B, Sq, Sk, H, D, blk = 1, (1 << 19) + 77, 130, 32, 128, 4096
    assert B * Sq * H * D > 2 ** 31
    gen = torch.Generator().manual_seed(31)
    q_blk, k, v = (workloads.randn(s, gen) for s in ((B, blk, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    reps = -(-Sq // blk)
    q = q_blk.cuda().repeat(1, reps, 1, 1)[:, :Sq].contiguous()
    out = torch.empty_like(q)
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    ctx.ctx_attn_lq_gkv(q, k.cuda(), v.cuda(), out, lse, workspace=ctx.attn_workspace(B, Sq, Sk, H, D))
    assert ctx.ctx_device_status() == 0
    rows_i = np.concatenate([workloads.sample_rows(Sq, 256), np.arange(Sq - 80, Sq)])
    rng = np.random.default_rng(31)
    bhi = np.stack([np.zeros(rows_i.size, np.int64), rng.integers(0, H, rows_i.size), rows_i], axis=1)
    src = bhi.copy()
    src[:, 2] %= blk  # row i of q is row i % blk of the block
    eo, el = orc.attention_rows(u16(q_blk), u16(k), u16(v), src)
    got_o = np.stack([out[0, i, h].float().cpu().numpy() for _, h, i in bhi])
    got_l = np.array([float(lse[0, h, i]) for _, h, i in bhi])
    err = np.abs(got_o - eo)
    assert err.max() <= O_MAX, err.max()
    assert err.mean() <= O_MEAN, err.mean()
    assert np.abs(got_l - el).max() <= LSE_TOL
