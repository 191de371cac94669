"""GPU parity of packed varlen metadata and varlen attention.

* ctx_varlen_remap on the vllm-omni page's worked example and on random
  document sets against the oracle (bit-exact integers);
* ctx_attn_varlen against the oracle's per-document attention (tolerance of
  the other attention tests); rows outside every document stay untouched;
* the AllGather-KV shard path: each rank remaps the global boundaries to its
  span and runs varlen attention of its local query rows against the full
  K/V; the ranks' outputs concatenate to the unsplit packed attention.
"""
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


def _remap(ctx, cu, lo, n, pad=None):
    g = torch.tensor(cu, dtype=torch.int32, device="cuda")
    out = torch.full((len(cu),), -7, dtype=torch.int32, device="cuda")
    pin = pout = None
    if pad is not None:
        pin = torch.tensor(pad, dtype=torch.int32, device="cuda")
        pout = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    ctx.ctx_varlen_remap(g, lo, n, out, pin, pout)
    torch.cuda.synchronize()
    return out.cpu().numpy(), (None if pout is None else pout.cpu().numpy())


def test_remap_worked_example(ctx):
    assert _remap(ctx, [0, 8, 12], 0, 6)[0].tolist() == [0, 6, 6]
    assert _remap(ctx, [0, 8, 12], 6, 6)[0].tolist() == [0, 2, 6]


@pytest.mark.parametrize("n_docs", [1, 7, 1024, 1025, 3000])
def test_remap_random_against_oracle(ctx, orc, n_docs):
    rng = np.random.default_rng(n_docs)
    lens = rng.integers(0, 40, n_docs)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    S = int(cu[-1]) + 3
    for A in (1, 2, 3):
        span = S // A
        for r in range(A):
            got, _ = _remap(ctx, cu.tolist(), r * span, span)
            assert np.array_equal(got, orc.varlen_remap(cu, r * span, span))


def test_padding_remap(ctx, orc):
    _, p0 = _remap(ctx, [0, 16], 0, 8, pad=[10, 6])
    _, p1 = _remap(ctx, [0, 16], 8, 8, pad=[10, 6])
    assert p0.tolist() == orc.padding_remap(10, 6, 0, 8).tolist() == [8, 0]
    assert p1.tolist() == orc.padding_remap(10, 6, 8, 8).tolist() == [2, 6]


def _run_varlen(ctx, q, k, v, cu_q, cu_k, max_q, mask=None):
    Sq, H, D = q.shape
    out = Guarded((Sq, H, D), q.dtype)
    lse = Guarded((H, Sq), torch.float32)
    m = None if mask is None else torch.from_numpy(mask).cuda()
    ctx.ctx_attn_varlen(q.cuda(), k.cuda(), v.cuda(), torch.tensor(cu_q, dtype=torch.int32, device="cuda"),
                        torch.tensor(cu_k, dtype=torch.int32, device="cuda"), max_q, out.t, lse.t, key_mask=m)
    assert ctx.ctx_device_status() == 0
    assert out.intact() and lse.intact()
    return out.t.float().cpu().numpy(), lse.t.cpu().numpy()


def _check(O, L, eO, eL):
    inside = ~np.isnan(eO[:, 0, 0])
    assert np.isnan(O[~inside]).all()            # rows outside every document untouched
    err = np.abs(O[inside] - eO[inside])
    assert err.max() <= O_MAX and err.mean() <= O_MEAN, err.max()
    fin = np.isfinite(eL)
    assert np.array_equal(np.isfinite(L) & ~np.isnan(L), fin)
    assert np.abs(L[fin] - eL[fin]).max() <= LSE_TOL


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "bf16"), (128, "fp16")])
def test_varlen_attention_against_oracle(ctx, orc, D, dtype):
    gen = torch.Generator().manual_seed(91)
    H = 3
    q_lens = [300, 0, 17, 513, 128, 1]
    k_lens = [700, 50, 0, 1000, 129, 5]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).tolist()
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).tolist()
    Sq, Sk = cu_q[-1] + 40, cu_k[-1] + 3           # padding rows / keys after the documents
    q, k, v = (workloads.randn(s, gen, dtype) for s in ((Sq, H, D), (Sk, H, D), (Sk, H, D)))
    O, L = _run_varlen(ctx, q, k, v, cu_q, cu_k, max(q_lens))
    eO, eL = orc.attention_varlen(u16(q), u16(k), u16(v), cu_q, cu_k, dtype=dtype)
    _check(O, L, eO, eL)


def test_varlen_attention_with_mask(ctx, orc):
    gen = torch.Generator().manual_seed(92)
    H, D = 2, 128
    cu_q, cu_k = [0, 200, 450], [0, 300, 1000]
    q, k, v = (workloads.randn(s, gen) for s in ((450, H, D), (1000, H, D), (1000, H, D)))
    mask = np.ones(1000, np.uint8)
    mask[250:300] = 0       # padded tail of document 0's keys
    mask[300:420] = 0       # a masked block at the start of document 1
    O, L = _run_varlen(ctx, q, k, v, cu_q, cu_k, 250, mask)
    eO, eL = orc.attention_varlen(u16(q), u16(k), u16(v), cu_q, cu_k, mask)
    _check(O, L, eO, eL)


@pytest.mark.parametrize("A", [2, 4])
def test_allgather_shard_path_equals_unsplit(ctx, orc, A):
    """Each rank: local query rows [r*S/A, (r+1)*S/A), boundaries remapped on
    the device, keys global; concatenated outputs == the unsplit attention."""
    gen = torch.Generator().manual_seed(93)
    H, D = 2, 128
    lens = [700, 120, 900, 6, 322]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    S = cu[-1]
    S -= S % A
    cu = [min(x, S) for x in cu]
    q, k, v = (workloads.randn((S, H, D), gen).cuda() for _ in range(3))
    cu_g = torch.tensor(cu, dtype=torch.int32, device="cuda")
    full = torch.empty_like(q)
    full_l = torch.empty((H, S), device="cuda")
    ctx.ctx_attn_varlen(q, k, v, cu_g, cu_g, max(lens), full, full_l)
    span = S // A
    parts, lparts = [], []
    for r in range(A):
        loc = torch.empty_like(cu_g)
        ctx.ctx_varlen_remap(cu_g, r * span, span, loc)
        qr = q[r * span:(r + 1) * span].contiguous()
        o = torch.empty_like(qr)
        l = torch.empty((H, span), device="cuda")
        # key boundaries stay global, so each document still sees all its keys
        ctx.ctx_attn_varlen(qr, k, v, loc, cu_g, max(lens), o, l)
        parts.append(o)
        lparts.append(l)
    assert ctx.ctx_device_status() == 0
    assert torch.equal(torch.cat(parts), full)          # rows are independent: bit for bit
    assert torch.equal(torch.cat(lparts, dim=1), full_l)
    eO, eL = orc.attention_varlen(u16(q.cpu()), u16(k.cpu()), u16(v.cpu()), cu, cu)
    _check(full.float().cpu().numpy(), full_l.cpu().numpy(), eO, eL)


def _varlen_pair(ctx, q, k, v, cu_q, cu_k, max_q, mask=None):
    """The same packed varlen call with one CTA per unit and with the balanced
    (key-split) schedule; the balanced one runs twice on one workspace."""
    Sq, H, D = q.shape
    cq = torch.tensor(cu_q, dtype=torch.int32, device="cuda")
    ck = torch.tensor(cu_k, dtype=torch.int32, device="cuda")
    m = None if mask is None else torch.from_numpy(mask).cuda()
    o1 = torch.full((Sq, H, D), float("nan"), dtype=q.dtype, device="cuda")
    l1 = torch.full((H, Sq), float("nan"), device="cuda")
    ctx.ctx_attn_varlen(q, k, v, cq, ck, max_q, o1, l1, key_mask=m)
    ws = ctx.varlen_workspace(len(cu_q) - 1, max_q, H, D)
    outs = []
    for _ in range(2):  # a second call on the same workspace: counters were left at zero
        o2 = Guarded((Sq, H, D), q.dtype)
        l2 = Guarded((H, Sq), torch.float32)
        ctx.ctx_attn_varlen(q, k, v, cq, ck, max_q, o2.t, l2.t, key_mask=m, workspace=ws)
        assert ctx.ctx_device_status() == 0
        assert o2.intact() and l2.intact()
        outs.append((o2.t, l2.t))
    n_units = ((max_q + 255) // 256) * H * (len(cu_q) - 1)
    assert int(ws[:n_units * 2 * 2 * 4].count_nonzero()) == 0  # arrived / written per tile
    return (o1, l1), outs


def _same_up_to_merge(a, b):
    """One CTA per unit vs the split schedule: rows not written stay NaN in
    both; written rows agree to fp32 rounding of the log-sum-exp merge."""
    (o1, l1), (o2, l2) = a, b
    assert torch.equal(torch.isnan(o1), torch.isnan(o2))
    w = ~torch.isnan(o1)
    d = (o1.float()[w] - o2.float()[w]).abs()
    if d.numel():
        assert float(d.max()) <= 2.0 ** -7 * max(1.0, float(o1.float()[w].abs().max()))
    lw = ~torch.isnan(l1)
    assert torch.equal(lw, ~torch.isnan(l2))
    fin = torch.isfinite(l1) & lw
    assert torch.equal(fin, torch.isfinite(l2) & lw)
    if fin.any():
        assert float((l1[fin] - l2[fin]).abs().max()) <= 1e-5


@pytest.mark.parametrize("D,dtype", [(128, "bf16"), (64, "bf16"), (128, "fp16")])
def test_balanced_varlen_matches_per_unit_and_oracle(ctx, orc, D, dtype):
    """Documents of uneven lengths, an empty one, one without keys, one
    without queries, padding rows after the last document."""
    gen = torch.Generator().manual_seed(94)
    H = 3
    q_lens = [1300, 0, 17, 513, 128, 1, 40, 600]
    k_lens = [2000, 50, 0, 1000, 129, 5, 0, 333]
    cu_q = np.concatenate([[0], np.cumsum(q_lens)]).tolist()
    cu_k = np.concatenate([[0], np.cumsum(k_lens)]).tolist()
    Sq, Sk = cu_q[-1] + 40, cu_k[-1] + 3
    q, k, v = (workloads.randn(s, gen, dtype).cuda() for s in ((Sq, H, D), (Sk, H, D), (Sk, H, D)))
    a, outs = _varlen_pair(ctx, q, k, v, cu_q, cu_k, max(q_lens))
    for b in outs:
        _same_up_to_merge(a, b)
    eO, eL = orc.attention_varlen(u16(q.cpu()), u16(k.cpu()), u16(v.cpu()), cu_q, cu_k, dtype=dtype)
    _check(outs[0][0].float().cpu().numpy(), outs[0][1].cpu().numpy(), eO, eL)


def test_balanced_varlen_with_mask_and_many_documents(ctx, orc):
    gen = torch.Generator().manual_seed(95)
    H, D = 2, 128
    rng = np.random.default_rng(95)
    lens = rng.integers(0, 700, 300).tolist()           # 300 documents, some empty
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    S = cu[-1]
    q, k, v = (workloads.randn((S, H, D), gen).cuda() for _ in range(3))
    mask = (rng.random(S) > 0.1).astype(np.uint8)
    a, outs = _varlen_pair(ctx, q, k, v, cu, cu, max(lens), mask)
    for b in outs:
        _same_up_to_merge(a, b)
    rows = workloads.sample_rows(S, 256)
    eO, eL = orc.attention_varlen(u16(q.cpu()), u16(k.cpu()), u16(v.cpu()), cu, cu, mask)
    got = outs[0][0].float().cpu().numpy()
    err = np.abs(got[rows] - eO[rows])
    assert err.max() <= O_MAX and err.mean() <= O_MEAN


@pytest.mark.parametrize("A", [4, 8])
def test_balanced_varlen_shard_path(ctx, orc, A):
    """One rank of an AllGather-KV group at a time, balanced: concatenated
    outputs equal the unsplit packed attention up to the merge rounding."""
    gen = torch.Generator().manual_seed(96)
    H, D = 4, 128
    lens = [12288, 8192, 6144, 4096, 2048]
    cu = np.concatenate([[0], np.cumsum(lens)]).tolist()
    S = cu[-1]
    q, k, v = (workloads.randn((S, H, D), gen).cuda() for _ in range(3))
    cu_g = torch.tensor(cu, dtype=torch.int32, device="cuda")
    full = torch.empty_like(q)
    full_l = torch.empty((H, S), device="cuda")
    ctx.ctx_attn_varlen(q, k, v, cu_g, cu_g, max(lens), full, full_l)
    span = S // A
    ws = ctx.varlen_workspace(len(lens), span, H, D)
    parts, lparts = [], []
    for r in range(A):
        loc = torch.empty_like(cu_g)
        ctx.ctx_varlen_remap(cu_g, r * span, span, loc)
        qr = q[r * span:(r + 1) * span].contiguous()
        o = torch.empty_like(qr)
        l = torch.empty((H, span), device="cuda")
        ctx.ctx_attn_varlen(qr, k, v, loc, cu_g, span, o, l, workspace=ws)
        parts.append(o)
        lparts.append(l)
    assert ctx.ctx_device_status() == 0
    d = (torch.cat(parts).float() - full.float()).abs()
    assert float(d.max()) <= 2.0 ** -7 * max(1.0, float(full.float().abs().max()))
    assert float((torch.cat(lparts, dim=1) - full_l).abs().max()) <= 1e-5
