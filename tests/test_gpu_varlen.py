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
