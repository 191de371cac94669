"""GPU parity of ctx_lse_merge: against the oracle's merge on the same
inputs, and end to end (attention over key segments, then the merge, equals
attention over all keys, within the attention tolerance)."""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import Guarded, u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import diffusion_transformer_context_gb300 as m
    m.build()
    return m


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("P,B,Sq,H,D", [(2, 1, 300, 3, 128), (5, 2, 17, 1, 64), (1, 1, 8, 2, 8), (3, 1, 4095, 12, 128),
                                       (4, 2, 100, 5, 128), (2, 3, 33, 7, 64)])
def test_merge_matches_oracle(ctx, orc, P, B, Sq, H, D, dtype):
    gen = torch.Generator().manual_seed(51)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    o = workloads.randn((P, B, Sq, H, D), gen, dtype)
    lse = torch.randn((P, B, H, Sq), generator=gen) * 3 + 10
    lse[0, :, :, :5] = -float("inf")            # an empty segment on some rows
    if P > 1:
        lse[:, :, :, 1] = -float("inf")         # rows with no valid key at all
    out = Guarded((B, Sq, H, D), tdt)
    lout = Guarded((B, H, Sq), torch.float32)
    ctx.ctx_lse_merge(o.cuda(), lse.cuda(), out.t, lout.t)
    torch.cuda.synchronize()
    assert out.intact() and lout.intact()
    eo, el = orc.lse_merge(u16(o), lse.double().numpy(), dtype)
    got = out.t.float().cpu().numpy()
    err = np.abs(got - eo)
    # fp32 arithmetic, one rounding of the result to the 16-bit type
    ulp = 2.0 ** -8 if dtype == "bf16" else 2.0 ** -11
    assert (err <= ulp * np.abs(eo) + 1e-5).all(), err.max()
    gl = lout.t.cpu().numpy()
    fin = np.isfinite(el)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.abs(gl[fin] - el[fin]).max() <= 1e-5
    if P > 1:
        assert (got[:, 1] == 0).all()


def test_segment_attention_plus_merge_equals_full_attention(ctx, orc):
    gen = torch.Generator().manual_seed(52)
    B, Sq, Sk, H, D = 1, 1000, 5000, 4, 128
    q, k, v = (workloads.randn(s, gen).cuda() for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    cuts = [0, 1700, 1701, 3333, 5000]
    P = len(cuts) - 1
    o_parts = torch.empty((P, B, Sq, H, D), dtype=torch.bfloat16, device="cuda")
    l_parts = torch.empty((P, B, H, Sq), dtype=torch.float32, device="cuda")
    for p in range(P):
        ctx.ctx_attn_lq_gkv(q, k[:, cuts[p]:cuts[p + 1]].contiguous(), v[:, cuts[p]:cuts[p + 1]].contiguous(),
                            o_parts[p], l_parts[p])
    out = torch.empty((B, Sq, H, D), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    ctx.ctx_lse_merge(o_parts, l_parts, out, lse)
    full_o = torch.empty_like(out)
    full_l = torch.empty_like(lse)
    ctx.ctx_attn_lq_gkv(q, k, v, full_o, full_l)
    assert ctx.ctx_device_status() == 0
    assert float((out.float() - full_o.float()).abs().max()) <= 2e-2
    assert float((lse - full_l).abs().max()) <= 1e-3
    rows = workloads.sample_rows(Sq, 160)
    bhi = np.stack([np.zeros_like(rows), rows % H, rows], axis=1)
    eo, el = orc.attention_rows(u16(q.cpu()), u16(k.cpu()), u16(v.cpu()), bhi)
    got = np.stack([out[0, i, h].float().cpu().numpy() for _, h, i in bhi])
    assert np.abs(got - eo).max() <= 2e-2 and np.abs(got - eo).mean() <= 2e-3
    assert np.abs(np.array([lse[0, h, i].item() for _, h, i in bhi]) - el).max() <= 1e-3
