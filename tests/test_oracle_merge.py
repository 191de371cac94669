"""Pins for the oracle's log-sum-exp merge of attention over key segments.

Attention over all keys equals the merge of attention over disjoint key
segments (the softmax denominator factorises over the segments). With V
constant inside each segment, every segment's output is that constant
exactly (representable in bf16), so the merge can be checked against full
attention to fp64 rounding.
"""
import numpy as np
import pytest
import torch

import workloads


def _bits(shape, gen):
    return workloads.as_u16(workloads.randn(shape, gen))


def _bf16(x):
    return workloads.as_u16(torch.tensor(x, dtype=torch.float32).to(torch.bfloat16))


@pytest.mark.parametrize("cuts", [[0, 40, 100], [0, 7, 8, 50, 100], [0, 100]])
def test_merge_of_segments_equals_full_attention(orc, cuts):
    gen = torch.Generator().manual_seed(41)
    B, Sq, Sk, H, D = 2, 9, 100, 3, 16
    q, k = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen)
    v = np.zeros((B, Sk, H, D), np.uint16)
    consts = [0.5, -1.25, 2.0, 0.375, -3.0]
    for p in range(len(cuts) - 1):
        v[:, cuts[p]:cuts[p + 1]] = _bf16(consts[p] * (1 + np.arange(D)) / D)[None, None, None, :]
    O, L = orc.attention(q, k, v)
    parts_o, parts_l = [], []
    for p in range(len(cuts) - 1):
        o, l = orc.attention(q, np.ascontiguousarray(k[:, cuts[p]:cuts[p + 1]]),
                             np.ascontiguousarray(v[:, cuts[p]:cuts[p + 1]]))
        # constant V per segment: the segment output is that constant exactly
        bits = workloads.as_u16(torch.from_numpy(o).float().to(torch.bfloat16))
        back = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
        assert np.allclose(back, o, rtol=0, atol=1e-12)
        parts_o.append(bits)
        parts_l.append(l)
    Om, Lm = orc.lse_merge(np.stack(parts_o), np.stack(parts_l))
    assert np.allclose(Om, O, rtol=0, atol=1e-12)
    assert np.allclose(Lm, L, rtol=0, atol=1e-12)


def test_merge_random_values_close_to_full(orc):
    gen = torch.Generator().manual_seed(42)
    B, Sq, Sk, H, D = 1, 5, 64, 2, 32
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    O, L = orc.attention(q, k, v)
    halves = [(0, 20), (20, 64)]
    po, pl = [], []
    for a, b in halves:
        o, l = orc.attention(q, np.ascontiguousarray(k[:, a:b]), np.ascontiguousarray(v[:, a:b]))
        po.append(workloads.as_u16(torch.from_numpy(o).float().to(torch.bfloat16)))
        pl.append(l)
    Om, Lm = orc.lse_merge(np.stack(po), np.stack(pl))
    assert np.abs(Om - O).max() < 2e-2          # bf16 rounding of the parts
    assert np.allclose(Lm, L, rtol=0, atol=1e-12)


def test_single_part_is_identity(orc):
    gen = torch.Generator().manual_seed(43)
    o = _bits((1, 2, 3, 4, 8), gen)
    l = np.random.default_rng(0).normal(size=(1, 2, 4, 3))
    Om, Lm = orc.lse_merge(o, l)
    widened = torch.from_numpy(o[0].view(np.int16)).view(torch.bfloat16).double().numpy()
    assert np.array_equal(Om, widened) and np.array_equal(Lm, l[0])


def test_empty_segments_are_ignored_and_order_does_not_matter(orc):
    gen = torch.Generator().manual_seed(44)
    o = _bits((3, 1, 4, 2, 8), gen)
    l = np.random.default_rng(1).normal(size=(3, 1, 2, 4))
    l[1] = -np.inf
    Om, Lm = orc.lse_merge(o, l)
    O2, L2 = orc.lse_merge(o[[0, 2]], l[[0, 2]])
    assert np.allclose(Om, O2, rtol=0, atol=1e-15) and np.allclose(Lm, L2, rtol=0, atol=1e-15)
    O3, L3 = orc.lse_merge(o[[2, 1, 0]], l[[2, 1, 0]])
    assert np.allclose(Om, O3, rtol=0, atol=1e-14) and np.allclose(Lm, L3, rtol=0, atol=1e-14)
    l[:] = -np.inf
    O4, L4 = orc.lse_merge(o, l)
    assert (O4 == 0).all() and np.isneginf(L4).all()
