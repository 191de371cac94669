"""Pins for packed varlen query metadata and varlen attention.

The remap is pinned by the worked example printed on the vllm-omni PR #7641
page (tests/golden/varlen_remap_example.txt); varlen attention by its
definition per document (a single document is plain attention; documents do
not see each other)."""
import os

import numpy as np
import pytest
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "varlen_remap_example.txt")


def _cases():
    out = []
    for line in open(GOLDEN):
        line = line.strip()
        if line and not line.startswith("#"):
            g, A, r, loc = line.split()
            out.append(([int(x) for x in g.split(",")], int(A), int(r), [int(x) for x in loc.split(",")]))
    return out


def test_golden_example_present():
    assert _cases() == [([0, 8, 12], 2, 0, [0, 6, 6]), ([0, 8, 12], 2, 1, [0, 2, 6])]


@pytest.mark.parametrize("case", _cases())
def test_remap_worked_example(orc, case):
    cu, A, r, local = case
    span = cu[-1] // A
    assert orc.varlen_remap(cu, r * span, span).tolist() == local


def test_remap_keeps_one_entry_per_document_and_covers_the_span(orc):
    rng = np.random.default_rng(0)
    for _ in range(50):
        n = int(rng.integers(1, 8))
        lens = rng.integers(0, 20, n)
        cu = np.concatenate([[0], np.cumsum(lens)]).astype(int)
        S = int(cu[-1]) + int(rng.integers(0, 5))   # trailing padding rows
        A = int(rng.integers(1, 5))
        S -= S % A
        span = S // A
        total = 0
        for r in range(A):
            loc = orc.varlen_remap(cu, r * span, span)
            assert len(loc) == n + 1 and loc[0] == 0 and (np.diff(loc) >= 0).all()
            total += int(loc[-1])
        assert total == min(int(cu[-1]), S)


def test_padding_remap(orc):
    # one document of 10 valid rows padded to 16, A = 2 (span 8)
    assert orc.padding_remap(10, 6, 0, 8).tolist() == [8, 0]
    assert orc.padding_remap(10, 6, 8, 8).tolist() == [2, 6]


def _bits(shape, gen):
    return workloads.as_u16(workloads.randn(shape, gen))


def test_single_document_is_plain_attention(orc):
    gen = torch.Generator().manual_seed(81)
    q, k, v = _bits((20, 2, 16), gen), _bits((33, 2, 16), gen), _bits((33, 2, 16), gen)
    O, L = orc.attention_varlen(q, k, v, [0, 20], [0, 33])
    eO, eL = orc.attention(q[None], k[None], v[None])
    assert np.array_equal(O, eO[0]) and np.array_equal(L, eL[0])


def test_documents_do_not_see_each_other(orc):
    gen = torch.Generator().manual_seed(82)
    q, k, v = _bits((12, 2, 8), gen), _bits((30, 2, 8), gen), _bits((30, 2, 8), gen)
    cu_q, cu_k = [0, 5, 5, 12], [0, 10, 14, 30]
    O, L = orc.attention_varlen(q, k, v, cu_q, cu_k)
    k2, v2 = k.copy(), v.copy()
    k2[0:10] = _bits((10, 2, 8), gen)   # document 0's keys
    O2, L2 = orc.attention_varlen(q, k2, v2, cu_q, cu_k)
    assert np.array_equal(O[5:], O2[5:]) and np.array_equal(L[:, 5:], L2[:, 5:])
    assert not np.allclose(O[:5], O2[:5])
    # document 2 alone
    e2, l2 = orc.attention(q[None, 5:12], k[None, 14:30], v[None, 14:30])
    assert np.array_equal(O[5:12], e2[0])


def test_empty_key_document_gives_zero_and_minus_inf(orc):
    gen = torch.Generator().manual_seed(83)
    q, k, v = _bits((6, 1, 8), gen), _bits((4, 1, 8), gen), _bits((4, 1, 8), gen)
    O, L = orc.attention_varlen(q, k, v, [0, 3, 6], [0, 4, 4])
    assert (O[3:] == 0).all() and np.isneginf(L[:, 3:]).all()
    assert np.isfinite(L[:, :3]).all()
