"""Pins for the oracle's local-Q / global-KV attention.

The attention of the vllm-omni PR #7641 page is plain non-causal softmax
attention of the local query rows against the gathered keys, with an
optional per-key validity mask. These checks fix the oracle against closed
forms and invariants rather than against a retyped copy of itself:
  * probabilities sum to 1; constant V gives O = V; Q = 0 gives the mean of
    the valid V rows and LSE = ln(#valid); a single valid key gives O = v_j
    and LSE = s_j; a two-key case in closed form (sigmoid weights);
  * known bf16 / fp16 bit patterns widen to their exact values;
  * masked keys behave as deleted keys; key order does not matter; other
    heads and batches do not leak in; a fully masked row gives O = 0 and
    LSE = -inf (reading chosen where the pages are silent);
  * the local-Q slices of the composed topology concatenate to the full
    attention bit for bit (rows are independent);
  * scipy's logsumexp / softmax (a library routine for the same quantity) on
    small random inputs.
"""
import math

import numpy as np
import pytest
import scipy.special
import torch

import workloads


def _bits(shape, gen, dtype="bf16"):
    return workloads.as_u16(workloads.randn(shape, gen, dtype))


def _bf16(x):
    """bf16 bit pattern of a float that is exactly representable."""
    t = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16)
    assert float(t) == x
    return workloads.as_u16(t)


def _as_f64(bits, dtype="bf16"):
    t = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16 if dtype == "bf16" else torch.float16)
    return t.double().numpy()


@pytest.mark.parametrize("masked", [False, True])
def test_probabilities_sum_to_one(orc, masked):
    gen = torch.Generator().manual_seed(21)
    B, Sq, Sk, H, D = 2, 5, 37, 3, 16
    q, k = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen)
    mask = None
    if masked:
        mask = (torch.rand(B, Sk, generator=gen) > 0.4).numpy().astype(np.uint8)
        mask[:, 0] = 1
    for (b, h, i) in [(0, 0, 0), (1, 2, 4), (1, 1, 2)]:
        p = orc.attention_probs(q, k, b, h, i, mask)
        assert abs(p.sum() - 1.0) < 1e-12
        assert (p >= 0).all()
        if mask is not None:
            assert (p[mask[b] == 0] == 0).all()


def test_constant_v_gives_v(orc):
    gen = torch.Generator().manual_seed(22)
    B, Sq, Sk, H, D = 2, 6, 41, 2, 8
    q, k = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen)
    row = _bits((1, 1, H, D), gen)
    v = np.ascontiguousarray(np.broadcast_to(row, (B, Sk, H, D)))
    mask = np.ones((B, Sk), np.uint8)
    mask[1, 10:] = 0
    O, _ = orc.attention(q, k, v, mask)
    expect = _as_f64(row)[0, 0]  # [H, D]
    for b in range(B):
        for i in range(Sq):
            assert np.allclose(O[b, i], expect, rtol=0, atol=1e-12)


def test_zero_q_gives_mean_of_valid_v_and_log_count(orc):
    gen = torch.Generator().manual_seed(23)
    B, Sq, Sk, H, D = 2, 3, 29, 3, 8
    q = np.zeros((B, Sq, H, D), np.uint16)
    k, v = _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    mask = np.ones((B, Sk), np.uint8)
    mask[0, ::3] = 0
    O, lse = orc.attention(q, k, v, mask)
    vf = _as_f64(v)
    for b in range(B):
        valid = mask[b].astype(bool)
        mean = vf[b, valid].mean(axis=0)  # [H, D]
        for i in range(Sq):
            assert np.allclose(O[b, i], mean, rtol=0, atol=1e-12)
        assert np.allclose(lse[b], math.log(valid.sum()), rtol=0, atol=1e-12)


def test_single_valid_key_closed_form(orc):
    B, Sq, Sk, H, D = 1, 1, 6, 2, 8
    q = np.zeros((B, Sq, H, D), np.uint16)
    k = np.zeros((B, Sk, H, D), np.uint16)
    gen = torch.Generator().manual_seed(24)
    v = _bits((B, Sk, H, D), gen)
    # head 1: q = (0.5, 3, 0...), key 4 = (2, -0.25, 0...) -> q.k = 1 - 0.75 = 0.25
    q[0, 0, 1, 0], q[0, 0, 1, 1] = _bf16(0.5), _bf16(3.0)
    k[0, 4, 1, 0], k[0, 4, 1, 1] = _bf16(2.0), _bf16(-0.25)
    mask = np.zeros((B, Sk), np.uint8)
    mask[0, 4] = 1
    scale = 0.5
    o, lse = orc.attention_rows(q, k, v, np.array([[0, 1, 0]]), mask, scale)
    assert lse[0] == pytest.approx(0.125, abs=1e-15)
    assert np.array_equal(o[0], _as_f64(v)[0, 4, 1])


def test_two_key_closed_form(orc):
    B, Sq, Sk, H, D = 2, 3, 2, 3, 8
    gen = torch.Generator().manual_seed(25)
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    b, h, i = 1, 2, 1
    q[b, i, h] = 0
    k[b, :, h] = 0
    v[b, :, h] = 0
    q[b, i, h, 0], q[b, i, h, 1] = _bf16(1.0), _bf16(2.0)
    k[b, 0, h, 0], k[b, 0, h, 1] = _bf16(0.5), _bf16(0.25)    # q.k0 = 1.0
    k[b, 1, h, 0], k[b, 1, h, 1] = _bf16(-1.0), _bf16(0.5)    # q.k1 = 0.0
    v[b, 0, h, 0], v[b, 0, h, 2] = _bf16(1.0), _bf16(-1.0)
    v[b, 1, h, 1], v[b, 1, h, 2] = _bf16(4.0), _bf16(2.0)
    scale = 1.0 / math.sqrt(D)
    s0, s1 = scale * 1.0, 0.0
    w0 = 1.0 / (1.0 + math.exp(s1 - s0))
    w1 = 1.0 - w0
    expect = np.zeros(D)
    expect[0], expect[1], expect[2] = w0, 4.0 * w1, -w0 + 2.0 * w1
    O, lse = orc.attention(q, k, v)
    assert np.allclose(O[b, i, h], expect, rtol=0, atol=1e-14)
    assert lse[b, h, i] == pytest.approx(math.log(math.exp(s0) + math.exp(s1)), abs=1e-14)


@pytest.mark.parametrize("dtype,bits,value", [
    ("bf16", 0x3F80, 1.0), ("bf16", 0xC000, -2.0), ("bf16", 0x4049, 3.140625),
    ("bf16", 0x3E80, 0.25), ("bf16", 0x0001, 2.0 ** -133),
    ("fp16", 0x3C00, 1.0), ("fp16", 0xC000, -2.0), ("fp16", 0x0001, 2.0 ** -24),
    ("fp16", 0x7BFF, 65504.0), ("fp16", 0x3555, 0.333251953125), ("fp16", 0x8400, -(2.0 ** -14)),
])
def test_widening_of_known_bit_patterns(orc, dtype, bits, value):
    """With one valid key k = e_0 (value 1) and scale 1, LSE = q_0 exactly."""
    one = 0x3F80 if dtype == "bf16" else 0x3C00
    q = np.zeros((1, 1, 1, 8), np.uint16)
    k = np.zeros((1, 3, 1, 8), np.uint16)
    v = np.zeros((1, 3, 1, 8), np.uint16)
    q[0, 0, 0, 0] = bits
    k[0, 1, 0, 0] = one
    v[0, 1, 0, 5] = bits
    mask = np.array([[0, 1, 0]], np.uint8)
    o, lse = orc.attention_rows(q, k, v, np.array([[0, 0, 0]]), mask, 1.0, dtype=dtype)
    assert lse[0] == value
    assert o[0, 5] == value


def test_masked_keys_equal_deleted_keys(orc):
    gen = torch.Generator().manual_seed(26)
    B, Sq, Sk, H, D = 1, 7, 50, 2, 16
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    keep = np.ones(Sk, bool)
    keep[[0, 7, 8, 31, 49]] = False
    O1, L1 = orc.attention(q, k, v, keep[None].astype(np.uint8))
    O2, L2 = orc.attention(q, np.ascontiguousarray(k[:, keep]), np.ascontiguousarray(v[:, keep]))
    assert np.allclose(O1, O2, rtol=0, atol=1e-13) and np.allclose(L1, L2, rtol=0, atol=1e-13)


def test_key_permutation_invariance(orc):
    gen = torch.Generator().manual_seed(27)
    B, Sq, Sk, H, D = 2, 4, 33, 2, 16
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    perm = np.random.default_rng(0).permutation(Sk)
    O1, L1 = orc.attention(q, k, v)
    O2, L2 = orc.attention(q, np.ascontiguousarray(k[:, perm]), np.ascontiguousarray(v[:, perm]))
    assert np.allclose(O1, O2, rtol=0, atol=1e-13) and np.allclose(L1, L2, rtol=0, atol=1e-13)


def test_other_heads_and_batches_do_not_leak(orc):
    gen = torch.Generator().manual_seed(28)
    B, Sq, Sk, H, D = 2, 3, 20, 3, 8
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    O1, L1 = orc.attention(q, k, v)
    k2, v2, q2 = k.copy(), v.copy(), q.copy()
    k2[:, :, 0] = _bits((B, Sk, D), gen)
    v2[1] = _bits((Sk, H, D), gen)
    q2[0, :, 2] = _bits((Sq, D), gen)
    O2, L2 = orc.attention(q2, k2, v2)
    # head 1 of batch 0 saw none of the changes
    assert np.array_equal(O1[0, :, 1], O2[0, :, 1]) and np.array_equal(L1[0, 1], L2[0, 1])
    # the changed ones did move
    assert not np.allclose(O1[0, :, 0], O2[0, :, 0])
    assert not np.allclose(O1[1, :, 1], O2[1, :, 1])
    assert not np.allclose(O1[0, :, 2], O2[0, :, 2])


def test_fully_masked_row(orc):
    gen = torch.Generator().manual_seed(29)
    B, Sq, Sk, H, D = 2, 2, 9, 1, 8
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    mask = np.ones((B, Sk), np.uint8)
    mask[1] = 0
    O, L = orc.attention(q, k, v, mask)
    assert (O[1] == 0).all() and np.isneginf(L[1]).all()
    assert np.isfinite(L[0]).all()


def test_local_q_slices_concatenate_to_full(orc):
    gen = torch.Generator().manual_seed(30)
    B, S, H, D, A = 1, 48, 2, 16, 3
    q, k, v = _bits((B, S, H, D), gen), _bits((B, S, H, D), gen), _bits((B, S, H, D), gen)
    O, L = orc.attention(q, k, v)
    parts = [orc.attention(np.ascontiguousarray(q[:, a * S // A:(a + 1) * S // A]), k, v) for a in range(A)]
    assert np.array_equal(np.concatenate([p[0] for p in parts], axis=1), O)
    assert np.array_equal(np.concatenate([p[1] for p in parts], axis=2), L)


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_against_scipy_logsumexp_and_softmax(orc, dtype):
    gen = torch.Generator().manual_seed(31)
    B, Sq, Sk, H, D = 2, 5, 70, 3, 32
    q, k, v = (_bits(s, gen, dtype) for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    mask = np.ones((B, Sk), np.uint8)
    mask[1, 60:] = 0
    scale = 0.37
    O, L = orc.attention(q, k, v, mask, scale, dtype=dtype)
    qf, kf, vf = _as_f64(q, dtype), _as_f64(k, dtype), _as_f64(v, dtype)
    for b in range(B):
        valid = mask[b].astype(bool)
        for h in range(H):
            s = scale * (kf[b][valid][:, h, :] @ qf[b, :, h, :].T)  # [Sk_valid, Sq]
            assert np.allclose(L[b, h], scipy.special.logsumexp(s, axis=0), rtol=0, atol=1e-12)
            p = scipy.special.softmax(s, axis=0)
            assert np.allclose(O[b, :, h], p.T @ vf[b][valid][:, h, :], rtol=0, atol=1e-12)


def test_pure_python_attention_twin(orc):
    gen = torch.Generator().manual_seed(32)
    B, Sq, Sk, H, D = 1, 3, 11, 2, 8
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    mask = np.ones((B, Sk), np.uint8)
    mask[0, 3] = 0
    O, L = orc.attention(q, k, v, mask)
    for (b, h, i) in [(0, 0, 0), (0, 1, 2)]:
        o, lse = orc.py_attention_row(q, k, v, b, h, i, mask)
        assert np.allclose(O[b, i, h], o, rtol=0, atol=1e-13)
        assert L[b, h, i] == pytest.approx(lse, abs=1e-13)


def test_sampled_rows_match_full(orc):
    gen = torch.Generator().manual_seed(33)
    B, Sq, Sk, H, D = 2, 9, 13, 2, 8
    q, k, v = _bits((B, Sq, H, D), gen), _bits((B, Sk, H, D), gen), _bits((B, Sk, H, D), gen)
    O, L = orc.attention(q, k, v)
    rows = np.array([[1, 0, 8], [0, 1, 3], [1, 1, 0]])
    o, lse = orc.attention_rows(q, k, v, rows)
    for n, (b, h, i) in enumerate(rows):
        assert np.array_equal(o[n], O[b, i, h]) and lse[n] == L[b, h, i]
