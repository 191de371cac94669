"""Pins for the oracle's composed U x A helpers (vllm-omni PR #7641, the
composed order: Ulysses all-to-all in the U group, K/V AllGather in the A
group, local-Q / global-KV attention, reverse Ulysses all-to-all; rank layout:
U groups are contiguous blocks of U ranks, A groups stride by U).

`ulysses_agkv_forward` and `ulysses_reverse` are the checkers of every
whole-layer GPU result, so each of their branches is fixed here against numpy
slicing of the GLOBAL tensors, which uses none of the oracle's pack, unpack or
exchange code:
  * rank g = a*U + u holds input rows [g*S_l, (g+1)*S_l);
  * its local query is rows [a*S/A, (a+1)*S/A) of padded heads
    [u*h_l, (u+1)*h_l) (heads beyond H are zero);
  * the gathered K/V of head group u is that head slice of every row, with the
    joint keys' head slice after (or before) the image rows.
A reverse exchange that indexed the U group u-major instead of a-major, a
joint slice taken before padding, or a layout-1 unpack that swapped Q and K
fails one of these.
"""
import numpy as np
import pytest
import torch

import workloads


def _bits(shape, gen):
    return workloads.as_u16(workloads.randn(shape, gen))


def _pad(x, H_pad):
    B, S, H, D = x.shape
    out = np.zeros((B, S, H_pad, D), np.uint16)
    out[:, :, :H] = x
    return out


def _global(U, A, B, S, H, D, J, seed):
    gen = torch.Generator().manual_seed(seed)
    full = [_bits((B, S, H, D), gen) for _ in range(3)]
    jk = jv = None
    if J:
        jk, jv = _bits((B, J, H, D), gen), _bits((B, J, H, D), gen)
    R = U * A
    S_l = S // R
    shards = [[x[:, g * S_l:(g + 1) * S_l].copy() for x in full] for g in range(R)]
    return full, jk, jv, shards


def _spec_local_q(full_q, U, A, g):
    B, S, H, D = full_q.shape
    h_l = -(-H // U)
    a, u = divmod(g, U)
    return _pad(full_q, U * h_l)[:, a * S // A:(a + 1) * S // A, u * h_l:(u + 1) * h_l]


CASES = [  # U, A, B, S, H, D
    (2, 2, 1, 32, 4, 8),
    (4, 2, 2, 64, 8, 8),
    (2, 3, 1, 36, 4, 8),
    (4, 2, 1, 64, 14, 8),   # 14 heads at U = 4: padded to 16
    (2, 3, 2, 36, 5, 8),    # 5 heads at U = 2: padded to 6
    (3, 2, 1, 30, 7, 16),
]


@pytest.mark.parametrize("U,A,B,S,H,D", CASES)
def test_reverse_of_global_local_q_slices_returns_every_input_shard(orc, U, A, B, S, H, D):
    """ulysses_reverse applied to each rank's local-Q slice (built by numpy
    slicing of the global tensor, i.e. the identity attention) gives every
    rank its own [B, S_l, H, D] input shard back, bit for bit."""
    full, _, _, shards = _global(U, A, B, S, H, D, 0, 81)
    R = U * A
    o_ranks = [np.ascontiguousarray(_spec_local_q(full[0], U, A, g)) for g in range(R)]
    back = orc.ulysses_reverse(o_ranks, U, A, H)
    for g in range(R):
        assert back[g].shape == (B, S // R, H, D)
        assert np.array_equal(back[g], shards[g][0]), f"rank {g}"


@pytest.mark.parametrize("U,A,B,S,H,D", CASES)
def test_forward_then_reverse_round_trip(orc, U, A, B, S, H, D):
    """The oracle's own forward local-Q slices equal the numpy spec, and the
    reverse of them is the input shards (all ranks, A > 1)."""
    full, _, _, shards = _global(U, A, B, S, H, D, 0, 82)
    R = U * A
    res = orc.ulysses_agkv_forward([s[0] for s in shards], [s[1] for s in shards], [s[2] for s in shards], U, A)
    for g in range(R):
        assert np.array_equal(res["q"][g], _spec_local_q(full[0], U, A, g)), f"local Q rank {g}"
    back = orc.ulysses_reverse(res["q"], U, A, H)
    for g in range(R):
        assert np.array_equal(back[g], shards[g][0])


def test_spec_rejects_a_u_major_reverse(orc):
    """A planted mistake, on the CPU: the reverse exchange with its U groups
    taken u-major (ranks u*A + a) instead of a-major. The spec of the test
    above rejects it, so the pin discriminates the rank layout."""
    U, A, B, S, H, D = 2, 3, 1, 36, 4, 8
    full, _, _, shards = _global(U, A, B, S, H, D, 0, 83)
    R = U * A
    o_ranks = [np.ascontiguousarray(_spec_local_q(full[0], U, A, g)) for g in range(R)]

    def reverse_u_major(o, U, A, H):
        sends = [orc.pack_out(o[g], U) for g in range(R)]
        out = [None] * R
        for a in range(A):
            grp = [u * A + a for u in range(U)]
            recvs = orc.all_to_all([sends[g] for g in grp])
            for u, g in enumerate(grp):
                out[g] = orc.unpack_out_ex(recvs[u], U, H)
        return out

    wrong = reverse_u_major(o_ranks, U, A, H)
    assert not all(np.array_equal(wrong[g], shards[g][0]) for g in range(R))
    right = orc.ulysses_reverse(o_ranks, U, A, H)
    assert all(np.array_equal(right[g], shards[g][0]) for g in range(R))


@pytest.mark.parametrize("front", [False, True], ids=["rear", "front"])
@pytest.mark.parametrize("U,A,H,J", [(4, 2, 14, 5), (2, 2, 5, 3), (4, 1, 14, 7), (3, 2, 7, 4)])
def test_padded_heads_with_joint_keys(orc, U, A, H, J, front):
    """Heads padded to U*ceil(H/U) and joint K/V re-attached: the gathered K
    and V of head group u are the padded global head slice of every image row
    plus the padded joint head slice (zeros on pad heads), in placement
    order."""
    B, S, D = 2, 16 * U * A, 8
    full, jk, jv, shards = _global(U, A, B, S, H, D, J, 84)
    h_l = -(-H // U)
    res = orc.ulysses_agkv_forward([s[0] for s in shards], [s[1] for s in shards], [s[2] for s in shards], U, A,
                                   jk, jv, joint_front=front)
    for u in range(U):
        hs = slice(u * h_l, (u + 1) * h_l)
        for t, (x, j) in enumerate(((full[1], jk), (full[2], jv))):
            img = _pad(x, U * h_l)[:, :, hs]
            jnt = _pad(j, U * h_l)[:, :, hs]
            spec = np.concatenate([jnt, img] if front else [img, jnt], axis=1)
            got = res["k" if t == 0 else "v"][u]
            assert got.shape == (B, S + J, h_l, D)
            assert np.array_equal(got, spec), f"{'kv'[t]} group {u}"
            # heads past H are zero in both segments
            for hh in range(h_l):
                if u * h_l + hh >= H:
                    assert (got[:, :, hh] == 0).all()


@pytest.mark.parametrize("U,A,B,S,H,D", CASES)
def test_interleaved_layout_composes_to_the_same_layer(orc, U, A, B, S, H, D):
    """The interleaved staging layout [U,B,S_l,h_l,3D] gives the same local
    Q and gathered K/V as [U,3,B,S_l,h_l,D], and both equal the numpy spec."""
    full, jk, jv, shards = _global(U, A, B, S, H, D, 3, 85)
    args = ([s[0] for s in shards], [s[1] for s in shards], [s[2] for s in shards], U, A, jk, jv)
    r0 = orc.ulysses_agkv_forward(*args, layout=orc.LAYOUT_TQKV)
    r1 = orc.ulysses_agkv_forward(*args, layout=orc.LAYOUT_INTERLEAVED)
    h_l = -(-H // U)
    for g in range(U * A):
        assert np.array_equal(r1["q"][g], r0["q"][g])
        assert np.array_equal(r1["q"][g], _spec_local_q(full[0], U, A, g))
    for u in range(U):
        hs = slice(u * h_l, (u + 1) * h_l)
        assert np.array_equal(r1["k"][u], r0["k"][u])
        assert np.array_equal(r1["v"][u], r0["v"][u])
        assert np.array_equal(r1["k"][u][:, :S], _pad(full[1], U * h_l)[:, :, hs])
        assert np.array_equal(r1["v"][u][:, :S], _pad(full[2], U * h_l)[:, :, hs])
