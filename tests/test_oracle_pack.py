"""Pins for the oracle's layout steps (pack, exchange, unpack, reverse).

Each check fixes the oracle against something other than itself:
  * the spec the sglang PR #33667 unit test compares with (rank r receives
    the whole sequence with heads [r*h_local, (r+1)*h_local)), computed here
    with numpy slicing, on the page's own shapes and seed;
  * the "packed exchange equals three separate exchanges" invariant, with the
    separate exchange written as numpy reshapes/transposes;
  * round trips (input exchange followed by the reverse exchange is the
    identity) and the U=1 identity;
  * the composed Ulysses-then-AllGather order of the vllm-omni PR #7641 page,
    and that the opposite order does NOT rebuild the sequence.
"""
import os

import numpy as np
import pytest
import torch

import workloads

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "usp_packed_qkv_cases.txt")


def _bits(shape, gen):
    return workloads.as_u16(workloads.randn(shape, gen))


def _page_cases():
    rows = []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(tuple(int(x) for x in line.split()))
    return rows


def test_golden_cases_present():
    assert _page_cases() == [(4, 1, 128, 8, 64), (2, 2, 48, 6, 32)]


@pytest.mark.parametrize("B,S_l,H,D,U", [(1, 5, 4, 8, 2), (2, 3, 6, 16, 3), (1, 7, 8, 24, 4), (2, 4, 3, 8, 1)])
def test_pack_is_head_slices_destination_major(orc, B, S_l, H, D, U):
    gen = torch.Generator().manual_seed(7)
    q, k, v = (_bits((B, S_l, H, D), gen) for _ in range(3))
    st = orc.pack_qkv(q, k, v, U)
    h_l = H // U
    assert st.shape == (U, 3, B, S_l, h_l, D)
    for r in range(U):
        for t, x in enumerate((q, k, v)):
            assert np.array_equal(st[r, t], x[:, :, r * h_l:(r + 1) * h_l])


@pytest.mark.parametrize("case", _page_cases())
def test_page_multirank_simulation_matches_spec(orc, case):
    """All ranks on one host, all_to_all_single chunk semantics, as the page's
    test does; rank r's unpacked Q/K/V must equal the global tensor's head
    slice r bit for bit."""
    world, b, s_global, h_global, d = case
    gen = torch.Generator().manual_seed(1234)
    full = [_bits((b, s_global, h_global, d), gen) for _ in range(3)]
    s_local, h_local = s_global // world, h_global // world
    shards = [[x[:, r * s_local:(r + 1) * s_local] for x in full] for r in range(world)]
    sends = [orc.pack_qkv(*shards[r], world) for r in range(world)]
    recvs = orc.all_to_all(sends)
    for r in range(world):
        got = orc.unpack_qkv(recvs[r], world)
        for i in range(3):
            spec = full[i][:, :, r * h_local:(r + 1) * h_local]
            assert got[i].shape == spec.shape
            assert np.array_equal(got[i], spec), f"rank{r} qkv[{i}]"


def _separate_exchange(shards, U):
    """One tensor's Ulysses input exchange without packing: each rank sends
    its head slices destination-major, all_to_all_single, and the receiver
    puts source rank r's rows at [r*S_l, (r+1)*S_l)."""
    B, S_l, H, D = shards[0].shape
    h_l = H // U
    sends = [np.ascontiguousarray(x.reshape(B, S_l, U, h_l, D).transpose(2, 0, 1, 3, 4)) for x in shards]
    out = []
    for j in range(U):
        chunks = [np.split(s.reshape(-1), U)[j].reshape(B, S_l, h_l, D) for s in sends]
        out.append(np.concatenate(chunks, axis=1))
    return out


@pytest.mark.parametrize("U,B,S_l,H,D", [(4, 1, 32, 8, 64), (2, 2, 24, 6, 32), (3, 2, 5, 9, 8)])
def test_packed_equals_three_separate_exchanges(orc, U, B, S_l, H, D):
    gen = torch.Generator().manual_seed(99)
    shards = [[_bits((B, S_l, H, D), gen) for _ in range(3)] for _ in range(U)]
    recvs = orc.all_to_all([orc.pack_qkv(*shards[r], U) for r in range(U)])
    packed = [orc.unpack_qkv(recvs[r], U) for r in range(U)]
    for t in range(3):
        sep = _separate_exchange([shards[r][t] for r in range(U)], U)
        for r in range(U):
            assert np.array_equal(packed[r][t], sep[r])


@pytest.mark.parametrize("U,B,S_l,H,D", [(1, 1, 9, 4, 16), (2, 1, 8, 4, 16), (4, 2, 5, 8, 8), (3, 1, 4, 6, 8)])
def test_round_trip_input_then_reverse_exchange(orc, U, B, S_l, H, D):
    """seq->head->seq: the reverse exchange gives every rank its input back."""
    gen = torch.Generator().manual_seed(5)
    shards = [[_bits((B, S_l, H, D), gen) for _ in range(3)] for _ in range(U)]
    recvs = orc.all_to_all([orc.pack_qkv(*shards[r], U) for r in range(U)])
    heads = [orc.unpack_qkv(recvs[r], U) for r in range(U)]
    for t in range(3):
        back = orc.all_to_all([orc.pack_out(heads[r][t], U) for r in range(U)])
        for r in range(U):
            y = orc.unpack_out(back[r], U)
            assert np.array_equal(y, shards[r][t])


def test_reverse_exchange_is_head_concat(orc):
    """unpack_out puts source rank r's slice at heads [r*h_l, (r+1)*h_l)."""
    U, B, S_l, h_l, D = 3, 2, 4, 2, 8
    gen = torch.Generator().manual_seed(11)
    recv = _bits((U, B, S_l, h_l, D), gen)
    y = orc.unpack_out(recv, U)
    for r in range(U):
        assert np.array_equal(y[:, :, r * h_l:(r + 1) * h_l], recv[r])
    o = _bits((B, U * S_l, h_l, D), gen)
    send = orc.pack_out(o, U)
    for r in range(U):
        assert np.array_equal(send[r], o[:, r * S_l:(r + 1) * S_l])


def test_pack_U1_is_a_copy(orc):
    gen = torch.Generator().manual_seed(3)
    q, k, v = (_bits((2, 7, 3, 16), gen) for _ in range(3))
    st = orc.pack_qkv(q, k, v, 1)
    assert np.array_equal(st[0, 0], q) and np.array_equal(st[0, 1], k) and np.array_equal(st[0, 2], v)
    back = orc.unpack_qkv(st, 1)
    for a, b in zip(back, (q, k, v)):
        assert np.array_equal(a, b)


@pytest.mark.parametrize("U,A,B,S,H,D", [(2, 2, 1, 32, 4, 8), (4, 2, 2, 64, 8, 8), (1, 4, 1, 24, 3, 8), (2, 3, 1, 36, 4, 8)])
def test_composed_ulysses_then_allgather_rebuilds_sequence(orc, U, A, B, S, H, D):
    gen = torch.Generator().manual_seed(1234)
    full = [_bits((B, S, H, D), gen) for _ in range(3)]
    R = U * A
    S_l = S // R
    sh = [[x[:, g * S_l:(g + 1) * S_l] for x in full] for g in range(R)]
    res = orc.ulysses_agkv_forward([s[0] for s in sh], [s[1] for s in sh], [s[2] for s in sh], U, A)
    h_l = H // U
    for u in range(U):
        assert np.array_equal(res["k"][u], full[1][:, :, u * h_l:(u + 1) * h_l])
        assert np.array_equal(res["v"][u], full[2][:, :, u * h_l:(u + 1) * h_l])
        for a in range(A):
            g = a * U + u
            rows = slice(a * S // A, (a + 1) * S // A)
            assert np.array_equal(res["q"][g], full[0][:, rows, u * h_l:(u + 1) * h_l])


def test_gather_before_ulysses_permutes_the_sequence(orc):
    """The opposite order (gather the pre-transform shards over the A group,
    then the Ulysses exchange) concatenates non-adjacent regions and does not
    rebuild the global sequence: the order is load-bearing."""
    U, A, B, S, H, D = 2, 2, 1, 16, 4, 8
    gen = torch.Generator().manual_seed(1234)
    full = [_bits((B, S, H, D), gen) for _ in range(3)]
    R, S_l, h_l = U * A, S // (U * A), H // U
    sh = [[x[:, g * S_l:(g + 1) * S_l] for x in full] for g in range(R)]
    gathered = [[orc.all_gather([sh[a * U + u][t] for a in range(A)]) for t in range(3)] for u in range(U)]
    recvs = orc.all_to_all([orc.pack_qkv(*gathered[u], U) for u in range(U)])
    k_u0 = orc.unpack_qkv(recvs[0], U)[1]
    spec = full[1][:, :, 0:h_l]
    assert k_u0.shape == spec.shape
    assert not np.array_equal(k_u0, spec)
    # it is a row permutation of the spec
    assert sorted(map(bytes, k_u0.reshape(S, -1))) == sorted(map(bytes, spec.reshape(S, -1)))


def test_joint_keys_appended_after_image(orc):
    U, A, B, S, H, D, J = 2, 2, 1, 16, 4, 8, 5
    gen = torch.Generator().manual_seed(2)
    full = [_bits((B, S, H, D), gen) for _ in range(3)]
    jk, jv = _bits((B, J, H, D), gen), _bits((B, J, H, D), gen)
    R, S_l, h_l = U * A, S // (U * A), H // U
    sh = [[x[:, g * S_l:(g + 1) * S_l] for x in full] for g in range(R)]
    res = orc.ulysses_agkv_forward([s[0] for s in sh], [s[1] for s in sh], [s[2] for s in sh], U, A, jk, jv)
    for u in range(U):
        assert res["k"][u].shape == (B, S + J, h_l, D)
        assert np.array_equal(res["k"][u][:, S:], jk[:, :, u * h_l:(u + 1) * h_l])
        assert np.array_equal(res["v"][u][:, :S], full[2][:, :, u * h_l:(u + 1) * h_l])


def test_pure_python_pack_twin(orc):
    gen = torch.Generator().manual_seed(4)
    q, k, v = (_bits((2, 3, 4, 8), gen) for _ in range(3))
    assert np.array_equal(orc.py_pack_qkv(q, k, v, 2), orc.pack_qkv(q, k, v, 2))


def test_pack_rejects_indivisible_heads(orc):
    gen = torch.Generator().manual_seed(4)
    q = _bits((1, 2, 6, 8), gen)
    with pytest.raises(ValueError):
        orc.pack_qkv(q, q, q, 4)
