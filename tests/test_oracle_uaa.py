"""Pins for uneven heads (head padding when H % U != 0, vllm-omni PR #7641
"advanced_uaa": e.g. 14 heads at U=4 are padded to 16) and for the
interleaved staging layout (U, rows, h_l, 3D) of the sglang PR #33667
excerpt. Expected values come from numpy slicing / concatenation, not from
the oracle's loops."""
import numpy as np
import pytest
import torch

import workloads


def _bits(shape, gen):
    return workloads.as_u16(workloads.randn(shape, gen))


def _padded(x, U):
    B, S, H, D = x.shape
    h_l = -(-H // U)
    out = np.zeros((B, S, U * h_l, D), np.uint16)
    out[:, :, :H] = x
    return out, h_l


@pytest.mark.parametrize("U,B,S_l,H,D", [(4, 1, 8, 14, 16), (3, 2, 5, 7, 8), (4, 1, 4, 16, 8), (2, 1, 3, 3, 8)])
def test_padded_pack_is_padded_head_slices(orc, U, B, S_l, H, D):
    gen = torch.Generator().manual_seed(61)
    q, k, v = (_bits((B, S_l, H, D), gen) for _ in range(3))
    st = orc.pack_qkv_ex(q, k, v, U)
    h_l = -(-H // U)
    assert st.shape == (U, 3, B, S_l, h_l, D)
    for t, x in enumerate((q, k, v)):
        xp, _ = _padded(x, U)
        for r in range(U):
            assert np.array_equal(st[r, t], xp[:, :, r * h_l:(r + 1) * h_l])


def test_fourteen_heads_at_u4_pad_to_sixteen(orc):
    """The page's case: 14 heads, U = 4 -> 16 padded heads (+14.3 % work);
    ranks 0-2 receive 4 real heads, rank 3 two real and two zero heads."""
    gen = torch.Generator().manual_seed(62)
    q = _bits((1, 6, 14, 8), gen)
    st = orc.pack_qkv_ex(q, q, q, 4)
    assert st.shape[4] == 4 and 4 * st.shape[4] == 16 and (16 - 14) / 14 == pytest.approx(0.143, abs=1e-3)
    assert (st[3, :, :, :, 2:] == 0).all() and (st[3, :, :, :, :2] != 0).any()
    assert np.array_equal(st[2, 0], q[:, :, 8:12])


@pytest.mark.parametrize("U,B,S_l,H,D", [(4, 1, 8, 8, 16), (2, 2, 5, 6, 8), (3, 1, 4, 7, 8)])
def test_interleaved_layout(orc, U, B, S_l, H, D):
    gen = torch.Generator().manual_seed(63)
    q, k, v = (_bits((B, S_l, H, D), gen) for _ in range(3))
    st = orc.pack_qkv_ex(q, k, v, U, orc.LAYOUT_INTERLEAVED)
    h_l = -(-H // U)
    assert st.shape == (U, B, S_l, h_l, 3 * D)
    qp, kp, vp = (_padded(x, U)[0] for x in (q, k, v))
    for r in range(U):
        sl = slice(r * h_l, (r + 1) * h_l)
        assert np.array_equal(st[r], np.concatenate([qp[:, :, sl], kp[:, :, sl], vp[:, :, sl]], axis=-1))
    # both layouts unpack to identical tensors after the exchange
    sends_i = [orc.pack_qkv_ex(q, k, v, U, orc.LAYOUT_INTERLEAVED) for _ in range(U)]
    sends_t = [orc.pack_qkv_ex(q, k, v, U, orc.LAYOUT_TQKV) for _ in range(U)]
    ri, rt = orc.all_to_all(sends_i), orc.all_to_all(sends_t)
    for r in range(U):
        a = orc.unpack_qkv_ex(ri[r], U, orc.LAYOUT_INTERLEAVED)
        b = orc.unpack_qkv_ex(rt[r], U, orc.LAYOUT_TQKV)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("U,B,S_l,H,D", [(4, 1, 6, 14, 8), (3, 2, 4, 5, 8)])
def test_padded_round_trip_drops_pad_heads(orc, U, B, S_l, H, D, layout):
    """Input exchange with padding, then the reverse exchange keeping H heads,
    returns every rank's input; the gathered K of rank r are the global
    padded head slice r."""
    gen = torch.Generator().manual_seed(64)
    shards = [[_bits((B, S_l, H, D), gen) for _ in range(3)] for _ in range(U)]
    recvs = orc.all_to_all([orc.pack_qkv_ex(*shards[r], U, layout) for r in range(U)])
    heads = [orc.unpack_qkv_ex(recvs[r], U, layout) for r in range(U)]
    h_l = -(-H // U)
    full_k = np.concatenate([shards[r][1] for r in range(U)], axis=1)
    kp, _ = _padded(full_k, U)
    for r in range(U):
        assert np.array_equal(heads[r][1], kp[:, :, r * h_l:(r + 1) * h_l])
    for t in range(3):
        back = orc.all_to_all([orc.pack_out(heads[r][t], U) for r in range(U)])
        for r in range(U):
            assert np.array_equal(orc.unpack_out_ex(back[r], U, H), shards[r][t])


def test_unpadded_ex_equals_plain_pack(orc):
    gen = torch.Generator().manual_seed(65)
    q, k, v = (_bits((2, 5, 8, 16), gen) for _ in range(3))
    assert np.array_equal(orc.pack_qkv_ex(q, k, v, 4), orc.pack_qkv(q, k, v, 4))
