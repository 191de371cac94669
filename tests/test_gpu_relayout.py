"""GPU parity of the layout steps against the oracle: bit-exact, every byte
of every output written (NaN prefill), nothing written outside the outputs
(guard bands), on the pages' shapes, the benchmark shapes and ragged ones."""
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


def _bits(shape, gen, dtype="bf16"):
    return workloads.randn(shape, gen, dtype)


CASES = [  # (B, S_l, H, D, U)
    (1, 32, 8, 64, 4),      # sglang page test, world 4
    (2, 24, 6, 32, 2),      # sglang page test, world 2
    (1, 256, 2, 128, 2),    # tiny
    (1, 1024, 24, 128, 4),  # pack workload, full size
    (1, 7, 9, 8, 3),        # ragged: odd rows, run of one 16-byte vector
    (2, 5, 40, 128, 4),     # long runs (10 heads x 128 -> several segments)
    (1, 13, 80, 128, 2),    # run of 40 heads: multi-segment
    (3, 3, 4, 16, 1),       # U = 1 identity
    (1, 20, 96, 128, 8),    # U = 8, 12 heads per destination
    (2, 9, 8, 64, 8),       # U = 8, one head per destination, ragged rows
]


@pytest.mark.parametrize("B,S_l,H,D,U", CASES)
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
def test_pack_unpack_bit_exact(ctx, orc, B, S_l, H, D, U, dtype):
    gen = torch.Generator().manual_seed(1234)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float16
    q, k, v = (_bits((B, S_l, H, D), gen, dtype) for _ in range(3))
    h_l = H // U
    st = Guarded((U, 3, B, S_l, h_l, D), tdt)
    ctx.ctx_pack_qkv(q.cuda(), k.cuda(), v.cuda(), st.t, U)
    torch.cuda.synchronize()
    expect = orc.pack_qkv(u16(q), u16(k), u16(v), U)
    assert st.intact()
    assert np.array_equal(u16(st.t), expect)
    outs = [Guarded((B, U * S_l, h_l, D), tdt) for _ in range(3)]
    ctx.ctx_unpack_qkv(st.t, outs[0].t, outs[1].t, outs[2].t, U)
    torch.cuda.synchronize()
    exp_un = orc.unpack_qkv(expect, U)
    for o, e in zip(outs, exp_un):
        assert o.intact()
        assert np.array_equal(u16(o.t), e)


def test_unpack_places_into_strided_global_buffers(ctx, orc):
    """Rank a's rows land at [a*U*S_l, ...) of a buffer with Sk rows per batch."""
    B, S_l, h_l, D, U, A, J = 2, 6, 3, 64, 2, 3, 5
    gen = torch.Generator().manual_seed(9)
    recv = _bits((U, 3, B, S_l, h_l, D), gen)
    S = U * A * S_l
    qg = Guarded((B, S, h_l, D), torch.bfloat16)
    kg = Guarded((B, S + J, h_l, D), torch.bfloat16)
    vg = Guarded((B, S + J, h_l, D), torch.bfloat16)
    a = 1
    r0 = a * U * S_l
    ctx.ctx_unpack_qkv(recv.cuda(), qg.t[:, r0:], kg.t[:, r0:], vg.t[:, r0:], U,
                       q_batch_stride_rows=S, kv_batch_stride_rows=S + J)
    torch.cuda.synchronize()
    eq, ek, ev = orc.unpack_qkv(u16(recv), U)
    assert np.array_equal(u16(qg.t)[:, r0:r0 + U * S_l], eq)
    assert np.array_equal(u16(kg.t)[:, r0:r0 + U * S_l], ek)
    assert np.array_equal(u16(vg.t)[:, r0:r0 + U * S_l], ev)
    # rows of other ranks untouched (still the NaN prefill)
    assert (u16(kg.t)[:, :r0] == 0xFFFF).all() and (u16(kg.t)[:, r0 + U * S_l:] == 0xFFFF).all()
    assert (u16(qg.t)[:, :r0] == 0xFFFF).all()
    assert qg.intact() and kg.intact() and vg.intact()


@pytest.mark.parametrize("B,S_l,h_l,D,U,stride_extra", [(1, 16, 2, 128, 4, 0), (2, 9, 10, 128, 4, 7),
                                                         (2, 5, 1, 8, 3, 0), (1, 2363, 10, 128, 4, 0)])
def test_reverse_exchange_bit_exact(ctx, orc, B, S_l, h_l, D, U, stride_extra):
    gen = torch.Generator().manual_seed(77)
    stride = U * S_l + stride_extra
    o_full = _bits((B, stride, h_l, D), gen)
    send = Guarded((U, B, S_l, h_l, D), torch.bfloat16)
    ctx.ctx_pack_out(o_full.cuda(), send.t, U, o_batch_stride_rows=stride)
    torch.cuda.synchronize()
    exp_send = orc.pack_out(u16(o_full[:, :U * S_l]), U)
    assert send.intact() and np.array_equal(u16(send.t), exp_send)
    y = Guarded((B, S_l, U * h_l, D), torch.bfloat16)
    ctx.ctx_unpack_out(send.t, y.t, U)
    torch.cuda.synchronize()
    assert y.intact() and np.array_equal(u16(y.t), orc.unpack_out(exp_send, U))


@pytest.mark.parametrize("G,U,chunk", [(1, 2, 16), (2, 4, 4096), (1, 4, 3 * 1024 * 6 * 128 * 2), (3, 3, 48)])
def test_sim_all_to_all_chunk_semantics(ctx, orc, G, U, chunk):
    gen = torch.Generator().manual_seed(5)
    send = torch.randint(0, 255, (G, U, U, chunk), generator=gen, dtype=torch.uint8)
    recv = Guarded((G, U, U, chunk), torch.uint8, fill_nan=False)
    recv.t.fill_(0x5A)
    ctx.ctx_sim_all_to_all(send.cuda(), recv.t, G, U)
    torch.cuda.synchronize()
    got = recv.t.cpu().numpy()
    s = send.numpy()
    for g in range(G):
        exp = orc.all_to_all([s[g, r] for r in range(U)])
        for j in range(U):
            assert np.array_equal(got[g, j], exp[j])
    assert recv.intact()


def test_wan14b_rank_pack_full_size(ctx, orc):
    """One rank of the Wan-14B-like workload at full size: [1,9450,40,128] x3, U=4."""
    wl = workloads.WORKLOADS["wan14b"]
    gen = torch.Generator().manual_seed(1234)
    q, k, v = (_bits((1, wl.S_l, wl.H, wl.D), gen) for _ in range(3))
    st = torch.empty((wl.U, 3, 1, wl.S_l, wl.h_l, wl.D), dtype=torch.bfloat16, device="cuda")
    ctx.ctx_pack_qkv(q.cuda(), k.cuda(), v.cuda(), st, wl.U)
    torch.cuda.synchronize()
    assert np.array_equal(u16(st), orc.pack_qkv(u16(q), u16(k), u16(v), wl.U))


def test_host_pointer_is_rejected(ctx):
    q = torch.zeros((1, 4, 2, 8), dtype=torch.bfloat16).pin_memory()
    st = torch.empty((2, 3, 1, 4, 1, 8), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(ctx.CtxError) as e:
        ctx.ctx_pack_qkv(q, q.clone().pin_memory(), q.clone().pin_memory(), st, 2)
    assert e.value.status == 1


@pytest.mark.parametrize("layout", [0, 1])
@pytest.mark.parametrize("B,S_l,H,D,U", [
    (1, 16, 14, 128, 4), (2, 5, 7, 64, 3), (1, 9, 8, 128, 4), (1, 3, 3, 8, 2),
    # heads of 9 and 17 vectors (D = 72, 136): the interleaved offsets carry a
    # remainder that is not a power of two
    (2, 3, 5, 72, 2), (1, 4, 33, 136, 2),
    # runs longer than one warp pass (40 x 128 and 33 x 136 elements per rank and part)
    (1, 6, 40, 128, 1), (1, 5, 33, 136, 1),
])
def test_pack_ex_bit_exact(ctx, orc, B, S_l, H, D, U, layout):
    gen = torch.Generator().manual_seed(71)
    q, k, v = (_bits((B, S_l, H, D), gen) for _ in range(3))
    h_l = -(-H // U)
    shape = (U, 3, B, S_l, h_l, D) if layout == 0 else (U, B, S_l, h_l, 3 * D)
    st = Guarded(shape, torch.bfloat16)
    ctx.ctx_pack_qkv_ex(q.cuda(), k.cuda(), v.cuda(), st.t, U, layout)
    torch.cuda.synchronize()
    expect = orc.pack_qkv_ex(u16(q), u16(k), u16(v), U, layout)
    assert st.intact() and np.array_equal(u16(st.t), expect)
    outs = [Guarded((B, U * S_l, h_l, D), torch.bfloat16) for _ in range(3)]
    ctx.ctx_unpack_qkv_ex(st.t, outs[0].t, outs[1].t, outs[2].t, U, B, S_l, h_l, D, layout)
    torch.cuda.synchronize()
    for o, e in zip(outs, orc.unpack_qkv_ex(expect, U, layout)):
        assert o.intact() and np.array_equal(u16(o.t), e)


@pytest.mark.parametrize("B,S_l,H,D,U", [(2, 7, 14, 128, 4), (2, 3, 40, 64, 1), (3, 5, 10, 72, 2)])
def test_interleaved_unpack_strided(ctx, orc, B, S_l, H, D, U):
    """The interleaved unpack placing every rank's rows inside larger gathered
    buffers (batch strides of U*S_l + 3 and U*S_l + 5 rows): placed rows equal
    the oracle's unpack, every other row stays untouched."""
    gen = torch.Generator().manual_seed(73)
    q, k, v = (_bits((B, S_l, H, D), gen) for _ in range(3))
    h_l = -(-H // U)
    staging = orc.pack_qkv_ex(u16(q), u16(k), u16(v), U, 1)
    st = torch.from_numpy(staging.view(np.int16)).view(torch.bfloat16).cuda()
    rows = U * S_l
    qs, ks = rows + 3, rows + 5
    outs = [Guarded((B, n, h_l, D), torch.bfloat16) for n in (qs, ks, ks)]
    for o in outs:
        o.t.view(torch.int16).fill_(-12345)
    ctx.ctx_unpack_qkv_ex(st, outs[0].t, outs[1].t, outs[2].t, U, B, S_l, h_l, D, 1,
                          q_batch_stride_rows=qs, kv_batch_stride_rows=ks)
    torch.cuda.synchronize()
    for o, e in zip(outs, orc.unpack_qkv_ex(staging, U, 1)):
        got = u16(o.t)
        assert o.intact()
        assert np.array_equal(got[:, :rows], e)
        assert (got[:, rows:] == np.uint16(np.int16(-12345).view(np.uint16))).all()


@pytest.mark.parametrize("B,S_l,h_l,H,D,U", [(1, 16, 4, 14, 128, 4), (2, 5, 3, 7, 64, 3), (1, 4, 2, 8, 8, 4)])
def test_unpack_out_ex_drops_pad_heads(ctx, orc, B, S_l, h_l, H, D, U):
    gen = torch.Generator().manual_seed(72)
    recv = _bits((U, B, S_l, h_l, D), gen)
    y = Guarded((B, S_l, H, D), torch.bfloat16)
    ctx.ctx_unpack_out_ex(recv.cuda(), y.t, U)
    torch.cuda.synchronize()
    assert y.intact() and np.array_equal(u16(y.t), orc.unpack_out_ex(u16(recv), U, H))


@pytest.mark.parametrize("layout", [0, 1], ids=["tqkv", "interleaved"])
def test_beyond_2pow31_elements(ctx, orc, layout):
    """Pack and unpack of tensors with more than 2^31 elements each (64-bit
    offsets): per-rank Q/K/V [1, 65541, 256, 128], U = 8 (staging 12.9 GB),
    in either staging layout. Each input is a seeded [1, 512, 256, 128] block
    repeated along the rows on the device; sampled rows (always the last ones)
    are compared bit for bit with the oracle applied to the same rows."""
    B, S_l, H, D, U, blk = 1, (1 << 16) + 5, 256, 128, 8, 512
    h_l = H // U
    assert B * S_l * H * D > 2 ** 31
    gen = torch.Generator().manual_seed(32)
    blocks = [_bits((B, blk, H, D), gen) for _ in range(3)]
    reps = -(-S_l // blk)
    q, k, v = (b.cuda().repeat(1, reps, 1, 1)[:, :S_l].contiguous() for b in blocks)
    shape = (U, 3, B, S_l, h_l, D) if layout == 0 else (U, B, S_l, h_l, 3 * D)
    st = torch.empty(shape, dtype=torch.bfloat16, device="cuda")
    ctx.ctx_pack_qkv_ex(q, k, v, st, U, layout)
    del q, k, v
    outs = [torch.empty((B, U * S_l, h_l, D), dtype=torch.bfloat16, device="cuda") for _ in range(3)]
    ctx.ctx_unpack_qkv_ex(st, *outs, U, B, S_l, h_l, D, layout)
    torch.cuda.synchronize()
    rows = np.concatenate([workloads.sample_rows(S_l, 64), np.arange(S_l - 8, S_l)])
    for s in rows:
        src = [u16(b[:, s % blk:s % blk + 1]) for b in blocks]
        exp_st = orc.pack_qkv_ex(*src, U, layout)           # the row s of every destination
        got_st = st[:, :, :, s:s + 1] if layout == 0 else st[:, :, s:s + 1]
        assert np.array_equal(u16(got_st), exp_st), s
        exp_un = orc.unpack_qkv_ex(exp_st, U, layout)       # 3 x [B, U, h_l, D]: row r <- source r
        for t in range(3):
            got = u16(outs[t][:, s::S_l][:, :U])
            assert np.array_equal(got, exp_un[t]), (s, t)
