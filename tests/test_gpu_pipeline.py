"""The whole simulated layer on the GPU (all U x A ranks: pack -> all-to-all
-> unpack into the gathered buffers -> attention -> reverse exchange)
against the oracle's composed pipeline (vllm-omni PR #7641 order).

Layout results are compared bit for bit; attention within the tolerance of
test_gpu_attention; the reverse exchange bit for bit on the GPU's own
attention output.
"""
import numpy as np
import pytest
import torch

import workloads
from gpu_util import u16

pytestmark = pytest.mark.gpu

O_MAX, O_MEAN, LSE_TOL = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module")
def ctx():
    import diffusion_transformer_context_gb300 as m
    m.build()
    return m


def _oracle_side(orc, inp, layout=0):
    wl = inp.wl
    R = wl.ranks
    sh = [[u16(inp.shard(t, g)) for t in (inp.q, inp.k, inp.v)] for g in range(R)]
    jk = u16(inp.jk) if inp.jk is not None else None
    jv = u16(inp.jv) if inp.jv is not None else None
    return orc.ulysses_agkv_forward([s[0] for s in sh], [s[1] for s in sh], [s[2] for s in sh],
                                    wl.U, wl.A, jk, jv, layout, joint_front=wl.joint_front)


def _check_layer(ctx, orc, wl, n_rows=None, layout=0, pack_view=True):
    from diffusion_transformer_context_gb300.simulate import SimLayer
    inp = workloads.make_inputs(wl)
    sim = SimLayer(wl, layout=layout, fuse_reverse=False, pack_view=pack_view)
    sim.load(inp)
    sim.step()
    st = ctx.ctx_device_status()
    assert st == 0, ctx.ctx_status_string(st)
    res = _oracle_side(orc, inp, layout)
    U, A = wl.U, wl.A
    # layout steps: bit-exact
    for u in range(U):
        assert np.array_equal(u16(sim.kg[u]), res["k"][u]), f"K group {u}"
        assert np.array_equal(u16(sim.vg[u]), res["v"][u]), f"V group {u}"
    for g in range(wl.ranks):
        assert np.array_equal(u16(sim.rank_q(g)), res["q"][g]), f"Q rank {g}"
    if not sim.attention:
        return
    # the key mask of the gathered layout: the oracle's merge of the raw masks,
    # and the library's (one per head group) bit for bit
    mask = orc.merge_joint_attn_mask(inp.image_mask, inp.joint_mask, wl.B, wl.S, wl.joint, wl.joint_front)
    if mask is None:
        assert sim.mask is None
    else:
        for u in range(U):
            assert np.array_equal(sim.mask[u * wl.B:(u + 1) * wl.B].cpu().numpy(), mask), f"key mask group {u}"
    # attention of every rank (rank g: its local-Q against its head group's K/V)
    out = sim.out.float().cpu().numpy()
    lse = sim.lse.cpu().numpy().reshape(U, wl.B, sim.h_l, wl.S)
    rows_per_rank = wl.S // A
    errs = []
    for g in range(wl.ranks):
        a, u = divmod(g, U)
        qg, kg, vg = res["q"][g], res["k"][u], res["v"][u]
        if n_rows is None:
            eO, eL = orc.attention(qg, kg, vg, mask)
            gO = out[u][:, a * rows_per_rank:(a + 1) * rows_per_rank]
            gL = lse[u][:, :, a * rows_per_rank:(a + 1) * rows_per_rank]
            errs.append(np.abs(gO - eO))
            assert np.abs(gL - eL).max() <= LSE_TOL
        else:
            rows_i = workloads.sample_rows(rows_per_rank, n_rows)
            rng = np.random.default_rng(g)
            bhi = np.stack([rng.integers(0, wl.B, rows_i.size), rng.integers(0, sim.h_l, rows_i.size),
                            rows_i], axis=1)
            eo, el = orc.attention_rows(qg, kg, vg, bhi, mask)
            go = np.stack([out[u][b, a * rows_per_rank + i, h] for b, h, i in bhi])
            gl = np.array([lse[u][b, h, a * rows_per_rank + i] for b, h, i in bhi])
            errs.append(np.abs(go - eo))
            assert np.abs(gl - el).max() <= LSE_TOL
    e = np.concatenate([x.ravel() for x in errs])
    assert e.max() <= O_MAX and e.mean() <= O_MEAN, (e.max(), e.mean())
    # reverse exchange of the GPU's own output: bit-exact
    o_ranks = [u16(sim.out[u][:, a * rows_per_rank:(a + 1) * rows_per_rank])
               for a in range(A) for u in range(U)]
    back = orc.ulysses_reverse(o_ranks, U, A, wl.H)
    for g in range(wl.ranks):
        assert np.array_equal(u16(sim.rank_output(g)), back[g]), f"reverse rank {g}"
    if U > 1:
        # the send-side relayout fused into the attention epilogue gives the same bits
        fused = SimLayer(wl, layout=layout, fuse_reverse=True)
        fused.load(inp)
        fused.step()
        assert ctx.ctx_device_status() == 0
        assert torch.equal(fused.lse, sim.lse)
        for g in range(wl.ranks):
            assert torch.equal(fused.rank_output(g), sim.rank_output(g)), f"fused reverse rank {g}"


def test_tiny(ctx, orc):
    _check_layer(ctx, orc, workloads.WORKLOADS["tiny"])


def test_pack_workload(ctx, orc):
    _check_layer(ctx, orc, workloads.WORKLOADS["pack"])


@pytest.mark.parametrize("wl", [
    workloads.custom("u2a2_joint_b2", B=2, S=512, H=8, D=128, U=2, A=2, joint=64, text_len_range=(1, 64)),
    workloads.custom("u4a2_d64", B=1, S=1024, H=8, D=64, U=4, A=2),
    workloads.custom("u1a4_ragged", B=1, S=1000, H=3, D=128, U=1, A=4),
    workloads.custom("u3a1", B=2, S=378, H=6, D=128, U=3, A=1),
    workloads.custom("u8a1_h16", B=1, S=1024, H=16, D=128, U=8, A=1),
    workloads.custom("u2a4_h12_joint", B=1, S=768, H=12, D=128, U=2, A=4, joint=48, text_len_range=(8, 48)),
], ids=lambda w: w.name)
def test_composed_small(ctx, orc, wl):
    _check_layer(ctx, orc, wl)


@pytest.mark.parametrize("wl", [
    workloads.custom("u1a4_ragged_packed", B=1, S=1000, H=3, D=128, U=1, A=4),
    workloads.custom("u1a8_b2_packed", B=2, S=1024, H=4, D=64, U=1, A=8),
], ids=lambda w: w.name)
def test_u1_pack_run(ctx, orc, wl):
    """U = 1 with the identity pack launched (the default views the input instead)."""
    _check_layer(ctx, orc, wl, pack_view=False)


@pytest.mark.parametrize("wl", [
    workloads.custom("uaa_u4_h14", B=1, S=1024, H=14, D=128, U=4, A=1),
    workloads.custom("uaa_u4a2_h14_joint", B=2, S=512, H=14, D=64, U=4, A=2, joint=32, text_len_range=(1, 32)),
    workloads.custom("uaa_u3_h7", B=1, S=384, H=7, D=128, U=3, A=1),
], ids=lambda w: w.name)
def test_uneven_heads(ctx, orc, wl):
    """H % U != 0: heads zero-padded to U*ceil(H/U) (vllm-omni "advanced_uaa")."""
    _check_layer(ctx, orc, wl)


@pytest.mark.parametrize("wl", [
    workloads.WORKLOADS["tiny"],
    workloads.custom("inter_u4a2", B=2, S=512, H=8, D=128, U=4, A=2),
    workloads.custom("inter_u4_h14", B=1, S=512, H=14, D=64, U=4, A=1),
], ids=lambda w: w.name)
def test_interleaved_staging_layout(ctx, orc, wl):
    _check_layer(ctx, orc, wl, layout=1)


@pytest.mark.parametrize("wl", [
    # a 2-D image mask (padded suffix of the global sequence) with text padding, joint keys in front
    workloads.custom("img_mask_front_u2a2", B=2, S=512, H=8, D=128, U=2, A=2, joint=64, text_len_range=(1, 64),
                     joint_front=True, image_pad_range=(1, 100)),
    # the same rear, uneven heads
    workloads.custom("img_mask_rear_u4a2_h14", B=2, S=512, H=14, D=64, U=4, A=2, joint=32, text_len_range=(4, 32),
                     image_pad_range=(10, 60)),
    # an image mask only (no joint keys): the key mask is the image mask
    workloads.custom("img_mask_only_u1a4", B=1, S=1000, H=3, D=128, U=1, A=4, image_pad_range=(200, 300)),
    # joint keys without any mask (cached K/V reuse: joint K/V, no joint query): no key mask at all
    workloads.custom("joint_nomask_front_u2a2", B=1, S=512, H=4, D=128, U=2, A=2, joint=48, joint_front=True),
    # joint keys without a joint mask but with an image mask: the joint segment is filled with True
    workloads.custom("joint_fill_u2a1", B=2, S=384, H=4, D=128, U=2, A=1, joint=40, image_pad_range=(0, 50)),
], ids=lambda w: w.name)
def test_mask_merge_layers(ctx, orc, wl):
    """The a4 step with non-trivial masks (vllm-omni PR #7641 follow-up
    review commit's cases): the merged key mask of every head group equals
    the oracle's bit for bit and the attention of every rank matches."""
    _check_layer(ctx, orc, wl)


def test_qwen_layer(ctx, orc):
    _check_layer(ctx, orc, workloads.WORKLOADS["qwen"], n_rows=128)


def test_wan480_layer(ctx, orc):
    _check_layer(ctx, orc, workloads.WORKLOADS["wan480"], n_rows=48)


def test_wan14b_layer(ctx, orc):
    _check_layer(ctx, orc, workloads.WORKLOADS["wan14b"], n_rows=24)
