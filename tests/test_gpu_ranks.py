"""The per-rank layer (one process per rank, collectives between the
library's calls) on the GPU. This pool gives one GPU per run, so the job here
is a single rank (U = A = 1, NCCL world of one): it exercises the library
path of RankLayer (its buffers, strides, joint re-attach, mask merge and the
attention) against the simulated layer and the oracle; the multi-rank wiring
is covered on CPU ranks over gloo (test_ranks_gloo.py)."""
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import workloads
from gpu_util import u16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import diffusion_transformer_context_gb300 as m
    m.build()
    return m


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("layout", [0, 1], ids=["tqkv", "interleaved"])
@pytest.mark.parametrize("wl", [
    workloads.custom("pr_u1a1", B=1, S=700, H=3, D=128, U=1, A=1),
    workloads.custom("pr_u1a1_joint_masks_front", B=1, S=512, H=4, D=128, U=1, A=1, joint=64,
                     text_len_range=(1, 64), joint_front=True, image_pad_range=(0, 40)),
], ids=lambda w: w.name)
def test_single_rank_job_matches_the_simulated_layer_and_the_oracle(ctx, orc, wl, layout):
    from diffusion_transformer_context_gb300.ranks import Groups, RankLayer
    from diffusion_transformer_context_gb300.simulate import SimLayer

    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{_free_port()}", rank=0, world_size=1,
                            device_id=torch.device("cuda", 0))
    try:
        inp = workloads.make_inputs(wl)
        layer = RankLayer(wl, Groups(1, 1), "cuda", layout=layout)
        layer.load(inp.q.cuda(), inp.k.cuda(), inp.v.cuda(), None if inp.jk is None else inp.jk.cuda(),
                   None if inp.jv is None else inp.jv.cuda(), inp.image_mask, inp.joint_mask)
        y = layer.step().clone()
        assert ctx.ctx_device_status() == 0
    finally:
        dist.destroy_process_group()
    sim = SimLayer(wl)
    sim.load(inp)
    sim.step()
    assert ctx.ctx_device_status() == 0
    assert torch.equal(y, sim.rank_output(0)), "per-rank layer differs from the simulated layer"
    mask = orc.merge_joint_attn_mask(inp.image_mask, inp.joint_mask, wl.B, wl.S, wl.joint, wl.joint_front)
    res = orc.ulysses_agkv_forward([u16(inp.q)], [u16(inp.k)], [u16(inp.v)], 1, 1,
                                   None if inp.jk is None else u16(inp.jk), None if inp.jv is None else u16(inp.jv),
                                   joint_front=wl.joint_front)
    eO, _ = orc.attention(res["q"][0], res["k"][0], res["v"][0], mask)
    err = np.abs(y.float().cpu().numpy() - eO)
    assert err.max() <= 2e-2 and err.mean() <= 2e-3, (err.max(), err.mean())
