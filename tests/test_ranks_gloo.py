"""The per-rank layer with real collectives (CPU, gloo): U x A processes, one
per rank g = a*U + u (vllm-omni PR #7641 rank layout: Ulysses groups are
contiguous blocks of U ranks, AllGather-KV groups stride by U). Each rank runs
diffusion_transformer_context_gb300.ranks.RankLayer with the oracle's steps
in place of the library's, so what is checked here is the host side: the
process groups, the all_to_all_single chunks, the all_gather into the
gathered rows, the joint re-attach and the reverse exchange. Every rank's
local Q, gathered K/V, key mask and final output must equal the
single-process composed oracle's bit for bit."""
import socket

import pytest
import torch.multiprocessing as mp

import workloads
from rank_worker import run_rank


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("wl", [
    workloads.custom("r_u2a2", B=1, S=64, H=4, D=16, U=2, A=2),
    workloads.custom("r_u4a1", B=1, S=64, H=8, D=16, U=4, A=1),
    workloads.custom("r_u1a4", B=1, S=64, H=3, D=16, U=1, A=4),
    workloads.custom("r_u2a2_h5_joint_masks_front", B=1, S=64, H=5, D=16, U=2, A=2, joint=6, text_len_range=(1, 6),
                     joint_front=True, image_pad_range=(1, 10)),
    workloads.custom("r_u2a2_joint_rear", B=1, S=48, H=4, D=8, U=2, A=2, joint=5, text_len_range=(2, 5)),
], ids=lambda w: w.name)
def test_ranks_as_processes_match_the_composed_oracle(wl):
    world = wl.U * wl.A
    mp.spawn(run_rank, args=(world, _free_port(), wl), nprocs=world, join=True)


@pytest.mark.parametrize("wl", [
    workloads.custom("ri_u2a2_h5_joint", B=1, S=64, H=5, D=16, U=2, A=2, joint=6, text_len_range=(1, 6)),
    workloads.custom("ri_u1a2", B=1, S=32, H=3, D=8, U=1, A=2),
], ids=lambda w: w.name)
def test_ranks_interleaved_staging_match_the_composed_oracle(wl):
    """The same job with the interleaved staging layout [U,B,S_l,h_l,3D]
    (sglang PR #33667 excerpt): the chunks the all-to-all moves change, the
    layer's results do not."""
    world = wl.U * wl.A
    mp.spawn(run_rank, args=(world, _free_port(), wl, 1), nprocs=world, join=True)
