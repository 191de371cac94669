"""Worker of tests/test_ranks_gloo.py: one CPU rank of the per-rank layer
(diffusion_transformer_context_gb300.ranks.RankLayer) over gloo, its compute
steps done by the oracle, checked against the single-process composed oracle."""
import os

import numpy as np
import torch
import torch.distributed as dist


def u16(t):
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def bf16(a):
    return torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(torch.bfloat16)


def round_bf16_bits(o):
    """fp64 attention output -> bf16 bit patterns (round to nearest even)."""
    return u16(torch.from_numpy(np.ascontiguousarray(o)).to(torch.bfloat16))


class OracleOps:
    """The layer's compute steps done by the oracle on CPU bf16 tensors."""

    def __init__(self, orc, H):
        self.orc, self.H = orc, H

    def pack(self, x, staging, U, layout=0):
        staging.copy_(bf16(self.orc.pack_qkv_ex(u16(x[0]), u16(x[1]), u16(x[2]), U, layout)))

    def unpack(self, src, q, k, v, U, B, S_l, h_l, D, layout=0):
        for dst, r in zip((q, k, v), self.orc.unpack_qkv_ex(u16(src), U, layout)):
            dst.copy_(bf16(r))

    def merge_mask(self, image_mask, joint_mask, B, S, J, front, out):
        m = self.orc.merge_joint_attn_mask(None if image_mask is None else image_mask.numpy(),
                                           None if joint_mask is None else joint_mask.numpy(), B, S, J, front)
        out.copy_(torch.from_numpy(m))

    def workspace(self, *args):
        return None

    def _attend(self, q, k, v, mask, lse):
        O, L = self.orc.attention(u16(q), u16(k), u16(v), None if mask is None else mask.numpy())
        lse.copy_(torch.from_numpy(L))
        return round_bf16_bits(O)

    def attention(self, q, k, v, out, lse, mask, workspace):
        out.copy_(bf16(self._attend(q, k, v, mask, lse)))

    def attention_pack_out(self, q, k, v, send, U, S_l, lse, mask, workspace):
        send.copy_(bf16(self.orc.pack_out(self._attend(q, k, v, mask, lse), U)))

    def unpack_out(self, recv, y, U):
        y.copy_(bf16(self.orc.unpack_out_ex(u16(recv), U, self.H)))


def run_rank(rank, world, port, wl, layout=0):
    import oracle
    import workloads
    from diffusion_transformer_context_gb300.ranks import Groups, RankLayer

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        oracle.build()
        inp = workloads.make_inputs(wl)
        G = Groups(wl.U, wl.A)
        layer = RankLayer(wl, G, "cpu", ops=OracleOps(oracle, wl.H), layout=layout)
        layer.load(inp.shard(inp.q, rank), inp.shard(inp.k, rank), inp.shard(inp.v, rank), inp.jk, inp.jv,
                   inp.image_mask, inp.joint_mask)
        y = layer.step()
        # the single-process composed oracle, whole layer, every rank
        R = wl.U * wl.A
        sh = [[u16(inp.shard(t, g)) for t in (inp.q, inp.k, inp.v)] for g in range(R)]
        jk = None if inp.jk is None else u16(inp.jk)
        jv = None if inp.jv is None else u16(inp.jv)
        res = oracle.ulysses_agkv_forward([s[0] for s in sh], [s[1] for s in sh], [s[2] for s in sh], wl.U, wl.A,
                                          jk, jv, joint_front=wl.joint_front)
        mask = oracle.merge_joint_attn_mask(inp.image_mask, inp.joint_mask, wl.B, wl.S, wl.joint, wl.joint_front)
        a, u = divmod(rank, wl.U)
        assert np.array_equal(u16(layer.q), res["q"][rank]), f"local Q of rank {rank}"
        assert np.array_equal(u16(layer.kg), res["k"][u]), f"gathered K of rank {rank}"
        assert np.array_equal(u16(layer.vg), res["v"][u]), f"gathered V of rank {rank}"
        if mask is None:
            assert layer.mask is None
        else:
            assert np.array_equal(layer.mask.numpy(), mask), f"key mask of rank {rank}"
        outs = [round_bf16_bits(oracle.attention(res["q"][g], res["k"][g % wl.U], res["v"][g % wl.U], mask)[0])
                for g in range(R)]
        back = oracle.ulysses_reverse(outs, wl.U, wl.A, wl.H)
        assert np.array_equal(u16(y), back[rank]), f"output of rank {rank}"
    finally:
        dist.destroy_process_group()
