"""All U x A virtual ranks of one context-parallel attention layer on one GPU.

Rank g = a*U + u (vllm-omni PR #7641: Ulysses groups are contiguous blocks of
U ranks, AllGather-KV groups stride by U) holds input rows [g*S_l, (g+1)*S_l)
of Q, K, V [B, S, H, D]. One step runs, through the C ABI only:

  1. ctx_pack_qkv_ex for every rank into its staging buffer (heads that do
     not divide by U are zero-padded, either staging layout);
  2. ctx_sim_all_to_all inside every U group (skipped at U = 1, where the
     exchange is the identity);
  3. ctx_unpack_qkv_ex for every rank, writing its local Q rows into the
     all-ranks query buffer and its K/V rows straight into the gathered K/V
     buffer of its head group at image rows [a*S/A, (a+1)*S/A): the K/V
     AllGather is this placement, no bytes are copied for it; then
     ctx_merge_joint_attn_mask builds the [B, S + joint] key mask of the
     gathered layout from the raw image and joint masks (when there are any);
  4. one ctx_attn_lq_gkv over all ranks: the ranks of head group u share the
     gathered K/V, so their local-Q slices stack into one [S, h_l] query set
     per u, batched over u (rows are independent, so this equals one launch
     per rank);
  5. the reverse exchange ctx_pack_out (fused into the attention epilogue
     by default: ctx_attn_lq_gkv_pack_out writes the send buffers) ->
     ctx_sim_all_to_all ->
     ctx_unpack_out_ex for every rank (at U = 1 the output rows already are the
     sequence-sharded result and step 5 is the identity).

The per-rank layout launches of a step (every rank's pack, every rank's
unpack) are issued on parallel streams, forked from and joined back into the
caller's stream: on a real deployment every rank runs its own on its own GPU
at the same time, and on one GPU the concurrent launches share the SMs
instead of queueing one behind the other.

Joint (text) keys and values are inputs every rank already holds; they are
written once, head-sliced, after the S image rows of each gathered K/V buffer
(or before them, for a workload with the joint segment in front: the
"re-attach" of the same page), and the merged key mask [B, S + joint] is
built once per head group.
"""
from __future__ import annotations

import numpy as np
import torch

from . import (CTX_LAYOUT_TQKV, attn_workspace, ctx_attn_lq_gkv, ctx_attn_lq_gkv_pack_out,
               ctx_merge_joint_attn_mask, ctx_pack_out, ctx_pack_qkv_ex, ctx_sim_all_to_all, ctx_unpack_out_ex,
               ctx_unpack_qkv_ex)


class SimLayer:
    def __init__(self, wl, device="cuda", dtype=torch.bfloat16, attention: bool | None = None,
                 balanced: bool = True, layout: int = CTX_LAYOUT_TQKV, fuse_reverse: bool = True,
                 pack_view: bool = True):
        self.wl = wl
        self.dev = torch.device(device)
        self.dtype = dtype
        self.layout = layout
        # U > 1: the attention epilogue writes the reverse exchange's send buffers directly
        self.fuse_reverse = fuse_reverse and wl.U > 1
        # U = 1 (AllGather-KV alone): a rank's [1, 3, B, S_l, H, D] staging buffer is
        # its [3, B, S_l, H, D] input bit for bit, so the unpack (the AllGather
        # placement) reads the input and no pack or all-to-all runs
        self.pack_view = pack_view and wl.U == 1 and layout == CTX_LAYOUT_TQKV
        U, A, B, S, H, D, J = wl.U, wl.A, wl.B, wl.S, wl.H, wl.D, wl.joint
        if S % (U * A):
            raise ValueError("S must divide by U*A")
        # heads that do not divide by U are zero-padded to U * ceil(H/U)
        self.R, self.S_l, self.h_l, self.Sk = U * A, S // (U * A), -(-H // U), S + J
        self.H_pad = U * self.h_l
        self.attention = wl.attention if attention is None else attention
        R, S_l, h_l, Sk = self.R, self.S_l, self.h_l, self.Sk
        kw = dict(dtype=dtype, device=self.dev)
        self.x = torch.empty((R, 3, B, S_l, H, D), **kw)           # per-rank inputs
        chunk = 3 * B * S_l * h_l * D
        if not self.pack_view:
            self.send = torch.empty((A, U, U, chunk), **kw)         # [group a, src u, dst chunk]
            self.recv = torch.empty_like(self.send) if U > 1 else self.send
        self.qg = torch.empty((U, B, S, h_l, D), **kw)              # local-Q of all ranks
        self.kg = torch.empty((U, B, Sk, h_l, D), **kw)             # gathered K (+ joint)
        self.vg = torch.empty((U, B, Sk, h_l, D), **kw)
        # gathered rows: image keys from img0, joint keys from j0 (joint segment in front or after)
        self.img0, self.j0 = (J, 0) if wl.joint_front else (0, S)
        u8 = dict(dtype=torch.uint8, device=self.dev)
        # raw masks as the model hands them over, and the merged key mask of every head group
        self.img_mask = torch.ones((B, S), **u8) if wl.image_pad_range is not None else None
        self.jnt_mask = torch.ones((B, J), **u8) if (J and wl.text_len_range is not None) else None
        has_mask = self.img_mask is not None or self.jnt_mask is not None
        self.mask = torch.empty((U * B, Sk), **u8) if has_mask else None
        self.out = torch.empty((U, B, S, h_l, D), **kw)
        self.lse = torch.empty((U * B, h_l, S), dtype=torch.float32, device=self.dev)
        # workspace of the balanced (persistent, key-split) attention schedule
        self.ws = attn_workspace(U * B, S, Sk, h_l, D, device=self.dev) if (balanced and self.attention) else None
        if U > 1:
            ochunk = B * S_l * h_l * D
            self.osend = torch.empty((A, U, U, ochunk), **kw)
            self.orecv = torch.empty_like(self.osend)
            self.y = torch.empty((R, B, S_l, H, D), **kw)
        # one stream per simulated rank (at most 8), for the per-rank layout launches
        self.lanes = [torch.cuda.Stream(self.dev) for _ in range(min(R, 8))]

    def _per_rank(self, stream, launch):
        """Runs launch(g, s) for every rank g on the rank streams, forked from
        and joined back into `stream` (default: the current stream)."""
        base = stream if stream is not None else torch.cuda.current_stream(self.dev)
        fork = torch.cuda.Event()
        fork.record(base)
        for lane in self.lanes:
            lane.wait_event(fork)
        for g in range(self.R):
            launch(g, self.lanes[g % len(self.lanes)])
        for lane in self.lanes:
            done = torch.cuda.Event()
            done.record(lane)
            base.wait_event(done)

    # ---------------------------------------------------------- inputs
    def load(self, inp, pinned: bool = False):
        """Copy per-rank shards, joint K/V and the key mask to the device."""
        wl, U = self.wl, self.wl.U
        for g in range(self.R):
            for t, src in enumerate((inp.q, inp.k, inp.v)):
                self.x[g, t].copy_(inp.shard(src, g))
        if wl.joint:
            J, h_l, H = wl.joint, self.h_l, wl.H
            j0, j1 = self.j0, self.j0 + J
            for u in range(U):
                lo, hi = u * h_l, min((u + 1) * h_l, H)
                self.kg[u, :, j0:j1].zero_()
                self.vg[u, :, j0:j1].zero_()
                if hi > lo:
                    self.kg[u, :, j0:j1, :hi - lo].copy_(inp.jk[:, :, lo:hi])
                    self.vg[u, :, j0:j1, :hi - lo].copy_(inp.jv[:, :, lo:hi])
        if self.img_mask is not None:
            self.img_mask.copy_(torch.from_numpy(np.ascontiguousarray(inp.image_mask)))
        if self.jnt_mask is not None:
            self.jnt_mask.copy_(torch.from_numpy(np.ascontiguousarray(inp.joint_mask)))
        torch.cuda.synchronize(self.dev)

    # ---------------------------------------------------------- one step
    def exchange_in(self, stream=None):
        """Steps 1-3: pack, all-to-all, unpack into the gathered buffers, and
        the key mask of the gathered layout."""
        wl = self.wl
        U, A, B, S = wl.U, wl.A, wl.B, wl.S
        if not self.pack_view:
            self.pack_ranks(stream)
        if U > 1:
            ctx_sim_all_to_all(self.send, self.recv, A, U, stream=stream)
        self.unpack_ranks(stream)
        if self.mask is not None:
            for u in range(U):
                ctx_merge_joint_attn_mask(self.img_mask, self.jnt_mask, B, S, wl.joint, self.mask[u * B:(u + 1) * B],
                                          joint_front=wl.joint_front, stream=stream)

    def pack_ranks(self, stream=None):
        """Step 1 alone: every rank's pack into its staging buffer."""
        U = self.wl.U

        def pack(g, s):
            a, u = divmod(g, U)
            x = self.x[g]
            ctx_pack_qkv_ex(x[0], x[1], x[2], self.send[a, u], U, self.layout, stream=s)

        self._per_rank(stream, pack)

    def unpack_ranks(self, stream=None):
        """Step 3 alone: every rank's unpack into the gathered buffers."""
        wl = self.wl
        U, B, S, D = wl.U, wl.B, wl.S, wl.D
        S_l, h_l, Sk = self.S_l, self.h_l, self.Sk

        def unpack(g, s):
            a, u = divmod(g, U)
            rq = a * U * S_l            # local-Q rows of rank (a, u) among all ranks' queries
            rk = self.img0 + rq         # its image rows in the gathered K/V (after joint keys in front)
            src = self.x[g] if self.pack_view else self.recv[a, u]
            ctx_unpack_qkv_ex(src, self.qg[u, :, rq:], self.kg[u, :, rk:], self.vg[u, :, rk:], U, B,
                              S_l, h_l, D, self.layout, q_batch_stride_rows=S, kv_batch_stride_rows=Sk, stream=s)

        self._per_rank(stream, unpack)

    def attend(self, stream=None):
        """Step 4: local-Q / global-KV attention of every rank."""
        if not self.attention:
            return
        wl = self.wl
        U, B, S, D = wl.U, wl.B, wl.S, wl.D
        h_l, Sk = self.h_l, self.Sk
        args = (self.qg.view(U * B, S, h_l, D), self.kg.view(U * B, Sk, h_l, D), self.vg.view(U * B, Sk, h_l, D))
        if self.fuse_reverse:
            ctx_attn_lq_gkv_pack_out(*args, self.osend, U, B, self.S_l, lse=self.lse, key_mask=self.mask,
                                     workspace=self.ws, stream=stream)
        else:
            ctx_attn_lq_gkv(*args, self.out.view(U * B, S, h_l, D), self.lse, key_mask=self.mask,
                            workspace=self.ws, stream=stream)

    def exchange_out(self, stream=None):
        """Step 5: the reverse exchange (identity at U = 1)."""
        wl = self.wl
        U, A, B, S, D = wl.U, wl.A, wl.B, wl.S, wl.D
        S_l, h_l = self.S_l, self.h_l
        if not self.attention or U == 1:
            return
        def pack_out(g, s):
            a, u = divmod(g, U)
            ctx_pack_out(self.out[u, :, a * U * S_l:], self.osend[a, u].view(U, B, S_l, h_l, D), U,
                         o_batch_stride_rows=S, stream=s)

        def unpack_out(g, s):
            a, u = divmod(g, U)
            ctx_unpack_out_ex(self.orecv[a, u].view(U, B, S_l, h_l, D), self.y[g], U, stream=s)

        if not self.fuse_reverse:
            self._per_rank(stream, pack_out)
        ctx_sim_all_to_all(self.osend, self.orecv, A, U, stream=stream)
        self._per_rank(stream, unpack_out)

    PHASES = ("exchange_in", "attend", "exchange_out")

    def step(self, stream=None):
        for name in self.PHASES:
            getattr(self, name)(stream=stream)

    # ---------------------------------------------------------- CUDA graphs
    def capture(self):
        """Captures each phase of the step as a CUDA graph (same kernels, same
        buffers: replay removes the host launch cost and the gaps between the
        back-to-back layout launches). Run one eager step first so that the
        library's per-device set-up happens outside the capture."""
        self.step()
        torch.cuda.synchronize(self.dev)
        self.graphs = {}
        for name in self.PHASES:
            if name == "exchange_out" and (not self.attention or self.wl.U == 1):
                continue  # the identity: nothing to launch
            if name == "attend" and not self.attention:
                continue
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                getattr(self, name)()
            self.graphs[name] = g
        torch.cuda.synchronize(self.dev)

    def replay(self, phase=None):
        for name in (self.PHASES if phase is None else (phase,)):
            g = self.graphs.get(name)
            if g is not None:
                g.replay()

    def launches_per_step(self) -> int:
        U, R = self.wl.U, self.R
        n = (R if self.pack_view else 2 * R) + (1 if U > 1 else 0) + (U if self.mask is not None else 0)
        if self.attention:
            n += 1
            if U > 1:
                n += (R + 1) if self.fuse_reverse else (2 * R + 1)
        return n

    # ---------------------------------------------------------- results
    def rank_output(self, g: int) -> torch.Tensor:
        """Rank g's sequence-sharded attention output [B, S_l, H, D]."""
        if self.wl.U > 1:
            return self.y[g]
        return self.out[0, :, g * self.S_l:(g + 1) * self.S_l, :self.wl.H]

    def rank_q(self, g: int) -> torch.Tensor:
        a, u = divmod(g, self.wl.U)
        rows = self.wl.S // self.wl.A
        return self.qg[u, :, a * rows:(a + 1) * rows]

    # ---------------------------------------------------------- work model
    def pack_bytes(self) -> int:
        """Algorithmic HBM bytes of all packs of one step: the real heads read,
        the padded heads written."""
        wl = self.wl
        if self.pack_view:
            return 0
        return 3 * self.R * wl.B * self.S_l * (wl.H + self.H_pad) * wl.D * 2

    def unpack_bytes(self) -> int:
        wl = self.wl
        return 2 * 3 * self.R * wl.B * self.S_l * self.H_pad * wl.D * 2

    def a2a_bytes(self) -> int:
        return self.unpack_bytes() if self.wl.U > 1 else 0

    def reverse_bytes(self) -> int:
        wl = self.wl
        if not self.attention or wl.U == 1:
            return 0
        one = self.R * wl.B * self.S_l * self.H_pad * wl.D * 2
        # pack_out (unless fused into the attention epilogue) and the all-to-all read + write
        # padded rows; unpack_out reads padded, writes real heads
        pack_out = 0 if self.fuse_reverse else 2 * one
        return pack_out + 2 * one + one + self.R * wl.B * self.S_l * wl.H * wl.D * 2

    def attn_flops(self, valid_keys=None, dense: bool = False) -> float:
        """4 * Sq * K_valid * D per head (QK^T and PV), summed over all ranks.
        valid_keys: per batch row, the keys the mask leaves valid (None or
        dense: every gathered key)."""
        wl = self.wl
        if not self.attention:
            return 0.0
        per_b = []
        for b in range(wl.B):
            kv = self.Sk
            if not dense and valid_keys is not None:
                kv = int(valid_keys[b])
            per_b.append(kv)
        # useful work: the real heads (padded heads are overhead, not counted)
        return float(sum(4.0 * wl.H * wl.S * kv * wl.D for kv in per_b))
