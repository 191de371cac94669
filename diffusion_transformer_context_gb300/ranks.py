"""One rank per process: the composed Ulysses x AllGather-KV layer with real
collectives between the library's calls.

vllm-omni PR #7641 ("Compose Ulysses with AllGather-KV as a 2D diffusion
SP") fixes the order and the rank layout: global rank g = a*U + u holds input
rows [g*S_l, (g+1)*S_l); Ulysses groups are the contiguous blocks
{a*U, ..., a*U + U-1}, AllGather-KV groups stride by U {u, U+u, ...}. One
step of rank (a, u):

  1. pack its Q/K/V [B, S_l, H, D] destination-major        (ctx_pack_qkv_ex)
  2. all_to_all_single inside its Ulysses group             (torch.distributed)
  3. unpack to [B, S/A, h_l, D] x3                          (ctx_unpack_qkv_ex)
  4. all_gather of K and V inside its AllGather-KV group into the gathered
     [B, S + joint, h_l, D] buffers; joint (text) keys re-attached before or
     after the image rows; the key mask of that layout      (ctx_merge_joint_attn_mask)
  5. local-Q / global-KV attention, the output written straight in the
     reverse exchange's send layout                         (ctx_attn_lq_gkv_pack_out)
  6. all_to_all_single inside the Ulysses group, then the reverse unpack to
     [B, S_l, H, D]                                         (ctx_unpack_out_ex)

Every data step runs in the library's kernels; torch.distributed moves the
bytes between ranks (NCCL on GPUs). The gathered rows of the A group are one
contiguous range only for B = 1, which every configuration of this method
uses; other batch sizes are refused.

The compute steps go through an `ops` object (LibraryOps by default), so
that the rank and group wiring can be exercised with other implementations of
the same steps (the tests run it on CPU ranks over gloo).
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import (CTX_LAYOUT_TQKV, attn_workspace, ctx_attn_lq_gkv, ctx_attn_lq_gkv_pack_out, ctx_merge_joint_attn_mask,
               ctx_pack_qkv_ex, ctx_unpack_out_ex, ctx_unpack_qkv_ex)


def rank_coords(g: int, U: int):
    """(a, u) of global rank g = a*U + u."""
    return divmod(g, U)


class Groups:
    """The two process groups of the calling rank. Every rank must build this
    at the same time (creating a group is a collective of the whole job)."""

    def __init__(self, U: int, A: int):
        world, g = dist.get_world_size(), dist.get_rank()
        if world != U * A:
            raise ValueError(f"world size {world} != U*A = {U * A}")
        self.U, self.A, self.g = U, A, g
        self.a, self.u = rank_coords(g, U)
        self.ulysses_ranks = [self.a * U + u for u in range(U)]
        self.agkv_ranks = [a * U + self.u for a in range(A)]
        self.ulysses = self.agkv = None
        for a in range(A):
            grp = dist.new_group([a * U + u for u in range(U)])
            if a == self.a:
                self.ulysses = grp
        for u in range(U):
            grp = dist.new_group([a * U + u for a in range(A)])
            if u == self.u:
                self.agkv = grp


class LibraryOps:
    """The layer's compute steps as calls of the C library (device tensors)."""

    def __init__(self, balanced: bool = True):
        self.balanced = balanced

    def pack(self, x, staging, U, layout=CTX_LAYOUT_TQKV):
        ctx_pack_qkv_ex(x[0], x[1], x[2], staging, U, layout)

    def unpack(self, src, q, k, v, U, B, S_l, h_l, D, layout=CTX_LAYOUT_TQKV):
        ctx_unpack_qkv_ex(src, q, k, v, U, B, S_l, h_l, D, layout)

    def merge_mask(self, image_mask, joint_mask, B, S, J, front, out):
        ctx_merge_joint_attn_mask(image_mask, joint_mask, B, S, J, out, joint_front=front)

    def workspace(self, B, Sq, Sk, H, D, device):
        return attn_workspace(B, Sq, Sk, H, D, device=device) if self.balanced else None

    def attention(self, q, k, v, out, lse, mask, workspace):
        ctx_attn_lq_gkv(q, k, v, out, lse, key_mask=mask, workspace=workspace)

    def attention_pack_out(self, q, k, v, send, U, S_l, lse, mask, workspace):
        ctx_attn_lq_gkv_pack_out(q, k, v, send, U, q.shape[0], S_l, lse=lse, key_mask=mask, workspace=workspace)

    def unpack_out(self, recv, y, U):
        ctx_unpack_out_ex(recv, y, U)


class RankLayer:
    """The layer as one rank of a U x A job runs it (see the module text).
    `layout` is the staging layout of the Ulysses exchange: [U,3,B,S_l,h_l,D]
    or the interleaved [U,B,S_l,h_l,3D]; either way chunk r of the flat
    buffer is what rank r of the group receives."""

    def __init__(self, wl, groups: Groups, device, ops=None, dtype=torch.bfloat16, layout=CTX_LAYOUT_TQKV):
        U, A, B, S, H, D, J = wl.U, wl.A, wl.B, wl.S, wl.H, wl.D, wl.joint
        if (groups.U, groups.A) != (U, A):
            raise ValueError("groups built for another U x A")
        if B != 1:
            raise ValueError("one rank per process needs B = 1 (the gathered rows of an A group are contiguous)")
        if S % (U * A):
            raise ValueError("S must divide by U*A")
        self.wl, self.G, self.dev, self.layout = wl, groups, torch.device(device), layout
        self.ops = ops if ops is not None else LibraryOps()
        self.S_l, self.h_l = S // (U * A), -(-H // U)
        self.rows = U * self.S_l                          # local query rows: S / A
        self.Sk = S + J
        self.img0, self.j0 = (J, 0) if wl.joint_front else (0, S)
        kw = dict(dtype=dtype, device=self.dev)
        S_l, h_l, Sk = self.S_l, self.h_l, self.Sk
        self.x = torch.zeros((3, B, S_l, H, D), **kw)     # this rank's input rows
        self.staging = torch.empty((U, 3, B, S_l, h_l, D) if layout == CTX_LAYOUT_TQKV else (U, B, S_l, h_l, 3 * D),
                                   **kw)
        self.recv = torch.empty_like(self.staging) if U > 1 else None
        self.q = torch.empty((B, self.rows, h_l, D), **kw)
        self.k_loc = torch.empty((B, self.rows, h_l, D), **kw)
        self.v_loc = torch.empty_like(self.k_loc)
        self.kg = torch.zeros((B, Sk, h_l, D), **kw)      # gathered K (+ joint rows)
        self.vg = torch.zeros((B, Sk, h_l, D), **kw)
        u8 = dict(dtype=torch.uint8, device=self.dev)
        self.img_mask = torch.ones((B, S), **u8) if wl.image_pad_range is not None else None
        self.jnt_mask = torch.ones((B, J), **u8) if (J and wl.text_len_range is not None) else None
        self.mask = torch.empty((B, Sk), **u8) if (self.img_mask is not None or self.jnt_mask is not None) else None
        self.lse = torch.empty((B, h_l, self.rows), dtype=torch.float32, device=self.dev)
        self.send = torch.empty((U, B, S_l, h_l, D), **kw)
        self.orecv = torch.empty_like(self.send) if U > 1 else None
        self.y = torch.empty((B, S_l, H, D), **kw)
        self.ws = self.ops.workspace(B, self.rows, Sk, h_l, D, self.dev)

    def load(self, q, k, v, jk=None, jv=None, image_mask=None, joint_mask=None):
        """This rank's input rows [B, S_l, H, D] x3; the joint K/V [B, J, H, D]
        and the raw masks, which every rank holds whole."""
        for t, src in enumerate((q, k, v)):
            self.x[t].copy_(src)
        u, h_l, H, J = self.G.u, self.h_l, self.wl.H, self.wl.joint
        if J:
            lo, hi = u * h_l, min((u + 1) * h_l, H)
            for buf, src in ((self.kg, jk), (self.vg, jv)):
                buf[:, self.j0:self.j0 + J].zero_()
                if hi > lo:
                    buf[:, self.j0:self.j0 + J, :hi - lo].copy_(src[:, :, lo:hi])
        if self.img_mask is not None:
            self.img_mask.copy_(torch.as_tensor(image_mask))
        if self.jnt_mask is not None:
            self.jnt_mask.copy_(torch.as_tensor(joint_mask))

    def step(self):
        wl, ops, G = self.wl, self.ops, self.G
        U, B, S, D = wl.U, wl.B, wl.S, wl.D
        S_l, h_l = self.S_l, self.h_l
        # 1-3: Ulysses exchange inside the U group (at U = 1 the [U,3,B,S_l,h_l,D]
        # staging buffer is the input bit for bit, so nothing is packed)
        if U > 1 or self.layout != CTX_LAYOUT_TQKV:
            ops.pack(self.x, self.staging, U, self.layout)
            src = self.staging
            if U > 1:
                dist.all_to_all_single(self.recv.view(-1), self.staging.view(-1), group=G.ulysses)
                src = self.recv
        else:
            src = self.x.view(1, 3, B, S_l, h_l, D)
        ops.unpack(src, self.q, self.k_loc, self.v_loc, U, B, S_l, h_l, D, self.layout)
        # 4: K/V AllGather inside the A group, straight into the gathered image rows
        img = slice(self.img0, self.img0 + S)  # one contiguous range at B = 1: gather flat
        dist.all_gather_into_tensor(self.kg[:, img].view(-1), self.k_loc.view(-1), group=G.agkv)
        dist.all_gather_into_tensor(self.vg[:, img].view(-1), self.v_loc.view(-1), group=G.agkv)
        if self.mask is not None:
            ops.merge_mask(self.img_mask, self.jnt_mask, B, S, wl.joint, wl.joint_front, self.mask)
        # 5-6: attention into the reverse exchange's send layout, exchange, unpack
        if U > 1:
            ops.attention_pack_out(self.q, self.kg, self.vg, self.send, U, S_l, self.lse, self.mask, self.ws)
            dist.all_to_all_single(self.orecv.view(-1), self.send.view(-1), group=G.ulysses)
            ops.unpack_out(self.orecv, self.y, U)
        else:
            ops.attention(self.q, self.kg, self.vg, self.y.view(B, S_l, h_l, D), self.lse, self.mask, self.ws)
        return self.y

    def attn_flops(self, valid_keys=None) -> float:
        """4 * rows * K_valid * D per real head of this rank."""
        wl = self.wl
        kv = self.Sk if valid_keys is None else int(valid_keys[0])
        heads = min(self.h_l, max(0, wl.H - self.G.u * self.h_l))
        return 4.0 * heads * self.rows * kv * wl.D
