"""Seeded synthetic inputs shared by the CUDA path's tests/bench and the oracle.

This module holds shapes and random draws only: no step of the method (no
pack, exchange, gather or attention arithmetic) lives here, so that both the
oracle and the CUDA path can take their inputs from it without sharing any of
the computation they are compared on.

Recipe (the same for every workload):
  * a ``torch.Generator`` seeded with 1234 (the seed of the single-card
    multi-rank test on the sglang PR #33667 page, "test_usp_packed_qkv_a2a");
  * ``randn`` in fp32, then a round-to-nearest-even cast to bf16 (or fp16);
  * Q, K, V are independent draws from the same generator, in that order,
    followed by the joint (text) K/V, the per-batch text lengths and, where a
    workload pads its image sequence, the per-batch image padding lengths;
  * masks are produced raw, one per side, as the model would hand them over:
    the joint (text) mask [B, joint] marks the first L_t text tokens valid,
    the image mask [B, S] marks a padded suffix of the global image sequence
    invalid; merging them into the gathered key layout is a step of the
    method (the oracle and the CUDA library each do it themselves);
  * the GLOBAL sequence ``[B, S, H, D]`` is generated once and split into the
    per-rank input shards, rank ``g = a*U + u`` holding rows
    ``[g*S_l, (g+1)*S_l)`` (vllm-omni PR #7641, "Compose Ulysses with
    AllGather-KV": Ulysses groups are contiguous blocks of U ranks, the flat
    contiguous sequence sharding gives each group one contiguous region).

The pages measure on real Wan 2.x / Qwen-Image latents; N(0,1) tensors of the
same shapes stand in for them (no dataset or weights are used).
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np
import torch

SEED = 1234


@dataclasses.dataclass(frozen=True)
class Workload:
    """One simulated context-parallel attention layer.

    name   : workload name
    B      : batch
    S      : global image/video sequence length (rows of the gathered K/V
             before joint tokens are attached)
    H      : global head count
    D      : head dim
    U      : Ulysses degree (head reshard group size)
    A      : AllGather-KV degree
    joint  : joint (text) tokens re-attached to the gathered K/V, 0 = none
    text_len_range : inclusive range of valid text lengths (joint padding
             mask), None = no joint mask
    attention : whether the workload runs the attention step
    joint_front : joint keys placed before the image keys (default after)
    image_pad_range : inclusive range of padded image tokens at the end of
             the global sequence (2-D image mask), None = no image mask
    """

    name: str
    B: int
    S: int
    H: int
    D: int
    U: int
    A: int
    joint: int = 0
    text_len_range: Optional[tuple] = None
    attention: bool = True
    joint_front: bool = False
    image_pad_range: Optional[tuple] = None

    @property
    def ranks(self) -> int:
        return self.U * self.A

    @property
    def S_l(self) -> int:  # per-rank input rows
        return self.S // (self.U * self.A)

    @property
    def h_l(self) -> int:  # per-rank heads after the Ulysses reshard
        return self.H // self.U

    @property
    def Sq_local(self) -> int:  # local-Q rows of one rank
        return self.S // self.A

    @property
    def Sk(self) -> int:  # gathered keys incl. joint tokens
        return self.S + self.joint


WORKLOADS = {
    # tiny: B=1, S=512, H=2, D=128, U=2 (per-rank [1,256,2,128]), full attention
    "tiny": Workload("tiny", B=1, S=512, H=2, D=128, U=2, A=1),
    # pack/unpack only: U=4, per-rank [1,1024,24,128] -> staging [4,3,1,1024,6,128]
    "pack": Workload("pack", B=1, S=4096, H=24, D=128, U=4, A=1, attention=False),
    # Qwen-Image-like 1024x1024, U=2 x A=2: local-Q [1,2048,12,128] vs
    # K/V [1,4096+256,12,128], text length uniform in [32,256]
    "qwen": Workload("qwen", B=1, S=4096, H=24, D=128, U=2, A=2, joint=256,
                     text_len_range=(32, 256)),
    # Wan-like 480p 81 frames, AllGather-KV CP8 (U=1): local-Q [1,4095,12,128]
    # vs global K/V [1,32760,12,128]
    "wan480": Workload("wan480", B=1, S=32760, H=12, D=128, U=1, A=8),
    # Wan-14B-like 720p, U=4 x A=2: per-rank [1,9450,40,128] -> [1,37800,10,128],
    # local-Q [1,37800,10,128] vs K/V [1,75600,10,128]
    "wan14b": Workload("wan14b", B=1, S=75600, H=40, D=128, U=4, A=2),
    # the vllm-omni PR #7641 topology comparison on 4 GPUs: 14 heads, D=128,
    # sequence 65536; Ulysses-4 pads 14 -> 16 heads ("advanced_uaa"),
    # Ulysses-2 x AllGather-2 divides evenly
    "uaa14_usp4": Workload("uaa14_usp4", B=1, S=65536, H=14, D=128, U=4, A=1),
    "uaa14_cp2usp2": Workload("uaa14_cp2usp2", B=1, S=65536, H=14, D=128, U=2, A=2),
    # the same comparison at the page's other sequence lengths (16384, 32768)
    "uaa14_usp4_s16k": Workload("uaa14_usp4_s16k", B=1, S=16384, H=14, D=128, U=4, A=1),
    "uaa14_cp2usp2_s16k": Workload("uaa14_cp2usp2_s16k", B=1, S=16384, H=14, D=128, U=2, A=2),
    "uaa14_usp4_s32k": Workload("uaa14_usp4_s32k", B=1, S=32768, H=14, D=128, U=4, A=1),
    "uaa14_cp2usp2_s32k": Workload("uaa14_cp2usp2_s32k", B=1, S=32768, H=14, D=128, U=2, A=2),
}


def custom(name: str, B: int, S: int, H: int, D: int, U: int, A: int = 1,
           joint: int = 0, text_len_range=None, attention: bool = True, joint_front: bool = False,
           image_pad_range=None) -> Workload:
    """A workload with explicit sizes (used for ragged / edge-case tests)."""
    return Workload(name, B, S, H, D, U, A, joint, text_len_range, attention, joint_front, image_pad_range)


def randn(shape, gen: torch.Generator, dtype: str = "bf16") -> torch.Tensor:
    """fp32 N(0,1) draw cast round-to-nearest-even to bf16/fp16 (CPU tensor)."""
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    return x.to(torch.bfloat16 if dtype == "bf16" else torch.float16)


@dataclasses.dataclass
class Inputs:
    wl: Workload
    q: torch.Tensor            # [B, S, H, D] global queries
    k: torch.Tensor            # [B, S, H, D]
    v: torch.Tensor            # [B, S, H, D]
    jk: Optional[torch.Tensor]  # [B, joint, H, D] joint (text) keys or None
    jv: Optional[torch.Tensor]  # [B, joint, H, D]
    text_len: Optional[np.ndarray]  # [B] valid text lengths (int64) or None
    dtype: str = "bf16"
    image_mask: Optional[np.ndarray] = None  # [B, S] uint8, 1 = valid image key, or None
    joint_mask: Optional[np.ndarray] = None  # [B, joint] uint8, 1 = valid text key, or None

    def shard(self, t: torch.Tensor, g: int) -> torch.Tensor:
        """Rank g's input rows [g*S_l, (g+1)*S_l) (contiguous copy)."""
        S_l = self.wl.S_l
        return t[:, g * S_l:(g + 1) * S_l].contiguous()


def make_inputs(wl: Workload, seed: int = SEED, dtype: str = "bf16") -> Inputs:
    gen = torch.Generator().manual_seed(seed)
    shape = (wl.B, wl.S, wl.H, wl.D)
    q = randn(shape, gen, dtype)
    k = randn(shape, gen, dtype)
    v = randn(shape, gen, dtype)
    jk = jv = None
    text_len = None
    joint_mask = image_mask = None
    if wl.joint:
        jshape = (wl.B, wl.joint, wl.H, wl.D)
        jk = randn(jshape, gen, dtype)
        jv = randn(jshape, gen, dtype)
        if wl.text_len_range is not None:
            lo, hi = wl.text_len_range
            text_len = torch.randint(lo, hi + 1, (wl.B,), generator=gen).numpy().astype(np.int64)
            joint_mask = np.zeros((wl.B, wl.joint), dtype=np.uint8)
            for b in range(wl.B):
                joint_mask[b, :int(text_len[b])] = 1
    if wl.image_pad_range is not None:
        lo, hi = wl.image_pad_range
        pad = torch.randint(lo, hi + 1, (wl.B,), generator=gen).numpy()
        image_mask = np.ones((wl.B, wl.S), dtype=np.uint8)
        for b in range(wl.B):
            image_mask[b, wl.S - int(pad[b]):] = 0
    return Inputs(wl, q, k, v, jk, jv, text_len, dtype, image_mask, joint_mask)


def as_u16(t: torch.Tensor) -> np.ndarray:
    """Bit pattern of a bf16/fp16 CPU tensor as a numpy uint16 array (no copy)."""
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def sample_rows(n_total: int, n_sample: int, tile: int = 128, seed: int = SEED) -> np.ndarray:
    """A fixed, seeded sample of query-row indices that always includes the
    first and last tile and the ragged tail rows (sorted, unique)."""
    rng = np.random.default_rng(seed)
    must = set(range(min(tile, n_total)))
    tail_start = (n_total // tile) * tile
    if tail_start == n_total:
        tail_start = max(0, n_total - tile)
    must.update(range(tail_start, n_total))
    rest = max(0, n_sample - len(must))
    if rest:
        must.update(rng.choice(n_total, size=min(rest, n_total), replace=False).tolist())
    return np.array(sorted(must), dtype=np.int64)
