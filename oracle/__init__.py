"""CPU oracle for the context-parallel attention hot path.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, by ``__graft_entry__.smoke()``
and by ``bench.py``'s CPU-baseline / reference leg. The CUDA library and its
Python binding never import this package, and this package never imports
them; the two share only the seeded input generators in ``workloads``.

The arithmetic lives in ``ctx_oracle.c`` (explicit index loops, fp64 softmax,
OpenMP over query rows); this module marshals numpy arrays into it and adds
two things that are plain data movement written from the pages:

* ``all_to_all``: ``all_to_all_single`` chunk semantics as the sglang PR
  #33667 unit test ("_run_all_ranks" / "fake_a2a") states them: every sender's
  flat buffer is cut into U equal chunks, chunk j goes to rank j, and the
  receiver concatenates what it got in source-rank order.
* ``all_gather``: the K/V AllGather of the vllm-omni PR #7641 composed order
  (concatenation over the A group in rank order).

``py_*`` functions are pure-Python loop twins for tiny shapes.

Every function is pinned by a CPU test against the pages' own test
construction, closed forms, invariants, numpy slicing of the global tensors
or a library routine for the same quantity (none against a retyped copy of
itself):

  pack_qkv, unpack_qkv, all_to_all  tests/test_oracle_pack.py (the sglang test's
                       construction and shapes against its head-slice spec;
                       packed == three separate exchanges)
  pack_out, unpack_out tests/test_oracle_pack.py (round trips, head concat)
  all_gather, ulysses_agkv_forward  tests/test_oracle_pack.py (the composed
                       order rebuilds the sequence, the reverse order does not),
                       tests/test_oracle_composed.py (padded heads + joint keys,
                       both placements, interleaved layout, against numpy slicing)
  ulysses_reverse      tests/test_oracle_composed.py (A > 1 and uneven heads
                       against the input shards; a planted u-major reverse fails)
  pack_qkv_ex, unpack_qkv_ex, unpack_out_ex  tests/test_oracle_uaa.py
  merge_joint_attn_mask  tests/test_oracle_mask.py (the page's case list)
  attention_rows, attention, attention_probs, py_attention_row
                       tests/test_oracle_attention.py (closed forms, invariants,
                       scipy logsumexp / softmax)
  lse_merge            tests/test_oracle_merge.py (segments == full attention)
  varlen_remap, padding_remap, attention_varlen  tests/test_oracle_varlen.py
                       (the page's worked example; documents are independent)
  py_pack_qkv          tests/test_oracle_pack.py (equals pack_qkv)
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "ctx_oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle_ctx.so")
_lib = None
_lock = threading.Lock()

BF16, FP16 = 0, 1
_DTYPES = {"bf16": BF16, "fp16": FP16}


def build(force: bool = False) -> str:
    """Compile ctx_oracle.c with gcc + OpenMP into liboracle_ctx.so."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-fPIC", "-shared", "-fopenmp", "-std=c11",
           "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            build()
            lib = ctypes.CDLL(_LIB_PATH)
            ll, p = ctypes.c_longlong, ctypes.c_void_p
            lib.orc_pack_qkv.argtypes = [p, p, p, p, ll, ll, ll, ll, ll]
            lib.orc_unpack_qkv.argtypes = [p, p, p, p, ll, ll, ll, ll, ll]
            lib.orc_pack_out.argtypes = [p, p, ll, ll, ll, ll, ll]
            lib.orc_unpack_out.argtypes = [p, p, ll, ll, ll, ll, ll]
            lib.orc_attention_rows.argtypes = [p, p, p, p, ctypes.c_int, ctypes.c_double,
                                               ll, ll, ll, ll, ll, ll, p, p, p]
            lib.orc_attention_probs.argtypes = [p, p, p, ctypes.c_int, ctypes.c_double,
                                                ll, ll, ll, ll, ll, ll, ll, ll, p]
            for f in (lib.orc_pack_qkv, lib.orc_unpack_qkv, lib.orc_pack_out,
                      lib.orc_unpack_out, lib.orc_attention_rows, lib.orc_attention_probs):
                f.restype = ctypes.c_int
            lib.orc_lse_merge.argtypes = [p, p, ctypes.c_int, ll, ll, ll, p, p]
            lib.orc_pack_qkv_ex.argtypes = [p, p, p, p, ll, ll, ll, ll, ll, ctypes.c_int]
            lib.orc_unpack_qkv_ex.argtypes = [p, p, p, p, ll, ll, ll, ll, ll, ctypes.c_int]
            lib.orc_unpack_out_ex.argtypes = [p, p, ll, ll, ll, ll, ll, ll]
            for f in (lib.orc_pack_qkv_ex, lib.orc_unpack_qkv_ex, lib.orc_unpack_out_ex):
                f.restype = ctypes.c_int
            lib.orc_lse_merge.restype = ctypes.c_int
            lib.orc_num_threads.restype = ctypes.c_int
            _lib = lib
    return _lib


def num_threads() -> int:
    return _load().orc_num_threads()


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle takes 16-bit float bit patterns as uint16 arrays")
    return a


# ---------------------------------------------------------------- exchanges

def pack_qkv(q, k, v, U: int) -> np.ndarray:
    """[B,S_l,H,D] x3 -> staging [U,3,B,S_l,H/U,D] (destination-major)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, S_l, H, D = q.shape
    if k.shape != q.shape or v.shape != q.shape or H % U:
        raise ValueError("pack_qkv: shape mismatch or H % U != 0")
    out = np.empty((U, 3, B, S_l, H // U, D), dtype=np.uint16)
    rc = _load().orc_pack_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S_l, H, D, U)
    assert rc == 0
    return out


def unpack_qkv(recv, U: int):
    """recv [U,3,B,S_l,h_l,D] -> (Q', K', V') each [B, U*S_l, h_l, D]."""
    recv = _u16(recv)
    U2, three, B, S_l, h_l, D = recv.shape
    assert U2 == U and three == 3
    outs = [np.empty((B, U * S_l, h_l, D), dtype=np.uint16) for _ in range(3)]
    rc = _load().orc_unpack_qkv(_ptr(recv), *(_ptr(o) for o in outs), B, S_l, h_l, D, U)
    assert rc == 0
    return tuple(outs)


def pack_out(o, U: int) -> np.ndarray:
    """O [B, U*S_l, h_l, D] -> send [U, B, S_l, h_l, D]."""
    o = _u16(o)
    B, rows, h_l, D = o.shape
    assert rows % U == 0
    S_l = rows // U
    out = np.empty((U, B, S_l, h_l, D), dtype=np.uint16)
    assert _load().orc_pack_out(_ptr(o), _ptr(out), B, S_l, h_l, D, U) == 0
    return out


def unpack_out(recv, U: int) -> np.ndarray:
    """recv [U, B, S_l, h_l, D] -> Y [B, S_l, U*h_l, D]."""
    recv = _u16(recv)
    U2, B, S_l, h_l, D = recv.shape
    assert U2 == U
    out = np.empty((B, S_l, U * h_l, D), dtype=np.uint16)
    assert _load().orc_unpack_out(_ptr(recv), _ptr(out), B, S_l, h_l, D, U) == 0
    return out


LAYOUT_TQKV, LAYOUT_INTERLEAVED = 0, 1


def pack_qkv_ex(q, k, v, U: int, layout: int = LAYOUT_TQKV) -> np.ndarray:
    """Pack with zero-padded heads (h_l = ceil(H/U)) and a choice of staging
    layout: 0 -> [U,3,B,S_l,h_l,D], 1 -> [U,B,S_l,h_l,3D]."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, S_l, H, D = q.shape
    h_l = -(-H // U)
    shape = (U, 3, B, S_l, h_l, D) if layout == LAYOUT_TQKV else (U, B, S_l, h_l, 3 * D)
    out = np.empty(shape, dtype=np.uint16)
    assert _load().orc_pack_qkv_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(out), B, S_l, H, D, U, layout) == 0
    return out


def unpack_qkv_ex(recv, U: int, layout: int = LAYOUT_TQKV):
    """Receive side for either layout -> (Q', K', V') each [B, U*S_l, h_l, D]."""
    recv = _u16(recv)
    if layout == LAYOUT_TQKV:
        U2, three, B, S_l, h_l, D = recv.shape
    else:
        U2, B, S_l, h_l, D3 = recv.shape
        D = D3 // 3
    assert U2 == U
    outs = [np.empty((B, U * S_l, h_l, D), dtype=np.uint16) for _ in range(3)]
    assert _load().orc_unpack_qkv_ex(_ptr(recv), *(_ptr(o) for o in outs), B, S_l, h_l, D, U, layout) == 0
    return tuple(outs)


def unpack_out_ex(recv, U: int, H: int) -> np.ndarray:
    """Reverse exchange receive side keeping the first H of the U*h_l heads."""
    recv = _u16(recv)
    U2, B, S_l, h_l, D = recv.shape
    out = np.empty((B, S_l, H, D), dtype=np.uint16)
    assert _load().orc_unpack_out_ex(_ptr(recv), _ptr(out), B, S_l, h_l, H, D, U) == 0
    return out


def all_to_all(sends):
    """all_to_all_single over one group: sends[r] is rank r's flat send
    buffer; returns recvs[j] = concat over r of chunk j of sends[r]."""
    U = len(sends)
    chunks = [np.split(np.ascontiguousarray(s).reshape(-1), U) for s in sends]
    return [np.concatenate([chunks[r][j] for r in range(U)]).reshape(sends[j].shape)
            for j in range(U)]


def all_gather(shards, axis: int = 1):
    """AllGather over one group: concatenation in rank order along ``axis``."""
    return np.concatenate([np.ascontiguousarray(s) for s in shards], axis=axis)


# ------------------------------------------------- joint-text key mask

class MaskMergeUnsupported(NotImplementedError):
    """A mask combination the merge refuses (fail closed): a 4-D image mask,
    alone (it belongs to a query-range slicing path outside this method's
    key-mask merge) or next to a 2-D joint mask."""


def merge_joint_attn_mask(image_mask, joint_mask, B: int, S_img: int, joint_len: int,
                          joint_front: bool = False):
    """The [B, K_final] key-validity mask of the gathered key layout
    (vllm-omni PR #7641, follow-up review commit that makes the joint-mask
    merge the single owner of 2-D key-mask handling after the K/V gather).

    image_mask : None or array; as a 2-D mask it must be [B, S_img] over the
                 gathered (global) image keys.
    joint_mask : None or array; must be 2-D [B, joint_len].
    joint_len  : joint keys re-attached after the gather, taken from the
                 joint KEY tensor (the joint query may be empty when cached
                 K/V is reused), 0 when there are none.
    joint_front: joint segment before the image keys (else after them).

    The steps, in the order the page gives them: ranks are checked joint
    side first (a joint mask that is not 2-D is invalid; a 4-D image mask is
    refused, with or without a joint mask); a joint mask needs joint K/V; each
    side's shape must equal (B, its segment length); a missing side is filled
    with True; the two segments are concatenated in placement order and
    normalised to 0/1. Returns None when neither side has a mask (every key
    valid), else uint8 [B, S_img + joint_len].
    Raises ValueError for invalid inputs, MaskMergeUnsupported for refused
    ones.
    """
    if image_mask is None and joint_mask is None:
        return None
    im = None if image_mask is None else np.asarray(image_mask)
    jm = None if joint_mask is None else np.asarray(joint_mask)
    if jm is not None and jm.ndim != 2:
        raise ValueError("joint mask must be 2-D [B, joint_len]")
    if im is not None and im.ndim == 4:
        raise MaskMergeUnsupported("4-D image mask: no key-mask merge (refused next to a joint mask)")
    if im is not None and im.ndim != 2:
        raise ValueError("image mask must be 2-D [B, S_img]")
    if jm is not None and joint_len == 0:
        raise ValueError("joint mask given without joint keys/values")
    if im is not None and tuple(im.shape) != (B, S_img):
        raise ValueError(f"image mask shape {im.shape} != {(B, S_img)}")
    if jm is not None and tuple(jm.shape) != (B, joint_len):
        raise ValueError(f"joint mask shape {jm.shape} != {(B, joint_len)}")
    K = S_img + joint_len
    out = np.zeros((B, K), dtype=np.uint8)
    for b in range(B):
        img_seg = [1 if im is None or im[b, i] else 0 for i in range(S_img)]
        jnt_seg = [1 if jm is None or jm[b, j] else 0 for j in range(joint_len)]
        row = jnt_seg + img_seg if joint_front else img_seg + jnt_seg
        for pos in range(K):
            out[b, pos] = row[pos]
    return out


# ---------------------------------------------------------------- attention

def default_scale(D: int) -> float:
    return 1.0 / math.sqrt(D)


def attention_rows(q, k, v, rows, mask=None, scale=None, dtype="bf16"):
    """fp64 attention for selected query rows.

    q [B,Sq,H,D], k/v [B,Sk,H,D] (uint16 bit patterns), mask None or
    [B,Sk] uint8 (nonzero = attend), rows an int64 array [n,3] of (b,h,i).
    Returns (O [n,D] float64, LSE [n] float64, natural log).
    """
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Sq, H, D = q.shape
    Bk, Sk, Hk, Dk = k.shape
    assert (Bk, Hk, Dk) == (B, H, D) and v.shape == k.shape
    if scale is None:
        scale = default_scale(D)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    n = rows.shape[0]
    m = None
    if mask is not None:
        m = np.ascontiguousarray(mask, dtype=np.uint8)
        assert m.shape == (B, Sk)
    out = np.empty((n, D), dtype=np.float64)
    lse = np.empty((n,), dtype=np.float64)
    rc = _load().orc_attention_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(m) if m is not None else None,
                                    _DTYPES[dtype], float(scale), B, Sq, Sk, H, D, n,
                                    _ptr(rows), _ptr(out), _ptr(lse))
    assert rc == 0, rc
    return out, lse


def all_rows(B: int, H: int, Sq: int) -> np.ndarray:
    """(b, h, i) triples for every query row, b-major then h then i."""
    b, h, i = np.meshgrid(np.arange(B), np.arange(H), np.arange(Sq), indexing="ij")
    return np.stack([b.ravel(), h.ravel(), i.ravel()], axis=1).astype(np.int64)


def attention(q, k, v, mask=None, scale=None, dtype="bf16"):
    """Full attention: O [B,Sq,H,D] float64, LSE [B,H,Sq] float64."""
    B, Sq, H, D = q.shape
    rows = all_rows(B, H, Sq)
    o, lse = attention_rows(q, k, v, rows, mask, scale, dtype)
    O = o.reshape(B, H, Sq, D).transpose(0, 2, 1, 3).copy()
    return O, lse.reshape(B, H, Sq)


def attention_probs(q, k, b, h, i, mask=None, scale=None, dtype="bf16") -> np.ndarray:
    """Softmax probabilities of query row (b, h, i) over all keys (fp64)."""
    q, k = _u16(q), _u16(k)
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    if scale is None:
        scale = default_scale(D)
    m = None if mask is None else np.ascontiguousarray(mask, dtype=np.uint8)
    p = np.empty((Sk,), dtype=np.float64)
    _load().orc_attention_probs(_ptr(q), _ptr(k), _ptr(m) if m is not None else None,
                                _DTYPES[dtype], float(scale), B, Sq, Sk, H, D, b, h, i, _ptr(p))
    return p


# ------------------------------------------------------ composed pipeline

def _pad_heads(x, H_pad):
    B, S, H, D = x.shape
    if H == H_pad:
        return x
    out = np.zeros((B, S, H_pad, D), np.uint16)
    out[:, :, :H] = x
    return out


def ulysses_agkv_forward(q_shards, k_shards, v_shards, U: int, A: int,
                         jk=None, jv=None, layout: int = LAYOUT_TQKV, joint_front: bool = False):
    """The composed U x A input side, all ranks (vllm-omni PR #7641 order):
    Ulysses all-to-all inside each U group (ranks a*U .. a*U+U-1), then the
    K/V AllGather inside each A group (ranks u, U+u, ...), then the joint
    (text) K/V re-attached after (or, joint_front, before) the gathered image
    keys. Heads that do not divide by U are zero-padded to U*ceil(H/U).

    Inputs are per-rank [B,S_l,H,D] uint16 shards indexed by g = a*U + u.
    Returns dict with, per rank g: 'q' [B,S/A,h_l,D] local-Q, and per head
    group u: 'k', 'v' [B,S(+joint),h_l,D] global K/V.
    """
    R = U * A
    assert len(q_shards) == R
    H = q_shards[0].shape[2]
    staging = [pack_qkv_ex(q_shards[g], k_shards[g], v_shards[g], U, layout) for g in range(R)]
    loc = [None] * R
    for a in range(A):
        grp = [a * U + u for u in range(U)]
        recvs = all_to_all([staging[g] for g in grp])
        for u, g in enumerate(grp):
            loc[g] = unpack_qkv_ex(recvs[u], U, layout)
    res = {"q": [loc[g][0] for g in range(R)], "k": [], "v": []}
    for u in range(U):
        grp = [a * U + u for a in range(A)]
        kg = all_gather([loc[g][1] for g in grp])
        vg = all_gather([loc[g][2] for g in grp])
        if jk is not None:
            h_l = kg.shape[2]
            jkp, jvp = _pad_heads(jk, U * h_l), _pad_heads(jv, U * h_l)
            jks = np.ascontiguousarray(jkp[:, :, u * h_l:(u + 1) * h_l])
            jvs = np.ascontiguousarray(jvp[:, :, u * h_l:(u + 1) * h_l])
            kg = np.concatenate([jks, kg] if joint_front else [kg, jks], axis=1)
            vg = np.concatenate([jvs, vg] if joint_front else [vg, jvs], axis=1)
        res["k"].append(kg)
        res["v"].append(vg)
    return res


def ulysses_reverse(o_ranks, U: int, A: int, H: int | None = None):
    """Reverse Ulysses exchange for all ranks: o_ranks[g] is rank g's output
    [B, S/A, h_l, D]; returns per-rank [B, S_l, H, D] sequence-sharded
    outputs (padded heads beyond H dropped)."""
    R = U * A
    sends = [pack_out(o_ranks[g], U) for g in range(R)]
    out = [None] * R
    for a in range(A):
        grp = [a * U + u for u in range(U)]
        recvs = all_to_all([sends[g] for g in grp])
        for u, g in enumerate(grp):
            out[g] = unpack_out(recvs[u], U) if H is None else unpack_out_ex(recvs[u], U, H)
    return out


def lse_merge(o_parts, lse_parts, dtype="bf16"):
    """Combine attention results over disjoint key segments.

    o_parts [P, B, Sq, H, D] uint16, lse_parts [P, B, H, Sq] float (natural
    log). Returns (O [B, Sq, H, D] float64, LSE [B, H, Sq] float64)."""
    o_parts = _u16(o_parts)
    P, B, Sq, H, D = o_parts.shape
    # row order (b, h, i) for both operands
    o_rows = np.ascontiguousarray(o_parts.transpose(0, 1, 3, 2, 4)).reshape(P, B * H * Sq, D)
    l_rows = np.ascontiguousarray(np.asarray(lse_parts, dtype=np.float64)).reshape(P, B * H * Sq)
    out = np.empty((B * H * Sq, D), dtype=np.float64)
    lse = np.empty((B * H * Sq,), dtype=np.float64)
    rc = _load().orc_lse_merge(_ptr(o_rows), _ptr(l_rows), _DTYPES[dtype], P, B * H * Sq, D, _ptr(out), _ptr(lse))
    assert rc == 0
    return out.reshape(B, H, Sq, D).transpose(0, 2, 1, 3).copy(), lse.reshape(B, H, Sq)


# ------------------------------------------------ packed varlen metadata

def varlen_remap(cu_global, span_begin: int, span_len: int):
    """Local query boundaries of one rank (vllm-omni PR #7641, packed query
    metadata under AllGather-KV): every global document [cu[d], cu[d+1]) is
    intersected with the rank's span [span_begin, span_begin + span_len); the
    rank keeps one (possibly empty) entry per document, prefix-summed from 0."""
    cu = [int(x) for x in cu_global]
    out = [0]
    lo, hi = span_begin, span_begin + span_len
    for d in range(len(cu) - 1):
        a, b = max(cu[d], lo), min(cu[d + 1], hi)
        out.append(out[-1] + max(0, b - a))
    return np.array(out, dtype=np.int32)


def padding_remap(real: int, pad: int, span_begin: int, span_len: int):
    """The single-document [real, pad] view of one rank: the query length
    narrows to the rank's valid prefix (the key length stays global)."""
    local_real = min(max(real - span_begin, 0), span_len)
    return np.array([local_real, span_len - local_real], dtype=np.int32)


def attention_varlen(q, k, v, cu_q, cu_k, mask=None, scale=None, dtype="bf16"):
    """Packed varlen attention: q [Sq,H,D], k/v [Sk,H,D]; query rows of
    document d (rows [cu_q[d], cu_q[d+1])) attend keys [cu_k[d], cu_k[d+1]).
    mask: None or [Sk] (nonzero = attend). Returns O [Sq,H,D] (rows outside
    every document stay NaN) and LSE [H,Sq]."""
    Sq, H, D = q.shape
    O = np.full((Sq, H, D), np.nan)
    L = np.full((H, Sq), np.nan)
    for d in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[d]), int(cu_q[d + 1]), int(cu_k[d]), int(cu_k[d + 1])
        if q1 <= q0:
            continue
        if k1 <= k0:
            O[q0:q1] = 0.0
            L[:, q0:q1] = -np.inf
            continue
        m = None if mask is None else np.ascontiguousarray(mask[k0:k1])[None]
        o, l = attention(np.ascontiguousarray(q[None, q0:q1]), np.ascontiguousarray(k[None, k0:k1]),
                         np.ascontiguousarray(v[None, k0:k1]), m, scale, dtype)
        O[q0:q1] = o[0]
        L[:, q0:q1] = l[0]
    return O, L


# ------------------------------------------------------- pure-Python twins

def _widen_py(x: int, dtype: str) -> float:
    if dtype == "bf16":
        return float(np.array([x << 16], dtype=np.uint32).view(np.float32)[0])
    return float(np.array([x], dtype=np.uint16).view(np.float16)[0])


def py_pack_qkv(q, k, v, U: int) -> np.ndarray:
    """Pure-Python loop twin of pack_qkv (tiny shapes only)."""
    B, S_l, H, D = q.shape
    h_l = H // U
    out = np.zeros((U, 3, B, S_l, h_l, D), dtype=np.uint16)
    src = (q, k, v)
    for r in range(U):
        for t in range(3):
            for b in range(B):
                for s in range(S_l):
                    for h in range(h_l):
                        for d in range(D):
                            out[r, t, b, s, h, d] = src[t][b, s, r * h_l + h, d]
    return out


def py_attention_row(q, k, v, b, h, i, mask=None, scale=None, dtype="bf16"):
    """Pure-Python twin of one attention row (tiny shapes only)."""
    D = q.shape[3]
    Sk = k.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(D)
    qs = [_widen_py(int(q[b, i, h, d]), dtype) for d in range(D)]
    s = []
    for j in range(Sk):
        if mask is not None and not mask[b, j]:
            continue
        s.append((j, scale * sum(qs[d] * _widen_py(int(k[b, j, h, d]), dtype) for d in range(D))))
    if not s:
        return [0.0] * D, -math.inf
    m = max(x for _, x in s)
    w = [(j, math.exp(x - m)) for j, x in s]
    l = sum(x for _, x in w)
    o = [sum(x * _widen_py(int(v[b, j, h, d]), dtype) for j, x in w) / l for d in range(D)]
    return o, m + math.log(l)
