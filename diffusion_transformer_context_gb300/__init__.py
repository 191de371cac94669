"""Python binding of libctx (include/ctx.h): argument marshalling only.

Every function here has the name of the C entry point it calls and does no
computation of its own: it reads shapes, dtypes, device pointers and the
current CUDA stream from torch tensors, calls the C ABI through ctypes and
raises ``CtxError`` on any status other than CTX_OK. There is no fallback: if
libctx.so has not been built, importing works but the first call raises.

torch is used only for device memory and streams.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

from .build import LIB_PATH, build  # noqa: F401  (re-exported for callers)

CTX_OK = 0
STATUS_NAMES = {0: "CTX_OK", 1: "CTX_ERR_INVALID_ARG", 2: "CTX_ERR_UNSUPPORTED", 3: "CTX_ERR_MISALIGNED",
                4: "CTX_ERR_ALIASING", 5: "CTX_ERR_CUDA", 6: "CTX_ERR_TIMEOUT"}
CTX_BF16, CTX_FP16 = 0, 1
CTX_LAYOUT_TQKV, CTX_LAYOUT_INTERLEAVED = 0, 1

# Every symbol include/ctx.h declares, with (restype, argtypes).
_P, _I, _LL, _F = ctypes.c_void_p, ctypes.c_int, ctypes.c_longlong, ctypes.c_float
SIGNATURES = {
    "ctx_pack_qkv": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_sim_all_to_all": (_I, [_P, _P, _I, _I, _LL, _P]),
    "ctx_pack_qkv_ex": (_I, [_P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_unpack_qkv_ex": (_I, [_P, _P, _P, _P, _LL, _LL, _I, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_unpack_out_ex": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_unpack_qkv": (_I, [_P, _P, _P, _P, _LL, _LL, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_attn_lq_gkv": (_I, [_P, _P, _P, _P, _F, _P, _P, _P, _LL, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_attn_lq_gkv_workspace_size": (_LL, [_I, _I, _I, _I, _I]),
    "ctx_attn_lq_gkv_pack_out": (_I, [_P, _P, _P, _P, _F, _P, _P, _P, _LL, _I, _I, _I, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_attn_lq_gkv_noalloc": (_I, [_P, _P, _P, _P, _F, _P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_pack_out": (_I, [_P, _P, _LL, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_unpack_out": (_I, [_P, _P, _I, _I, _I, _I, _I, _I, _P]),
    "ctx_lse_merge": (_I, [_P, _P, _I, _P, _P, _I, _I, _I, _I, _I, _P]),
    "ctx_merge_joint_attn_mask": (_I, [_P, _I, _P, _P, _I, _P, _I, _I, _I, _I, _P, _P]),
    "ctx_varlen_remap": (_I, [_P, _I, _LL, _LL, _P, _P, _P, _P]),
    "ctx_attn_varlen": (_I, [_P, _P, _P, _P, _P, _I, _I, _P, _F, _P, _P, _P, _LL, _I, _I, _I, _I, _I, _P]),
    "ctx_attn_varlen_workspace_size": (_LL, [_I, _I, _I, _I]),
    "ctx_status_string": (ctypes.c_char_p, [_I]),
    "ctx_device_status": (_I, [_P]),
    "ctx_last_cuda_error": (_I, []),
    "ctx_selftest_wait_timeout": (_I, [_LL, _P]),
    "ctx_version": (_I, []),
}

_lib = None
_lock = threading.Lock()


class CtxError(RuntimeError):
    def __init__(self, fn: str, status: int, cuda_error: int = 0):
        self.status = status
        self.cuda_error = cuda_error
        msg = f"{fn} failed: {STATUS_NAMES.get(status, status)}"
        if cuda_error:
            msg += f" (cudaError {cuda_error})"
        super().__init__(msg)


def lib():
    """The loaded libctx (ctypes.CDLL). Raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(f"libctx.so not found at {LIB_PATH}: build it first "
                                   "(python -c 'import __graft_entry__ as g; g.build()')")
            handle = ctypes.CDLL(LIB_PATH)
            for name, (res, args) in SIGNATURES.items():
                f = getattr(handle, name)
                f.restype = res
                f.argtypes = args
            _lib = handle
    return _lib


def _check(fn: str, status: int):
    if status != CTX_OK:
        raise CtxError(fn, status, lib().ctx_last_cuda_error() if status == 5 else 0)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return CTX_BF16
    if t.dtype == torch.float16:
        return CTX_FP16
    raise TypeError(f"libctx moves bf16/fp16 tensors, got {t.dtype}")


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return getattr(stream, "cuda_stream", stream)


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check_span(name: str, t, nbytes: int):
    """A strided output addressed from t.data_ptr() must lie inside t's
    storage: the C library sees only the pointer, so a view too short for
    the rows it is asked to write is refused here, before the call."""
    have = t.untyped_storage().nbytes() - t.storage_offset() * t.element_size()
    if nbytes > have:
        raise ValueError(f"{name}: {nbytes} bytes addressed from the tensor's first element, storage holds {have}")


def ctx_pack_qkv(q, k, v, staging, U: int, stream=None):
    """q, k, v [B,S_l,H,D] -> staging [U,3,B,S_l,H/U,D] (all contiguous CUDA tensors)."""
    B, S_l, H, D = q.shape
    _check("ctx_pack_qkv", lib().ctx_pack_qkv(_ptr(q), _ptr(k), _ptr(v), _ptr(staging), B, S_l, H, D, U,
                                              _dtype(q), _stream(stream)))
    return staging


def ctx_pack_qkv_ex(q, k, v, staging, U: int, layout: int = CTX_LAYOUT_TQKV, stream=None):
    """q, k, v [B,S_l,H,D] (H % U allowed: zero-padded heads) -> staging in `layout`."""
    B, S_l, H, D = q.shape
    _check("ctx_pack_qkv_ex", lib().ctx_pack_qkv_ex(_ptr(q), _ptr(k), _ptr(v), _ptr(staging), B, S_l, H, D, U,
                                                    layout, _dtype(q), _stream(stream)))
    return staging


def ctx_unpack_qkv_ex(recv, q, k, v, U: int, B: int, S_l: int, h_l: int, D: int, layout: int = CTX_LAYOUT_TQKV,
                      q_batch_stride_rows: int | None = None, kv_batch_stride_rows: int | None = None, stream=None):
    """recv in `layout` -> q, k, v bases of [B, stride_rows, h_l, D] buffers."""
    qs = U * S_l if q_batch_stride_rows is None else q_batch_stride_rows
    ks = U * S_l if kv_batch_stride_rows is None else kv_batch_stride_rows
    row = h_l * D * recv.element_size()
    _check_span("ctx_unpack_qkv_ex q", q, ((B - 1) * qs + U * S_l) * row)
    for name, t in (("k", k), ("v", v)):
        _check_span("ctx_unpack_qkv_ex " + name, t, ((B - 1) * ks + U * S_l) * row)
    _check("ctx_unpack_qkv_ex", lib().ctx_unpack_qkv_ex(_ptr(recv), _ptr(q), _ptr(k), _ptr(v), qs, ks, B, S_l, h_l,
                                                        D, U, layout, _dtype(recv), _stream(stream)))


def ctx_unpack_out_ex(recv, y, U: int, stream=None):
    """recv [U,B,S_l,h_l,D] -> y [B,S_l,H,D] keeping the first H = y.shape[2] heads."""
    U2, B, S_l, h_l, D = recv.shape
    H = y.shape[2]
    _check("ctx_unpack_out_ex", lib().ctx_unpack_out_ex(_ptr(recv), _ptr(y), B, S_l, h_l, H, D, U, _dtype(recv),
                                                        _stream(stream)))
    return y


def ctx_sim_all_to_all(send, recv, G: int, U: int, stream=None):
    """send/recv [G, U, U, chunk] (any dtype): recv[g][j][r] = send[g][r][j]."""
    chunk_bytes = send.numel() * send.element_size() // (G * U * U)
    _check("ctx_sim_all_to_all", lib().ctx_sim_all_to_all(_ptr(send), _ptr(recv), G, U, chunk_bytes,
                                                          _stream(stream)))
    return recv


def ctx_unpack_qkv(recv, q, k, v, U: int, q_batch_stride_rows: int | None = None,
                   kv_batch_stride_rows: int | None = None, stream=None):
    """recv [U,3,B,S_l,h_l,D] -> q, k, v: bases of [B, stride_rows, h_l, D] buffers
    (default strides U*S_l: contiguous [B, U*S_l, h_l, D] outputs)."""
    U2, three, B, S_l, h_l, D = recv.shape
    assert U2 == U and three == 3
    qs = U * S_l if q_batch_stride_rows is None else q_batch_stride_rows
    ks = U * S_l if kv_batch_stride_rows is None else kv_batch_stride_rows
    row = h_l * D * recv.element_size()
    _check_span("ctx_unpack_qkv q", q, ((B - 1) * qs + U * S_l) * row)
    for name, t in (("k", k), ("v", v)):
        _check_span("ctx_unpack_qkv " + name, t, ((B - 1) * ks + U * S_l) * row)
    _check("ctx_unpack_qkv", lib().ctx_unpack_qkv(_ptr(recv), _ptr(q), _ptr(k), _ptr(v), qs, ks,
                                                  B, S_l, h_l, D, U, _dtype(recv), _stream(stream)))


def ctx_attn_lq_gkv(q, k, v, out, lse=None, key_mask=None, scale: float | None = None, workspace=None,
                    stream=None):
    """q [B,Sq,H,D], k/v [B,Sk,H,D] -> out [B,Sq,H,D], lse [B,H,Sq] fp32 (optional).
    workspace: None, or a zero-filled device buffer of at least
    ctx_attn_lq_gkv_workspace_size(...) bytes for the balanced schedule."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    s = float("nan") if scale is None else float(scale)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ctx_attn_lq_gkv", lib().ctx_attn_lq_gkv(_ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), s, _ptr(out),
                                                    _ptr(lse), _ptr(workspace), wb, B, Sq, Sk, H, D, _dtype(q),
                                                    _stream(stream)))
    return out


def ctx_attn_lq_gkv_pack_out(q, k, v, send, U: int, B_rank: int, S_l: int, lse=None, key_mask=None,
                             scale: float | None = None, workspace=None, stream=None):
    """Attention whose output goes straight into the reverse exchange's send
    layout: q [B,Sq,H,D] (B = U'*B_rank, Sq = A*U*S_l), send [A,U',U,B_rank,S_l,H,D]."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    s = float("nan") if scale is None else float(scale)
    wb = 0 if workspace is None else workspace.numel() * workspace.element_size()
    _check("ctx_attn_lq_gkv_pack_out", lib().ctx_attn_lq_gkv_pack_out(
        _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), s, _ptr(send), _ptr(lse), _ptr(workspace), wb, B, Sq, Sk, H, D,
        U, B_rank, S_l, _dtype(q), _stream(stream)))
    return send


def ctx_attn_lq_gkv_workspace_size(B: int, Sq: int, Sk: int, H: int, D: int) -> int:
    n = lib().ctx_attn_lq_gkv_workspace_size(B, Sq, Sk, H, D)
    if n < 0:
        raise CtxError("ctx_attn_lq_gkv_workspace_size", 1)
    return n


def ctx_attn_lq_gkv_noalloc(q, k, v, out, lse=None, key_mask=None, scale: float | None = None, stream=None):
    """ctx_attn_lq_gkv with the balanced schedule and the library's own fixed
    scratch array: nothing is allocated by anyone. Calls that can overlap on
    the GPU must be serialised by the caller."""
    B, Sq, H, D = q.shape
    Sk = k.shape[1]
    s = float("nan") if scale is None else float(scale)
    _check("ctx_attn_lq_gkv_noalloc", lib().ctx_attn_lq_gkv_noalloc(
        _ptr(q), _ptr(k), _ptr(v), _ptr(key_mask), s, _ptr(out), _ptr(lse), B, Sq, Sk, H, D, _dtype(q),
        _stream(stream)))
    return out


def attn_workspace(B: int, Sq: int, Sk: int, H: int, D: int, device="cuda"):
    """A zero-filled workspace tensor of the size the balanced schedule needs."""
    n = ctx_attn_lq_gkv_workspace_size(B, Sq, Sk, H, D)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def ctx_pack_out(o, send, U: int, o_batch_stride_rows: int | None = None, stream=None):
    """o: base of a [B, stride_rows, h_l, D] buffer whose first U*S_l rows per
    batch are this rank's output -> send [U, B, S_l, h_l, D]."""
    Us, B, S_l, h_l, D = send.shape
    assert Us == U
    st = U * S_l if o_batch_stride_rows is None else o_batch_stride_rows
    _check_span("ctx_pack_out o", o, ((B - 1) * st + U * S_l) * h_l * D * send.element_size())
    _check("ctx_pack_out", lib().ctx_pack_out(_ptr(o), _ptr(send), st, B, S_l, h_l, D, U, _dtype(send),
                                              _stream(stream)))
    return send


def ctx_unpack_out(recv, y, U: int, stream=None):
    """recv [U, B, S_l, h_l, D] -> y [B, S_l, U*h_l, D]."""
    U2, B, S_l, h_l, D = recv.shape
    _check("ctx_unpack_out", lib().ctx_unpack_out(_ptr(recv), _ptr(y), B, S_l, h_l, D, U, _dtype(recv),
                                                  _stream(stream)))
    return y


def ctx_lse_merge(o_parts, lse_parts, out, lse=None, stream=None):
    """o_parts [P,B,Sq,H,D], lse_parts [P,B,H,Sq] fp32 -> out [B,Sq,H,D], lse [B,H,Sq] (optional)."""
    P, B, Sq, H, D = o_parts.shape
    _check("ctx_lse_merge", lib().ctx_lse_merge(_ptr(o_parts), _ptr(lse_parts), P, _ptr(out), _ptr(lse), B, Sq, H,
                                                D, _dtype(o_parts), _stream(stream)))
    return out


def _mask_arg(t):
    """(pointer, rank, host array of sizes) of an optional mask tensor."""
    if t is None:
        return None, 0, None
    dims = (ctypes.c_longlong * t.dim())(*t.shape)
    return t.data_ptr(), t.dim(), dims


def ctx_merge_joint_attn_mask(image_mask, joint_mask, B: int, S_img: int, J: int, key_mask,
                              joint_front: bool = False, stream=None):
    """Optional image mask [B, S_img] and joint mask [B, J] (uint8 or bool CUDA
    tensors, nonzero = attend) -> key_mask [B, S_img + J] uint8 0/1, the joint
    segment first when joint_front. The masks' ranks and sizes are passed as
    they are; the library checks them."""
    ip, ind, idims = _mask_arg(image_mask)
    jp, jnd, jdims = _mask_arg(joint_mask)
    _check("ctx_merge_joint_attn_mask", lib().ctx_merge_joint_attn_mask(
        ip, ind, None if idims is None else ctypes.cast(idims, ctypes.c_void_p),
        jp, jnd, None if jdims is None else ctypes.cast(jdims, ctypes.c_void_p),
        B, S_img, J, 1 if joint_front else 0, _ptr(key_mask), _stream(stream)))
    return key_mask


def ctx_varlen_remap(cu_seqlens_q, span_begin: int, span_len: int, cu_seqlens_q_local, packed_padding=None,
                     packed_padding_local=None, stream=None):
    """int32 device tensors: [n_docs+1] global -> [n_docs+1] local boundaries of one rank."""
    n_docs = cu_seqlens_q.numel() - 1
    _check("ctx_varlen_remap", lib().ctx_varlen_remap(_ptr(cu_seqlens_q), n_docs, span_begin, span_len,
                                                      _ptr(cu_seqlens_q_local), _ptr(packed_padding),
                                                      _ptr(packed_padding_local), _stream(stream)))
    return cu_seqlens_q_local


def ctx_attn_varlen(q, k, v, cu_seqlens_q, cu_seqlens_k, max_seqlen_q: int, out, lse=None, key_mask=None,
                    scale: float | None = None, workspace=None, stream=None):
    """q [Sq,H,D], k/v [Sk,H,D], int32 cu tensors [n_docs+1] -> out [Sq,H,D], lse [H,Sq]; `workspace`: a
    zero-filled uint8 device tensor of ctx_attn_varlen_workspace_size(...) bytes for the balanced schedule."""
    Sq, H, D = q.shape
    Sk = k.shape[0]
    s = float("nan") if scale is None else float(scale)
    wsb = workspace.numel() * workspace.element_size() if workspace is not None else 0
    _check("ctx_attn_varlen", lib().ctx_attn_varlen(_ptr(q), _ptr(k), _ptr(v), _ptr(cu_seqlens_q),
                                                    _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, max_seqlen_q,
                                                    _ptr(key_mask), s, _ptr(out), _ptr(lse), _ptr(workspace), wsb,
                                                    Sq, Sk, H, D, _dtype(q), _stream(stream)))
    return out


def ctx_attn_varlen_workspace_size(n_docs: int, max_seqlen_q: int, H: int, D: int) -> int:
    n = lib().ctx_attn_varlen_workspace_size(n_docs, max_seqlen_q, H, D)
    if n < 0:
        raise CtxError("ctx_attn_varlen_workspace_size", 1)
    return n


def varlen_workspace(n_docs: int, max_seqlen_q: int, H: int, D: int, device="cuda"):
    """A zero-filled workspace tensor of the size the balanced varlen schedule needs."""
    n = ctx_attn_varlen_workspace_size(n_docs, max_seqlen_q, H, D)
    return torch.zeros(max(n, 256), dtype=torch.uint8, device=device)


def ctx_device_status(stream=None) -> int:
    return lib().ctx_device_status(_stream(stream))


def ctx_selftest_wait_timeout(limit_ns: int, stream=None) -> int:
    return lib().ctx_selftest_wait_timeout(int(limit_ns), _stream(stream))


def ctx_status_string(status: int) -> str:
    return lib().ctx_status_string(status).decode()


def ctx_version() -> int:
    return lib().ctx_version()


def ctx_last_cuda_error() -> int:
    return lib().ctx_last_cuda_error()
