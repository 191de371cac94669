"""The C-ABI library builds, loads and exports every symbol include/ctx.h
declares; host-side validation fails closed before touching the GPU.

These run without a GPU: every call below is rejected by the host checks,
which come before any CUDA runtime call.
"""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "ctx.h")

OK, INVALID, UNSUPPORTED, MISALIGNED, ALIASING = 0, 1, 2, 3, 4


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(ctx_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    import diffusion_transformer_context_gb300 as ctx
    ctx.build()
    return ctx.lib()


def test_header_declares_the_hot_path():
    syms = declared_symbols()
    for s in ("ctx_pack_qkv", "ctx_unpack_qkv", "ctx_attn_lq_gkv", "ctx_pack_out", "ctx_unpack_out",
              "ctx_sim_all_to_all", "ctx_status_string", "ctx_device_status"):
        assert s in syms


def test_library_exports_every_declared_symbol(lib):
    import diffusion_transformer_context_gb300 as ctx
    for name in declared_symbols():
        assert hasattr(lib, name), name
        assert name in ctx.SIGNATURES, f"binding lacks {name}"
    assert set(ctx.SIGNATURES) == set(declared_symbols())


def test_binding_names_match_the_c_entry_points():
    import diffusion_transformer_context_gb300 as ctx
    for name in declared_symbols():
        assert callable(getattr(ctx, name)), name


def test_status_strings_and_version(lib):
    import diffusion_transformer_context_gb300 as ctx
    for code, name in ctx.STATUS_NAMES.items():
        assert ctx.ctx_status_string(code) == name
    assert ctx.ctx_status_string(99) == "CTX_ERR_UNKNOWN"
    assert ctx.ctx_version() >= 100


# fake, never dereferenced addresses: validation rejects before any CUDA call
A0 = 0x10000000
MB = 1 << 20


def test_pack_validation(lib):
    f = lib.ctx_pack_qkv
    assert f(None, A0, A0, A0, 1, 4, 4, 8, 2, 0, None) == INVALID
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 1, 4, 6, 8, 4, 0, None) == INVALID   # H % U
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 0, 4, 4, 8, 2, 0, None) == INVALID   # B = 0
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 1, 4, 4, 8, 2, 7, None) == INVALID   # dtype
    assert f(A0 + 8, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 1, 4, 4, 8, 2, 0, None) == MISALIGNED
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 1, 4, 4, 12, 2, 0, None) == MISALIGNED  # D % 8
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 64, 1, 4, 4, 8, 2, 0, None) == ALIASING


def test_unpack_validation(lib):
    f = lib.ctx_unpack_qkv
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 4, 8, 1, 4, 2, 8, 2, 0, None) == INVALID  # q stride < U*S_l
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, 8, 4, 1, 4, 2, 8, 2, 0, None) == INVALID  # kv stride
    # k overlaps v
    assert f(A0, A0 + MB, A0 + 2 * MB, A0 + 2 * MB + 16, 8, 8, 1, 4, 2, 8, 2, 0, None) == ALIASING
    # recv overlaps q
    assert f(A0, A0 + 32, A0 + 2 * MB, A0 + 3 * MB, 8, 8, 1, 4, 2, 8, 2, 0, None) == ALIASING


def test_attention_validation(lib):
    f = lib.ctx_attn_lq_gkv
    q, k, v, o, l = A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, A0 + 4 * MB
    w = A0 + 8 * MB
    nan = float("nan")
    assert f(q, k, v, None, nan, o, l, None, 0, 1, 16, 16, 2, 96, 0, None) == UNSUPPORTED
    assert f(q, k, v, None, -1.0, o, l, None, 0, 1, 16, 16, 2, 128, 0, None) == INVALID
    assert f(q, k, v, None, float("inf"), o, l, None, 0, 1, 16, 16, 2, 128, 0, None) == INVALID
    assert f(q, k, v, None, nan, o, l, None, 0, 1, 0, 16, 2, 128, 0, None) == INVALID
    assert f(q, k, v, None, nan, o, l, None, 0, 1, 16, -1, 2, 128, 0, None) == INVALID
    assert f(q, k, v, None, nan, None, l, None, 0, 1, 16, 16, 2, 128, 0, None) == INVALID
    assert f(q, k, v, None, nan, o, l, w, 0, 1, 16, 16, 2, 128, 0, None) == INVALID      # workspace, no size
    assert f(q + 4, k, v, None, nan, o, l, None, 0, 1, 16, 16, 2, 128, 0, None) == MISALIGNED
    assert f(q, k, v, None, nan, o, l + 2, None, 0, 1, 16, 16, 2, 128, 0, None) == MISALIGNED
    assert f(q, k, v, None, nan, o, l, w + 16, MB, 1, 16, 16, 2, 128, 0, None) == MISALIGNED
    assert f(q, k, v, None, nan, q + 64, l, None, 0, 1, 16, 16, 2, 128, 0, None) == ALIASING
    assert f(q, k, v, None, nan, o, o + 16, None, 0, 1, 16, 16, 2, 128, 0, None) == ALIASING
    assert f(q, k, v, None, nan, o, l, k, MB, 1, 16, 16, 2, 128, 0, None) == ALIASING    # workspace over K


def test_workspace_size_rejects_bad_sizes(lib):
    assert lib.ctx_attn_lq_gkv_workspace_size(1, 0, 16, 2, 128) == -1
    assert lib.ctx_attn_lq_gkv_workspace_size(1, 16, 16, 2, 96) == -1


def test_reverse_and_a2a_validation(lib):
    assert lib.ctx_pack_out(A0, A0 + MB, 3, 1, 2, 2, 8, 2, 0, None) == INVALID  # stride < U*S_l
    assert lib.ctx_pack_out(A0, A0 + 16, 4, 1, 2, 2, 8, 2, 0, None) == ALIASING
    assert lib.ctx_unpack_out(A0, A0 + MB, 1, 2, 2, 12, 2, 0, None) == MISALIGNED
    assert lib.ctx_unpack_out(A0, None, 1, 2, 2, 8, 2, 0, None) == INVALID
    assert lib.ctx_sim_all_to_all(A0, A0 + MB, 1, 2, 24, None) == MISALIGNED
    assert lib.ctx_sim_all_to_all(A0, A0 + 16, 1, 2, 32, None) == ALIASING
    assert lib.ctx_sim_all_to_all(A0, A0 + MB, 0, 2, 32, None) == INVALID


def test_selftest_limit_validation(lib):
    assert lib.ctx_selftest_wait_timeout(10, None) == INVALID
    assert lib.ctx_selftest_wait_timeout(10 ** 10, None) == INVALID


def test_product_path_has_no_oracle_or_fallback():
    """The CUDA package never imports the oracle and has no CPU path."""
    pkg = os.path.join(ROOT, "diffusion_transformer_context_gb300")
    for dirpath, _, files in os.walk(pkg):
        for fn in files:
            if fn.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, fn)).read()
                assert "import oracle" not in src and "from oracle" not in src, fn
                assert "ctx_oracle" not in src, fn


def test_lse_merge_validation(lib):
    f = lib.ctx_lse_merge
    o, l, out, lo = A0, A0 + 8 * MB, A0 + 16 * MB, A0 + 24 * MB
    assert f(o, l, 0, out, lo, 1, 4, 2, 8, 0, None) == INVALID          # P = 0
    assert f(o, l, 2, out, lo, 1, 4, 2, 12, 0, None) == MISALIGNED     # D % 8
    assert f(o + 8, l, 2, out, lo, 1, 4, 2, 8, 0, None) == MISALIGNED
    assert f(o, l, 2, o + 16, lo, 1, 4, 2, 8, 0, None) == ALIASING      # out inside the parts
    assert f(o, l, 2, out, l, 1, 4, 2, 8, 0, None) == ALIASING          # lse over lse_parts


def test_varlen_validation(lib):
    f = lib.ctx_attn_varlen
    q, k, v, cq, ck, o, l = A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB, A0 + 3 * MB + 256, A0 + 4 * MB, A0 + 5 * MB
    nan = float("nan")
    assert f(q, k, v, cq, ck, 0, 16, None, nan, o, l, None, 0, 16, 16, 2, 128, 0, None) == INVALID   # no documents
    assert f(q, k, v, cq, ck, 2, 0, None, nan, o, l, None, 0, 16, 16, 2, 128, 0, None) == INVALID   # max_seqlen_q
    assert f(q, k, v, cq, ck, 2, 16, None, nan, o, l, None, 0, 16, 16, 2, 96, 0, None) == UNSUPPORTED
    assert f(q, k, v, cq + 2, ck, 2, 16, None, nan, o, l, None, 0, 16, 16, 2, 128, 0, None) == MISALIGNED
    assert f(q, k, v, cq, ck, 2, 16, None, nan, cq, l, None, 0, 16, 16, 2, 128, 0, None) == ALIASING
    ws = A0 + 8 * MB
    assert f(q, k, v, cq, ck, 2, 16, None, nan, o, l, ws, 0, 16, 16, 2, 128, 0, None) == INVALID    # no size
    assert f(q, k, v, cq, ck, 2, 16, None, nan, o, l, ws + 16, MB, 16, 16, 2, 128, 0, None) == MISALIGNED
    assert f(q, k, v, cq, ck, 2, 16, None, nan, o, l, o, MB, 16, 16, 2, 128, 0, None) == ALIASING   # over out
    assert lib.ctx_attn_varlen_workspace_size(0, 16, 2, 128) == -1
    assert lib.ctx_attn_varlen_workspace_size(2, 16, 2, 96) == -1
    r = lib.ctx_varlen_remap
    assert r(cq, 0, 0, 8, ck, None, None, None) == INVALID
    assert r(cq, 2, -1, 8, ck, None, None, None) == INVALID
    assert r(cq, 2, 0, 8, cq + 4, None, None, None) == ALIASING
    assert r(cq, 2, 0, 8, ck, A0 + 6 * MB, None, None) == INVALID      # padding in without out


def test_pack_out_fused_validation(lib):
    f = lib.ctx_attn_lq_gkv_pack_out
    q, k, v, o = A0, A0 + MB, A0 + 2 * MB, A0 + 3 * MB
    nan = float("nan")
    # Sq = 30 not a multiple of U*S_l = 4*8
    assert f(q, k, v, None, nan, o, None, None, 0, 1, 30, 16, 2, 128, 4, 1, 8, 0, None) == INVALID
    # B = 3 not a multiple of B_rank = 2
    assert f(q, k, v, None, nan, o, None, None, 0, 3, 32, 16, 2, 128, 4, 2, 8, 0, None) == INVALID
    # more batch blocks (B / B_rank = 5) than destinations U = 4
    assert f(q, k, v, None, nan, o, None, None, 0, 5, 32, 16, 2, 128, 4, 1, 8, 0, None) == INVALID
    assert f(q, k, v, None, nan, o, None, None, 0, 1, 32, 16, 2, 96, 4, 1, 8, 0, None) == UNSUPPORTED


def test_mask_merge_validation(lib):
    """The page's fail-closed cases, rejected on the host in the page's order
    (joint rank first, then the image rank, joint keys, shapes)."""
    f = lib.ctx_merge_joint_attn_mask
    im, jm, out = A0, A0 + MB, A0 + 2 * MB
    L = ctypes.c_longlong

    def dims(*d):
        return ctypes.cast((L * len(d))(*d), ctypes.c_void_p)

    B, S, J = 2, 100, 8
    assert f(im, 2, dims(B, S), jm, 3, dims(B, 1, J), B, S, J, 0, out, None) == INVALID      # joint mask 3-D
    assert f(im, 4, dims(B, 1, 5, S), jm, 3, dims(B, 1, J), B, S, J, 0, out, None) == INVALID  # joint rank first
    assert f(im, 4, dims(B, 1, 5, S), jm, 2, dims(B, J), B, S, J, 0, out, None) == UNSUPPORTED  # 4-D + joint
    assert f(im, 4, dims(B, 1, 5, S), None, 0, None, B, S, J, 0, out, None) == UNSUPPORTED     # 4-D alone
    assert f(im, 1, dims(S), None, 0, None, B, S, J, 0, out, None) == INVALID                  # image 1-D
    assert f(None, 0, None, jm, 2, dims(B, J), B, S, 0, 0, out, None) == INVALID               # joint mask, no keys
    assert f(im, 2, dims(B, S + 1), None, 0, None, B, S, J, 0, out, None) == INVALID           # image length
    assert f(im, 2, dims(B + 1, S), None, 0, None, B, S, J, 0, out, None) == INVALID           # image batch
    assert f(None, 0, None, jm, 2, dims(B, J - 1), B, S, J, 0, out, None) == INVALID           # joint length
    assert f(None, 0, None, jm, 2, dims(1, J), B, S, J, 0, out, None) == INVALID               # joint batch
    assert f(im, 2, None, None, 0, None, B, S, J, 0, out, None) == INVALID                     # no dims
    assert f(None, 0, None, None, 0, None, B, S, J, 0, None, None) == INVALID                  # no output
    assert f(None, 0, None, None, 0, None, 0, S, J, 0, out, None) == INVALID                   # B = 0
    assert f(im, 2, dims(B, S), None, 0, None, B, S, J, 0, im + 50, None) == ALIASING           # out over image


def test_binding_refuses_views_that_overrun_their_storage(lib):
    """The library sees only a pointer, so the binding checks that the rows a
    strided output addresses lie inside the tensor's storage, before the call
    (here on host tensors: the refusal comes first)."""
    import torch

    import diffusion_transformer_context_gb300 as ctx
    U, B, S_l, h_l, D = 2, 1, 4, 2, 8
    recv = torch.zeros((U, 3, B, S_l, h_l, D), dtype=torch.bfloat16)
    big = torch.zeros((1, 16, h_l, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        # 8 rows from row 10 of a 16-row buffer
        ctx.ctx_unpack_qkv_ex(recv, big[:, 10:], big[:, :8], big[:, :8], U, B, S_l, h_l, D)
    o = torch.zeros((1, 6, h_l, D), dtype=torch.bfloat16)
    send = torch.zeros((U, B, S_l, h_l, D), dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ctx.ctx_pack_out(o, send, U)  # U*S_l = 8 rows of a 6-row output
