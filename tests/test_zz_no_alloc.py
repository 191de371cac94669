"""The allocation-free attention entry point.

Some callers of this library cannot allocate device memory: a host framework
that owns every device buffer and gives a plugin only its inputs and outputs,
a C program embedding the library without a device allocator, or a path that
must not call cudaMalloc because it can synchronise the device.
ctx_attn_lq_gkv_noalloc serves them with the library's own fixed scratch
array. This test calls it through the C ABI twice in a row and checks each
result against ctx_attn_lq_gkv with a caller-provided workspace, within the
attention tolerance the other GPU tests use (O max-abs 2e-2, mean-abs 2e-3,
LSE 1e-3). The second call checks that the shared scratch left by the first
call does not leak into the next result.

It sits in a file of its own that pytest collects last, and it depends on
nothing earlier tests leave behind.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def ctx():
    import diffusion_transformer_context_gb300 as m
    m.build()
    return m


CASES = [  # B, Sq, Sk, H, masked
    (1, 4095, 8192, 4, False),   # 64 work units < SMs: every unit split and merged
    (2, 700, 1300, 3, True),     # text-padding mask, ragged tails
]


@pytest.mark.parametrize("B,Sq,Sk,H,masked", CASES)
def test_noalloc_matches_the_workspace_entry_point_twice(ctx, B, Sq, Sk, H, masked):
    D = 128
    lib = ctx.lib()
    gen = torch.Generator().manual_seed(1234)
    q, k, v = (workloads.randn(s, gen).cuda() for s in ((B, Sq, H, D), (B, Sk, H, D), (B, Sk, H, D)))
    mask = None
    if masked:
        m = np.ones((B, Sk), np.uint8)
        m[0, Sk - 200:] = 0
        m[1, :50] = 0
        mask = torch.from_numpy(m).cuda()
    stream = torch.cuda.current_stream().cuda_stream
    nan = float("nan")
    mptr = None if mask is None else mask.data_ptr()

    ref_o = torch.empty_like(q)
    ref_l = torch.empty((B, H, Sq), dtype=torch.float32, device="cuda")
    ws = torch.zeros(lib.ctx_attn_lq_gkv_workspace_size(B, Sq, Sk, H, D), dtype=torch.uint8, device="cuda")
    assert lib.ctx_attn_lq_gkv(q.data_ptr(), k.data_ptr(), v.data_ptr(), mptr, nan, ref_o.data_ptr(),
                               ref_l.data_ptr(), ws.data_ptr(), ws.numel(), B, Sq, Sk, H, D, 0, stream) == 0

    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((B, H, Sq), float("nan"), dtype=torch.float32, device="cuda")
        st = lib.ctx_attn_lq_gkv_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), mptr, nan, out.data_ptr(),
                                         lse.data_ptr(), B, Sq, Sk, H, D, 0, stream)
        assert st == 0, ctx.ctx_status_string(st)
        assert lib.ctx_device_status(stream) == 0
        err = (out.float() - ref_o.float()).abs()
        assert float(err.max()) <= 2e-2 and float(err.mean()) <= 2e-3, (call, float(err.max()))
        assert float((lse - ref_l).abs().max()) <= 1e-3, call


def test_noalloc_rejects_problems_beyond_its_scratch(ctx):
    """Sizes whose workspace would exceed the fixed scratch array are refused
    up front (CTX_ERR_UNSUPPORTED), before anything is enqueued."""
    lib = ctx.lib()
    q = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    need = lib.ctx_attn_lq_gkv_workspace_size(4096, 65536, 1024, 1, 128)  # 1M work units
    assert need > 44 * 2 ** 20
    st = lib.ctx_attn_lq_gkv_noalloc(q.data_ptr(), q.data_ptr(), q.data_ptr(), None, float("nan"), q.data_ptr(),
                                     None, 4096, 65536, 1024, 1, 128, 0, None)
    assert st == 2, ctx.ctx_status_string(st)
