"""GPU parity of ctx_merge_joint_attn_mask against the oracle's merge
(vllm-omni PR #7641, follow-up review commit: the joint-mask merge owns the
2-D key mask of the gathered layout). Byte work: bit-exact. Invalid inputs:
the library's status must be the oracle's verdict (INVALID_ARG for a
ValueError, UNSUPPORTED for a refused combination), with nothing written.
"""
import numpy as np
import pytest
import torch

pytestmark = pytest.mark.gpu

INVALID, UNSUPPORTED = 1, 2


@pytest.fixture(scope="module")
def ctx():
    import diffusion_transformer_context_gb300 as m
    m.build()
    return m


def _rand(rng, shape, p):
    return ((rng.random(shape) < p) * rng.integers(1, 256, shape)).astype(np.uint8)


def _gpu(ctx, im, jm, B, S, J, front):
    out = torch.full((B, S + J), 0x5A, dtype=torch.uint8, device="cuda")
    imt = None if im is None else torch.from_numpy(np.ascontiguousarray(im)).cuda()
    jmt = None if jm is None else torch.from_numpy(np.ascontiguousarray(jm)).cuda()
    ctx.ctx_merge_joint_attn_mask(imt, jmt, B, S, J, out, joint_front=front)
    assert ctx.ctx_device_status() == 0
    return out.cpu().numpy()


CASES = [  # B, S_img, J, image?, joint?
    (1, 4096, 256, False, True),      # the Qwen-like layer: text padding only
    (2, 4096, 256, True, True),
    (3, 1000, 0, True, False),        # image mask, no joint keys
    (2, 777, 33, True, False),        # joint keys, no joint mask: filled with True
    (4, 1, 1, True, True),
    (1, 75600, 512, True, True),      # the longest gathered key range
    (5, 129, 1000, False, True),
]


@pytest.mark.parametrize("front", [False, True], ids=["rear", "front"])
@pytest.mark.parametrize("B,S,J,has_img,has_jnt", CASES)
def test_merge_bit_exact(ctx, orc, B, S, J, has_img, has_jnt, front):
    rng = np.random.default_rng(B * 7 + S + J)
    im = _rand(rng, (B, S), 0.8) if has_img else None
    jm = _rand(rng, (B, J), 0.5) if has_jnt else None
    got = _gpu(ctx, im, jm, B, S, J, front)
    want = orc.merge_joint_attn_mask(im, jm, B, S, J, front)
    assert np.array_equal(got, want)


def test_no_mask_writes_all_valid(ctx, orc):
    """No mask on either side: the oracle has no mask at all and the library
    writes the all-valid mask (the same attention)."""
    assert orc.merge_joint_attn_mask(None, None, 2, 50, 7, False) is None
    assert (_gpu(ctx, None, None, 2, 50, 7, False) == 1).all()


def _status(ctx, im_shape, jm_shape, B, S, J):
    lib = ctx.lib()
    import ctypes
    out = torch.full((B, S + max(J, 0)), 0x5A, dtype=torch.uint8, device="cuda")
    keep = []

    def arg(shape):
        if shape is None:
            return None, 0, None
        t = torch.ones(shape, dtype=torch.uint8, device="cuda")
        d = (ctypes.c_longlong * len(shape))(*shape)
        keep.append((t, d))
        return t.data_ptr(), len(shape), ctypes.cast(d, ctypes.c_void_p)

    ip, ind, idims = arg(im_shape)
    jp, jnd, jdims = arg(jm_shape)
    st = lib.ctx_merge_joint_attn_mask(ip, ind, idims, jp, jnd, jdims, B, S, J, 0, out.data_ptr(),
                                       torch.cuda.current_stream().cuda_stream)
    torch.cuda.synchronize()
    untouched = bool((out == 0x5A).all())
    return st, untouched


@pytest.mark.parametrize("im_shape,jm_shape,J", [
    ((2, 11), None, 4),              # image length
    ((3, 10), None, 4),              # image batch
    (None, (2, 3), 4),               # joint length
    (None, (1, 4), 4),               # joint batch
    (None, (2, 4), 0),               # joint mask without joint keys
    (None, (2, 1, 4), 4),            # joint mask 3-D
    ((2, 1, 10), None, 4),           # image mask 3-D
    ((2, 1, 3, 10), (2, 4), 4),      # 4-D image mask next to a joint mask
    ((2, 1, 3, 10), None, 4),        # 4-D image mask alone
    ((2, 1, 3, 10), (2, 1, 4), 4),   # joint rank reported first
])
def test_invalid_inputs_same_verdict_as_the_oracle(ctx, orc, im_shape, jm_shape, J):
    B, S = 2, 10
    im = None if im_shape is None else np.ones(im_shape, np.uint8)
    jm = None if jm_shape is None else np.ones(jm_shape, np.uint8)
    with pytest.raises((ValueError, orc.MaskMergeUnsupported)) as ei:
        orc.merge_joint_attn_mask(im, jm, B, S, J, False)
    want = UNSUPPORTED if isinstance(ei.value, orc.MaskMergeUnsupported) else INVALID
    st, untouched = _status(ctx, im_shape, jm_shape, B, S, J)
    assert st == want and untouched
