"""Pins for the oracle's joint-text key-mask merge (vllm-omni PR #7641,
follow-up review commit: the joint-mask merge is the single owner of 2-D
key-mask handling against the final, post-gather key layout).

The page lists the cases its own tests cover: image-only, joint-only (front
and rear), both masks, cached K/V (joint keys without joint queries), both
layouts, and invalid shapes (length, batch, joint mask without joint K/V),
plus the refusal of a 4-D image mask next to a 2-D joint mask. Each case is
pinned here against a construction that does not use the oracle's loops:
numpy comparisons and concatenation, closed-form counts of valid keys, and,
end to end, attention with masked keys equal to attention with those keys
deleted, in both placements.
"""
import numpy as np
import pytest
import torch

import workloads


def _rand_mask(rng, shape, p=0.6):
    # nonzero byte values other than 1 as well: the merge normalises to 0/1
    return ((rng.random(shape) < p) * rng.integers(1, 256, shape)).astype(np.uint8)


@pytest.mark.parametrize("B,S,J", [(1, 7, 0), (3, 40, 0), (2, 33, 5)])
def test_image_only(orc, B, S, J):
    """A 2-D image mask alone: the image segment is the mask normalised to
    0/1; a joint segment of joint_len keys (if any) is all True."""
    rng = np.random.default_rng(1)
    im = _rand_mask(rng, (B, S))
    for front in (False, True):
        m = orc.merge_joint_attn_mask(im, None, B, S, J, front)
        assert m.shape == (B, S + J) and m.dtype == np.uint8
        img = m[:, J:] if front else m[:, :S]
        jnt = m[:, :J] if front else m[:, S:]
        assert np.array_equal(img, (im != 0).astype(np.uint8))
        assert (jnt == 1).all()


@pytest.mark.parametrize("front", [False, True], ids=["rear", "front"])
def test_joint_only(orc, front):
    """Text padding carried only by the joint mask (the Qwen-Image case of
    the page, attn_mask None): image keys all valid, joint keys as given."""
    B, S, J = 2, 50, 12
    rng = np.random.default_rng(2)
    jm = _rand_mask(rng, (B, J))
    m = orc.merge_joint_attn_mask(None, jm, B, S, J, front)
    img = m[:, J:] if front else m[:, :S]
    jnt = m[:, :J] if front else m[:, S:]
    assert (img == 1).all()
    assert np.array_equal(jnt, (jm != 0).astype(np.uint8))


@pytest.mark.parametrize("front", [False, True], ids=["rear", "front"])
def test_both_masks_concatenate_in_placement_order(orc, front):
    B, S, J = 3, 21, 9
    rng = np.random.default_rng(3)
    im, jm = _rand_mask(rng, (B, S)), _rand_mask(rng, (B, J))
    m = orc.merge_joint_attn_mask(im, jm, B, S, J, front)
    parts = [(jm != 0), (im != 0)] if front else [(im != 0), (jm != 0)]
    assert np.array_equal(m, np.concatenate(parts, axis=1).astype(np.uint8))


def test_text_padding_counts(orc):
    """Text lengths L_b of a [B, J] joint mask with a valid prefix: row b has
    exactly (valid image keys) + L_b valid keys, in either placement."""
    B, S, J = 4, 64, 32
    L = [0, 1, 17, 32]
    jm = np.zeros((B, J), np.uint8)
    for b in range(B):
        jm[b, :L[b]] = 1
    im = np.ones((B, S), np.uint8)
    im[1, 60:] = 0
    for front in (False, True):
        m = orc.merge_joint_attn_mask(im, jm, B, S, J, front)
        assert [int(x) for x in m.sum(axis=1)] == [S + L[0], S - 4 + L[1], S + L[2], S + L[3]]


def test_cached_kv_sizes_joint_segment_from_keys(orc):
    """Cached K/V reuse: joint keys exist but the joint query is empty, and
    there is no joint mask. The joint segment is sized from the joint keys
    and filled with True; an image mask still applies to the image keys."""
    B, S, J = 2, 16, 6
    im = np.ones((B, S), np.uint8)
    im[0, :3] = 0
    m = orc.merge_joint_attn_mask(im, None, B, S, J, False)
    assert m.shape == (B, S + J)
    assert (m[:, S:] == 1).all() and int(m[0].sum()) == S + J - 3


def test_no_mask_at_all_is_none(orc):
    assert orc.merge_joint_attn_mask(None, None, 2, 10, 4, False) is None
    assert orc.merge_joint_attn_mask(None, None, 2, 10, 0, True) is None


@pytest.mark.parametrize("case", ["image_len", "image_batch", "joint_len", "joint_batch", "joint_without_kv",
                                  "joint_3d", "image_3d", "image_1d"])
def test_invalid_shapes_raise(orc, case):
    B, S, J = 2, 10, 4
    im, jm, jl = np.ones((B, S), np.uint8), np.ones((B, J), np.uint8), J
    if case == "image_len":
        im = np.ones((B, S + 1), np.uint8)
    elif case == "image_batch":
        im = np.ones((B + 1, S), np.uint8)
    elif case == "joint_len":
        jm = np.ones((B, J - 1), np.uint8)
    elif case == "joint_batch":
        jm = np.ones((1, J), np.uint8)
    elif case == "joint_without_kv":
        jl = 0
    elif case == "joint_3d":
        jm = np.ones((B, 1, J), np.uint8)
    elif case == "image_3d":
        im = np.ones((B, 1, S), np.uint8)
    elif case == "image_1d":
        im = np.ones((S,), np.uint8)
    with pytest.raises(ValueError):
        orc.merge_joint_attn_mask(im, jm, B, S, jl, False)


def test_4d_image_mask_refused(orc):
    """A 4-D image mask is refused next to a 2-D joint mask (fail closed),
    and on its own too: it has no key-mask form."""
    B, S, J = 1, 8, 2
    im4 = np.ones((B, 1, 3, S), np.uint8)
    with pytest.raises(orc.MaskMergeUnsupported):
        orc.merge_joint_attn_mask(im4, np.ones((B, J), np.uint8), B, S, J, False)
    with pytest.raises(orc.MaskMergeUnsupported):
        orc.merge_joint_attn_mask(im4, None, B, S, J, False)
    # rank checks run joint side first: a bad joint rank is reported even next to a 4-D image mask
    with pytest.raises(ValueError):
        orc.merge_joint_attn_mask(im4, np.ones((B, 1, J), np.uint8), B, S, J, False)


def test_merged_mask_equals_deleting_keys_in_both_placements(orc):
    """End to end: attention over the composed layer's gathered keys with the
    merged mask equals attention over only the valid keys, and the joint
    placement (front or rear) does not change the result."""
    U, A, B, S, H, D, J = 2, 2, 2, 32, 4, 16, 6
    gen = torch.Generator().manual_seed(71)
    u16 = workloads.as_u16
    full = [u16(workloads.randn((B, S, H, D), gen)) for _ in range(3)]
    jk, jv = u16(workloads.randn((B, J, H, D), gen)), u16(workloads.randn((B, J, H, D), gen))
    rng = np.random.default_rng(71)
    im = (rng.random((B, S)) > 0.25).astype(np.uint8)
    jm = np.zeros((B, J), np.uint8)
    jm[0, :4] = 1
    jm[1, :1] = 1
    R, S_l, h_l = U * A, S // (U * A), H // U
    sh = [[x[:, g * S_l:(g + 1) * S_l] for x in full] for g in range(R)]
    outs = {}
    for front in (False, True):
        res = orc.ulysses_agkv_forward([s[0] for s in sh], [s[1] for s in sh], [s[2] for s in sh], U, A,
                                       jk, jv, joint_front=front)
        mask = orc.merge_joint_attn_mask(im, jm, B, S, J, front)
        outs[front] = [orc.attention(res["q"][g], res["k"][g % U], res["v"][g % U], mask) for g in range(R)]
    for g in range(R):
        assert np.allclose(outs[False][g][0], outs[True][g][0], rtol=0, atol=1e-12)
        assert np.allclose(outs[False][g][1], outs[True][g][1], rtol=0, atol=1e-12)
    # rank 0 (a = 0, u = 0), batch 1: only the valid keys, gathered by numpy slicing
    b, u = 1, 0
    keep_img = np.nonzero(im[b])[0]
    kk = np.concatenate([full[1][b:b + 1, keep_img, u * h_l:(u + 1) * h_l], jk[b:b + 1, :1, u * h_l:(u + 1) * h_l]], 1)
    vv = np.concatenate([full[2][b:b + 1, keep_img, u * h_l:(u + 1) * h_l], jv[b:b + 1, :1, u * h_l:(u + 1) * h_l]], 1)
    qq = full[0][b:b + 1, :S // A, u * h_l:(u + 1) * h_l]
    eO, eL = orc.attention(np.ascontiguousarray(qq), np.ascontiguousarray(kk), np.ascontiguousarray(vv))
    assert np.allclose(outs[False][0][0][b], eO[0], rtol=0, atol=1e-12)
    assert np.allclose(outs[False][0][1][b], eL[0], rtol=0, atol=1e-12)
