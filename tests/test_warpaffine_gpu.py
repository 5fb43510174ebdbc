"""GPU parity of the warpaffine kernels (include/wa.h) with the oracle.

wa_warpaffine_u8 truncates a float to uint8, and both sides compute that
float with the same fp32 steps (wa.h), so its output must equal the oracle's
bit for bit. wa_preprocess writes normalised floats: within fp32 rounding of
the oracle's double normalisation. Cases: the page's 1080p -> 640x640
letterbox with random rotation and zoom, sizes that do not fill the 32x8
blocks, upscaling, a 1x1 source, the identity, and an empty batch.
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def da():
    import deformable_view_feature_gb300 as m
    m.build.build()
    m.load_library()
    assert torch.cuda.is_available(), "the warpaffine tests need a CUDA GPU"
    return m


def _both(da, inp):
    dev = torch.device("cuda")
    src, d2i = inp.src.to(dev), inp.d2i.to(dev)
    u8 = da.warpaffine_u8(src, d2i, inp.dst_hw, inp.fill).cpu().numpy()
    pre = da.warpaffine_preprocess(src, d2i, inp.dst_hw, inp.fill, inp.mean.tolist(), inp.std.tolist())
    torch.cuda.synchronize()
    ref_u8 = oracle.warpaffine_u8(inp.src.numpy(), inp.d2i.numpy(), inp.dst_hw, inp.fill)
    ref_pre = oracle.warpaffine_preprocess(inp.src.numpy(), inp.d2i.numpy(), inp.dst_hw, inp.fill,
                                           inp.mean.numpy(), inp.std.numpy())
    return u8, pre.cpu().numpy(), ref_u8, ref_pre


def _check(da, inp):
    u8, pre, ref_u8, ref_pre = _both(da, inp)
    bad = u8 != ref_u8
    assert not bad.any(), f"{int(bad.sum())} uint8 values differ, first at {np.argwhere(bad)[0]}"
    # fp32 normalisation (two roundings of v/255, one of the subtraction, one
    # of the reciprocal and one of the product) against double.
    np.testing.assert_allclose(pre, ref_pre, rtol=4e-7, atol=1e-6)


def test_1080p_letterbox_with_jitter(da):
    _check(da, da_inputs.make_warpaffine_inputs(batch=3, seed=21))


@pytest.mark.parametrize("src_hw,dst_hw", [((37, 53), (19, 45)), ((20, 30), (61, 77)), ((1, 1), (5, 7)),
                                           ((64, 48), (33, 9))])
def test_ragged_and_upscaled_sizes(da, src_hw, dst_hw):
    _check(da, da_inputs.make_warpaffine_inputs(batch=2, src_hw=src_hw, dst_hw=dst_hw, seed=22))


def test_identity_returns_the_source(da):
    inp = da_inputs.make_warpaffine_inputs(batch=2, src_hw=(31, 70), dst_hw=(31, 70), seed=23, jitter=False)
    inp.d2i = torch.tensor([[1, 0, 0, 0, 1, 0]] * 2, dtype=torch.float32)
    u8, _, _, _ = _both(da, inp)
    np.testing.assert_array_equal(u8, inp.src.numpy())


def test_empty_batch(da):
    dev = torch.device("cuda")
    src = torch.empty(0, 4, 4, 3, dtype=torch.uint8, device=dev)
    d2i = torch.empty(0, 6, dtype=torch.float32, device=dev)
    assert da.warpaffine_u8(src, d2i, (2, 2)).shape == (0, 2, 2, 3)
    assert da.warpaffine_preprocess(src, d2i, (2, 2)).shape == (0, 3, 2, 2)


def test_bad_arguments_raise(da):
    dev = torch.device("cuda")
    src = torch.zeros(1, 4, 4, 3, dtype=torch.uint8, device=dev)
    d2i = torch.zeros(1, 6, dtype=torch.float32, device=dev)
    with pytest.raises(da.DaError, match="DA_ERR_SHAPE"):
        da.warpaffine_preprocess(src, d2i, (2, 2), std=(0.2, 0.0, 0.2))
    with pytest.raises(ValueError):
        da.warpaffine_u8(src.float(), d2i, (2, 2))
