"""Pins for the warpaffine oracle (oracle.warpaffine_u8 and
oracle.warpaffine_preprocess), checked against facts other than itself:

  * the identity matrix returns the source exactly, and the fused
    preprocessing then equals its closed form (channels reversed, (v/255 -
    mean)/std) computed here from the source bytes;
  * an integer shift moves the pixels and fills what falls outside;
  * a 2x reduction sampled at the centre of each 2x2 block gives
    floor(block sum / 4), exactly (an integer pin of the weights and of the
    uint8 truncation);
  * at the right edge, a point half a pixel inside blends the last column
    with the fill value (the constant border);
  * inside the image, a random rotation and zoom matches torch grid_sample in
    float64 (which fails if two corners' weights are swapped, the slip of the
    page's printed listing).
The definitions are those of the page "Hand-written warpaffine kernel",
§2.1 (the 2x3 matrix and its inverse), §2.2 (bilinear interpolation), §3.2
(fill value, uint8 output) and §4.2 (the fused preprocessing).
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle

MEAN = np.array([0.406, 0.456, 0.485], np.float32)
STD = np.array([0.225, 0.224, 0.229], np.float32)


def _src(B=2, H=9, W=14, seed=0):
    return np.random.default_rng(seed).integers(0, 256, (B, H, W, 3)).astype(np.uint8)


def _closed_form(src_like):
    v = src_like.astype(np.float64)[..., ::-1]  # RGB
    out = (v / 255.0 - MEAN[::-1].astype(np.float64)) / STD[::-1].astype(np.float64)
    return out.transpose(0, 3, 1, 2).astype(np.float32)


def test_identity_returns_the_source_and_the_closed_form():
    src = _src()
    B, H, W, _ = src.shape
    eye = np.tile(np.array([1, 0, 0, 0, 1, 0], np.float32), (B, 1))
    np.testing.assert_array_equal(oracle.warpaffine_u8(src, eye, (H, W), 7), src)
    np.testing.assert_allclose(oracle.warpaffine_preprocess(src, eye, (H, W), 7, MEAN, STD), _closed_form(src),
                               rtol=1e-6, atol=1e-6)


def test_integer_shift_moves_pixels_and_fills_outside():
    src = _src(1, 8, 10, seed=1)
    tx, ty = 3, -2
    m = np.array([[1, 0, tx, 0, 1, ty]], np.float32)
    out = oracle.warpaffine_u8(src, m, (8, 10), 200)
    want = np.full_like(src, 200)
    for y in range(8):
        for x in range(10):
            sx, sy = x + tx, y + ty
            if 0 <= sx < 10 and 0 <= sy < 8:
                want[0, y, x] = src[0, sy, sx]
    np.testing.assert_array_equal(out, want)


def test_half_size_at_block_centres_is_floor_of_block_mean():
    src = _src(2, 12, 16, seed=2)
    m = np.tile(np.array([2, 0, 0.5, 0, 2, 0.5], np.float32), (2, 1))
    out = oracle.warpaffine_u8(src, m, (6, 8), 0)
    blocks = src.astype(np.int64).reshape(2, 6, 2, 8, 2, 3).sum(axis=(2, 4))
    np.testing.assert_array_equal(out, (blocks // 4).astype(np.uint8))


def test_right_edge_blends_with_the_fill_value():
    src = _src(1, 4, 6, seed=3)
    fill = 250
    # dst (0, 0) -> src (W - 0.5, 1): half the last column, half the fill.
    m = np.array([[1, 0, 5.5, 0, 1, 1]], np.float32)
    out = oracle.warpaffine_u8(src, m, (1, 1), fill)
    want = np.floor(0.5 * src[0, 1, 5].astype(np.float64) + 0.5 * fill).astype(np.uint8)
    np.testing.assert_array_equal(out[0, 0, 0], want)
    # A point at x = W is outside: the fill value alone.
    m = np.array([[1, 0, 6.0, 0, 1, 1]], np.float32)
    np.testing.assert_array_equal(oracle.warpaffine_u8(src, m, (1, 1), fill)[0, 0, 0], [fill] * 3)


def test_random_rotation_matches_grid_sample_inside_the_image():
    inp = da_inputs.make_warpaffine_inputs(batch=2, src_hw=(45, 80), dst_hw=(32, 32), seed=4)
    src = inp.src.numpy()
    d2i = inp.d2i.numpy()
    Hd, Wd = inp.dst_hw
    got = oracle.warpaffine_preprocess(src, d2i, (Hd, Wd), inp.fill, MEAN, STD)
    B, H, W, _ = src.shape
    dy, dx = np.meshgrid(np.arange(Hd, dtype=np.float64), np.arange(Wd, dtype=np.float64), indexing="ij")
    m = d2i.astype(np.float64)
    sx = m[:, 0, None, None] * dx + m[:, 1, None, None] * dy + m[:, 2, None, None]
    sy = m[:, 3, None, None] * dx + m[:, 4, None, None] * dy + m[:, 5, None, None]
    # grid_sample (align_corners=False) samples input pixel ((g + 1) * W - 1) / 2.
    grid = torch.tensor(np.stack([(2 * sx + 1) / W - 1, (2 * sy + 1) / H - 1], -1))
    img = torch.tensor(src, dtype=torch.float64).permute(0, 3, 1, 2)
    v = torch.nn.functional.grid_sample(img, grid, mode="bilinear", padding_mode="zeros",
                                        align_corners=False).numpy()  # [B, 3, Hd, Wd] in BGR
    ref = (v[:, ::-1] / 255.0 - MEAN[::-1, None, None]) / STD[::-1, None, None]
    interior = (sx >= 0) & (sy >= 0) & (sx <= W - 1) & (sy <= H - 1)
    interior = np.broadcast_to(interior[:, None], ref.shape)
    assert interior.mean() > 0.3  # the letterbox bars are outside
    # The oracle rounds the source coordinates in fp32 (three roundings each),
    # torch works in float64: a coordinate error e moves a value by at most
    # 255 * e per axis (pixel steps are at most 255), i.e. by
    # (e_x + e_y) / std in normalised units.
    u = 2.0 ** -24
    ex = 3 * u * (np.abs(m[:, 0, None, None] * dx) + np.abs(m[:, 1, None, None] * dy) + np.abs(m[:, 2, None, None]))
    ey = 3 * u * (np.abs(m[:, 3, None, None] * dx) + np.abs(m[:, 4, None, None] * dy) + np.abs(m[:, 5, None, None]))
    tol = np.broadcast_to(((ex + ey)[:, None] / STD.min()), ref.shape) + 1e-6
    err = np.abs(got - ref)
    assert (err[interior] <= tol[interior] + 1e-5 * np.abs(ref[interior])).all(), float(err[interior].max())
    outside = ~((sx >= 0) & (sy >= 0) & (sx < W) & (sy < H))
    fill_val = (inp.fill / 255.0 - MEAN[::-1]) / STD[::-1]
    for o in range(3):
        np.testing.assert_allclose(got[:, o][outside], fill_val[o], rtol=1e-6)
