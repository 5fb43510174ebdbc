"""Pins for the CPU oracle, checked against facts other than the oracle itself.

Each test pins the oracle to something independent of it:
  * hand-worked golden cases;
  * closed forms (integer-centre locations, constant maps, affine ramps);
  * linearity and adjoint identities;
  * brute-force Jacobians and finite differences on tiny inputs;
  * torch.nn.functional.grid_sample, which computes the same bilinear sample
    for one map; with several cameras and scales the operator is a weighted
    sum of grid_samples.
Together they fail on a dropped corner, a wrong sign, a swapped x/y or H/W,
a wrong level offset or a transposed operand.

The definitions pinned are those on the page "Inside Sparse4D's CUDA core:
deformable_aggregation bilinear interpolation and gradient back-propagation":
the bilinear step (§3.2), the gradients (§4.1) and the HWC layout (§3.1).
"""
import json
import os

import numpy as np
import pytest
import torch

import da_inputs
import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "hand_worked.json")


def _tables(shapes_ks):
    """spatial_shape / level_start_index for an explicit [K][S] list of (H, W)."""
    K, S = len(shapes_ks), len(shapes_ks[0])
    ss = np.zeros((K, S, 2), np.int32)
    ls = np.zeros((K, S), np.int32)
    row = 0
    for k in range(K):
        for s in range(S):
            ss[k, s] = shapes_ks[k][s]
            ls[k, s] = row
            row += shapes_ks[k][s][0] * shapes_ks[k][s][1]
    return ss, ls, row


def _rand_problem(rng, B, shapes_ks, C, G, A, P, lo=-0.1, hi=1.1):
    ss, ls, rows = _tables(shapes_ks)
    K, S = ss.shape[:2]
    feat = rng.standard_normal((B, rows, C)).astype(np.float32)
    loc = rng.uniform(lo, hi, (B, A, P, K, 2)).astype(np.float32)
    w = rng.standard_normal((B, A, P, K, S, G)).astype(np.float32)
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    return feat, ss, ls, loc, w, go


# --------------------------------------------------------------------------- golden

@pytest.mark.parametrize("case", json.load(open(GOLDEN))["cases"], ids=lambda c: c["name"])
def test_hand_worked_golden(case):
    H, W, C = case["H"], case["W"], case["C"]
    feat = np.array(case["map"], np.float32).reshape(1, H * W, C)
    ss = np.array([[[H, W]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    loc = np.array([case["x"], case["y"]], np.float32).reshape(1, 1, 1, 1, 2)
    w = np.full((1, 1, 1, 1, 1, 1), case["weight"], np.float32)
    go = np.full((1, 1, C), case["grad_out"], np.float32)
    out = oracle.forward(feat, ss, ls, loc, w)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)
    np.testing.assert_array_equal(out.ravel(), np.array(case["out"], np.float32))
    np.testing.assert_array_equal(gf.ravel(), np.array(case["grad_feat"], np.float32))
    np.testing.assert_array_equal(gl.ravel(), np.array(case["grad_loc"], np.float32))
    np.testing.assert_array_equal(gw.ravel(), np.array([case["grad_weight"]], np.float32))


# --------------------------------------------------------------------------- closed forms

def test_integer_centres_return_pixel_values_exactly():
    """Locations at pixel centres of power-of-two maps give h_im, w_im integers,
    so the sample is the pixel itself (lh = lw = 0)."""
    rng = np.random.default_rng(11)
    shapes = [[(16, 32)], [(8, 8)], [(32, 4)]]  # three cameras, one scale each
    ss, ls, rows = _tables(shapes)
    B, A, P, K, C, G = 2, 5, 3, 3, 8, 2
    feat = rng.standard_normal((B, rows, C)).astype(np.float32)
    ii = np.zeros((B, A, P, K), np.int64)
    jj = np.zeros((B, A, P, K), np.int64)
    loc = np.zeros((B, A, P, K, 2), np.float32)
    for k, ((H, W),) in enumerate(shapes):
        ii[..., k] = rng.integers(0, H, (B, A, P))
        jj[..., k] = rng.integers(0, W, (B, A, P))
        loc[..., k, 0] = (jj[..., k] + 0.5) / W
        loc[..., k, 1] = (ii[..., k] + 0.5) / H
    w = rng.standard_normal((B, A, P, K, 1, G)).astype(np.float32)
    out = oracle.forward(feat, ss, ls, loc, w)
    D = C // G
    expect = np.zeros((B, A, C))
    for k, ((H, W),) in enumerate(shapes):
        pix = ls[k, 0] + ii[..., k] * W + jj[..., k]  # [B, A, P]
        vals = feat[np.arange(B)[:, None, None], pix].astype(np.float64)  # [B,A,P,C]
        wk = np.repeat(w[:, :, :, k, 0, :].astype(np.float64), D, axis=-1)  # [B,A,P,C]
        expect += (wk * vals).sum(axis=2)
    np.testing.assert_allclose(out, expect, rtol=1e-6, atol=1e-7)
    # One point, one camera: a single product, rounded once.
    out1 = oracle.forward(feat[:, :, :], ss[:1], ls[:1], loc[:, :, :1, :1], w[:, :, :1, :1])
    pix = ls[0, 0] + ii[:, :, 0, 0] * shapes[0][0][1] + jj[:, :, 0, 0]
    v = feat[np.arange(B)[:, None], pix].astype(np.float64)
    e1 = (np.repeat(w[:, :, 0, 0, 0, :].astype(np.float64), D, axis=-1) * v).astype(np.float32)
    np.testing.assert_array_equal(out1[:, :, :], e1)


def test_constant_maps_sum_weights_and_zero_loc_grad():
    """A constant map kappa_ks gives kappa_ks times the sum of the in-bounds
    corner weights: exactly kappa_ks for interior samples. grad_loc is then 0."""
    rng = np.random.default_rng(12)
    shapes = [[(8, 12), (4, 6)], [(10, 7), (5, 3)]]
    ss, ls, rows = _tables(shapes)
    B, A, P, K, S, C, G = 2, 4, 3, 2, 2, 6, 3
    kappa = rng.uniform(1, 2, (K, S))
    feat = np.zeros((B, rows, C), np.float32)
    for k in range(K):
        for s in range(S):
            H, W = shapes[k][s]
            feat[:, ls[k, s]:ls[k, s] + H * W, :] = np.float32(kappa[k, s])
    kappa = kappa.astype(np.float32).astype(np.float64)
    # interior at every scale: 0.5/H <= y <= 1 - 0.5/H for the smallest H (3)
    loc = rng.uniform(0.17, 0.83, (B, A, P, K, 2)).astype(np.float32)
    w = rng.standard_normal((B, A, P, K, S, G)).astype(np.float32)
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    out = oracle.forward(feat, ss, ls, loc, w)
    expect = np.einsum("bapksg,ks->bag", w.astype(np.float64), kappa)
    expect = np.repeat(expect, C // G, axis=-1)
    np.testing.assert_allclose(out, expect, rtol=1e-6, atol=1e-7)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)
    assert np.all(gl == 0.0)
    # grad_weight = sum over the group's channels of grad_out * kappa
    gsum = go.astype(np.float64).reshape(B, A, G, C // G).sum(-1)
    e_gw = np.broadcast_to(np.einsum("bag,ks->baksg", gsum, kappa)[:, :, None], gw.shape)
    np.testing.assert_allclose(gw, e_gw, rtol=1e-6, atol=1e-6)


def test_partially_outside_sample_keeps_only_inside_corners():
    """h_im in (-1, 0): the two corners in row -1 read 0, so a constant map
    gives kappa * lh (the inside weight lh*hw + lh*lw)."""
    H, W, C = 6, 5, 4
    kappa = 3.0
    feat = np.full((1, H * W, C), kappa, np.float32)
    ss = np.array([[[H, W]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    y = np.float32(0.05)  # h_im = 0.3 - 0.5 = -0.2, h_low = -1, lh = 0.8
    x = np.float32(0.5)  # interior column
    loc = np.array([x, y], np.float32).reshape(1, 1, 1, 1, 2)
    w = np.ones((1, 1, 1, 1, 1, 1), np.float32)
    out = oracle.forward(feat, ss, ls, loc, w)
    h_im = np.float32(np.float32(y * np.float32(H)) - np.float32(0.5))
    lh = np.float64(h_im - np.floor(h_im))
    np.testing.assert_allclose(out.ravel(), np.full(C, kappa * lh), rtol=1e-7)
    # Fully outside (h_im <= -1): nothing is read.
    loc2 = np.array([0.5, -0.2], np.float32).reshape(1, 1, 1, 1, 2)
    assert np.all(oracle.forward(feat, ss, ls, loc2, w) == 0.0)
    # Not finite: nothing is read and all gradients vanish.
    loc3 = np.array([np.nan, 0.5], np.float32).reshape(1, 1, 1, 1, 2)
    assert np.all(oracle.forward(feat, ss, ls, loc3, w) == 0.0)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc3, w, np.ones((1, 1, C), np.float32))
    assert np.all(gf == 0) and np.all(gl == 0) and np.all(gw == 0)


def test_affine_ramp_pins_axes_and_location_gradient():
    """Bilinear interpolation reproduces an affine map exactly inside the map:
    F(r, c) = alpha*r + beta*c + gamma gives val = alpha*h_im + beta*w_im +
    gamma. So grad_loc = (W*beta, H*alpha) * top_grad, summed over channels.
    H != W and alpha != beta, so swapping x/y or H/W fails this test."""
    rng = np.random.default_rng(13)
    shapes = [[(12, 20), (6, 10)], [(9, 14), (3, 7)]]
    ss, ls, rows = _tables(shapes)
    B, A, P, K, S, C, G = 1, 3, 2, 2, 2, 4, 2
    D = C // G
    alpha = rng.uniform(-2, 2, C)
    beta = rng.uniform(-2, 2, C)
    gamma = rng.uniform(-2, 2, C)
    feat = np.zeros((B, rows, C), np.float32)
    for k in range(K):
        for s in range(S):
            H, W = shapes[k][s]
            r, c = np.meshgrid(np.arange(H), np.arange(W), indexing="ij")
            f = alpha * r[..., None] + beta * c[..., None] + gamma
            feat[0, ls[k, s]:ls[k, s] + H * W] = f.reshape(H * W, C)
    loc = rng.uniform(0.2, 0.8, (B, A, P, K, 2)).astype(np.float32)
    w = rng.standard_normal((B, A, P, K, S, G)).astype(np.float32)
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    out = oracle.forward(feat, ss, ls, loc, w)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)
    exp_out = np.zeros((B, A, C))
    exp_gl = np.zeros((B, A, P, K, 2))
    exp_gw = np.zeros((B, A, P, K, S, G))
    for k in range(K):
        for s in range(S):
            H, W = shapes[k][s]
            y = loc[..., k, 1].astype(np.float32)
            x = loc[..., k, 0].astype(np.float32)
            h_im = (np.float32(y * np.float32(H)) - np.float32(0.5)).astype(np.float64)
            w_im = (np.float32(x * np.float32(W)) - np.float32(0.5)).astype(np.float64)
            val = alpha * h_im[..., None] + beta * w_im[..., None] + gamma  # [B,A,P,C]
            wc = np.repeat(w[:, :, :, k, s, :].astype(np.float64), D, axis=-1)
            exp_out += (wc * val).sum(axis=2)
            tg = wc * go[:, :, None, :]
            exp_gl[..., k, 0] += W * (beta * tg).sum(-1)
            exp_gl[..., k, 1] += H * (alpha * tg).sum(-1)
            exp_gw[..., k, s, :] = (go[:, :, None, :] * val).reshape(B, A, P, G, D).sum(-1)
    # The stored map is the fp32 rounding of the affine function: allow for it.
    np.testing.assert_allclose(out, exp_out, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gl, exp_gl, rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(gw, exp_gw, rtol=1e-5, atol=1e-5)


# --------------------------------------------------------------------------- identities

def test_linear_in_weights_and_in_features():
    rng = np.random.default_rng(14)
    feat, ss, ls, loc, w, go = _rand_problem(rng, 2, [[(9, 11), (4, 6)], [(7, 5), (3, 3)]],
                                             C=8, G=2, A=4, P=3)
    w2 = rng.standard_normal(w.shape).astype(np.float32)
    f2 = rng.standard_normal(feat.shape).astype(np.float32)
    o1 = oracle.forward(feat, ss, ls, loc, w).astype(np.float64)
    o2 = oracle.forward(feat, ss, ls, loc, w2).astype(np.float64)
    o12 = oracle.forward(feat, ss, ls, loc, (w + w2).astype(np.float32)).astype(np.float64)
    np.testing.assert_allclose(o12, o1 + o2, rtol=1e-5, atol=1e-5)
    o3 = oracle.forward(f2, ss, ls, loc, w).astype(np.float64)
    o13 = oracle.forward((feat + f2).astype(np.float32), ss, ls, loc, w).astype(np.float64)
    np.testing.assert_allclose(o13, o1 + o3, rtol=1e-5, atol=1e-5)


def test_adjoint_identity_for_grad_feat():
    """forward is linear in feat, so <grad_out, fwd(feat)> = <grad_feat, feat>."""
    rng = np.random.default_rng(15)
    feat, ss, ls, loc, w, go = _rand_problem(rng, 2, [[(9, 11), (4, 6)], [(7, 5), (3, 3)]],
                                             C=8, G=4, A=5, P=3)
    out = oracle.forward(feat, ss, ls, loc, w)
    gf, _, _ = oracle.backward(feat, ss, ls, loc, w, go)
    lhs = np.dot(go.ravel().astype(np.float64), out.ravel().astype(np.float64))
    rhs = np.dot(gf.ravel().astype(np.float64), feat.ravel().astype(np.float64))
    assert abs(lhs - rhs) <= 1e-5 * (abs(lhs) + 1.0)


def test_grad_feat_equals_brute_force_jacobian():
    """grad_feat[col] = sum_i grad_out[i] * d out[i] / d feat[col], one column
    at a time, with feat = e_col (forward is linear in feat)."""
    rng = np.random.default_rng(16)
    shapes = [[(5, 6), (3, 2)]]
    feat, ss, ls, loc, w, go = _rand_problem(rng, 1, shapes, C=4, G=2, A=3, P=3)
    gf, _, _ = oracle.backward(feat, ss, ls, loc, w, go)
    B, rows, C = feat.shape
    expect = np.zeros_like(gf, dtype=np.float64)
    e = np.zeros_like(feat)
    for r in range(rows):
        for c in range(C):
            e[0, r, c] = 1.0
            col = oracle.forward(e, ss, ls, loc, w).astype(np.float64)
            expect[0, r, c] = np.sum(go.astype(np.float64) * col)
            e[0, r, c] = 0.0
    np.testing.assert_allclose(gf, expect, rtol=1e-6, atol=1e-7)


def test_grad_weight_equals_one_hot_forward():
    """forward is linear in the weights: grad_weight[i] = <grad_out, fwd(e_i)>."""
    rng = np.random.default_rng(17)
    feat, ss, ls, loc, w, go = _rand_problem(rng, 2, [[(6, 7), (3, 4)], [(5, 5), (2, 3)]],
                                             C=6, G=3, A=2, P=2)
    _, _, gw = oracle.backward(feat, ss, ls, loc, w, go)
    e = np.zeros_like(w)
    flat = e.reshape(-1)
    expect = np.zeros(w.size)
    for i in range(w.size):
        flat[i] = 1.0
        expect[i] = np.sum(go.astype(np.float64)
                           * oracle.forward(feat, ss, ls, loc, e).astype(np.float64))
        flat[i] = 0.0
    np.testing.assert_allclose(gw.ravel(), expect, rtol=1e-6, atol=1e-6)


def test_grad_loc_matches_central_difference_inside_cells():
    """Inside one cell the sample is bilinear in (h_im, w_im), so it is linear
    along each axis. A central difference whose step stays in the cell is then
    exact up to rounding."""
    rng = np.random.default_rng(18)
    shapes = [[(7, 9), (4, 5)], [(6, 6), (3, 4)]]
    feat, ss, ls, loc, w, go = _rand_problem(rng, 1, shapes, C=4, G=2, A=3, P=2,
                                             lo=-0.05, hi=1.05)
    _, gl, _ = oracle.backward(feat, ss, ls, loc, w, go)
    go64 = go.astype(np.float64)
    step = np.float32(2.0 ** -12)
    hmax = 16.0  # largest map side here is 9 < 16
    checked = 0
    for idx in np.ndindex(*loc.shape):
        k = idx[3]
        # Keep the perturbation inside the cell at every scale.
        ok = True
        for s in range(ss.shape[1]):
            n = ss[k, s, 1 if idx[4] == 0 else 0]
            t = loc[idx] * n - 0.5
            fr = t - np.floor(t)
            if not (0.05 < fr < 0.95):
                ok = False
        if not ok:
            continue
        lp = loc.copy()
        lm = loc.copy()
        lp[idx] += step
        lm[idx] -= step
        fp = np.sum(go64 * oracle.forward(feat, ss, ls, lp, w).astype(np.float64))
        fm = np.sum(go64 * oracle.forward(feat, ss, ls, lm, w).astype(np.float64))
        d = (fp - fm) / (float(lp[idx]) - float(lm[idx]))
        assert abs(d - gl[idx]) <= 2e-3 * abs(gl[idx]) + 2e-3 * hmax, (idx, d, gl[idx])
        checked += 1
    assert checked > loc.size // 4


# --------------------------------------------------------------------------- library special case

@pytest.mark.parametrize("B,H,W,C,G,A,P", [(2, 11, 17, 8, 2, 6, 4), (1, 16, 16, 32, 1, 16, 4)])
def test_single_map_matches_grid_sample(B, H, W, C, G, A, P):
    """With one camera and one scale, the bilinear sample is grid_sample's
    (bilinear, zero padding, align_corners=False) at grid = 2*loc - 1. Its
    unnormalised coordinate is ((g+1)*W - 1)/2 = x*W - 0.5. Autograd of
    grid_sample gives the independent reference backward; grad_loc =
    2 * grad_grid."""
    rng = np.random.default_rng(19)
    D = C // G
    feat = rng.standard_normal((B, H * W, C)).astype(np.float32)
    loc = rng.uniform(-0.1, 1.1, (B, A, P, 1, 2)).astype(np.float32)
    w = rng.standard_normal((B, A, P, 1, 1, G)).astype(np.float32)
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    ss = np.array([[[H, W]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    out = oracle.forward(feat, ss, ls, loc, w)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)

    f = torch.tensor(feat, dtype=torch.float64).view(B, H, W, C).permute(0, 3, 1, 2)
    f.requires_grad_(True)
    grid = (2.0 * torch.tensor(loc, dtype=torch.float64).view(B, A * P, 1, 2) - 1.0)
    grid.requires_grad_(True)
    wt = torch.tensor(w, dtype=torch.float64).view(B, A, P, G).requires_grad_(True)
    samp = torch.nn.functional.grid_sample(f, grid, mode="bilinear", padding_mode="zeros",
                                           align_corners=False)  # [B, C, A*P, 1]
    samp = samp.view(B, G, D, A, P).permute(0, 3, 4, 1, 2)  # [B, A, P, G, D]
    ref = (wt[..., None] * samp).sum(2).reshape(B, A, C)
    ref.backward(torch.tensor(go, dtype=torch.float64))
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-5, atol=1e-5)
    ref_gf = f.grad.permute(0, 2, 3, 1).reshape(B, H * W, C).numpy()
    np.testing.assert_allclose(gf, ref_gf, rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gl.reshape(B, A, P, 2),
                               2.0 * grid.grad.view(B, A, P, 2).numpy(), rtol=1e-4, atol=1e-3)
    np.testing.assert_allclose(gw.reshape(B, A, P, G), wt.grad.numpy(), rtol=1e-5, atol=1e-5)


@pytest.mark.parametrize("B,shapes,C,G,A,P", [
    (2, [[(7, 9), (4, 5)], [(6, 11), (3, 2)], [(5, 5), (2, 7)]], 8, 2, 5, 3),
    (1, [[(12, 10), (6, 5), (3, 3)], [(9, 14), (5, 7), (2, 4)]], 16, 4, 4, 2),
])
def test_many_maps_match_a_sum_of_grid_samples(B, shapes, C, G, A, P):
    """With several cameras and scales, out is the sum over (p, k, s) of
    w[b,a,p,k,s,g] times grid_sample of map (k, s) at camera k's location of
    point p, the same location at every scale of the camera (page §5.1's sum
    over the sampling dimensions). Every map has its own (H, W), so a
    transposed camera/scale index or a location taken per scale fails. Each
    map is a view of one packed float64 leaf, so autograd gives grad_feat in
    the packed layout and grad_loc summed over the scales."""
    rng = np.random.default_rng(21)
    feat, ss, ls, loc, w, go = _rand_problem(rng, B, shapes, C, G, A, P)
    K, S = ss.shape[:2]
    D = C // G
    out = oracle.forward(feat, ss, ls, loc, w)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)

    f = torch.tensor(feat, dtype=torch.float64, requires_grad=True)
    lt = torch.tensor(loc, dtype=torch.float64, requires_grad=True)
    wt = torch.tensor(w, dtype=torch.float64, requires_grad=True)
    ref = torch.zeros(B, A, G, D, dtype=torch.float64)
    for k in range(K):
        grid = (2.0 * lt[:, :, :, k, :] - 1.0).reshape(B, A * P, 1, 2)
        for s in range(S):
            H, W, r0 = int(ss[k, s, 0]), int(ss[k, s, 1]), int(ls[k, s])
            m = f[:, r0:r0 + H * W].reshape(B, H, W, C).permute(0, 3, 1, 2)
            samp = torch.nn.functional.grid_sample(m, grid, mode="bilinear", padding_mode="zeros",
                                                   align_corners=False)  # [B, C, A*P, 1]
            samp = samp.view(B, G, D, A, P).permute(0, 3, 4, 1, 2)  # [B, A, P, G, D]
            ref = ref + (wt[:, :, :, k, s, :, None] * samp).sum(2)
    ref = ref.reshape(B, A, C)
    ref.backward(torch.tensor(go, dtype=torch.float64))
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gf, f.grad.numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gl, lt.grad.numpy(), rtol=1e-4, atol=1e-3)
    np.testing.assert_allclose(gw, wt.grad.numpy(), rtol=1e-5, atol=1e-5)


# --------------------------------------------------------------------------- layout & edges

def test_level_start_index_selects_the_right_map():
    """Permuting how the maps are packed (and the start table with it) must
    not change the result."""
    rng = np.random.default_rng(20)
    shapes = [[(6, 8), (3, 4)], [(5, 7), (2, 3)]]
    feat, ss, ls, loc, w, go = _rand_problem(rng, 2, shapes, C=4, G=2, A=3, P=2)
    out = oracle.forward(feat, ss, ls, loc, w)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)
    # Re-pack in reverse order with a gap of 3 spare rows in front.
    K, S = ss.shape[:2]
    order = [(k, s) for k in range(K) for s in range(S)][::-1]
    rows2 = 3 + feat.shape[1]
    feat2 = rng.standard_normal((feat.shape[0], rows2, feat.shape[2])).astype(np.float32)
    ls2 = np.zeros_like(ls)
    r = 3
    for k, s in order:
        n = ss[k, s, 0] * ss[k, s, 1]
        feat2[:, r:r + n] = feat[:, ls[k, s]:ls[k, s] + n]
        ls2[k, s] = r
        r += n
    out2 = oracle.forward(feat2, ss, ls2, loc, w)
    gf2, gl2, gw2 = oracle.backward(feat2, ss, ls2, loc, w, go)
    np.testing.assert_array_equal(out, out2)
    np.testing.assert_array_equal(gl, gl2)
    np.testing.assert_array_equal(gw, gw2)
    for k, s in order:
        n = ss[k, s, 0] * ss[k, s, 1]
        np.testing.assert_array_equal(gf[:, ls[k, s]:ls[k, s] + n], gf2[:, ls2[k, s]:ls2[k, s] + n])
    assert np.all(gf2[:, :3] == 0)


def test_bf16_features_are_widened_exactly():
    inp = da_inputs.make_inputs(da_inputs.small_variant("large_bf16", num_anchors=3))
    as_f32 = inp.feat.to(torch.float32).numpy()
    args = (inp.spatial_shape.numpy(), inp.level_start_index.numpy(), inp.loc.numpy(),
            inp.weights.numpy())
    np.testing.assert_array_equal(oracle.forward(inp.feat_numpy(), *args),
                                  oracle.forward(as_f32, *args))


def test_f16_decoder_reads_every_bit_pattern_like_numpy():
    # One 1x1 map whose single pixel holds all 65536 binary16 bit patterns as
    # channels; a sample at the pixel centre with weight 1 returns them. numpy's
    # float16 -> float64 conversion is the independent reference.
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    feat = bits.view(np.float16).reshape(1, 1, 65536)
    ss = np.array([[[1, 1]]], np.int32)
    ls = np.array([[0]], np.int32)
    loc = np.full((1, 1, 1, 1, 2), 0.5, np.float32)
    w = np.ones((1, 1, 1, 1, 1, 1), np.float32)
    out = oracle.forward(feat, ss, ls, loc, w).reshape(-1)
    with np.errstate(invalid="ignore"):  # the NaN patterns cast to NaN, as intended
        want = feat.reshape(-1).astype(np.float64).astype(np.float32)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(out), nan)
    np.testing.assert_array_equal(out[~nan], want[~nan])
    assert nan.sum() == 2 * 1023  # every exponent-31 pattern with a non-zero fraction


def test_f16_features_are_widened_exactly():
    wl = da_inputs.small_variant("dcnv4", batch=1).replace(feat_dtype="f16")
    inp = da_inputs.make_inputs(wl)
    assert inp.feat.dtype == torch.float16
    as_f32 = inp.feat.to(torch.float32).numpy()
    args = (inp.spatial_shape.numpy(), inp.level_start_index.numpy(), inp.loc.numpy(),
            inp.weights.numpy())
    np.testing.assert_array_equal(oracle.forward(inp.feat_numpy(), *args), oracle.forward(as_f32, *args))
    go = inp.grad_out.numpy()
    for a, b in zip(oracle.backward(inp.feat_numpy(), *args, go), oracle.backward(as_f32, *args, go)):
        np.testing.assert_array_equal(a, b)


def test_anchor_range_matches_full_run():
    inp = da_inputs.make_inputs(da_inputs.small_variant("sp4d_train", batch=2, num_anchors=5))
    full = oracle.run_inputs(inp)
    part = oracle.run_inputs(inp, ba_range=(3, 7))
    A = inp.wl.num_anchors
    np.testing.assert_array_equal(part["out"], full["out"].reshape(2 * A, -1)[3:7])
    np.testing.assert_array_equal(part["grad_loc"],
                                  full["grad_loc"].reshape((2 * A,) + full["grad_loc"].shape[2:])[3:7])
    np.testing.assert_array_equal(part["grad_weight"],
                                  full["grad_weight"].reshape((2 * A,) + full["grad_weight"].shape[2:])[3:7])


@pytest.mark.parametrize("B,A,P", [(0, 4, 3), (2, 0, 3), (2, 4, 0)])
def test_empty_inputs(B, A, P):
    rng = np.random.default_rng(21)
    feat, ss, ls, loc, w, go = _rand_problem(rng, max(B, 1), [[(4, 4)]], C=8, G=2, A=max(A, 1),
                                             P=max(P, 1))
    feat = feat[:B]
    loc = loc[:B, :A, :P]
    w = w[:B, :A, :P]
    go = go[:B, :A]
    out = oracle.forward(feat, ss, ls, loc, w)
    assert out.shape == (B, A, 8) and np.all(out == 0)
    gf, gl, gw = oracle.backward(feat, ss, ls, loc, w, go)
    assert gf.shape == feat.shape and np.all(gf == 0)
    assert gl.shape == loc.shape and gw.shape == w.shape


def test_workload_shapes():
    """The five workloads have the sizes the configuration names."""
    W = da_inputs.WORKLOADS
    assert W["sp4d_train"].num_feat_rows == 6 * 14960
    assert W["sp4d_train"].num_samples == 13_478_400
    assert W["sp4d_inf"].num_samples == 2_246_400
    assert W["large_bf16"].num_samples == 4_492_800
    assert W["dcnv4"].num_samples == 903_168
    assert W["tiny"].num_samples == 64


# --------------------------------------------------------------------------- tolerance helper

def test_grad_loc_magnitude_bounds_and_hand_value():
    """The error-bound helper: it bounds |grad_loc|, and on the 2x2 centre
    case it equals the hand-worked sum of |terms|. With W = H = 2,
    |top_grad| = 2 and lh = lw = hh = hw = 0.5:
    x: 2*2*(0.5*(4+3) + 0.5*(2+1)) = 20; y: 2*2*(0.5*(4+2) + 0.5*(3+1)) = 20."""
    feat = np.array([1.0, 2.0, 3.0, 4.0], np.float32).reshape(1, 4, 1)
    ss = np.array([[[2, 2]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    loc = np.array([0.5, 0.5], np.float32).reshape(1, 1, 1, 1, 2)
    w = np.full((1, 1, 1, 1, 1, 1), 2.0, np.float32)
    go = np.ones((1, 1, 1), np.float32)
    m = oracle.grad_loc_magnitude(feat, ss, ls, loc, w, go)
    np.testing.assert_array_equal(m.ravel(), np.array([20.0, 20.0], np.float32))
    rng = np.random.default_rng(22)
    feat, ss, ls, loc, w, go = _rand_problem(rng, 2, [[(7, 9), (3, 4)], [(5, 6), (2, 2)]],
                                             C=8, G=2, A=5, P=3)
    _, gl, _ = oracle.backward(feat, ss, ls, loc, w, go)
    m = oracle.grad_loc_magnitude(feat, ss, ls, loc, w, go)
    assert np.all(np.abs(gl) <= m * (1 + 1e-6) + 1e-30)
    m2 = oracle.grad_loc_magnitude(feat, ss, ls, loc, w, (-3.0 * go).astype(np.float32))
    np.testing.assert_allclose(m2, 3.0 * m, rtol=1e-6)


def test_row_counts_hand_values_and_brute_force():
    """The grad_feat error-bound helper counts, per feature row, the in-map
    corners that land there (§3.2's four corners, §4.1's scatter).
    Hand values on a 2x2 map: the centre (0.5, 0.5) has h_im = w_im = 0.5,
    so all four pixels get one corner each; the origin (0, 0) has
    h_im = w_im = -0.5, so only pixel (0, 0), as corner 4, is in the map.
    Then a brute-force count on a random two-camera, two-scale problem, with
    the corner test written out here in numpy fp32."""
    ss = np.array([[[2, 2]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    feat = np.zeros((1, 4, 1), np.float32)
    w = np.ones((1, 2, 1, 1, 1, 1), np.float32)
    loc = np.array([[0.5, 0.5], [0.0, 0.0]], np.float32).reshape(1, 2, 1, 1, 2)
    np.testing.assert_array_equal(oracle.row_counts(feat, ss, ls, loc, w), [[2, 1, 1, 1]])

    rng = np.random.default_rng(23)
    shapes = [[(7, 9), (3, 4)], [(5, 6), (2, 2)]]
    feat, ss, ls, loc, w, _ = _rand_problem(rng, 2, shapes, C=4, G=2, A=6, P=5, lo=-0.3, hi=1.3)
    B, A, P, K = loc.shape[:4]
    expect = np.zeros((B, feat.shape[1]), np.int64)
    for b in range(B):
        for a in range(A):
            for p in range(P):
                for k in range(K):
                    x, y = loc[b, a, p, k]
                    for s in range(len(shapes[k])):
                        H, W = (int(v) for v in ss[k, s])
                        h_im = np.float32(np.float32(y * np.float32(H)) - np.float32(0.5))
                        w_im = np.float32(np.float32(x * np.float32(W)) - np.float32(0.5))
                        h0, w0 = int(np.floor(h_im)), int(np.floor(w_im))
                        for r, c in ((h0, w0), (h0, w0 + 1), (h0 + 1, w0), (h0 + 1, w0 + 1)):
                            if 0 <= r < H and 0 <= c < W:
                                expect[b, ls[k, s] + r * W + c] += 1
    got = oracle.row_counts(feat, ss, ls, loc, w)
    np.testing.assert_array_equal(got, expect)
    assert 0 < got.sum() < 4 * B * A * P * sum(len(s) for s in shapes)
