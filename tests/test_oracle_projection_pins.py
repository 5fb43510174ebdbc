"""Pins for the oracle of the upstream step: the projection of anchor key
points into the cameras and the softmax that turns logits into weights
(oracle.project, softmax_weights, projected_chain, backward_projected).

The Sparse4D page says that each 3D anchor is projected into the 2D views
before the aggregation (§1, §6) but prints no formula; the reading is the
pinhole projection by a 4x4 matrix (see dao_project). It is pinned by:
  * closed forms: a point on a camera's axis lands on the principal point, a
    lateral offset moves it by focal * offset / depth, and points behind a
    camera read nothing;
  * torch: the same projection in float64, torch.softmax, and autograd of
    both for the chain rule;
  * end to end, with one camera and one scale: torch grid_sample of the
    projected points, weighted by torch.softmax, differentiated by autograd.
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle


def test_axis_point_lands_on_the_principal_point_and_offsets_scale_with_depth():
    W, H = 704.0, 256.0
    rig = da_inputs.camera_rig(6, W, H, focal_px=300.0, height_m=1.6).astype(np.float32)
    proj = rig[None]  # [1, 6, 4, 4]
    depth, side, up = 20.0, 3.0, 1.0
    # Straight ahead of camera 0 (yaw 0, looking along +x), at camera height;
    # then 3 m to the right (-y) and 1 m up (+z).
    kp = np.array([[[[depth, 0.0, 1.6], [depth, -side, 1.6 + up]]]], np.float32)
    loc = oracle.project(kp, proj, W, H)  # [1, 1, 2, 6, 2]
    np.testing.assert_allclose(loc[0, 0, 0, 0], [0.5, 0.5], rtol=0, atol=1e-7)
    np.testing.assert_allclose(loc[0, 0, 1, 0], [(W / 2 + 300.0 * side / depth) / W,
                                                 (H / 2 - 300.0 * up / depth) / H], rtol=1e-6)
    # Camera 3 (yaw 180 degrees) sees both points from behind: nothing.
    assert np.isnan(loc[0, 0, :, 3]).all()


def test_projection_matches_float64_within_fp32_rounding():
    inp = da_inputs.make_projected_inputs(da_inputs.small_variant("sp4d_proj", batch=2, num_anchors=40))
    loc = oracle.project(inp.keypoints.numpy(), inp.projection.numpy(), inp.image_w, inp.image_h)
    kp = inp.keypoints.to(torch.float64)
    M = inp.projection.to(torch.float64)
    hom = torch.cat([kp, torch.ones_like(kp[..., :1])], -1)  # [B, A, P, 4]
    q = torch.einsum("bkij,bapj->bapki", M, hom)  # [B, A, P, K, 4]
    d = q[..., 2]
    ref = torch.stack([q[..., 0] / d / inp.image_w, q[..., 1] / d / inp.image_h], -1).numpy()
    front = (d > 1e-5).numpy()
    assert front.mean() > 0.3 and (~front).mean() > 0.3
    assert np.isnan(loc[~front]).all()
    # fp32 error bound of the steps: each row sum carries up to 4 roundings of
    # terms of total size T, the divisions two more: with u = 2^-24,
    # |dx| <= 8u * (T_u / (|d| W) + |x| * T_d / |d|) + 2u |x| (likewise y).
    u = 2.0 ** -24
    absterm = torch.einsum("bkij,bapj->bapki", M.abs(), hom.abs()).numpy()  # T per row
    dd = d.abs().numpy()
    bound = np.stack([8 * u * (absterm[..., 0] / (dd * inp.image_w) + np.abs(ref[..., 0]) * absterm[..., 2] / dd),
                      8 * u * (absterm[..., 1] / (dd * inp.image_h) + np.abs(ref[..., 1]) * absterm[..., 2] / dd)],
                     -1) + 2 * u * np.abs(ref)
    err = np.abs(loc.astype(np.float64) - ref)
    assert (err[front] <= bound[front]).all(), float((err[front] / bound[front]).max())
    # Inside the image the bound is a few parts in 10^7.
    vis = front[..., None] & (np.abs(ref - 0.5) < 0.6)
    assert (err[vis] <= 1e-6).all()


def test_softmax_matches_torch_and_sums_to_one():
    z = np.random.default_rng(3).standard_normal((2, 5, 3, 2, 4, 8)).astype(np.float32) * 4
    w = oracle.softmax_weights(z)
    t = torch.tensor(z, dtype=torch.float64).permute(0, 1, 5, 2, 3, 4).reshape(2, 5, 8, -1).softmax(-1)
    ref = t.reshape(2, 5, 8, 3, 2, 4).permute(0, 1, 3, 4, 5, 2).numpy()
    np.testing.assert_allclose(w, ref, rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(w.astype(np.float64).sum(axis=(2, 3, 4)), 1.0, rtol=1e-6)


def test_chain_rule_matches_autograd():
    inp = da_inputs.make_projected_inputs(da_inputs.small_variant("sp4d_proj", batch=1, num_anchors=30))
    rng = np.random.default_rng(4)
    B, A, P, _ = inp.keypoints.shape
    K, S, G = 6, 4, 8
    w = oracle.softmax_weights(inp.logits.numpy())
    gl = rng.standard_normal((B, A, P, K, 2)).astype(np.float32)
    gw = rng.standard_normal((B, A, P, K, S, G)).astype(np.float32)
    gkp, glg = oracle.projected_chain(inp.keypoints.numpy(), inp.projection.numpy(), inp.image_w, inp.image_h,
                                      w, gl, gw)
    kp = inp.keypoints.to(torch.float64).requires_grad_(True)
    z = inp.logits.to(torch.float64).requires_grad_(True)
    M = inp.projection.to(torch.float64)
    hom = torch.cat([kp, torch.ones_like(kp[..., :1])], -1)
    q = torch.einsum("bkij,bapj->bapki", M, hom)
    d = q[..., 2]
    front = d > 1e-5
    x = torch.where(front, q[..., 0] / d / inp.image_w, torch.zeros_like(d))
    y = torch.where(front, q[..., 1] / d / inp.image_h, torch.zeros_like(d))
    wt = z.permute(0, 1, 5, 2, 3, 4).reshape(B, A, G, -1).softmax(-1).reshape(B, A, G, P, K, S)
    wt = wt.permute(0, 1, 3, 4, 5, 2)
    obj = (x * torch.tensor(gl[..., 0], dtype=torch.float64)).sum() + \
          (y * torch.tensor(gl[..., 1], dtype=torch.float64)).sum() + \
          (wt * torch.tensor(gw, dtype=torch.float64)).sum()
    obj.backward()
    np.testing.assert_allclose(gkp, kp.grad.numpy(), rtol=1e-5, atol=1e-6)
    np.testing.assert_allclose(glg, z.grad.numpy(), rtol=1e-5, atol=1e-7)


def test_end_to_end_single_camera_matches_grid_sample_autograd():
    """One camera, one scale: out = sum_p softmax(z)_p * grid_sample(map, 2*(x, y) - 1)."""
    B, A, P, C, G = 1, 12, 5, 16, 2
    H, W = 24, 40
    image_w, image_h = 4.0 * W, 4.0 * H
    rng = np.random.default_rng(5)
    D = C // G
    feat = rng.standard_normal((B, H * W, C)).astype(np.float32)
    proj = da_inputs.camera_rig(1, image_w, image_h, focal_px=120.0).astype(np.float32)[None]
    kp = np.stack([rng.uniform(6, 30, (B, A, P)), rng.uniform(-8, 8, (B, A, P)), rng.uniform(-1, 3, (B, A, P))],
                  -1).astype(np.float32)
    z = rng.standard_normal((B, A, P, 1, 1, G)).astype(np.float32)
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    ss = np.array([[[H, W]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    out, loc, _ = oracle.forward_projected(feat, ss, ls, kp, proj, image_w, image_h, z)
    gf, gl, gw, gkp, glg = oracle.backward_projected(feat, ss, ls, kp, proj, image_w, image_h, z, go)
    inside = ((loc >= 0) & (loc <= 1)).all(-1)
    assert inside.mean() > 0.5

    f = torch.tensor(feat, dtype=torch.float64).view(B, H, W, C).permute(0, 3, 1, 2).requires_grad_(True)
    t_kp = torch.tensor(kp, dtype=torch.float64).requires_grad_(True)
    t_z = torch.tensor(z, dtype=torch.float64).requires_grad_(True)
    M = torch.tensor(proj[0, 0], dtype=torch.float64)
    q = t_kp @ M[:3, :3].T + M[:3, 3]
    xy = torch.stack([q[..., 0] / q[..., 2] / image_w, q[..., 1] / q[..., 2] / image_h], -1)  # [B, A, P, 2]
    samp = torch.nn.functional.grid_sample(f, (2 * xy - 1).view(B, A * P, 1, 2), mode="bilinear",
                                           padding_mode="zeros", align_corners=False)
    samp = samp.view(B, G, D, A, P).permute(0, 3, 4, 1, 2)  # [B, A, P, G, D]
    wt = t_z.view(B, A, P, G).softmax(2)
    ref = (wt[..., None] * samp).sum(2).reshape(B, A, C)
    ref.backward(torch.tensor(go, dtype=torch.float64))
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gf, f.grad.permute(0, 2, 3, 1).reshape(B, H * W, C).numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(glg.reshape(B, A, P, G), t_z.grad.view(B, A, P, G).numpy(), rtol=1e-4, atol=1e-5)
    np.testing.assert_allclose(gkp, t_kp.grad.numpy(), rtol=1e-3, atol=1e-4)
