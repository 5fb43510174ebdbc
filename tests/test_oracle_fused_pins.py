"""Pins for the oracle of the DCNv4 form (per-group locations fused with the
weights; oracle.forward_fused / oracle.backward_fused).

The DCNv4 page writes the operator as y_g(p0) = sum_k m_gk x_g(p0 + p_k + dp_gk)
("Defining the problem"): the groups are independent, and each uses only its
own channels, points and weights. Two facts pin the fused oracle without
reference to itself:
  * the per-group split: group g's output channels equal the standard
    (already pinned) oracle run on that group's channel slice, with that
    group's locations and weights, and the gradients split the same way;
  * the library special case: with one camera and one scale every group is a
    torch grid_sample of its channel slice at its own grid, and autograd of
    that gives every gradient.
A swapped group index, a location read from another group, a transposed
(x, y) pair or a weight read at the wrong scale breaks one of them.
"""
import numpy as np
import pytest
import torch

import oracle


def _tables(shapes_ks):
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


def _problem(seed, shapes_ks, B, C, G, A, P, lo=-0.2, hi=1.2):
    rng = np.random.default_rng(seed)
    ss, ls, rows = _tables(shapes_ks)
    K, S = ss.shape[:2]
    feat = rng.standard_normal((B, rows, C)).astype(np.float32)
    lw = np.empty((B, A, G, P, K, 2 + S), np.float32)
    lw[..., :2] = rng.uniform(lo, hi, (B, A, G, P, K, 2))
    lw[..., 2:] = rng.standard_normal((B, A, G, P, K, S))
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    return feat, ss, ls, lw, go


def _split_group(lw, g):
    """Group g's locations [B,A,P,K,2] and weights [B,A,P,K,S,1]."""
    loc = np.ascontiguousarray(lw[:, :, g, :, :, :2])
    w = np.ascontiguousarray(lw[:, :, g, :, :, 2:])[..., None]
    return loc, w


@pytest.mark.parametrize("shapes,B,C,G,A,P", [
    ([[(7, 9), (3, 5)], [(6, 11), (2, 2)]], 2, 32, 4, 5, 3),
    ([[(12, 10)]], 1, 16, 2, 9, 9),
    ([[(5, 6), (3, 3), (1, 2)]], 2, 24, 3, 4, 2),
])
def test_fused_equals_per_group_standard_operator(shapes, B, C, G, A, P):
    feat, ss, ls, lw, go = _problem(1, shapes, B, C, G, A, P)
    D = C // G
    out = oracle.forward_fused(feat, ss, ls, lw)
    gf, glw = oracle.backward_fused(feat, ss, ls, lw, go)
    for g in range(G):
        sl = slice(g * D, (g + 1) * D)
        loc, w = _split_group(lw, g)
        fs = np.ascontiguousarray(feat[..., sl])
        np.testing.assert_array_equal(out[..., sl], oracle.forward(fs, ss, ls, loc, w))
        gf_g, gl_g, gw_g = oracle.backward(fs, ss, ls, loc, w, np.ascontiguousarray(go[..., sl]))
        np.testing.assert_array_equal(gf[..., sl], gf_g)
        # (x, y) gradients sum over scales and channels in another grouping
        # of the same double-precision terms: equal up to the final rounding.
        np.testing.assert_allclose(glw[:, :, g, :, :, :2], gl_g, rtol=3e-7, atol=1e-6)
        np.testing.assert_array_equal(glw[:, :, g, :, :, 2:], gw_g[..., 0])


def test_groups_do_not_see_each_others_points():
    # Moving group 1's points changes group 1's channels only.
    feat, ss, ls, lw, go = _problem(2, [[(8, 8)]], 1, 16, 2, 6, 4)
    out = oracle.forward_fused(feat, ss, ls, lw)
    lw2 = lw.copy()
    lw2[:, :, 1, :, :, :2] = np.random.default_rng(3).uniform(0, 1, lw2[:, :, 1, :, :, :2].shape)
    out2 = oracle.forward_fused(feat, ss, ls, lw2)
    np.testing.assert_array_equal(out[..., :8], out2[..., :8])
    assert not np.allclose(out[..., 8:], out2[..., 8:])


@pytest.mark.parametrize("B,H,W,C,G,A,P", [(2, 11, 17, 16, 4, 6, 9), (1, 14, 14, 8, 2, 20, 3)])
def test_fused_single_map_matches_grid_sample_per_group(B, H, W, C, G, A, P):
    """One camera, one scale: group g's output is sum_p w_gp * grid_sample of
    channels [gD, (g+1)D) at grid 2*(x, y) - 1 (bilinear, zero padding,
    align_corners=False). Autograd gives grad_feat, the location gradients
    (2 * grad_grid) and the weight gradients."""
    rng = np.random.default_rng(29)
    D = C // G
    feat = rng.standard_normal((B, H * W, C)).astype(np.float32)
    lw = np.empty((B, A, G, P, 1, 3), np.float32)
    lw[..., :2] = rng.uniform(-0.1, 1.1, (B, A, G, P, 1, 2))
    lw[..., 2] = rng.standard_normal((B, A, G, P, 1))
    go = rng.standard_normal((B, A, C)).astype(np.float32)
    ss = np.array([[[H, W]]], np.int32)
    ls = np.zeros((1, 1), np.int32)
    out = oracle.forward_fused(feat, ss, ls, lw)
    gf, glw = oracle.backward_fused(feat, ss, ls, lw, go)

    f = torch.tensor(feat, dtype=torch.float64).view(B, H, W, C).permute(0, 3, 1, 2).requires_grad_(True)
    t_lw = torch.tensor(lw, dtype=torch.float64).requires_grad_(True)
    outs = []
    for g in range(G):
        grid = 2.0 * t_lw[:, :, g, :, 0, :2].reshape(B, A * P, 1, 2) - 1.0
        samp = torch.nn.functional.grid_sample(f[:, g * D:(g + 1) * D], grid, mode="bilinear",
                                               padding_mode="zeros", align_corners=False)  # [B, D, A*P, 1]
        samp = samp.view(B, D, A, P).permute(0, 2, 3, 1)  # [B, A, P, D]
        outs.append((t_lw[:, :, g, :, 0, 2][..., None] * samp).sum(2))  # [B, A, D]
    ref = torch.cat(outs, dim=-1)
    ref.backward(torch.tensor(go, dtype=torch.float64))
    np.testing.assert_allclose(out, ref.detach().numpy(), rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(gf, f.grad.permute(0, 2, 3, 1).reshape(B, H * W, C).numpy(), rtol=1e-5,
                               atol=1e-5)
    # d/d(grid) -> d/d(loc): grid = 2*loc - 1, and autograd already applied it.
    np.testing.assert_allclose(glw[..., :2], t_lw.grad[..., :2].numpy(), rtol=1e-4, atol=1e-3)
    np.testing.assert_allclose(glw[..., 2], t_lw.grad[..., 2].numpy(), rtol=1e-5, atol=1e-5)
