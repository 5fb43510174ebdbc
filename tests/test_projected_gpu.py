"""GPU parity of the projected layout (da_forward_projected /
da_backward_projected): key points projected into the cameras and softmax
weights computed inside the forward, and the chain rule back to key points
and logits after the backward.

Stage by stage, against the oracle (pinned in test_oracle_projection_pins.py):
  * the locations the kernel wrote equal the oracle's bit for bit (the same
    fp32 steps; NaN behind a camera), the weights agree to fp32 rounding;
  * out, grad_feat, grad_loc, grad_weight against the oracle run on the
    oracle's locations and weights, with the usual parity tolerances;
  * grad_keypoints and grad_logits against the oracle's chain rule applied to
    the kernel's own grad_loc / grad_weight / weights, with fp32 error bounds
    derived from the chain rule's arithmetic;
  * and end to end against the oracle's chain rule applied to the oracle's
    own weights, grad_loc and grad_weight, with the parity tolerance of those
    carried through the (linear) chain rule.
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle
from parity_util import TOL, conditioning_atol, to_np, violations, widened_violations

pytestmark = pytest.mark.gpu
U32 = 2.0 ** -24


@pytest.fixture(scope="module")
def da():
    import deformable_view_feature_gb300 as m
    m.build.build()
    m.load_library()
    assert torch.cuda.is_available(), "the projected-layout tests need a CUDA GPU"
    return m


def _run(da, inp, path="binned", deterministic=False):
    dev = torch.device("cuda")
    feat, kp, pr, z, go = (t.to(dev) for t in (inp.feat, inp.keypoints, inp.projection, inp.logits, inp.grad_out))
    ss, ls = inp.spatial_shape, inp.level_start_index
    out, loc, w = da.da_forward_projected(feat, ss, ls, kp, pr, inp.image_w, inp.image_h, z)
    gf, gl, gw, gkp, glg = da.da_backward_projected(feat, ss, ls, kp, pr, inp.image_w, inp.image_h, loc, w, go,
                                                    path=path, deterministic=deterministic)
    torch.cuda.synchronize()
    names = ("out", "loc", "weights", "grad_feat", "grad_loc", "grad_weight", "grad_keypoints", "grad_logits")
    return dict(zip(names, (to_np(t) for t in (out, loc, w, gf, gl, gw, gkp, glg))))


def _chain_abs(inp, w, gl_abs, gw_abs):
    """The chain rule applied to magnitudes: (|w| * (gw_abs + sum |w| gw_abs)
    per (b, a, g), and sum over cameras of |J_k|^T gl_abs), the two factors
    that carry an error in grad_weight / grad_loc (or a rounding) into
    grad_logits and grad_keypoints."""
    w = np.abs(np.asarray(w, np.float64))
    gw_abs = np.asarray(gw_abs, np.float64)
    B, A, P, K, S, G = w.shape
    wg = (w * gw_abs).sum(axis=(2, 3, 4), keepdims=True)
    glg = w * (gw_abs + wg)
    kp = inp.keypoints.numpy().astype(np.float64)
    M = inp.projection.numpy().astype(np.float64)
    hom = np.concatenate([kp, np.ones_like(kp[..., :1])], -1)
    q = np.einsum("bkij,bapj->bapki", M[:, :, :3], hom)  # [B, A, P, K, 3]
    d = q[..., 2]
    ok = d > 1e-5
    dd = np.where(ok, d, 1.0)
    uv = q[..., :2] / dd[..., None]
    gl = np.asarray(gl_abs, np.float64)
    size = np.array([inp.image_w, inp.image_h])
    kpb = np.zeros(kp.shape)
    for i in range(3):
        mi = np.abs(M[:, None, None, :, :2, i])  # [B,1,1,K,2]
        m2 = np.abs(M[:, None, None, :, 2, i])[..., None]                # [B,1,1,K,1]
        term = gl * (mi + np.abs(uv) * m2) / (dd[..., None] * size)
        kpb[..., i] = np.where(ok[..., None], term, 0.0).sum(axis=(3, 4))
    return glg, kpb


def _chain_bounds(inp, got):
    """fp32 error bounds of the two chain-rule outputs (per element)."""
    B, A, P, K, S, G = got["weights"].shape
    glg, kpb = _chain_abs(inp, got["weights"], np.abs(got["grad_loc"]), np.abs(got["grad_weight"]))
    return (P * K * S + 8) * U32 * glg, 16 * U32 * kpb


def _check(inp, got):
    feat, ss, ls = inp.feat_numpy(), inp.spatial_shape.numpy(), inp.level_start_index.numpy()
    kp, pr, z, go = inp.keypoints.numpy(), inp.projection.numpy(), inp.logits.numpy(), inp.grad_out.numpy()
    loc = oracle.project(kp, pr, inp.image_w, inp.image_h)
    assert np.array_equal(np.isnan(got["loc"]), np.isnan(loc))
    assert np.array_equal(got["loc"][~np.isnan(loc)], loc[~np.isnan(loc)]), "locations differ"
    w = oracle.softmax_weights(z)
    n, msg = violations(got["weights"], w, 2e-6, 1e-12, "weights")
    assert n == 0, msg
    ref = oracle.run_inputs(da_inputs.Inputs(inp.wl, inp.feat, inp.spatial_shape, inp.level_start_index,
                                             torch.from_numpy(loc), torch.from_numpy(w), inp.grad_out))
    sub = da_inputs.Inputs(inp.wl, inp.feat, inp.spatial_shape, inp.level_start_index, torch.from_numpy(loc),
                           torch.from_numpy(w), inp.grad_out)
    extra = conditioning_atol(sub)
    msgs = []
    for name in ("out", "grad_feat", "grad_loc", "grad_weight"):
        rtol, atol = TOL[inp.wl.feat_dtype][name]
        msgs += widened_violations(got[name], ref[name], rtol, atol, extra.get(name), name)
    gkp, glg = oracle.projected_chain(kp, pr, inp.image_w, inp.image_h, got["weights"], got["grad_loc"],
                                      got["grad_weight"])
    glg_bound, kp_bound = _chain_bounds(inp, got)
    for name, r, bound in (("grad_logits", glg, glg_bound), ("grad_keypoints", gkp, kp_bound)):
        n, msg = violations(got[name], r, 1e-5, 1e-9 + bound, name)
        if n:
            msgs.append(msg)
    # End to end: the oracle's chain rule on the oracle's own weights,
    # grad_loc and grad_weight. The kernel's inputs to the chain may differ
    # from those by their parity tolerance (and the weights by 2e-6
    # relative); the chain carries that difference in linearly, so the bound
    # is the chain applied to the tolerance envelope, plus its own rounding.
    e_gkp, e_glg = oracle.projected_chain(kp, pr, inp.image_w, inp.image_h, w, ref["grad_loc"], ref["grad_weight"])
    tol = {}
    for name in ("grad_loc", "grad_weight"):
        rtol, atol = TOL[inp.wl.feat_dtype][name]
        tol[name] = rtol * np.abs(ref[name].astype(np.float64)) + atol + extra[name].reshape(ref[name].shape)
    p_glg, p_kp = _chain_abs(inp, w, tol["grad_loc"], tol["grad_weight"])
    w_glg, _ = _chain_abs(inp, w, np.zeros_like(tol["grad_loc"]), np.abs(ref["grad_weight"]))
    for name, r, bound in (("grad_logits e2e", e_glg, p_glg + 4e-6 * w_glg + glg_bound),
                           ("grad_keypoints e2e", e_gkp, p_kp + kp_bound)):
        key = name.split()[0]
        n, msg = violations(got[key], r, 1e-5, 1e-9 + bound, name)
        print(f"{name}: max |gpu - oracle| = {np.max(np.abs(got[key] - r)):.3e}, "
              f"max bound = {np.max(bound):.3e}")
        if n:
            msgs.append(msg)
    assert not msgs, " | ".join(msgs)


def test_training_shape_full_size(da):
    inp = da_inputs.make_projected_inputs("sp4d_proj")
    _check(inp, _run(da, inp))


@pytest.mark.parametrize("path,deterministic", [("scatter", False), ("binned", True)])
def test_small_shape_both_backward_paths(da, path, deterministic):
    inp = da_inputs.make_projected_inputs(da_inputs.small_variant("sp4d_proj", batch=2, num_anchors=25), seed=9)
    _check(inp, _run(da, inp, path=path, deterministic=deterministic))


# G = 3 takes the per-(anchor, group) logits kernel; C = 48 is not a power of
# two, so its backward takes the scatter path.
@pytest.mark.parametrize("C,G,path", [(64, 4, "binned"), (48, 3, "scatter")])
def test_one_camera_one_scale_bf16(da, C, G, path):
    wl = da_inputs.WORKLOADS["sp4d_proj"].replace(name="proj_k1", batch=1, num_cams=1, shapes=((32, 80),),
                                                  num_embeds=C, num_groups=G, num_anchors=50, num_pts=7,
                                                  feat_dtype="bf16")
    inp = da_inputs.make_projected_inputs(wl, seed=10)
    _check(inp, _run(da, inp, path=path))


def test_forward_without_kept_samples_gives_the_same_out(da):
    inp = da_inputs.make_projected_inputs(da_inputs.small_variant("sp4d_proj", num_anchors=30), seed=11)
    dev = torch.device("cuda")
    args = (inp.feat.to(dev), inp.spatial_shape, inp.level_start_index, inp.keypoints.to(dev),
            inp.projection.to(dev), inp.image_w, inp.image_h, inp.logits.to(dev))
    a, loc, w = da.da_forward_projected(*args)
    b, none_loc, none_w = da.da_forward_projected(*args, keep_samples=False)
    assert none_loc is None and none_w is None
    assert torch.equal(a, b)
    # And the standard forward on the written samples gives the same result:
    # within the fp32 forward tolerance, since at six cameras the standard
    # forward sums two camera halves (another association of the same sum).
    c = da.da_forward(args[0], inp.spatial_shape, inp.level_start_index, loc, w)
    n, msg = violations(to_np(a), to_np(c), 1e-5, 1e-6, "out")
    assert n == 0, msg


def test_bad_image_size_refused(da):
    inp = da_inputs.make_projected_inputs(da_inputs.small_variant("sp4d_proj", num_anchors=4), seed=12)
    dev = torch.device("cuda")
    with pytest.raises(da.DaError, match="DA_ERR_SHAPE"):
        da.da_forward_projected(inp.feat.to(dev), inp.spatial_shape, inp.level_start_index, inp.keypoints.to(dev),
                                inp.projection.to(dev), 0.0, inp.image_h, inp.logits.to(dev))
