"""GPU test of the bounds-checking build (libda_debug.so, DA_DEBUG_BOUNDS).

A child process with DA_DEBUG_BOUNDS=1 builds and loads the bounds-checking
library and runs every kind of entry point once on valid inputs: forward,
both backward paths and the deterministic mode, the binning on its own, the
DCNv4 form (both paths, fp16 features), the projected layout, the warpaffine
kernels and a map table with gaps, odd sides and reversed order. With valid
inputs no kernel may compute an index outside its tensor, so every call must
return DA_OK (a set bit in the device error word would come back as
DA_ERR_DEVICE_BOUNDS, raised as DaError), and the results must still match
the CPU oracle. No case here feeds the kernels bad indices.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import numpy as np
import torch
import da_inputs
import oracle
import deformable_view_feature_gb300 as da
from parity_util import TOL, conditioning_atol, to_np, widened_violations

assert da.build.build().endswith("libda_debug.so")
da.load_library()
dev = torch.device("cuda", 0)


def check(inp, got, ref, what):
    extra = conditioning_atol(inp) if "grad_loc" in ref else {}
    msgs = []
    for k in ref:
        rtol, atol = TOL[inp.wl.feat_dtype][k]
        msgs += widened_violations(got[k], ref[k], rtol, atol, extra.get(k), f"{what} {k}")
    assert not msgs, " | ".join(msgs)


def standard(inp, what):
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    ss, ls = inp.spatial_shape, inp.level_start_index
    ref = oracle.run_inputs(inp)
    out = da.da_forward(feat, ss, ls, loc, w)
    for path, det in (("binned", False), ("binned", True), ("scatter", False)):
        gf, gl, gw = da.da_backward(feat, ss, ls, loc, w, go, path=path, deterministic=det)
        got = {"out": to_np(out), "grad_feat": to_np(gf), "grad_loc": to_np(gl), "grad_weight": to_np(gw)}
        check(inp, got, ref, f"{what} {path}{' det' if det else ''}")
    ws = da.da_backward_bin(feat, ss, ls, loc, w)
    da.da_backward(feat, ss, ls, loc, w, go, path="binned", workspace=ws, binned_ready=True)
    torch.cuda.synchronize()


standard(da_inputs.make_inputs(da_inputs.small_variant("sp4d_train", batch=2, num_anchors=24)), "sp4d_train")
standard(da_inputs.make_inputs(da_inputs.small_variant("large_bf16", batch=1, num_anchors=16)), "large_bf16")
standard(da_inputs.make_inputs("tiny"), "tiny")

# A map table with rows outside every map, odd sides and reversed order.
g = torch.Generator().manual_seed(5)
maps = [[(62, 9, 4), (53, 1, 9)], [(13, 5, 7), (3, 3, 3)]]
rows, B, C, G, A, P = 105, 2, 64, 4, 12, 5
ss = torch.tensor([[[H, W] for (_, H, W) in r] for r in maps], dtype=torch.int32)
ls = torch.tensor([[st for (st, _, _) in r] for r in maps], dtype=torch.int32)
wts = torch.softmax(torch.randn(B, A, P * 4, G, generator=g), dim=2).reshape(B, A, P, 2, 2, G)
inp = da_inputs.Inputs(da_inputs.WORKLOADS["tiny"].replace(name="tables"), torch.randn(B, rows, C, generator=g),
                       ss, ls, -0.2 + 1.4 * torch.rand(B, A, P, 2, 2, generator=g), wts,
                       torch.randn(B, A, C, generator=g))
standard(inp, "tables")

# The DCNv4 form, fp16 features, both backward paths.
fi = da_inputs.make_fused_inputs(da_inputs.small_variant("dcnv4", batch=1).replace(feat_dtype="f16"))
feat, lw, go = fi.feat.to(dev), fi.loc_weight.to(dev), fi.grad_out.to(dev)
out = da.da_forward_fused(feat, fi.spatial_shape, fi.level_start_index, lw)
want = oracle.forward_fused(fi.feat_numpy(), fi.spatial_shape.numpy(), fi.level_start_index.numpy(),
                            fi.loc_weight.numpy())
assert np.allclose(to_np(out), want, rtol=1e-5, atol=1e-6)
for path in ("binned", "scatter"):
    da.da_backward_fused(feat, fi.spatial_shape, fi.level_start_index, lw, go, path=path)
torch.cuda.synchronize()

# The projected layout.
pi = da_inputs.make_projected_inputs(da_inputs.small_variant("sp4d_proj", batch=1, num_anchors=16))
feat, kp, pr, z, go = (t.to(dev) for t in (pi.feat, pi.keypoints, pi.projection, pi.logits, pi.grad_out))
out, loc, w = da.da_forward_projected(feat, pi.spatial_shape, pi.level_start_index, kp, pr, pi.image_w,
                                      pi.image_h, z)
da.da_backward_projected(feat, pi.spatial_shape, pi.level_start_index, kp, pr, pi.image_w, pi.image_h, loc, w, go)
torch.cuda.synchronize()

# The warpaffine kernels.
wi = da_inputs.make_warpaffine_inputs(batch=2)
src, d2i = wi.src.to(dev), wi.d2i.to(dev)
da.warpaffine_u8(src, d2i, wi.dst_hw, wi.fill)
da.warpaffine_preprocess(src, d2i, wi.dst_hw, wi.fill)
torch.cuda.synchronize()
print("DEBUG_BOUNDS_OK")
"""


def test_bounds_checking_build_runs_every_entry_point_clean():
    env = dict(os.environ)
    env["DA_DEBUG_BOUNDS"] = "1"
    env["PYTHONPATH"] = os.pathsep.join([ROOT, os.path.join(ROOT, "tests"), env.get("PYTHONPATH", "")])
    r = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=1200)
    assert r.returncode == 0 and "DEBUG_BOUNDS_OK" in r.stdout, (r.stdout[-3000:] + "\n" + r.stderr[-6000:])
