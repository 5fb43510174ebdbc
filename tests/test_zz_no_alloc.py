"""GPU test of da_backward_noalloc, the backward entry point that allocates nothing.

Some callers cannot call cudaMalloc: a runtime whose device memory is fixed at
start-up, a plug-in whose host framework owns all device memory, or code that
cannot take the synchronisation an allocation may cause. For them the library
keeps its backward scratch in a fixed array in device memory.

This test calls that entry point through the C ABI. It checks the result
against the regular da_backward (given a workspace) with the parity
tolerances the other GPU tests use, on two calls in a row: the second call
reuses an array the first one left behind. It also checks that a problem too
large for the array is refused before anything is launched.

The file name puts it last in collection, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import da_inputs
from parity_util import TOL, conditioning_atol, to_np, violations

pytestmark = pytest.mark.gpu


def _lib():
    import deformable_view_feature_gb300 as da
    da.build.build()
    lib = da.load_library()
    vp = ctypes.c_void_p
    lib.da_backward_noalloc.argtypes = [ctypes.POINTER(da.DaDims), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.da_backward_noalloc.restype = ctypes.c_int
    return da, lib


def test_noalloc_matches_da_backward_on_two_calls():
    da, lib = _lib()
    assert torch.cuda.is_available()
    dev = torch.device("cuda", 0)
    # The 6-camera, 4-scale Sparse4D shape at B = 1 fits the built-in scratch.
    inp = da_inputs.make_inputs("sp4d_inf")
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    ss = inp.spatial_shape.contiguous()
    ls = inp.level_start_index.contiguous()
    dims = da._dims(feat, ss, loc, w)
    assert da.backward_workspace_size(dims) <= 64 << 20

    # Reference: the regular entry point with a caller-provided workspace.
    ref = da.da_backward(feat, ss, ls, loc, w, go, path="binned")
    torch.cuda.synchronize(dev)
    ref = {k: to_np(t) for k, t in zip(("grad_feat", "grad_loc", "grad_weight"), ref)}
    extra = conditioning_atol(inp)

    stream = torch.cuda.current_stream(dev).cuda_stream
    for call in range(2):
        gf = torch.full(feat.shape, float("nan"), device=dev)
        gl = torch.full(loc.shape, float("nan"), device=dev)
        gw = torch.full(w.shape, float("nan"), device=dev)
        st = lib.da_backward_noalloc(ctypes.byref(dims), feat.data_ptr(), ss.data_ptr(), ls.data_ptr(),
                                     loc.data_ptr(), w.data_ptr(), go.data_ptr(), gf.data_ptr(),
                                     gl.data_ptr(), gw.data_ptr(), stream or None)
        assert st == 0, lib.da_last_error()
        torch.cuda.synchronize(dev)
        got = {"grad_feat": to_np(gf), "grad_loc": to_np(gl), "grad_weight": to_np(gw)}
        for name, r in ref.items():
            rtol, atol = TOL["f32"][name]
            if name in extra:
                atol = atol + extra[name].reshape(r.shape)
            n, msg = violations(got[name], r, rtol, atol, f"call {call} {name}")
            assert n == 0, msg
            assert np.isfinite(got[name]).all()


def test_noalloc_refuses_problems_larger_than_its_array():
    da, lib = _lib()
    wl = da_inputs.WORKLOADS["sp4d_train"]  # about 300 MB of scratch
    dims = da.DaDims(wl.batch, wl.num_cams, wl.num_scales, wl.num_embeds, wl.num_groups,
                     wl.num_anchors, wl.num_pts, 0, wl.num_feat_rows)
    assert da.backward_workspace_size(dims) > 64 << 20
    fake = 0x7F0000000000  # never dereferenced: the size check comes first
    st = lib.da_backward_noalloc(ctypes.byref(dims), fake, None, None, *([fake] * 6), None)
    assert st == 6  # DA_ERR_WORKSPACE
    assert b"built-in array" in lib.da_last_error()
