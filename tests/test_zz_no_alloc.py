"""GPU test of da_backward_noalloc, the backward entry point that allocates nothing.

Some callers cannot call cudaMalloc: a runtime whose device memory is fixed at
start-up, a plug-in whose host framework owns all device memory, or code that
cannot take the synchronisation an allocation may cause. For them the library
keeps its backward scratch in a fixed array in device memory.

This test calls that entry point through the C ABI, on two checked calls of
one problem with a call on other inputs in between, so the second checked
call finds the array full of another problem's records and counts. Each
checked call must match the CPU oracle with the parity tolerances the other
GPU tests use, and also the regular da_backward given a workspace. A problem
too large for the array must be refused before anything is launched.

The file name puts it last in collection, so a run that stops at the first
failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import da_inputs
import oracle
from parity_util import TOL, conditioning_atol, to_np, widened_violations

pytestmark = pytest.mark.gpu

NAMES = ("grad_feat", "grad_loc", "grad_weight")


def _lib():
    import deformable_view_feature_gb300 as da
    da.build.build()
    lib = da.load_library()
    vp = ctypes.c_void_p
    lib.da_backward_noalloc.argtypes = [ctypes.POINTER(da.DaDims), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.da_backward_noalloc.restype = ctypes.c_int
    return da, lib


def _noalloc(da, lib, inp, dev):
    """One da_backward_noalloc call on inp; outputs start as NaN."""
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    ss = inp.spatial_shape.contiguous()
    ls = inp.level_start_index.contiguous()
    dims = da._dims(feat, ss, loc, w)
    assert da.backward_workspace_size(dims) <= 64 << 20
    gf = torch.full(feat.shape, float("nan"), device=dev)
    gl = torch.full(loc.shape, float("nan"), device=dev)
    gw = torch.full(w.shape, float("nan"), device=dev)
    stream = torch.cuda.current_stream(dev).cuda_stream
    st = lib.da_backward_noalloc(ctypes.byref(dims), feat.data_ptr(), ss.data_ptr(), ls.data_ptr(),
                                 loc.data_ptr(), w.data_ptr(), go.data_ptr(), gf.data_ptr(),
                                 gl.data_ptr(), gw.data_ptr(), stream or None)
    assert st == 0, lib.da_last_error()
    torch.cuda.synchronize(dev)
    return dict(zip(NAMES, (to_np(gf), to_np(gl), to_np(gw))))


def _check(got, ref, extra, what):
    msgs = []
    for name, r in ref.items():
        rtol, atol = TOL["f32"][name]
        assert np.isfinite(got[name]).all(), f"{what} {name}: non-finite output"
        msgs += widened_violations(got[name], r, rtol, atol, extra.get(name), f"{what} {name}")
    assert not msgs, " | ".join(msgs)


def test_noalloc_matches_oracle_and_da_backward_on_two_calls():
    da, lib = _lib()
    assert torch.cuda.is_available()
    dev = torch.device("cuda", 0)
    # The 6-camera, 4-scale Sparse4D shape at B = 1 fits the built-in scratch.
    inp = da_inputs.make_inputs("sp4d_inf")
    # Another draw of the same shape (other locations, weights, grad_out):
    # its call leaves different records, offsets and counts in the array.
    other = da_inputs.make_inputs("sp4d_inf", seed=101)

    want = oracle.run_inputs(inp, backward_pass=True)
    want = {k: want[k] for k in NAMES}
    extra = conditioning_atol(inp)

    # The regular entry point with a caller-provided workspace.
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    ref = da.da_backward(feat, inp.spatial_shape, inp.level_start_index, loc, w, go, path="binned")
    torch.cuda.synchronize(dev)
    ref = dict(zip(NAMES, (to_np(t) for t in ref)))
    _check(ref, want, extra, "da_backward")

    first = _noalloc(da, lib, inp, dev)
    _check(first, want, extra, "noalloc call 1 vs oracle")
    _check(first, ref, extra, "noalloc call 1 vs da_backward")

    between = _noalloc(da, lib, other, dev)
    assert not np.array_equal(between["grad_weight"], first["grad_weight"])

    second = _noalloc(da, lib, inp, dev)
    _check(second, want, extra, "noalloc call 2 vs oracle")
    _check(second, ref, extra, "noalloc call 2 vs da_backward")


def test_noalloc_refuses_problems_larger_than_its_array():
    da, lib = _lib()
    wl = da_inputs.WORKLOADS["sp4d_train"]  # a few hundred MB of scratch
    dims = da.DaDims(wl.batch, wl.num_cams, wl.num_scales, wl.num_embeds, wl.num_groups,
                     wl.num_anchors, wl.num_pts, 0, wl.num_feat_rows)
    assert da.backward_workspace_size(dims) > 64 << 20
    fake = 0x7F0000000000  # never dereferenced: the size check comes first
    st = lib.da_backward_noalloc(ctypes.byref(dims), fake, None, None, *([fake] * 6), None)
    assert st == 6  # DA_ERR_WORKSPACE
    assert b"built-in array" in lib.da_last_error()
