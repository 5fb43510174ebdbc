"""Host-side checks of the C ABI; no GPU is needed and nothing is launched.

* libda.so builds (nvcc cross-compiles) and loads.
* It exports every function that include/da.h declares.
* Argument validation returns the documented status codes.
Every call here fails validation, or has nothing to do, before any CUDA call.
Fake device addresses are safe for that reason: they are never dereferenced.
"""
import ctypes
import os
import re
import subprocess

import pytest

import deformable_view_feature_gb300 as da

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "da.h")

DA_OK, DA_ERR_NULL, DA_ERR_SHAPE, DA_ERR_ALIGN, DA_ERR_UNSUPPORTED = 0, 1, 2, 3, 4
FAKE = 0x7F0000000000  # 256-byte aligned stand-in for a device address


@pytest.fixture(scope="module")
def lib():
    da.build.build()
    return da.load_library()


def _declared_functions():
    names = set()
    for h in sorted(os.listdir(os.path.dirname(HEADER))):
        if h.endswith(".h"):
            text = open(os.path.join(os.path.dirname(HEADER), h)).read()
            text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
            names |= set(re.findall(r"\b((?:da|wa)_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_library_exports_every_declared_function(lib):
    names = _declared_functions()
    assert {"da_forward", "da_backward", "da_status_string", "da_last_error", "da_version",
            "wa_warpaffine_u8", "wa_preprocess"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", da.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\bT ((?:da|wa)_\w+)", out))
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared in da.h but not exported: {missing}"
    for n in names:
        getattr(lib, n)  # resolvable through ctypes


def test_header_compiles_as_plain_c(tmp_path):
    src = tmp_path / "use.c"
    src.write_text('#include "da.h"\n#include "wa.h"\n'
                   'int main(void){ da_dims d = {0}; wa_dims w = {0}; (void)d; (void)w; return (int)DA_OK; }\n')
    subprocess.run(["gcc", "-std=c99", "-Wall", "-Werror", "-I", os.path.dirname(HEADER), "-c",
                    str(src), "-o", str(tmp_path / "use.o")], check=True)


def test_status_strings_and_version(lib):
    assert lib.da_status_string(0) == b"DA_OK"
    assert lib.da_status_string(4) == b"DA_ERR_UNSUPPORTED"
    assert lib.da_version() >= 100


def _dims(**kw):
    d = dict(batch=1, num_cams=1, num_scales=1, num_embeds=32, num_groups=1, num_anchors=4,
             num_pts=2, feat_dtype=0, num_feat_rows=16)
    d.update(kw)
    return da.DaDims(**d)


def _tables(H=4, W=4, start=0):
    ss = (ctypes.c_int32 * 2)(H, W)
    ls = (ctypes.c_int32 * 1)(start)
    return ss, ls


def _fwd(lib, dims, ss=None, ls=None, feat=FAKE, loc=FAKE, w=FAKE, out=FAKE):
    if ss is None:
        ss, ls = _tables()
    return lib.da_forward(ctypes.byref(dims) if dims is not None else None, feat, ss, ls, loc, w,
                          out, None)


def _bwd(lib, dims, feat=FAKE, loc=FAKE, w=FAKE, go=FAKE, gf=FAKE, gl=FAKE, gw=FAKE, ws=None,
         ws_bytes=0):
    ss, ls = _tables()
    return lib.da_backward(ctypes.byref(dims), feat, ss, ls, loc, w, go, gf, gl, gw, ws, ws_bytes, None)


def test_null_dims(lib):
    assert _fwd(lib, None) == DA_ERR_NULL


@pytest.mark.parametrize("kw", [dict(batch=-1), dict(num_groups=3), dict(num_embeds=0),
                                dict(feat_dtype=7), dict(num_feat_rows=-5),
                                dict(num_feat_rows=(1 << 30) + 1)])
def test_bad_sizes(lib, kw):
    assert _fwd(lib, _dims(**kw)) == DA_ERR_SHAPE
    assert b"" != lib.da_last_error()


def test_map_must_fit_rows(lib):
    ss, ls = _tables(H=4, W=5)  # 20 rows > 16
    assert _fwd(lib, _dims(), ss, ls) == DA_ERR_SHAPE
    ss, ls = _tables(H=0, W=5)
    assert _fwd(lib, _dims(), ss, ls) == DA_ERR_SHAPE
    ss, ls = _tables(start=-1)
    assert _fwd(lib, _dims(), ss, ls) == DA_ERR_SHAPE


@pytest.mark.parametrize("C,G,dt", [(12, 1, 0), (64, 1, 0), (8, 2, 1), (256, 2, 1), (40, 2, 0)])
def test_unsupported_group_width(lib, C, G, dt):
    assert _fwd(lib, _dims(num_embeds=C, num_groups=G, feat_dtype=dt)) == DA_ERR_UNSUPPORTED
    assert b"group width" in lib.da_last_error()


def test_too_many_maps(lib):
    ss = (ctypes.c_int32 * (2 * 65))(*([1, 1] * 65))
    ls = (ctypes.c_int32 * 65)(*range(65))
    d = _dims(num_cams=65, num_feat_rows=65)
    assert _fwd(lib, d, ss, ls) == DA_ERR_UNSUPPORTED


def test_null_pointers(lib):
    assert _fwd(lib, _dims(), feat=None) == DA_ERR_NULL
    assert _fwd(lib, _dims(), loc=None) == DA_ERR_NULL
    assert _fwd(lib, _dims(), out=None) == DA_ERR_NULL
    assert _bwd(lib, _dims(), go=None) == DA_ERR_NULL
    assert _bwd(lib, _dims(), gf=None) == DA_ERR_NULL
    assert _bwd(lib, _dims(), gl=None) == DA_ERR_NULL
    assert _bwd(lib, _dims(), gw=None) == DA_ERR_NULL
    ss, ls = _tables()
    assert lib.da_forward(ctypes.byref(_dims()), FAKE, None, ls, FAKE, FAKE, FAKE, None) == DA_ERR_NULL


def test_misaligned_pointers(lib):
    assert _fwd(lib, _dims(), feat=FAKE + 4) == DA_ERR_ALIGN
    assert _fwd(lib, _dims(), loc=FAKE + 4) == DA_ERR_ALIGN
    assert _fwd(lib, _dims(), w=FAKE + 2) == DA_ERR_ALIGN
    assert _fwd(lib, _dims(), out=FAKE + 8) == DA_ERR_ALIGN
    assert _bwd(lib, _dims(), go=FAKE + 8) == DA_ERR_ALIGN
    assert _bwd(lib, _dims(), gf=FAKE + 8) == DA_ERR_ALIGN
    assert _bwd(lib, _dims(), gl=FAKE + 2) == DA_ERR_ALIGN
    assert _bwd(lib, _dims(), gw=FAKE + 1) == DA_ERR_ALIGN


def test_workspace_size_and_errors(lib):
    n = ctypes.c_size_t(0)
    d = _dims(batch=6, num_cams=6, num_scales=4, num_embeds=256, num_groups=8, num_anchors=900,
              num_pts=13, num_feat_rows=6 * 14960)
    assert lib.da_backward_workspace_size(ctypes.byref(d), ctypes.byref(n)) == DA_OK
    nsid = 6 * 900 * 13 * 6 * 4
    # records (key + weight) and dpix for 8 groups: 4*nsid*(4+4) + 4*nsid*8*4,
    # plus the deterministic sort's row lists (rows of > 8, > 128, > 2048 records)
    # and the pull's leftover-row list (one int32 per feature row)
    ncap = 4 * nsid
    lists = 4 * (ncap // 9 + ncap // 129 + ncap // 2049 + 3) + 4 * 6 * 14960
    assert n.value >= nsid * (32 + 128) + lists
    assert n.value < nsid * (32 + 128) + lists + 4 * 1024 * 1024
    assert lib.da_backward_workspace_size(None, ctypes.byref(n)) == DA_ERR_NULL
    big = _dims(batch=1 << 20, num_anchors=1 << 10, num_pts=4)
    assert lib.da_backward_workspace_size(ctypes.byref(big), ctypes.byref(n)) == DA_ERR_UNSUPPORTED
    # too small / misaligned workspace: rejected before any launch
    assert _bwd(lib, _dims(), ws=FAKE, ws_bytes=16) == 6
    assert _bwd(lib, _dims(), ws=FAKE + 16, ws_bytes=1 << 30) == 6
    assert lib.da_status_string(6) == b"DA_ERR_WORKSPACE"


def test_backward_ex_flags(lib):
    vp = ctypes.c_void_p
    lib.da_backward_ex.argtypes = [ctypes.POINTER(da.DaDims)] + [vp] * 10 + [ctypes.c_size_t, ctypes.c_uint32, vp]
    ss, ls = _tables()

    def call(flags, ws=None, ws_bytes=0):
        return lib.da_backward_ex(ctypes.byref(_dims()), FAKE, ss, ls, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, ws,
                                  ws_bytes, flags, None)
    assert call(4) == DA_ERR_SHAPE  # unknown flag
    assert b"flags" in lib.da_last_error()
    assert call(1) == 6  # deterministic without a workspace
    assert b"DETERMINISTIC" in lib.da_last_error()
    assert call(1, FAKE, 16) == 6  # workspace too small


def test_empty_problem_needs_no_pointers(lib):
    """With B = 0 every tensor is empty: NULL pointers are fine and nothing is
    enqueued (no CUDA call is made, so this passes without a GPU)."""
    d = _dims(batch=0)
    assert _fwd(lib, d, feat=None, loc=None, w=None, out=None) == DA_OK
    assert _bwd(lib, d, feat=None, loc=None, w=None, go=None, gf=None, gl=None, gw=None) == DA_OK


def test_binding_rejects_host_tensors():
    import torch
    feat = torch.zeros(1, 16, 32)
    loc = torch.zeros(1, 4, 2, 1, 2)
    w = torch.zeros(1, 4, 2, 1, 1, 1)
    with pytest.raises((ValueError, RuntimeError)):
        da.da_forward(feat, [[[4, 4]]], [[0]], loc, w, out=torch.zeros(1, 4, 32))


def test_pipeline_validation_before_any_cuda_call(lib):
    vp = ctypes.c_void_p
    lib.da_pipeline_create.argtypes = [ctypes.POINTER(da.DaDims), vp, vp, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(vp)]
    lib.da_pipeline_submit.argtypes = [vp] * 9
    lib.da_pipeline_sync.argtypes = [vp]
    lib.da_pipeline_destroy.argtypes = [vp]
    ss, ls = _tables()
    h = vp(None)
    assert lib.da_pipeline_create(ctypes.byref(_dims()), ss, ls, 1, 2, None) == DA_ERR_NULL
    assert lib.da_pipeline_create(ctypes.byref(_dims()), ss, ls, 1, 0, ctypes.byref(h)) == DA_ERR_SHAPE
    assert lib.da_pipeline_create(ctypes.byref(_dims()), ss, ls, 1, 5, ctypes.byref(h)) == DA_ERR_SHAPE
    assert lib.da_pipeline_create(ctypes.byref(_dims()), ss, ls, 2, 2, ctypes.byref(h)) == DA_ERR_SHAPE
    assert lib.da_pipeline_create(ctypes.byref(_dims(num_groups=3)), ss, ls, 1, 2, ctypes.byref(h)) == DA_ERR_SHAPE
    big_ss, big_ls = _tables(H=4, W=5)  # 20 rows > 16
    assert lib.da_pipeline_create(ctypes.byref(_dims()), big_ss, big_ls, 0, 2, ctypes.byref(h)) == DA_ERR_SHAPE
    assert lib.da_pipeline_create(ctypes.byref(_dims(num_embeds=12)), ss, ls, 0, 2,
                                  ctypes.byref(h)) == DA_ERR_UNSUPPORTED
    assert not h.value  # nothing was created
    assert lib.da_pipeline_submit(None, *([None] * 8)) == DA_ERR_NULL
    assert lib.da_pipeline_sync(None) == DA_ERR_NULL
    assert lib.da_pipeline_destroy(None) == DA_OK


@pytest.mark.skipif(__import__("torch").cuda.is_available(), reason="checks the behaviour without a GPU")
def test_pipeline_create_without_gpu_fails_cleanly(lib):
    vp = ctypes.c_void_p
    lib.da_pipeline_create.argtypes = [ctypes.POINTER(da.DaDims), vp, vp, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(vp)]
    ss, ls = _tables()
    h = vp(None)
    assert lib.da_pipeline_create(ctypes.byref(_dims()), ss, ls, 1, 2, ctypes.byref(h)) == 5  # DA_ERR_CUDA
    assert not h.value
    assert b"pipeline set-up" in lib.da_last_error()


def test_binding_signatures_reach_validation(lib):
    """Every entry point called through the argtypes the Python binding
    declares: arguments that fail validation come back as the documented
    status before any CUDA call, which also checks the declared argument
    counts."""
    bl = da.load_library()
    ss, ls = _tables()
    d = ctypes.byref(_dims())
    F = FAKE
    # Fused layout: a misaligned loc_weight.
    assert bl.da_forward_fused(d, F, ss, ls, F + 2, F, None) == DA_ERR_ALIGN
    assert bl.da_backward_fused(d, F, ss, ls, F + 2, F, F, F, None, 0, None) == DA_ERR_ALIGN
    # Projected layout: a zero image width.
    assert bl.da_forward_projected(d, F, ss, ls, F, F, 0.0, 4.0, F, F, None, None, None) == DA_ERR_SHAPE
    assert bl.da_backward_projected(d, F, ss, ls, F, F, 0.0, 4.0, F, F, F, F, F, F, F, F, None, 0, 0,
                                    None) == DA_ERR_SHAPE
    assert bl.da_backward_ex(d, F, ss, ls, F, F, F, F, F, F, None, 0, 4, None) == DA_ERR_SHAPE
    assert b"flags" in bl.da_last_error()


def test_warpaffine_validation_without_gpu(lib):
    bl = da.load_library()
    bad = da.WaDims(1, 0, 4, 2, 2)  # zero source height
    assert bl.wa_warpaffine_u8(ctypes.byref(bad), FAKE, FAKE, 0, FAKE, None) == DA_ERR_SHAPE
    ok = da.WaDims(1, 4, 4, 2, 2)
    assert bl.wa_warpaffine_u8(ctypes.byref(ok), FAKE, FAKE + 2, 0, FAKE, None) == DA_ERR_ALIGN
    assert bl.wa_warpaffine_u8(ctypes.byref(ok), None, FAKE, 0, FAKE, None) == DA_ERR_NULL
    mean = (ctypes.c_float * 3)(0.5, 0.5, 0.5)
    std = (ctypes.c_float * 3)(0.2, -1.0, 0.2)
    assert bl.wa_preprocess(ctypes.byref(ok), FAKE, FAKE, 0, mean, std, FAKE, None) == DA_ERR_SHAPE
    assert bl.wa_preprocess(ctypes.byref(ok), FAKE, FAKE, 0, mean, mean, FAKE + 2, None) == DA_ERR_ALIGN
    empty = da.WaDims(0, 4, 4, 2, 2)
    assert bl.wa_warpaffine_u8(ctypes.byref(empty), None, None, 0, None, None) == DA_OK


def test_fused_workspace_size(lib):
    bl = da.load_library()
    n = ctypes.c_size_t(0)
    # The DCNv4 page's benchmark: B=64, one 56x56 map, C=128, G=4, 3136 anchors, 9 points.
    d = _dims(batch=64, num_cams=1, num_scales=1, num_embeds=128, num_groups=4, num_anchors=3136, num_pts=9,
              num_feat_rows=3136)
    assert bl.da_backward_fused_workspace_size(ctypes.byref(d), ctypes.byref(n)) == DA_OK
    nsid = 64 * 3136 * 4 * 9  # samples of the rewrite: one per (anchor, group, point)
    ncap = 4 * nsid
    # records (8 bytes) and d (one group: 4 bytes) per record, plus the sort's row lists
    base = ncap * (8 + 4) + 4 * (ncap // 9 + ncap // 129 + ncap // 2049 + 3)
    assert base <= n.value < base + 4 * 64 * 3136 * 4 + (8 << 20)
    bad = _dims(num_embeds=48, num_groups=4)  # D = 12: not a power of two
    assert bl.da_backward_fused_workspace_size(ctypes.byref(bad), ctypes.byref(n)) == DA_ERR_UNSUPPORTED


def test_binning_entry_validation(lib):
    bl = da.load_library()
    ss, ls = _tables()
    d = ctypes.byref(_dims())
    assert bl.da_backward_bin(d, ss, ls, FAKE, FAKE, 1 << 30, 2, None) == DA_ERR_SHAPE  # READY is not a bin flag
    assert bl.da_backward_bin(d, ss, ls, FAKE + 4, FAKE, 1 << 30, 0, None) == DA_ERR_ALIGN
    assert bl.da_backward_bin(d, ss, ls, FAKE, FAKE, 16, 0, None) == 6  # workspace too small
    # READY without a workspace
    assert bl.da_backward_ex(d, FAKE, ss, ls, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, None, 0, 2, None) == 6


def test_last_error_is_per_thread(lib):
    """da_last_error() reports the calling thread's own last failure: threads
    that fail at the same time with different sizes each read their own
    message (ctypes releases the GIL during the calls, so they interleave)."""
    import threading
    bad = []

    def worker(i):
        rows = -(1000 + i)
        d = _dims(num_feat_rows=rows)
        for _ in range(300):
            if _fwd(lib, d) != DA_ERR_SHAPE:
                bad.append((i, "status"))
                return
            if str(rows).encode() not in lib.da_last_error():
                bad.append((i, lib.da_last_error()))
                return

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not bad, bad[:3]
