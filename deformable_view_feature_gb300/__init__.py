"""GB300 deformable aggregation: thin Python binding of libda.so.

The functions here only marshal arguments. They check tensor shapes, pick the
stream, allocate outputs with torch and call the C ABI (include/da.h). Every
step of the operator runs in the library's CUDA kernels. There is no fallback:
if libda.so has not been built, or the tensors are not on a CUDA device, the
call raises.

    out = da_forward(mc_ms_feat, spatial_shape, level_start_index,
                     sampling_location, weights)
    grad_feat, grad_loc, grad_weight = da_backward(
        mc_ms_feat, spatial_shape, level_start_index, sampling_location,
        weights, grad_out)

``DeformableAggregationFunction`` wraps the two as a torch autograd function.
It takes the inputs of the op of the same name on the page "Inside Sparse4D's
CUDA core" (§6).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional, Tuple

import torch

from . import build as _build

__all__ = ["da_forward", "da_backward", "da_forward_fused", "da_backward_fused", "da_forward_projected",
           "da_backward_projected", "warpaffine_u8", "warpaffine_preprocess", "backward_workspace_size",
           "backward_path", "da_backward_bin", "DeformableAggregationFunction", "HostPipeline", "DaError", "library_path", "load_library", "da_version"]

DA_F32, DA_BF16, DA_F16 = 0, 1, 2
_STATUS = {0: "DA_OK", 1: "DA_ERR_NULL", 2: "DA_ERR_SHAPE", 3: "DA_ERR_ALIGN",
           4: "DA_ERR_UNSUPPORTED", 5: "DA_ERR_CUDA", 6: "DA_ERR_WORKSPACE", 7: "DA_ERR_DEVICE_BOUNDS"}


class DaError(RuntimeError):
    """A non-OK status from libda.so."""

    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS.get(status, status)}: {message}")
        self.status = status


class DaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("num_cams", ctypes.c_int32),
                ("num_scales", ctypes.c_int32), ("num_embeds", ctypes.c_int32),
                ("num_groups", ctypes.c_int32), ("num_anchors", ctypes.c_int32),
                ("num_pts", ctypes.c_int32), ("feat_dtype", ctypes.c_int32),
                ("num_feat_rows", ctypes.c_int64)]


class WaDims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("src_h", ctypes.c_int32), ("src_w", ctypes.c_int32),
                ("dst_h", ctypes.c_int32), ("dst_w", ctypes.c_int32)]


_lib = None


def library_path() -> str:
    """libda.so, or the bounds-checking libda_debug.so when the environment
    variable DA_DEBUG_BOUNDS is 1 (build it with
    `python -m deformable_view_feature_gb300.build --debug-bounds`)."""
    return _build.DEBUG_LIB if os.environ.get("DA_DEBUG_BOUNDS") == "1" else _build.LIB


def load_library():
    """Load libda.so (it must already be built: ``deformable_view_feature_gb300.build``)."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if not os.path.exists(path):
        raise RuntimeError(f"libda.so is not built ({path}); run "
                           "`python -m deformable_view_feature_gb300.build`")
    lib = ctypes.CDLL(path)
    vp = ctypes.c_void_p
    lib.da_forward.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, vp, vp]
    lib.da_forward.restype = ctypes.c_int
    lib.da_backward.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                ctypes.c_size_t, vp]
    lib.da_backward.restype = ctypes.c_int
    lib.da_backward_ex.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, vp, vp, vp, vp, vp,
                                   ctypes.c_size_t, ctypes.c_uint32, vp]
    lib.da_backward_ex.restype = ctypes.c_int
    lib.da_forward_fused.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, vp]
    lib.da_forward_fused.restype = ctypes.c_int
    lib.da_backward_fused.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_size_t, vp]
    lib.da_backward_fused.restype = ctypes.c_int
    f32 = ctypes.c_float
    lib.da_forward_projected.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, f32, f32, vp, vp, vp, vp, vp]
    lib.da_forward_projected.restype = ctypes.c_int
    lib.da_backward_projected.argtypes = ([ctypes.POINTER(DaDims), vp, vp, vp, vp, vp, f32, f32]
                                          + [vp] * 9 + [ctypes.c_size_t, ctypes.c_uint32, vp])
    lib.da_backward_projected.restype = ctypes.c_int
    lib.wa_warpaffine_u8.argtypes = [ctypes.POINTER(WaDims), vp, vp, ctypes.c_uint8, vp, vp]
    lib.wa_warpaffine_u8.restype = ctypes.c_int
    lib.wa_preprocess.argtypes = [ctypes.POINTER(WaDims), vp, vp, ctypes.c_uint8, vp, vp, vp, vp]
    lib.wa_preprocess.restype = ctypes.c_int
    lib.da_backward_bin.argtypes = [ctypes.POINTER(DaDims), vp, vp, vp, vp, ctypes.c_size_t, ctypes.c_uint32, vp]
    lib.da_backward_bin.restype = ctypes.c_int
    lib.da_backward_fused_workspace_size.argtypes = [ctypes.POINTER(DaDims), ctypes.POINTER(ctypes.c_size_t)]
    lib.da_backward_fused_workspace_size.restype = ctypes.c_int
    lib.da_backward_workspace_size.argtypes = [ctypes.POINTER(DaDims), ctypes.POINTER(ctypes.c_size_t)]
    lib.da_backward_workspace_size.restype = ctypes.c_int
    lib.da_status_string.argtypes = [ctypes.c_int]
    lib.da_status_string.restype = ctypes.c_char_p
    lib.da_last_error.argtypes = []
    lib.da_last_error.restype = ctypes.c_char_p
    lib.da_version.argtypes = []
    lib.da_version.restype = ctypes.c_int32
    lib.da_pipeline_create.argtypes = [ctypes.POINTER(DaDims), vp, vp, ctypes.c_int32, ctypes.c_int32,
                                       ctypes.POINTER(vp)]
    lib.da_pipeline_create.restype = ctypes.c_int
    lib.da_pipeline_submit.argtypes = [vp] * 9
    lib.da_pipeline_submit.restype = ctypes.c_int
    lib.da_pipeline_sync.argtypes = [vp]
    lib.da_pipeline_sync.restype = ctypes.c_int
    lib.da_pipeline_destroy.argtypes = [vp]
    lib.da_pipeline_destroy.restype = ctypes.c_int
    _lib = lib
    return lib


def da_version() -> int:
    return load_library().da_version()


def _check(status: int):
    if status != 0:
        raise DaError(status, load_library().da_last_error().decode(errors="replace"))


def _host_i32(t) -> torch.Tensor:
    """The small map tables travel as host int32 arrays (copied if on a device)."""
    t = torch.as_tensor(t)
    return t.detach().to(device="cpu", dtype=torch.int32).contiguous()


def _dptr(t: Optional[torch.Tensor]) -> Optional[int]:
    if t is None or t.numel() == 0:
        return None
    if not t.is_cuda:
        raise ValueError("device tensors must live on a CUDA device")
    if not t.is_contiguous():
        raise ValueError("tensors must be contiguous")
    return t.data_ptr()


def _stream_handle(stream) -> Optional[int]:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream or None


def _dims(feat: torch.Tensor, ss: torch.Tensor, loc: torch.Tensor, weights: torch.Tensor) -> DaDims:
    if feat.dim() != 3:
        raise ValueError("mc_ms_feat must be [B, rows, C]")
    B, rows, C = feat.shape
    if loc.dim() != 5 or loc.shape[-1] != 2:
        raise ValueError("sampling_location must be [B, A, P, K, 2]")
    _, A, P, K, _ = loc.shape
    if ss.dim() != 3 or ss.shape[0] != K or ss.shape[2] != 2:
        raise ValueError("spatial_shape must be [K, S, 2]")
    S = ss.shape[1]
    if weights.dim() != 6 or tuple(weights.shape[:5]) != (B, A, P, K, S):
        raise ValueError("weights must be [B, A, P, K, S, G]")
    if loc.shape[0] != B:
        raise ValueError("batch sizes differ")
    G = weights.shape[5]
    if feat.dtype == torch.float32:
        dt = DA_F32
    elif feat.dtype == torch.bfloat16:
        dt = DA_BF16
    elif feat.dtype == torch.float16:
        dt = DA_F16
    else:
        raise TypeError("mc_ms_feat must be float32, bfloat16 or float16")
    if loc.dtype != torch.float32 or weights.dtype != torch.float32:
        raise TypeError("sampling_location and weights must be float32")
    return DaDims(B, K, S, C, G, A, P, dt, rows)


def da_forward(mc_ms_feat: torch.Tensor, spatial_shape, level_start_index,
               sampling_location: torch.Tensor, weights: torch.Tensor,
               out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """Forward pass on the current (or given) CUDA stream; returns out [B, A, C] fp32."""
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims(mc_ms_feat, ss, sampling_location, weights)
    if out is None:
        out = torch.empty(d.batch, d.num_anchors, d.num_embeds, device=mc_ms_feat.device,
                          dtype=torch.float32)
    elif out.shape != (d.batch, d.num_anchors, d.num_embeds) or out.dtype != torch.float32:
        raise ValueError("out must be float32 [B, A, C]")
    _check(lib.da_forward(ctypes.byref(d), _dptr(mc_ms_feat), ss.data_ptr() if ss.numel() else None,
                          ls.data_ptr() if ls.numel() else None, _dptr(sampling_location),
                          _dptr(weights), _dptr(out), _stream_handle(stream)))
    return out


def backward_workspace_size(dims: DaDims) -> int:
    """Bytes of device scratch the binned backward needs (da_backward_workspace_size)."""
    n = ctypes.c_size_t(0)
    _check(load_library().da_backward_workspace_size(ctypes.byref(dims), ctypes.byref(n)))
    return n.value


# One reusable workspace per (device, stream): calls on one stream are ordered,
# so they may share it.
_workspaces = {}


def _workspace(device: torch.device, stream_handle, nbytes: int) -> torch.Tensor:
    key = (device.index, stream_handle)
    ws = _workspaces.get(key)
    if ws is None or ws.numel() < nbytes:
        ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)
        _workspaces[key] = ws
    return ws


def da_backward_bin(mc_ms_feat: torch.Tensor, spatial_shape, level_start_index, sampling_location: torch.Tensor,
                    weights: torch.Tensor, workspace: Optional[torch.Tensor] = None, deterministic: bool = False,
                    stream=None) -> torch.Tensor:
    """da_backward_bin: the location-only half of the binned backward, into
    workspace (allocated if None; returned). mc_ms_feat and weights only give
    the sizes. Finish with da_backward(..., path="binned", workspace=...,
    binned_ready=True) ordered after it."""
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims(mc_ms_feat, ss, sampling_location, weights)
    need = backward_workspace_size(d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=sampling_location.device)
    if workspace.numel() < need:
        raise ValueError(f"workspace holds {workspace.numel()} bytes; {need} are needed")
    _check(lib.da_backward_bin(ctypes.byref(d), ss.data_ptr() if ss.numel() else None,
                               ls.data_ptr() if ls.numel() else None, _dptr(sampling_location), _dptr(workspace),
                               workspace.numel(), 1 if deterministic else 0, _stream_handle(stream)))
    return workspace


# Samples per (anchor, group) up to which the scatter backward is the faster
# one: its small-task kernels serve these shapes (the DCNv4 form's 3x3 points,
# the tiny test shapes), and a binned pass costs more than it saves there.
SMALL_TASK_SAMPLES = 16


def backward_path(dims: DaDims) -> str:
    """The backward algorithm path="auto" takes for these sizes: "binned"
    when the binned kernels serve them (C a power of two in [8, 256], D a
    multiple of 8, record indices within int32) and each (anchor, group) has
    more than SMALL_TASK_SAMPLES samples; "scatter" otherwise."""
    if dims.num_pts * dims.num_cams * dims.num_scales <= SMALL_TASK_SAMPLES:
        return "scatter"
    n = ctypes.c_size_t(0)
    st = load_library().da_backward_workspace_size(ctypes.byref(dims), ctypes.byref(n))
    return "binned" if st == 0 else "scatter"


def da_backward(mc_ms_feat: torch.Tensor, spatial_shape, level_start_index,
                sampling_location: torch.Tensor, weights: torch.Tensor, grad_out: torch.Tensor,
                grad_feat: Optional[torch.Tensor] = None, grad_loc: Optional[torch.Tensor] = None,
                grad_weight: Optional[torch.Tensor] = None, stream=None, path: str = "auto",
                workspace: Optional[torch.Tensor] = None,
                deterministic: bool = False,
                binned_ready: bool = False) -> Tuple[torch.Tensor, torch.Tensor, torch.Tensor]:
    """Backward pass; returns (grad_feat fp32, grad_loc, grad_weight).

    path="binned" sorts the corner contributions by feature row in a device
    workspace (allocated through torch and reused, or passed in) and writes
    every grad_feat row once; path="scatter" needs no workspace and scatters
    grad_feat with vector reductions; path="auto" (default) takes the one
    backward_path() names for the sizes. deterministic=True (binned only)
    fixes the order of every row's contributions, so the gradients are the
    same bit for bit on every run (DA_BACKWARD_DETERMINISTIC).
    """
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims(mc_ms_feat, ss, sampling_location, weights)
    if path == "auto":
        path = "binned" if (deterministic or binned_ready) else backward_path(d)
    if (deterministic or binned_ready) and path != "binned":
        raise ValueError("deterministic=True and binned_ready=True need path='binned'")
    if binned_ready and workspace is None:
        raise ValueError("binned_ready=True needs the workspace da_backward_bin filled")
    dev = mc_ms_feat.device
    if tuple(grad_out.shape) != (d.batch, d.num_anchors, d.num_embeds) or grad_out.dtype != torch.float32:
        raise ValueError("grad_out must be float32 [B, A, C]")
    if grad_feat is None:
        grad_feat = torch.empty(mc_ms_feat.shape, device=dev, dtype=torch.float32)
    if grad_loc is None:
        grad_loc = torch.empty(sampling_location.shape, device=dev, dtype=torch.float32)
    if grad_weight is None:
        grad_weight = torch.empty(weights.shape, device=dev, dtype=torch.float32)
    for name, t, shape in (("grad_feat", grad_feat, mc_ms_feat.shape),
                           ("grad_loc", grad_loc, sampling_location.shape),
                           ("grad_weight", grad_weight, weights.shape)):
        if t.shape != shape or t.dtype != torch.float32:
            raise ValueError(f"{name} must be float32 {tuple(shape)}")
    sh = _stream_handle(stream)
    ws_ptr, ws_bytes = None, 0
    if path == "binned":
        need = backward_workspace_size(d)
        if workspace is None:
            workspace = _workspace(mc_ms_feat.device, sh, need)
        ws_bytes = workspace.numel() * workspace.element_size()
        if ws_bytes < need:
            raise ValueError(f"workspace holds {ws_bytes} bytes; {need} are needed")
        ws_ptr = _dptr(workspace)
    elif path != "scatter":
        raise ValueError("path must be 'binned' or 'scatter'")
    _check(lib.da_backward_ex(ctypes.byref(d), _dptr(mc_ms_feat), ss.data_ptr() if ss.numel() else None,
                              ls.data_ptr() if ls.numel() else None, _dptr(sampling_location),
                              _dptr(weights), _dptr(grad_out), _dptr(grad_feat), _dptr(grad_loc),
                              _dptr(grad_weight), ws_ptr, ws_bytes,
                              (1 if deterministic else 0) | (2 if binned_ready else 0), sh))
    return grad_feat, grad_loc, grad_weight


def _hptr(t: Optional[torch.Tensor], name: str, shape, dtype) -> Optional[int]:
    if t is None:
        if int(torch.Size(shape).numel()) == 0:
            return None
        raise ValueError(f"{name} is required")
    if t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if not t.is_contiguous() or tuple(t.shape) != tuple(shape) or t.dtype != dtype:
        raise ValueError(f"{name} must be a contiguous {dtype} host tensor of shape {tuple(shape)}")
    return t.data_ptr() if t.numel() else None


class HostPipeline:
    """da_pipeline_* (include/da.h): steps whose tensors are HOST tensors.

    Each ``submit`` copies a step's inputs to the device, runs the forward
    (and backward), and copies the outputs back into the given host tensors.
    Copies in, kernels and copies out of consecutive steps overlap on three
    streams. Host tensors should be pinned (``tensor.pin_memory()``); the
    outputs are valid, and the inputs may change, after ``sync()``.
    """

    def __init__(self, dims: DaDims, spatial_shape, level_start_index, backward: bool = True,
                 depth: int = 2, device: Optional[torch.device] = None):
        lib = load_library()
        self._ss, self._ls = _host_i32(spatial_shape), _host_i32(level_start_index)
        self.dims = dims
        self.backward = backward
        self._handle = ctypes.c_void_p(None)
        self._inflight = []
        dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        with torch.cuda.device(dev):
            _check(lib.da_pipeline_create(ctypes.byref(dims), self._ss.data_ptr() if self._ss.numel() else None,
                                          self._ls.data_ptr() if self._ls.numel() else None,
                                          int(backward), depth, ctypes.byref(self._handle)))
        self.device = dev

    def shapes(self):
        d = self.dims
        fdt = {DA_BF16: torch.bfloat16, DA_F16: torch.float16}.get(d.feat_dtype, torch.float32)
        S, G = d.num_scales, d.num_groups
        B, A, P, K, C = d.batch, d.num_anchors, d.num_pts, d.num_cams, d.num_embeds
        return {"mc_ms_feat": ((B, d.num_feat_rows, C), fdt),
                "sampling_location": ((B, A, P, K, 2), torch.float32),
                "weights": ((B, A, P, K, S, G), torch.float32),
                "grad_out": ((B, A, C), torch.float32), "out": ((B, A, C), torch.float32),
                "grad_feat": ((B, d.num_feat_rows, C), torch.float32),
                "grad_loc": ((B, A, P, K, 2), torch.float32),
                "grad_weight": ((B, A, P, K, S, G), torch.float32)}

    def submit(self, mc_ms_feat, sampling_location, weights, out, grad_out=None, grad_feat=None,
               grad_loc=None, grad_weight=None):
        if not self._handle:
            raise RuntimeError("pipeline is closed")
        sh = self.shapes()
        args = {"mc_ms_feat": mc_ms_feat, "sampling_location": sampling_location, "weights": weights,
                "grad_out": grad_out, "out": out, "grad_feat": grad_feat, "grad_loc": grad_loc,
                "grad_weight": grad_weight}
        grads = ("grad_out", "grad_feat", "grad_loc", "grad_weight")
        ptrs = {}
        for name, t in args.items():
            if name in grads and not self.backward:
                ptrs[name] = None
                continue
            ptrs[name] = _hptr(t, name, *sh[name])
        _check(load_library().da_pipeline_submit(
            self._handle, ptrs["mc_ms_feat"], ptrs["sampling_location"], ptrs["weights"], ptrs["grad_out"],
            ptrs["out"], ptrs["grad_feat"], ptrs["grad_loc"], ptrs["grad_weight"]))
        # The copies read and write these tensors until the next sync.
        self._inflight.append(tuple(t for t in args.values() if t is not None))

    def sync(self):
        if self._handle:
            _check(load_library().da_pipeline_sync(self._handle))
        self._inflight.clear()

    def close(self):
        if self._handle:
            st = load_library().da_pipeline_destroy(self._handle)
            self._handle = ctypes.c_void_p(None)
            self._inflight.clear()
            _check(st)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _dims_fused(feat: torch.Tensor, ss: torch.Tensor, loc_weight: torch.Tensor) -> DaDims:
    if loc_weight.dim() != 6:
        raise ValueError("loc_weight must be [B, A, G, P, K, 2 + S]")
    B, A, G, P, K, E = loc_weight.shape
    if ss.dim() != 3 or ss.shape[0] != K or ss.shape[2] != 2 or E != 2 + ss.shape[1]:
        raise ValueError("spatial_shape must be [K, S, 2] with loc_weight's last dim 2 + S")
    if loc_weight.dtype != torch.float32:
        raise TypeError("loc_weight must be float32")
    # The standard dims, read off stand-in shapes.
    d = _dims(feat, ss, torch.empty(B, A, P, K, 2, device="meta"),
              torch.empty(B, A, P, K, ss.shape[1], G, device="meta"))
    return d


def da_forward_fused(mc_ms_feat: torch.Tensor, spatial_shape, level_start_index, loc_weight: torch.Tensor,
                     out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The DCNv4 form (da_forward_fused): per-group points fused with their
    weights, loc_weight [B, A, G, P, K, 2 + S] = (x, y, w_0 .. w_{S-1})."""
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims_fused(mc_ms_feat, ss, loc_weight)
    if out is None:
        out = torch.empty(d.batch, d.num_anchors, d.num_embeds, device=mc_ms_feat.device, dtype=torch.float32)
    elif out.shape != (d.batch, d.num_anchors, d.num_embeds) or out.dtype != torch.float32:
        raise ValueError("out must be float32 [B, A, C]")
    _check(lib.da_forward_fused(ctypes.byref(d), _dptr(mc_ms_feat), ss.data_ptr() if ss.numel() else None,
                                ls.data_ptr() if ls.numel() else None, _dptr(loc_weight), _dptr(out),
                                _stream_handle(stream)))
    return out


def da_backward_fused(mc_ms_feat: torch.Tensor, spatial_shape, level_start_index, loc_weight: torch.Tensor,
                      grad_out: torch.Tensor, grad_feat: Optional[torch.Tensor] = None,
                      grad_loc_weight: Optional[torch.Tensor] = None,
                      stream=None, path: str = "scatter") -> Tuple[torch.Tensor, torch.Tensor]:
    """Backward of the DCNv4 form; returns (grad_feat fp32, grad_loc_weight).
    path="binned" takes the gather-form backward (a workspace from torch,
    reused per stream), path="scatter" the vector-reduction one."""
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims_fused(mc_ms_feat, ss, loc_weight)
    dev = mc_ms_feat.device
    if tuple(grad_out.shape) != (d.batch, d.num_anchors, d.num_embeds) or grad_out.dtype != torch.float32:
        raise ValueError("grad_out must be float32 [B, A, C]")
    if grad_feat is None:
        grad_feat = torch.empty(mc_ms_feat.shape, device=dev, dtype=torch.float32)
    if grad_loc_weight is None:
        grad_loc_weight = torch.empty(loc_weight.shape, device=dev, dtype=torch.float32)
    if grad_feat.shape != mc_ms_feat.shape or grad_feat.dtype != torch.float32:
        raise ValueError("grad_feat must be float32 with mc_ms_feat's shape")
    if grad_loc_weight.shape != loc_weight.shape or grad_loc_weight.dtype != torch.float32:
        raise ValueError("grad_loc_weight must be float32 with loc_weight's shape")
    sh = _stream_handle(stream)
    ws_ptr, ws_bytes = None, 0
    if path == "binned":
        n = ctypes.c_size_t(0)
        _check(lib.da_backward_fused_workspace_size(ctypes.byref(d), ctypes.byref(n)))
        ws = _workspace(dev, sh, n.value)
        ws_ptr, ws_bytes = _dptr(ws), ws.numel()
    elif path != "scatter":
        raise ValueError("path must be 'binned' or 'scatter'")
    _check(lib.da_backward_fused(ctypes.byref(d), _dptr(mc_ms_feat), ss.data_ptr() if ss.numel() else None,
                                 ls.data_ptr() if ls.numel() else None, _dptr(loc_weight), _dptr(grad_out),
                                 _dptr(grad_feat), _dptr(grad_loc_weight), ws_ptr, ws_bytes, sh))
    return grad_feat, grad_loc_weight


def _dims_projected(feat, ss, keypoints, logits) -> DaDims:
    if keypoints.dim() != 4 or keypoints.shape[-1] != 3:
        raise ValueError("keypoints must be [B, A, P, 3]")
    if logits.dim() != 6:
        raise ValueError("weight_logits must be [B, A, P, K, S, G]")
    B, A, P, K, S, G = logits.shape
    if tuple(keypoints.shape[:3]) != (B, A, P):
        raise ValueError("keypoints and weight_logits disagree on B, A, P")
    if keypoints.dtype != torch.float32 or logits.dtype != torch.float32:
        raise TypeError("keypoints and weight_logits must be float32")
    return _dims(feat, ss, torch.empty(B, A, P, K, 2, device="meta"), torch.empty(B, A, P, K, S, G, device="meta"))


def da_forward_projected(mc_ms_feat, spatial_shape, level_start_index, keypoints, projection, image_w: float,
                         image_h: float, weight_logits, keep_samples: bool = True, stream=None):
    """Key points projected into the cameras and softmax weights, fused into
    the forward (da_forward_projected). Returns (out, sampling_location,
    weights); the last two are None unless keep_samples (the backward needs
    them)."""
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims_projected(mc_ms_feat, ss, keypoints, weight_logits)
    dev = mc_ms_feat.device
    if tuple(projection.shape) != (d.batch, d.num_cams, 4, 4) or projection.dtype != torch.float32:
        raise ValueError("projection must be float32 [B, K, 4, 4]")
    out = torch.empty(d.batch, d.num_anchors, d.num_embeds, device=dev, dtype=torch.float32)
    loc = w = None
    if keep_samples:
        loc = torch.empty(d.batch, d.num_anchors, d.num_pts, d.num_cams, 2, device=dev, dtype=torch.float32)
        w = torch.empty(weight_logits.shape, device=dev, dtype=torch.float32)
    _check(lib.da_forward_projected(ctypes.byref(d), _dptr(mc_ms_feat), ss.data_ptr() if ss.numel() else None,
                                    ls.data_ptr() if ls.numel() else None, _dptr(keypoints), _dptr(projection),
                                    float(image_w), float(image_h), _dptr(weight_logits), _dptr(out),
                                    _dptr(loc), _dptr(w), _stream_handle(stream)))
    return out, loc, w


def da_backward_projected(mc_ms_feat, spatial_shape, level_start_index, keypoints, projection, image_w: float,
                          image_h: float, sampling_location, weights, grad_out, path: str = "binned",
                          deterministic: bool = False, stream=None):
    """Backward of da_forward_projected: returns (grad_feat, grad_loc,
    grad_weight, grad_keypoints, grad_logits)."""
    lib = load_library()
    ss, ls = _host_i32(spatial_shape), _host_i32(level_start_index)
    d = _dims(mc_ms_feat, ss, sampling_location, weights)
    dev = mc_ms_feat.device
    if tuple(keypoints.shape) != (d.batch, d.num_anchors, d.num_pts, 3) or keypoints.dtype != torch.float32:
        raise ValueError("keypoints must be float32 [B, A, P, 3]")
    if tuple(projection.shape) != (d.batch, d.num_cams, 4, 4) or projection.dtype != torch.float32:
        raise ValueError("projection must be float32 [B, K, 4, 4]")
    gf = torch.empty(mc_ms_feat.shape, device=dev, dtype=torch.float32)
    gl = torch.empty(sampling_location.shape, device=dev, dtype=torch.float32)
    gw = torch.empty(weights.shape, device=dev, dtype=torch.float32)
    gkp = torch.empty(keypoints.shape, device=dev, dtype=torch.float32)
    glg = torch.empty(weights.shape, device=dev, dtype=torch.float32)
    sh = _stream_handle(stream)
    ws_ptr, ws_bytes = None, 0
    if path == "binned":
        need = backward_workspace_size(d)
        ws = _workspace(dev, sh, need)
        ws_ptr, ws_bytes = _dptr(ws), ws.numel()
    elif path != "scatter" or deterministic:
        raise ValueError("path must be 'binned' or 'scatter' (deterministic needs 'binned')")
    _check(lib.da_backward_projected(ctypes.byref(d), _dptr(mc_ms_feat), ss.data_ptr() if ss.numel() else None,
                                     ls.data_ptr() if ls.numel() else None, _dptr(keypoints), _dptr(projection),
                                     float(image_w), float(image_h), _dptr(sampling_location), _dptr(weights),
                                     _dptr(grad_out), _dptr(gf), _dptr(gl), _dptr(gw), _dptr(gkp), _dptr(glg),
                                     ws_ptr, ws_bytes, 1 if deterministic else 0, sh))
    return gf, gl, gw, gkp, glg


def _wa_args(src: torch.Tensor, d2i: torch.Tensor, dst_hw) -> WaDims:
    if src.dim() != 4 or src.shape[-1] != 3 or src.dtype != torch.uint8:
        raise ValueError("src must be uint8 [B, H, W, 3]")
    B, H, W, _ = src.shape
    if tuple(d2i.shape) != (B, 6) or d2i.dtype != torch.float32:
        raise ValueError("d2i must be float32 [B, 6]")
    return WaDims(B, H, W, int(dst_hw[0]), int(dst_hw[1]))


def warpaffine_u8(src: torch.Tensor, d2i: torch.Tensor, dst_hw, fill: int = 114, stream=None) -> torch.Tensor:
    """wa_warpaffine_u8: frames [B, H, W, 3] uint8 warped by the destination ->
    source matrices d2i [B, 6] into [B, Hd, Wd, 3] uint8."""
    lib = load_library()
    d = _wa_args(src, d2i, dst_hw)
    dst = torch.empty(d.batch, d.dst_h, d.dst_w, 3, dtype=torch.uint8, device=src.device)
    _check(lib.wa_warpaffine_u8(ctypes.byref(d), _dptr(src), _dptr(d2i), int(fill), _dptr(dst),
                                _stream_handle(stream)))
    return dst


def warpaffine_preprocess(src: torch.Tensor, d2i: torch.Tensor, dst_hw, fill: int = 114, mean=(0.406, 0.456, 0.485),
                          std=(0.225, 0.224, 0.229), stream=None) -> torch.Tensor:
    """wa_preprocess: warp, BGR -> RGB, (v/255 - mean)/std, HWC -> CHW: [B, 3, Hd, Wd] float32.
    mean and std are in the source's (BGR) channel order."""
    lib = load_library()
    d = _wa_args(src, d2i, dst_hw)
    m = torch.tensor(mean, dtype=torch.float32)
    s = torch.tensor(std, dtype=torch.float32)
    if m.numel() != 3 or s.numel() != 3:
        raise ValueError("mean and std take 3 values")
    dst = torch.empty(d.batch, 3, d.dst_h, d.dst_w, dtype=torch.float32, device=src.device)
    _check(lib.wa_preprocess(ctypes.byref(d), _dptr(src), _dptr(d2i), int(fill), m.data_ptr(), s.data_ptr(),
                             _dptr(dst), _stream_handle(stream)))
    return dst


class DeformableAggregationFunction(torch.autograd.Function):
    """Autograd wrapper with the argument list of Sparse4D's op:
    (mc_ms_feat, spatial_shape, scale_start_index, sampling_location, weights).
    The backward takes da_backward's path="auto": the binned algorithm at the
    Sparse4D shapes, the scatter one for a few samples per anchor and group."""

    @staticmethod
    def forward(ctx, mc_ms_feat, spatial_shape, scale_start_index, sampling_location, weights):
        mc_ms_feat = mc_ms_feat.contiguous()
        sampling_location = sampling_location.contiguous().float()
        weights = weights.contiguous().float()
        ss, ls = _host_i32(spatial_shape), _host_i32(scale_start_index)
        ctx.save_for_backward(mc_ms_feat, sampling_location, weights)
        ctx.tables = (ss, ls)
        return da_forward(mc_ms_feat, ss, ls, sampling_location, weights)

    @staticmethod
    def backward(ctx, grad_output):
        mc_ms_feat, sampling_location, weights = ctx.saved_tensors
        ss, ls = ctx.tables
        gf, gl, gw = da_backward(mc_ms_feat, ss, ls, sampling_location, weights,
                                 grad_output.contiguous().float(), path="auto")
        if mc_ms_feat.dtype != torch.float32:
            gf = gf.to(mc_ms_feat.dtype)
        return gf, None, None, gl, gw
