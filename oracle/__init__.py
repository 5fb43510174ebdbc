"""CPU oracle for the deformable-aggregation operator (test infrastructure).

This package wraps ``da_oracle.c``, a plain single-threaded C implementation
of what the operator computes, and ``wa_oracle.c``, the same for the
warpaffine preprocessing kernels, through ctypes. Only these may import it:

* the tests;
* ``__graft_entry__.smoke()``;
* the CPU-baseline and reference legs of ``bench.py``.

The product path (``deformable_view_feature_gb300``) never imports it.

``da_oracle.c`` names the page passages each step follows.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional, Tuple

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "da_oracle.c")
_SRCS = [_SRC, os.path.join(_HERE, "wa_oracle.c")]
_LIB = os.path.join(_HERE, "_build", "libda_oracle.so")

# -ffp-contract=off: the coordinate step must round twice (see da_oracle.c).
CFLAGS = ["-O3", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc into ``oracle/_build``; return the .so path."""
    if (not force and os.path.exists(_LIB)
            and all(os.path.getmtime(_LIB) >= os.path.getmtime(src) for src in _SRCS)):
        return _LIB
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    tmp = _LIB + f".tmp{os.getpid()}"
    subprocess.run(["gcc", *CFLAGS, *_SRCS, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        lib = ctypes.CDLL(build())
        i32, i64, vp = ctypes.c_int, ctypes.c_int64, ctypes.c_void_p
        lib.dao_forward.argtypes = [i32] * 7 + [i64, vp, vp, vp, i32, vp, vp, i64, i64, vp]
        lib.dao_forward.restype = i32
        lib.dao_backward.argtypes = ([i32] * 7 + [i64, vp, vp, vp, i32, vp, vp, vp, i64, i64,
                                                  vp, vp, vp])
        lib.dao_backward.restype = i32
        lib.dao_grad_loc_magnitude.argtypes = ([i32] * 7 + [i64, vp, vp, vp, i32, vp, vp, vp,
                                                            i64, i64, vp])
        lib.dao_grad_loc_magnitude.restype = i32
        lib.dao_row_counts.argtypes = [i32] * 7 + [i64, vp, vp, vp, vp]
        lib.dao_row_counts.restype = i32
        lib.dao_forward_fused.argtypes = [i32] * 7 + [i64, vp, vp, vp, i32, vp, vp]
        lib.dao_forward_fused.restype = i32
        lib.dao_backward_fused.argtypes = [i32] * 7 + [i64, vp, vp, vp, i32, vp, vp, vp, vp]
        lib.dao_backward_fused.restype = i32
        f32 = ctypes.c_float
        lib.dao_project.argtypes = [i32, i32, i32, i32, vp, vp, f32, f32, vp]
        lib.dao_project.restype = i32
        lib.dao_softmax_weights.argtypes = [i32] * 6 + [vp, vp]
        lib.dao_softmax_weights.restype = i32
        lib.dao_projected_chain.argtypes = [i32] * 6 + [vp, vp, f32, f32, vp, vp, vp, vp, vp]
        lib.dao_projected_chain.restype = i32
        lib.wao_warpaffine_u8.argtypes = [i32] * 5 + [vp, vp, ctypes.c_uint8, vp]
        lib.wao_warpaffine_u8.restype = i32
        lib.wao_warpaffine_preprocess.argtypes = [i32] * 5 + [vp, vp, ctypes.c_uint8, vp, vp, vp]
        lib.wao_warpaffine_preprocess.restype = i32
        lib.dao_bilinear.argtypes = [vp, i32, i32, i32, i32, ctypes.c_float, ctypes.c_float]
        lib.dao_bilinear.restype = ctypes.c_double
        _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _prep(feat, spatial_shape, level_start_index, loc, weights):
    feat = np.ascontiguousarray(feat)
    # feat kind passed to the C oracle: 0 fp32, 1 bf16 bits, 2 fp16 bits
    if feat.dtype == np.uint16:
        bf16 = 1
    elif feat.dtype == np.float16:
        feat, bf16 = feat.view(np.uint16), 2
    elif feat.dtype == np.float32:
        bf16 = 0
    else:
        raise TypeError("feat must be float32, float16, or uint16 holding bf16 bits")
    ss = np.ascontiguousarray(spatial_shape, dtype=np.int32)
    ls = np.ascontiguousarray(level_start_index, dtype=np.int32)
    loc = np.ascontiguousarray(loc, dtype=np.float32)
    weights = np.ascontiguousarray(weights, dtype=np.float32)
    B, rows, C = feat.shape
    _, A, P, K, _ = loc.shape
    S = ss.shape[1] if ss.ndim == 3 else 0
    G = weights.shape[-1]
    assert weights.shape == (B, A, P, K, S, G), weights.shape
    assert ss.shape == (K, S, 2) and ls.shape == (K, S)
    return feat, bf16, ss, ls, loc, weights, (B, K, S, C, G, A, P, rows)


def forward(feat, spatial_shape, level_start_index, loc, weights,
            ba_range: Optional[Tuple[int, int]] = None) -> np.ndarray:
    """out [B, A, C] float32 (or [n, C] rows for ``ba_range=(begin, end)``
    over flat anchor index b*A+a)."""
    feat, bf16, ss, ls, loc, weights, dims = _prep(feat, spatial_shape, level_start_index,
                                                   loc, weights)
    B, K, S, C, G, A, P, rows = dims
    lo, hi = (0, B * A) if ba_range is None else ba_range
    out = np.empty((hi - lo, C), dtype=np.float32)
    rc = _load().dao_forward(B, K, S, C, G, A, P, rows, _ptr(ss), _ptr(ls), _ptr(feat), bf16,
                             _ptr(loc), _ptr(weights), lo, hi, _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle forward rejected its arguments (code {rc})")
    return out.reshape(B, A, C) if ba_range is None else out


def backward(feat, spatial_shape, level_start_index, loc, weights, grad_out,
             ba_range: Optional[Tuple[int, int]] = None):
    """(grad_feat [B, rows, C], grad_loc, grad_weight), all float32.

    With ``ba_range``, grad_feat holds the selected anchors' contributions and
    grad_loc / grad_weight hold the selected anchors' rows only.
    """
    feat, bf16, ss, ls, loc, weights, dims = _prep(feat, spatial_shape, level_start_index,
                                                   loc, weights)
    B, K, S, C, G, A, P, rows = dims
    grad_out = np.ascontiguousarray(grad_out, dtype=np.float32)
    assert grad_out.shape == (B, A, C)
    lo, hi = (0, B * A) if ba_range is None else ba_range
    gf = np.empty((B, rows, C), dtype=np.float32)
    gl = np.empty((hi - lo, P, K, 2), dtype=np.float32)
    gw = np.empty((hi - lo, P, K, S, G), dtype=np.float32)
    rc = _load().dao_backward(B, K, S, C, G, A, P, rows, _ptr(ss), _ptr(ls), _ptr(feat), bf16,
                              _ptr(loc), _ptr(weights), _ptr(grad_out), lo, hi,
                              _ptr(gf), _ptr(gl), _ptr(gw))
    if rc != 0:
        raise ValueError(f"oracle backward rejected its arguments (code {rc})")
    if ba_range is None:
        gl = gl.reshape(B, A, P, K, 2)
        gw = gw.reshape(B, A, P, K, S, G)
    return gf, gl, gw


def grad_loc_magnitude(feat, spatial_shape, level_start_index, loc, weights, grad_out):
    """Sum of |terms| of every grad_loc element (an error-bound helper for the
    parity tests; see dao_grad_loc_magnitude in da_oracle.c)."""
    feat, bf16, ss, ls, loc, weights, dims = _prep(feat, spatial_shape, level_start_index,
                                                   loc, weights)
    B, K, S, C, G, A, P, rows = dims
    grad_out = np.ascontiguousarray(grad_out, dtype=np.float32)
    mag = np.empty((B, A, P, K, 2), dtype=np.float32)
    rc = _load().dao_grad_loc_magnitude(B, K, S, C, G, A, P, rows, _ptr(ss), _ptr(ls), _ptr(feat),
                                        bf16, _ptr(loc), _ptr(weights), _ptr(grad_out), 0, B * A,
                                        _ptr(mag))
    if rc != 0:
        raise ValueError(f"oracle magnitude rejected its arguments (code {rc})")
    return mag


def row_counts(feat, spatial_shape, level_start_index, loc, weights):
    """int32 [B, rows]: how many in-map corners of the samples land on each
    feature row (an error-bound helper for the parity tests; see
    dao_row_counts in da_oracle.c)."""
    feat, _, ss, ls, loc, weights, dims = _prep(feat, spatial_shape, level_start_index, loc, weights)
    B, K, S, C, G, A, P, rows = dims
    count = np.empty((B, rows), dtype=np.int32)
    rc = _load().dao_row_counts(B, K, S, C, G, A, P, rows, _ptr(ss), _ptr(ls), _ptr(loc), _ptr(count))
    if rc != 0:
        raise ValueError(f"oracle row counts rejected its arguments (code {rc})")
    return count


def _prep_fused(feat, spatial_shape, level_start_index, loc_weight):
    ss = np.ascontiguousarray(spatial_shape, dtype=np.int32)
    S = ss.shape[1]
    lw = np.ascontiguousarray(loc_weight, dtype=np.float32)
    B, A, G, P, K, E = lw.shape
    assert E == 2 + S, (E, S)
    # The standard-layout checks with stand-in loc/weights of the right shapes.
    feat, kind, ss, ls, _, _, dims = _prep(feat, ss, level_start_index, np.zeros((B, A, P, K, 2), np.float32),
                                           np.zeros((B, A, P, K, S, G), np.float32))
    return feat, kind, ss, ls, lw, dims


def forward_fused(feat, spatial_shape, level_start_index, loc_weight) -> np.ndarray:
    """The DCNv4 form (per-group locations fused with the weights):
    loc_weight [B, A, G, P, K, 2 + S] -> out [B, A, C] float32."""
    feat, kind, ss, ls, lw, dims = _prep_fused(feat, spatial_shape, level_start_index, loc_weight)
    B, K, S, C, G, A, P, rows = dims
    out = np.empty((B, A, C), dtype=np.float32)
    rc = _load().dao_forward_fused(B, K, S, C, G, A, P, rows, _ptr(ss), _ptr(ls), _ptr(feat), kind, _ptr(lw),
                                   _ptr(out))
    if rc != 0:
        raise ValueError(f"oracle fused forward rejected its arguments (code {rc})")
    return out


def backward_fused(feat, spatial_shape, level_start_index, loc_weight, grad_out):
    """(grad_feat [B, rows, C], grad_loc_weight [B, A, G, P, K, 2 + S]) of the DCNv4 form."""
    feat, kind, ss, ls, lw, dims = _prep_fused(feat, spatial_shape, level_start_index, loc_weight)
    B, K, S, C, G, A, P, rows = dims
    grad_out = np.ascontiguousarray(grad_out, dtype=np.float32)
    gf = np.empty((B, rows, C), dtype=np.float32)
    glw = np.empty(lw.shape, dtype=np.float32)
    rc = _load().dao_backward_fused(B, K, S, C, G, A, P, rows, _ptr(ss), _ptr(ls), _ptr(feat), kind, _ptr(lw),
                                    _ptr(grad_out), _ptr(gf), _ptr(glw))
    if rc != 0:
        raise ValueError(f"oracle fused backward rejected its arguments (code {rc})")
    return gf, glw


def project(keypoints, projection, image_w: float, image_h: float) -> np.ndarray:
    """Key points [B, A, P, 3] seen through the cameras [B, K, 4, 4]: the
    normalised locations [B, A, P, K, 2] (NaN behind a camera); see
    dao_project in da_oracle.c for the exact fp32 steps."""
    kp = np.ascontiguousarray(keypoints, dtype=np.float32)
    pr = np.ascontiguousarray(projection, dtype=np.float32)
    B, A, P, _ = kp.shape
    K = pr.shape[1]
    assert pr.shape == (B, K, 4, 4), pr.shape
    loc = np.empty((B, A, P, K, 2), dtype=np.float32)
    if _load().dao_project(B, K, A, P, _ptr(kp), _ptr(pr), float(image_w), float(image_h), _ptr(loc)) != 0:
        raise ValueError("oracle projection rejected its arguments")
    return loc


def softmax_weights(logits) -> np.ndarray:
    """Softmax of logits [B, A, P, K, S, G] over (P, K, S) for every (b, a, g)."""
    z = np.ascontiguousarray(logits, dtype=np.float32)
    B, A, P, K, S, G = z.shape
    w = np.empty_like(z)
    if _load().dao_softmax_weights(B, A, P, K, S, G, _ptr(z), _ptr(w)) != 0:
        raise ValueError("oracle softmax rejected its arguments")
    return w


def projected_chain(keypoints, projection, image_w, image_h, weights, grad_loc, grad_weight):
    """(grad_keypoints [B, A, P, 3], grad_logits [B, A, P, K, S, G]) from the
    operator's grad_loc and grad_weight."""
    kp = np.ascontiguousarray(keypoints, dtype=np.float32)
    pr = np.ascontiguousarray(projection, dtype=np.float32)
    w = np.ascontiguousarray(weights, dtype=np.float32)
    gl = np.ascontiguousarray(grad_loc, dtype=np.float32)
    gw = np.ascontiguousarray(grad_weight, dtype=np.float32)
    B, A, P, K, S, G = w.shape
    gkp = np.empty(kp.shape, dtype=np.float32)
    glg = np.empty(w.shape, dtype=np.float32)
    rc = _load().dao_projected_chain(B, K, S, G, A, P, _ptr(kp), _ptr(pr), float(image_w), float(image_h), _ptr(w),
                                     _ptr(gl), _ptr(gw), _ptr(gkp), _ptr(glg))
    if rc != 0:
        raise ValueError("oracle chain rule rejected its arguments")
    return gkp, glg


def forward_projected(feat, spatial_shape, level_start_index, keypoints, projection, image_w, image_h, logits):
    """The operator fed by the projection and the softmax: (out, loc, weights)."""
    loc = project(keypoints, projection, image_w, image_h)
    w = softmax_weights(logits)
    return forward(feat, spatial_shape, level_start_index, loc, w), loc, w


def backward_projected(feat, spatial_shape, level_start_index, keypoints, projection, image_w, image_h, logits,
                       grad_out):
    """(grad_feat, grad_loc, grad_weight, grad_keypoints, grad_logits)."""
    loc = project(keypoints, projection, image_w, image_h)
    w = softmax_weights(logits)
    gf, gl, gw = backward(feat, spatial_shape, level_start_index, loc, w, grad_out)
    gkp, glg = projected_chain(keypoints, projection, image_w, image_h, w, gl, gw)
    return gf, gl, gw, gkp, glg


def warpaffine_u8(src, d2i, dst_hw, fill: int) -> np.ndarray:
    """src [B, H, W, 3] uint8, d2i [B, 6] (destination -> source) -> [B, Hd, Wd, 3] uint8."""
    src = np.ascontiguousarray(src, dtype=np.uint8)
    d2i = np.ascontiguousarray(d2i, dtype=np.float32).reshape(-1, 6)
    B, H, W, C = src.shape
    assert C == 3 and d2i.shape[0] == B
    Hd, Wd = dst_hw
    dst = np.empty((B, Hd, Wd, 3), np.uint8)
    if _load().wao_warpaffine_u8(B, H, W, Hd, Wd, _ptr(src), _ptr(d2i), int(fill), _ptr(dst)) != 0:
        raise ValueError("oracle warpaffine rejected its arguments")
    return dst


def warpaffine_preprocess(src, d2i, dst_hw, fill: int, mean, std) -> np.ndarray:
    """The fused preprocessing: [B, 3, Hd, Wd] float32, RGB planes normalised."""
    src = np.ascontiguousarray(src, dtype=np.uint8)
    d2i = np.ascontiguousarray(d2i, dtype=np.float32).reshape(-1, 6)
    mean = np.ascontiguousarray(mean, dtype=np.float32)
    std = np.ascontiguousarray(std, dtype=np.float32)
    B, H, W, C = src.shape
    assert C == 3 and d2i.shape[0] == B and mean.shape == (3,) and std.shape == (3,)
    Hd, Wd = dst_hw
    dst = np.empty((B, 3, Hd, Wd), np.float32)
    if _load().wao_warpaffine_preprocess(B, H, W, Hd, Wd, _ptr(src), _ptr(d2i), int(fill), _ptr(mean), _ptr(std),
                                         _ptr(dst)) != 0:
        raise ValueError("oracle preprocess rejected its arguments")
    return dst


def bilinear(fmap: np.ndarray, c: int, x: float, y: float) -> float:
    """One bilinear sample of channel c of an HWC float32 map at normalised (x, y)."""
    fmap = np.ascontiguousarray(fmap, dtype=np.float32)
    H, W, C = fmap.shape
    return _load().dao_bilinear(_ptr(fmap), H, W, C, c, float(x), float(y))


def run_inputs(inp, backward_pass: bool = True, ba_range=None):
    """Run the oracle on a ``da_inputs.Inputs`` draw; returns a dict of arrays."""
    args = (inp.feat_numpy(), inp.spatial_shape.numpy(), inp.level_start_index.numpy(),
            inp.loc.numpy(), inp.weights.numpy())
    res = {"out": forward(*args, ba_range=ba_range)}
    if backward_pass:
        gf, gl, gw = backward(*args, inp.grad_out.numpy(), ba_range=ba_range)
        res.update(grad_feat=gf, grad_loc=gl, grad_weight=gw)
    return res
