"""Seeded synthetic inputs for the deformable-aggregation operator.

This module holds workload tables and random draws only. None of the
operator's arithmetic (coordinate transform, bilinear weights, sums,
gradients) lives here. The CUDA path's tests and bench, and the CPU oracle's
tests, all draw their inputs from this one module. That way both sides see the
same bytes.

Layouts follow the Sparse4D deformable_aggregation op. The page "Inside
Sparse4D's CUDA core: deformable_aggregation bilinear interpolation and
gradient back-propagation" fixes the HWC layout (§3.1) and the flattened
multi-camera, multi-scale feature tensor built by feature_maps_format (§6):

* ``mc_ms_feat``        [B, K*NPIX, C]   one row per pixel; camera-major,
                                        then scale, then row-major pixels
* ``spatial_shape``     [K, S, 2] int32  (H, W) of map (k, s)
* ``level_start_index`` [K, S]    int32  first row of map (k, s)
* ``sampling_location`` [B, A, P, K, 2]  normalised (x, y); x pairs with W
* ``weights``           [B, A, P, K, S, G]
* ``grad_out``          [B, A, C]

The five workloads mirror the shapes and value distributions the pages work
with: a 16x16 toy; the 6-camera, 4-scale Sparse4D head at inference (B=1) and
training (B=6) sizes; a larger-image bf16-feature variant; and DCNv4-style
dense queries (one anchor per pixel of a 56x56 map, 3x3 grid plus noise,
unnormalised weights, see the DCNv4 page, "Solving the problem: 1. remove
softmax"). No dataset is involved: everything is drawn from a seeded
``torch.Generator``.
"""
from __future__ import annotations

import dataclasses
from typing import Dict, Optional, Tuple

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    num_cams: int
    shapes: Tuple[Tuple[int, int], ...]  # (H, W) per scale, shared by every camera
    num_embeds: int
    num_groups: int
    num_anchors: int
    num_pts: int
    feat_dtype: str  # "f32", "bf16" or "f16"
    loc_kind: str  # "uniform", "dcnv4_grid" or "projected" (make_projected_inputs only)
    loc_lo: float
    loc_hi: float
    weight_kind: str  # "uniform01", "softmax", "normal" or "logits" (make_projected_inputs only)
    weight_sigma: float
    backward: bool
    seed: int
    offset_sigma_px: float = 0.0  # dcnv4_grid only

    @property
    def num_scales(self) -> int:
        return len(self.shapes)

    @property
    def npix(self) -> int:
        return sum(h * w for h, w in self.shapes)

    @property
    def num_feat_rows(self) -> int:
        return self.num_cams * self.npix

    @property
    def depth(self) -> int:
        return self.num_embeds // self.num_groups

    @property
    def num_samples(self) -> int:
        """Bilinear samples per pass: one per (b, a, p, k, s, g), each a D-vector."""
        return (self.batch * self.num_anchors * self.num_pts * self.num_cams
                * self.num_scales * self.num_groups)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


SP4D_SHAPES = ((64, 176), (32, 88), (16, 44), (8, 22))
LARGE_SHAPES = ((80, 200), (40, 100), (20, 50), (10, 25))

WORKLOADS: Dict[str, Workload] = {
    "tiny": Workload("tiny", 1, 1, ((16, 16),), 32, 1, 16, 4, "f32",
                     "uniform", -0.1, 1.1, "uniform01", 0.0, True, 0),
    "sp4d_inf": Workload("sp4d_inf", 1, 6, SP4D_SHAPES, 256, 8, 900, 13, "f32",
                         "uniform", 0.0, 1.0, "softmax", 0.0, False, 1),
    "sp4d_train": Workload("sp4d_train", 6, 6, SP4D_SHAPES, 256, 8, 900, 13, "f32",
                           "uniform", -0.05, 1.05, "softmax", 0.0, True, 2),
    "large_bf16": Workload("large_bf16", 1, 6, LARGE_SHAPES, 256, 8, 1800, 13, "bf16",
                           "uniform", 0.0, 1.0, "softmax", 0.0, True, 3),
    "dcnv4": Workload("dcnv4", 8, 1, ((56, 56),), 64, 4, 56 * 56, 9, "f32",
                      "dcnv4_grid", 0.0, 0.0, "normal", 0.5, True, 4, offset_sigma_px=1.5),
    # The training shape fed from one step upstream: key points, a camera
    # ring and weight logits (make_projected_inputs).
    "sp4d_proj": Workload("sp4d_proj", 6, 6, SP4D_SHAPES, 256, 8, 900, 13, "f32",
                          "projected", 0.0, 0.0, "logits", 0.0, True, 6),
    # The DCNv4 page's kernel benchmark (its Table 10 excerpt, "Solving the
    # problem: 2"): input 56x56x128, batch 64, 4 groups of 32 channels,
    # 3x3 points. Measured in the DCNv4 form (per-group points).
    "dcnv4_table10": Workload("dcnv4_table10", 64, 1, ((56, 56),), 128, 4, 56 * 56, 9, "f32",
                              "dcnv4_grid", 0.0, 0.0, "normal", 0.5, True, 5, offset_sigma_px=1.5),
}

# The order in which the workloads are listed by the project's configuration.
WORKLOAD_ORDER = ("tiny", "sp4d_inf", "sp4d_train", "large_bf16", "dcnv4")


@dataclasses.dataclass
class Inputs:
    """One draw of every operator input, as CPU tensors."""
    wl: Workload
    feat: torch.Tensor  # [B, rows, C] float32 or bfloat16
    spatial_shape: torch.Tensor  # [K, S, 2] int32
    level_start_index: torch.Tensor  # [K, S] int32
    loc: torch.Tensor  # [B, A, P, K, 2] float32
    weights: torch.Tensor  # [B, A, P, K, S, G] float32
    grad_out: Optional[torch.Tensor]  # [B, A, C] float32

    def feat_numpy(self) -> np.ndarray:
        """Feature bytes for a consumer without bf16 support: float32, or the
        raw uint16 bit patterns of bf16 values."""
        if self.feat.dtype == torch.bfloat16:
            return self.feat.view(torch.int16).numpy().view(np.uint16)
        return self.feat.numpy()  # float32 or float16


def map_tables(num_cams: int, shapes) -> Tuple[torch.Tensor, torch.Tensor]:
    """spatial_shape [K,S,2] and level_start_index [K,S] for maps packed
    camera-major, then scale (the feature_maps_format packing)."""
    k_n, s_n = num_cams, len(shapes)
    ss = torch.zeros(k_n, s_n, 2, dtype=torch.int32)
    ls = torch.zeros(k_n, s_n, dtype=torch.int32)
    row = 0
    for k in range(k_n):
        for s, (h, w) in enumerate(shapes):
            ss[k, s, 0] = h
            ss[k, s, 1] = w
            ls[k, s] = row
            row += h * w
    return ss, ls


def _draw_loc(wl: Workload, g: torch.Generator) -> torch.Tensor:
    B, A, P, K = wl.batch, wl.num_anchors, wl.num_pts, wl.num_cams
    if wl.loc_kind == "uniform":
        u = torch.rand(B, A, P, K, 2, generator=g, dtype=torch.float64)
        return (wl.loc_lo + (wl.loc_hi - wl.loc_lo) * u).to(torch.float32)
    if wl.loc_kind == "dcnv4_grid":
        # One anchor per pixel (i, j) of the single map; point p sits on the
        # 3x3 grid around it, plus a Gaussian offset in pixels.
        assert K == 1 and wl.num_scales == 1 and P == 9
        H, W = wl.shapes[0]
        assert A == H * W
        a = torch.arange(A)
        i = (a // W).to(torch.float64).view(1, A, 1)
        j = (a % W).to(torch.float64).view(1, A, 1)
        p = torch.arange(P)
        dy = (p // 3 - 1).to(torch.float64).view(1, 1, P)
        dx = (p % 3 - 1).to(torch.float64).view(1, 1, P)
        off = torch.randn(B, A, P, 2, generator=g, dtype=torch.float64) * wl.offset_sigma_px
        x = (j + 0.5 + dx + off[..., 0]) / W
        y = (i + 0.5 + dy + off[..., 1]) / H
        return torch.stack([x, y], dim=-1).view(B, A, P, 1, 2).to(torch.float32).contiguous()
    raise ValueError(wl.loc_kind)


def _draw_weights(wl: Workload, g: torch.Generator) -> torch.Tensor:
    B, A, P, K, S, G = (wl.batch, wl.num_anchors, wl.num_pts, wl.num_cams,
                        wl.num_scales, wl.num_groups)
    if wl.weight_kind == "uniform01":
        return torch.rand(B, A, P, K, S, G, generator=g, dtype=torch.float32)
    if wl.weight_kind == "normal":
        return (torch.randn(B, A, P, K, S, G, generator=g, dtype=torch.float32)
                * wl.weight_sigma)
    if wl.weight_kind == "softmax":
        # Logits N(0,1), normalised over (P, K, S) for every (b, a, g): the
        # Sparse4D head's weight normalisation. The operator itself never
        # normalises (the DCNv4 page removes softmax altogether).
        z = torch.randn(B, A, P, K, S, G, generator=g, dtype=torch.float64)
        z = z.permute(0, 1, 5, 2, 3, 4).reshape(B, A, G, P * K * S).softmax(-1)
        z = z.reshape(B, A, G, P, K, S).permute(0, 1, 3, 4, 5, 2)
        return z.to(torch.float32).contiguous()
    raise ValueError(wl.weight_kind)


def make_inputs(wl: Workload | str, seed: Optional[int] = None) -> Inputs:
    """Draw every input of ``wl`` from ``torch.Generator().manual_seed(seed)``.

    Draw order is fixed (feat, loc, weights, grad_out), so a workload's bytes
    depend only on its fields and seed.
    """
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    g = torch.Generator().manual_seed(wl.seed if seed is None else seed)
    B, C = wl.batch, wl.num_embeds
    feat = torch.randn(B, wl.num_feat_rows, C, generator=g, dtype=torch.float32)
    if wl.feat_dtype == "bf16":
        feat = feat.to(torch.bfloat16)  # round to nearest even
    elif wl.feat_dtype == "f16":
        feat = feat.to(torch.float16)  # round to nearest even
    ss, ls = map_tables(wl.num_cams, wl.shapes)
    loc = _draw_loc(wl, g)
    w = _draw_weights(wl, g)
    grad_out = torch.randn(B, wl.num_anchors, C, generator=g, dtype=torch.float32)
    return Inputs(wl, feat, ss, ls, loc, w, grad_out)


@dataclasses.dataclass
class FusedInputs:
    """Inputs of the DCNv4 form: every group has its own points, and the
    points and weights share one tensor (the DCNv4 page, "Solving the
    problem: 1": one linear layer yields offsets and weights together)."""
    wl: Workload
    feat: torch.Tensor  # [B, rows, C]
    spatial_shape: torch.Tensor  # [K, S, 2] int32
    level_start_index: torch.Tensor  # [K, S] int32
    loc_weight: torch.Tensor  # [B, A, G, P, K, 2 + S] float32: (x, y, w_0 .. w_{S-1})
    grad_out: torch.Tensor  # [B, A, C] float32

    def feat_numpy(self) -> np.ndarray:
        return Inputs.feat_numpy(self)  # same rule: bf16 travels as its bits


def make_fused_inputs(wl: Workload | str, seed: Optional[int] = None) -> FusedInputs:
    """The workload's draws with per-group points: the location recipe runs
    once per group (in group order), the weight recipe once for all groups,
    and both are packed into loc_weight."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    g = torch.Generator().manual_seed((wl.seed if seed is None else seed) + 1000)
    B, C, G, S = wl.batch, wl.num_embeds, wl.num_groups, wl.num_scales
    feat = torch.randn(B, wl.num_feat_rows, C, generator=g, dtype=torch.float32)
    if wl.feat_dtype == "bf16":
        feat = feat.to(torch.bfloat16)
    elif wl.feat_dtype == "f16":
        feat = feat.to(torch.float16)
    ss, ls = map_tables(wl.num_cams, wl.shapes)
    locs = [_draw_loc(wl, g) for _ in range(G)]  # G x [B, A, P, K, 2]
    w = _draw_weights(wl, g)  # [B, A, P, K, S, G]
    lw = torch.empty(B, wl.num_anchors, G, wl.num_pts, wl.num_cams, 2 + S, dtype=torch.float32)
    for gi in range(G):
        lw[:, :, gi, :, :, :2] = locs[gi]
        lw[:, :, gi, :, :, 2:] = w[..., gi]
    grad_out = torch.randn(B, wl.num_anchors, C, generator=g, dtype=torch.float32)
    return FusedInputs(wl, feat, ss, ls, lw.contiguous(), grad_out)


@dataclasses.dataclass
class ProjectedInputs:
    """Inputs one step upstream of the operator, as the Sparse4D head holds
    them (the Sparse4D page, §1 and §6: 3D anchors' key points are projected
    into the camera views): key points in the ego frame, one 4x4 projection
    matrix per camera, and weight logits that a softmax turns into weights."""
    wl: Workload
    feat: torch.Tensor  # [B, rows, C]
    spatial_shape: torch.Tensor  # [K, S, 2] int32
    level_start_index: torch.Tensor  # [K, S] int32
    keypoints: torch.Tensor  # [B, A, P, 3] float32, metres, ego frame (x forward, y left, z up)
    projection: torch.Tensor  # [B, K, 4, 4] float32, ego point -> (u*d, v*d, d, 1) in pixels
    image_w: float
    image_h: float
    logits: torch.Tensor  # [B, A, P, K, S, G] float32
    grad_out: torch.Tensor  # [B, A, C] float32

    def feat_numpy(self) -> np.ndarray:
        return Inputs.feat_numpy(self)


def camera_rig(num_cams: int, image_w: float, image_h: float, focal_px: float = 300.0,
               height_m: float = 1.6) -> np.ndarray:
    """A ring of num_cams pinhole cameras at the ego origin, height_m above the
    ground, looking out at evenly spaced yaws (the first one straight ahead).
    Returns [K, 4, 4] float64 matrices: ego (X, Y, Z, 1) -> (u*d, v*d, d, 1),
    with the principal point at the image centre. Input construction only."""
    cx, cy = image_w / 2.0, image_h / 2.0
    mats = np.zeros((num_cams, 4, 4))
    t = np.array([0.0, 0.0, height_m])
    for k in range(num_cams):
        yaw = 2.0 * np.pi * k / num_cams
        fwd = np.array([np.cos(yaw), np.sin(yaw), 0.0])
        right = np.array([np.sin(yaw), -np.cos(yaw), 0.0])
        down = np.array([0.0, 0.0, -1.0])
        rows = [focal_px * right + cx * fwd, focal_px * down + cy * fwd, fwd]
        for r, vec in enumerate(rows):
            mats[k, r, :3] = vec
            mats[k, r, 3] = -vec @ t
        mats[k, 3, 3] = 1.0
    return mats


def make_projected_inputs(wl: Workload | str, seed: Optional[int] = None) -> ProjectedInputs:
    """Anchors uniform in a 100 m x 100 m square around the ego car (centres
    0.5 m below to 2 m above the ground); each anchor's P key points spread
    up to +-2 m (x, y) and +-1 m (z) around its centre; a six-camera ring;
    logits N(0, 1). The image is four times the finest map (stride 4)."""
    if isinstance(wl, str):
        wl = WORKLOADS[wl]
    g = torch.Generator().manual_seed((wl.seed if seed is None else seed) + 2000)
    B, C, A, P, K = wl.batch, wl.num_embeds, wl.num_anchors, wl.num_pts, wl.num_cams
    feat = torch.randn(B, wl.num_feat_rows, C, generator=g, dtype=torch.float32)
    if wl.feat_dtype == "bf16":
        feat = feat.to(torch.bfloat16)
    elif wl.feat_dtype == "f16":
        feat = feat.to(torch.float16)
    ss, ls = map_tables(K, wl.shapes)
    image_h, image_w = 4.0 * wl.shapes[0][0], 4.0 * wl.shapes[0][1]
    lo = torch.tensor([-50.0, -50.0, -0.5], dtype=torch.float64)
    hi = torch.tensor([50.0, 50.0, 2.0], dtype=torch.float64)
    centre = lo + (hi - lo) * torch.rand(B, A, 1, 3, generator=g, dtype=torch.float64)
    spread = torch.tensor([2.0, 2.0, 1.0], dtype=torch.float64)
    kp = centre + spread * (2.0 * torch.rand(B, A, P, 3, generator=g, dtype=torch.float64) - 1.0)
    rig = torch.from_numpy(camera_rig(K, image_w, image_h)).to(torch.float32)
    projection = rig.unsqueeze(0).expand(B, K, 4, 4).contiguous()
    logits = torch.randn(B, A, P, K, wl.num_scales, wl.num_groups, generator=g, dtype=torch.float32)
    grad_out = torch.randn(B, A, C, generator=g, dtype=torch.float32)
    return ProjectedInputs(wl, feat, ss, ls, kp.to(torch.float32).contiguous(), projection, image_w, image_h,
                           logits, grad_out)


@dataclasses.dataclass
class WarpAffineInputs:
    """Inputs of the warpaffine preprocessing (the warpaffine page, §3-§4):
    8-bit BGR frames in HWC layout, one destination->source affine matrix per
    frame, the fill value and the per-channel normalisation."""
    src: torch.Tensor  # [B, H, W, 3] uint8
    d2i: torch.Tensor  # [B, 6] float32: src_x = m0*dx + m1*dy + m2, src_y = m3*dx + m4*dy + m5
    dst_hw: Tuple[int, int]
    fill: int
    mean: torch.Tensor  # [3] float32, source channel order (B, G, R)
    std: torch.Tensor  # [3] float32


# The page's benchmark: 1920x1080 frames resized to 640x640 (its §4.3).
WARPAFFINE_SRC_HW = (1080, 1920)
WARPAFFINE_DST_HW = (640, 640)


def letterbox_d2i(src_hw, dst_hw) -> np.ndarray:
    """The destination->source matrix of a letterbox resize: scale by
    s = min(Wd/W, Hd/H) and centre (input construction, float64; the inverse
    of i2d = [s, 0, (Wd - s*W)/2; 0, s, (Hd - s*H)/2])."""
    (H, W), (Hd, Wd) = src_hw, dst_hw
    s = min(Wd / W, Hd / H)
    tx, ty = (Wd - s * W) / 2.0, (Hd - s * H) / 2.0
    return np.array([1.0 / s, 0.0, -tx / s, 0.0, 1.0 / s, -ty / s])


def make_warpaffine_inputs(batch: int = 64, src_hw=WARPAFFINE_SRC_HW, dst_hw=WARPAFFINE_DST_HW, seed: int = 7,
                           jitter: bool = True) -> WarpAffineInputs:
    """Uniform random bytes for the frames. Every frame gets the letterbox
    matrix, and with jitter also a small random rotation (up to 5 degrees)
    and zoom (up to 10 %) about the destination centre, as an augmenting
    pipeline would."""
    g = torch.Generator().manual_seed(seed)
    H, W = src_hw
    src = torch.randint(0, 256, (batch, H, W, 3), generator=g, dtype=torch.int32).to(torch.uint8)
    base = letterbox_d2i(src_hw, dst_hw)
    mats = np.empty((batch, 6))
    r = torch.rand(batch, 2, generator=g, dtype=torch.float64).numpy()
    for b in range(batch):
        m = base.copy()
        if jitter:
            ang = np.deg2rad(10.0 * r[b, 0] - 5.0)
            zoom = 0.9 + 0.2 * r[b, 1]
            cx, cy = dst_hw[1] / 2.0, dst_hw[0] / 2.0
            # destination pixel -> rotated/zoomed destination pixel -> source
            c, s_ = np.cos(ang) / zoom, np.sin(ang) / zoom
            rot = np.array([[c, -s_, cx - c * cx + s_ * cy], [s_, c, cy - s_ * cx - c * cy], [0, 0, 1.0]])
            full = np.vstack([m.reshape(2, 3), [0, 0, 1.0]]) @ rot
            m = full[:2].reshape(6)
        mats[b] = m
    return WarpAffineInputs(src, torch.from_numpy(mats).to(torch.float32), tuple(dst_hw), 114,
                            torch.tensor([0.406, 0.456, 0.485]), torch.tensor([0.225, 0.224, 0.229]))


def small_variant(name: str, batch: int = 1, num_anchors: int = 24) -> Workload:
    """A cut-down copy of a named workload with the same maps, channels and
    distributions but few anchors, for fast CPU/GPU parity runs."""
    wl = WORKLOADS[name]
    if wl.loc_kind == "dcnv4_grid":
        return wl.replace(name=name + "_small", batch=batch)
    return wl.replace(name=name + "_small", batch=batch, num_anchors=num_anchors)
