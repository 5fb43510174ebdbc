"""GPU parity of the DCNv4 form (da_forward_fused / da_backward_fused): every
group has its own points, fused with their weights in one tensor
loc_weight [B, A, G, P, K, 2 + S].

Each case is compared element by element with the oracle of the DCNv4 form
(oracle.forward_fused / backward_fused, pinned in test_oracle_fused_pins.py):
the DCNv4 workload at full size in fp32, fp16 and bf16, the Sparse4D shape
cut to a few anchors, and ragged shapes. A consistency case checks that the
fused forward equals the standard forward when every group is given the same
points: bit for bit where the standard forward runs as one camera part.
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle
from parity_util import TOL, conditioning_atol, to_np, violations, widened_violations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def da():
    import deformable_view_feature_gb300 as m
    m.build.build()
    m.load_library()
    assert torch.cuda.is_available(), "the fused-layout tests need a CUDA GPU"
    return m


def _binned_ok(inp):
    """The binned path serves D = C/G a power of two in [8, 256]."""
    D = inp.wl.num_embeds // inp.wl.num_groups
    return 8 <= D <= 256 and D & (D - 1) == 0


def _run(da, inp, path="scatter"):
    dev = torch.device("cuda")
    feat, lw, go = inp.feat.to(dev), inp.loc_weight.to(dev), inp.grad_out.to(dev)
    out = da.da_forward_fused(feat, inp.spatial_shape, inp.level_start_index, lw)
    gf, glw = da.da_backward_fused(feat, inp.spatial_shape, inp.level_start_index, lw, go, path=path)
    torch.cuda.synchronize()
    return {"out": to_np(out), "grad_feat": to_np(gf), "grad_loc_weight": to_np(glw)}


def _conditioning(inp):
    """kappa*u*M of every grad_loc_weight entry, from the standard helper run
    per group (the groups are independent; see the fused oracle pins)."""
    wl = inp.wl
    B, A, G, P, K, E = inp.loc_weight.shape
    D = wl.num_embeds // G
    atol = np.zeros(inp.loc_weight.shape, np.float64)
    for g in range(G):
        sl = slice(g * D, (g + 1) * D)
        sub = da_inputs.Inputs(wl.replace(num_embeds=D, num_groups=1), inp.feat[..., sl].contiguous(),
                               inp.spatial_shape, inp.level_start_index,
                               inp.loc_weight[:, :, g, :, :, :2].contiguous(),
                               inp.loc_weight[:, :, g, :, :, 2:].unsqueeze(-1).contiguous(),
                               inp.grad_out[..., sl].contiguous())
        extra = conditioning_atol(sub)
        atol[:, :, g, :, :, :2] = extra["grad_loc"].reshape(B, A, P, K, 2)
        atol[:, :, g, :, :, 2:] = extra["grad_weight"].reshape(B, A, P, K, E - 2)
    return atol


def _check(inp, got):
    kind = inp.wl.feat_dtype
    out = oracle.forward_fused(inp.feat_numpy(), inp.spatial_shape.numpy(), inp.level_start_index.numpy(),
                               inp.loc_weight.numpy())
    gf, glw = oracle.backward_fused(inp.feat_numpy(), inp.spatial_shape.numpy(), inp.level_start_index.numpy(),
                                    inp.loc_weight.numpy(), inp.grad_out.numpy())
    msgs = []
    for name, ref, tol in (("out", out, TOL[kind]["out"]), ("grad_feat", gf, TOL[kind]["grad_feat"])):
        n, msg = violations(got[name], ref, tol[0], tol[1], name)
        if n:
            msgs.append(msg)
    # Location entries take grad_loc's tolerance, weight entries grad_weight's.
    rt_l, at_l = TOL[kind]["grad_loc"]
    rt_w, at_w = TOL[kind]["grad_weight"]
    cond = _conditioning(inp)
    for name, sl, rt, at in (("grad_loc_weight[xy]", np.s_[..., :2], rt_l, at_l),
                             ("grad_loc_weight[w]", np.s_[..., 2:], rt_w, at_w)):
        msgs += widened_violations(got["grad_loc_weight"][sl], glw[sl], rt, at, cond[sl], name)
    assert not msgs, f"{inp.wl.name}: " + " | ".join(msgs)


PATHS = ("scatter", "binned")


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("dtype", ["f32", "f16", "bf16"])
def test_dcnv4_full_size(da, dtype, path):
    wl = da_inputs.WORKLOADS["dcnv4"].replace(feat_dtype=dtype)
    inp = da_inputs.make_fused_inputs(wl)
    _check(inp, _run(da, inp, path))


@pytest.mark.parametrize("path", PATHS)
def test_sparse4d_shape_per_group_points(da, path):
    inp = da_inputs.make_fused_inputs(da_inputs.small_variant("sp4d_train", batch=2, num_anchors=30))
    _check(inp, _run(da, inp, path))


@pytest.mark.parametrize("path", PATHS)
@pytest.mark.parametrize("C,G,dtype", [(24, 3, "f32"), (64, 16, "f32"), (128, 2, "f16"), (32, 4, "bf16"),
                                       (64, 4, "f32")])
def test_ragged_shapes(da, C, G, dtype, path):
    wl = da_inputs.WORKLOADS["tiny"].replace(name=f"tiny_c{C}g{G}", num_embeds=C, num_groups=G, batch=2,
                                             num_anchors=13, num_pts=5, shapes=((9, 7), (3, 4)),
                                             num_cams=2, feat_dtype=dtype)
    inp = da_inputs.make_fused_inputs(wl, seed=7)
    if path == "binned" and not _binned_ok(inp):
        with pytest.raises(da.DaError, match="DA_ERR_UNSUPPORTED"):
            _run(da, inp, path)
        return
    _check(inp, _run(da, inp, path))


@pytest.mark.parametrize("channels,groups", [(128, 4), (256, 8)])
@pytest.mark.parametrize("cams", [2, 6])
def test_shared_points_match_standard_forward(da, cams, channels, groups):
    """The DCNv4 form with every group on the same points is the standard
    operator. With two cameras (one camera part in the standard forward) and
    128 channels in 4 groups of 32 both run the same per-group decomposition
    and the bits agree.
    At six cameras the standard forward sums two camera halves, and with 256
    channels it sums each lane's channels sample by sample in one warp per
    anchor: other associations of the same sum, so the two agree within the
    fp32 forward tolerance."""
    wl = da_inputs.small_variant("sp4d_inf", num_anchors=40).replace(num_cams=cams, num_embeds=channels,
                                                                     num_groups=groups)
    inp = da_inputs.make_inputs(wl)
    B, A, P, K, _ = inp.loc.shape
    S, G = inp.weights.shape[4], inp.weights.shape[5]
    lw = torch.empty(B, A, G, P, K, 2 + S)
    for g in range(G):
        lw[:, :, g, :, :, :2] = inp.loc
        lw[:, :, g, :, :, 2:] = inp.weights[..., g]
    dev = torch.device("cuda")
    feat = inp.feat.to(dev)
    a = da.da_forward_fused(feat, inp.spatial_shape, inp.level_start_index, lw.to(dev))
    b = da.da_forward(feat, inp.spatial_shape, inp.level_start_index, inp.loc.to(dev), inp.weights.to(dev))
    if cams == 2 and channels != 256:
        assert torch.equal(a, b)
    else:
        n, msg = violations(to_np(a), to_np(b), 1e-5, 1e-6, "out")
        assert n == 0, msg


@pytest.mark.parametrize("path", PATHS)
def test_empty_batch(da, path):
    wl = da_inputs.WORKLOADS["tiny"].replace(name="tiny_b0", batch=0)
    inp = da_inputs.make_fused_inputs(wl)
    got = _run(da, inp, path)
    assert all(v.size == 0 for v in got.values())


def test_binned_workspace_too_small_refused(da):
    import ctypes
    inp = da_inputs.make_fused_inputs(da_inputs.WORKLOADS["tiny"])
    dev = torch.device("cuda")
    lib = da.load_library()
    d = da._dims_fused(inp.feat, da._host_i32(inp.spatial_shape), inp.loc_weight)
    feat, lw, go = inp.feat.to(dev), inp.loc_weight.to(dev), inp.grad_out.to(dev)
    gf, glw = torch.empty_like(feat), torch.empty_like(lw)
    ws = torch.empty(4096, dtype=torch.uint8, device=dev)
    ss, ls = da._host_i32(inp.spatial_shape), da._host_i32(inp.level_start_index)
    st = lib.da_backward_fused(ctypes.byref(d), feat.data_ptr(), ss.data_ptr(), ls.data_ptr(), lw.data_ptr(),
                               go.data_ptr(), gf.data_ptr(), glw.data_ptr(), ws.data_ptr(), ws.numel(), None)
    assert st == 6  # DA_ERR_WORKSPACE


@pytest.mark.parametrize("path", PATHS)
def test_no_scales(da, path):
    """S = 0: loc_weight [B,A,G,P,K,2] holds locations with no weights; the
    output is 0 and so is every location gradient."""
    g = torch.Generator().manual_seed(51)
    B, A, G, P, K, C = 2, 5, 4, 3, 2, 64
    dev = torch.device("cuda")
    feat = torch.randn(B, 6, C, generator=g).to(dev)
    ss, ls = torch.zeros(K, 0, 2, dtype=torch.int32), torch.zeros(K, 0, dtype=torch.int32)
    lw = torch.rand(B, A, G, P, K, 2, generator=g).to(dev)
    go = torch.randn(B, A, C, generator=g).to(dev)
    out = da.da_forward_fused(feat, ss, ls, lw)
    gf, glw = da.da_backward_fused(feat, ss, ls, lw, go, path=path)
    torch.cuda.synchronize()
    assert torch.all(out == 0) and torch.all(gf == 0) and torch.all(glw == 0)


@pytest.mark.parametrize("i", range(12))
def test_random_shapes(da, i):
    """Seeded random shapes of the DCNv4 form through both backward paths (the
    binned one where it is served): K, S in 1..4 with map sides 1..20, a group
    width of 16/32/64/128 bytes, G in 1..8, B in 1..3, A in 1..30, P in 1..13;
    per-group points in [-0.3, 1.3] and softmax weights."""
    r = np.random.default_rng(3000 + i)
    dtype = ["f32", "bf16", "f16"][r.integers(3)]
    elem = 4 if dtype == "f32" else 2
    while True:
        D = int(r.choice([16, 32, 64, 128])) // elem
        G = int(r.choice([1, 2, 3, 4, 8]))
        if D * G <= 256:
            break
    S = int(r.integers(1, 5))
    wl = da_inputs.WORKLOADS["tiny"].replace(
        name=f"fused_random{i}", batch=int(r.integers(1, 4)), num_cams=int(r.integers(1, 5)),
        shapes=tuple((int(r.integers(1, 21)), int(r.integers(1, 21))) for _ in range(S)),
        num_embeds=D * G, num_groups=G, num_anchors=int(r.integers(1, 31)), num_pts=int(r.integers(1, 14)),
        feat_dtype=dtype, loc_lo=-0.3, loc_hi=1.3, weight_kind="softmax")
    inp = da_inputs.make_fused_inputs(wl, seed=4000 + i)
    for path in PATHS:
        if path == "binned" and not _binned_ok(inp):
            continue
        _check(inp, _run(da, inp, path))
