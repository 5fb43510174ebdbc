"""GPU tests of the deterministic binned backward (DA_BACKWARD_DETERMINISTIC).

In this mode the records of every feature row are put in a fixed order before
they are summed. The tests check that
  * the gradients still match the oracle within the parity tolerances, at the
    full training shape and on cases whose rows fall in each tier of the
    per-row sort (up to 8, 9..128, 129..2048 and more records per row);
  * two runs give the same bits, even when the workspace holds different
    garbage before each run and the calls go to different streams;
  * the result agrees with the default (unordered) binned mode within the
    parity tolerances.
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle
from parity_util import TOL, conditioning_atol, to_np, violations, widened_violations

pytestmark = pytest.mark.gpu

NAMES = ("grad_feat", "grad_loc", "grad_weight")


@pytest.fixture(scope="module")
def da():
    import deformable_view_feature_gb300 as m
    m.build.build()
    m.load_library()
    assert torch.cuda.is_available(), "the deterministic-mode tests need a CUDA GPU"
    return m


def _backward(da, inp, deterministic=True, garbage_seed=None, stream=None):
    dev = torch.device("cuda")
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    dims = da._dims(feat, da._host_i32(inp.spatial_shape), loc, w)
    ws = torch.empty(max(da.backward_workspace_size(dims), 256), dtype=torch.uint8, device=dev)
    if garbage_seed is not None:
        g = torch.Generator(device=dev).manual_seed(garbage_seed)
        ws.copy_(torch.randint(0, 256, ws.shape, generator=g, device=dev, dtype=torch.int32).to(torch.uint8))
    res = da.da_backward(feat, inp.spatial_shape, inp.level_start_index, loc, w, go, path="binned",
                         workspace=ws, deterministic=deterministic, stream=stream)
    torch.cuda.synchronize()
    return dict(zip(NAMES, (to_np(t) for t in res)))


def _check_oracle(inp, got, crowded=False):
    ref = oracle.run_inputs(inp, backward_pass=True)
    # Crowded rows sum thousands of signed products: grad_feat then gets the
    # fp32 summation bound too, with each row's own record count. On the
    # four rows around the spot (thousands of records) it no longer sees one
    # missing record; the spread rows (tens of records) still do, and the
    # run-to-run bit equality below and the uncrowded cases keep the
    # per-record check everywhere.
    extra = conditioning_atol(inp, ("grad_loc", "grad_weight", "grad_feat") if crowded else
                              ("grad_loc", "grad_weight"))
    msgs = []
    for name in NAMES:
        rtol, atol = TOL[inp.wl.feat_dtype][name]
        msgs += widened_violations(got[name], ref[name], rtol, atol, extra.get(name), f"{inp.wl.name} {name}")
    assert not msgs, " | ".join(msgs)


def _same_bits(a, b):
    for name in NAMES:
        assert np.array_equal(a[name].view(np.uint32), b[name].view(np.uint32)), name


def _crowded(seed, n_spot, H=16, W=16, A=600, P=8, C=64, G=2, softmax_w=False):
    """One 16x16 map and A*P = 4800 locations. The first n_spot*P sit on one
    spot, the rest are spread uniformly. A pixel then gets about
    4*(4800 - n_spot*P)/256 records from the spread locations, and the four
    pixels around the spot n_spot*P more. softmax_w: the weights of each
    (anchor, group) are a softmax over its P points, as in the Sparse4D
    workloads, instead of N(0, 1) draws."""
    g = torch.Generator().manual_seed(seed)
    ss, ls = da_inputs.map_tables(1, [(H, W)])
    feat = torch.randn(1, H * W, C, generator=g)
    loc = torch.rand(1, A, P, 1, 2, generator=g)
    loc.view(1, A * P, 2)[:, :n_spot * P] = torch.tensor([0.37, 0.61])
    w = torch.randn(1, A, P, 1, 1, G, generator=g)
    if softmax_w:
        w = w.softmax(dim=2)
    go = torch.randn(1, A, C, generator=g)
    wl = da_inputs.WORKLOADS["tiny"].replace(name=f"crowded{n_spot}", batch=1, num_embeds=C, num_groups=G,
                                             num_anchors=A, num_pts=P, shapes=((H, W),))
    return da_inputs.Inputs(wl, feat, ss, ls, loc, w, go)


@pytest.mark.parametrize("n_spot", [0, 10, 100, 600])
def test_crowded_rows_every_sort_tier(da, n_spot):
    # Spread rows hold about 75, 74, 62 and 0 records (the warp tier); the
    # spot's rows about 75, 154, 862 (the shared-memory CTA tier) and 4800
    # (the global-memory CTA tier). Border pixels get fewer.
    inp = _crowded(70 + n_spot, n_spot)
    a = _backward(da, inp, garbage_seed=1)
    _check_oracle(inp, a, crowded=True)
    b = _backward(da, inp, garbage_seed=2, stream=torch.cuda.Stream())
    _same_bits(a, b)


@pytest.mark.parametrize("n_spot", [0, 100, 600])
@pytest.mark.parametrize("deterministic", [False, True])
def test_crowded_pixel_runs_hand_rows_on(da, n_spot, deterministic):
    # C = 256 on a 64x64 map: about 4.7 records per row from the spread
    # locations, so the pull walks the map in runs of 16 pixels per warp.
    # The runs around the spot hold up to 4800 records, beyond a run's cap:
    # their rows past the cap go to the leftover list and its own launch.
    # Softmax weights: 8 groups of 32 channels sum many signed products per
    # grad_loc element, and N(0, 1) weights on top of that put about 0.1 % of
    # them past the plain bound through cancellation alone.
    inp = _crowded(90 + n_spot, n_spot, H=64, W=64, C=256, G=8, softmax_w=True)
    a = _backward(da, inp, deterministic=deterministic, garbage_seed=7)
    _check_oracle(inp, a, crowded=True)
    b = _backward(da, inp, deterministic=deterministic, garbage_seed=8, stream=torch.cuda.Stream())
    if deterministic:
        _same_bits(a, b)
    else:
        _check_oracle(inp, b, crowded=True)


def test_pull_twice_on_one_binning(da):
    # The leftover-row count lives in the workspace: the epilogue clears it,
    # so a second pull of the same binned workspace hands on the same rows
    # and gives the same bits.
    inp = _crowded(95, 600, H=64, W=64, C=256, G=8, softmax_w=True)
    dev = torch.device("cuda")
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    ws = da.da_backward_bin(feat, inp.spatial_shape, inp.level_start_index, loc, w, deterministic=True)
    outs = []
    for _ in range(2):
        res = da.da_backward(feat, inp.spatial_shape, inp.level_start_index, loc, w, go, path="binned",
                             workspace=ws, deterministic=True, binned_ready=True)
        torch.cuda.synchronize()
        outs.append(dict(zip(NAMES, (to_np(t) for t in res))))
    _same_bits(outs[0], outs[1])
    _check_oracle(inp, outs[0], crowded=True)


def test_short_rows_and_many_maps(da):
    # A Sparse4D-like cut (4 scales, 6 cameras): rows of every length from 1
    # record up, mostly the thread-per-row tier.
    wl = da_inputs.small_variant("sp4d_train", batch=2, num_anchors=50)
    inp = da_inputs.make_inputs(wl, seed=81)
    a = _backward(da, inp, garbage_seed=3)
    _check_oracle(inp, a)
    _same_bits(a, _backward(da, inp, garbage_seed=4))


@pytest.mark.parametrize("name", ["sp4d_train", "large_bf16", "dcnv4"])
def test_full_size_reproducible_and_close_to_default(da, name):
    inp = da_inputs.make_inputs(name)
    a = _backward(da, inp, garbage_seed=5)
    b = _backward(da, inp, garbage_seed=6)
    _same_bits(a, b)
    c = _backward(da, inp, deterministic=False)
    rtol, atol = TOL[inp.wl.feat_dtype]["grad_feat"]
    n, msg = violations(a["grad_feat"], c["grad_feat"], rtol, atol, f"{name} grad_feat vs default")
    assert n == 0, msg


def test_full_size_training_shape_against_oracle(da):
    inp = da_inputs.make_inputs("sp4d_train")
    _check_oracle(inp, _backward(da, inp))


def test_deterministic_needs_binned(da):
    inp = da_inputs.make_inputs("tiny")
    dev = torch.device("cuda")
    with pytest.raises(ValueError):
        da.da_backward(inp.feat.to(dev), inp.spatial_shape, inp.level_start_index, inp.loc.to(dev),
                       inp.weights.to(dev), inp.grad_out.to(dev), path="scatter", deterministic=True)


@pytest.mark.parametrize("name", ["sp4d_train", "tiny"])
def test_binning_on_a_side_stream_during_the_forward(da, name):
    """da_backward_bin on a second stream while da_forward runs, then the rest
    of the backward with binned_ready: with the deterministic order on both
    sides, the same bits as the one-call deterministic backward."""
    inp = da_inputs.make_inputs(name)
    dev = torch.device("cuda")
    feat, loc, w, go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
    ss, ls = inp.spatial_shape, inp.level_start_index
    ref = _backward(da, inp, garbage_seed=7)
    main, side = torch.cuda.Stream(), torch.cuda.Stream()
    ws = None
    for rep in range(2):  # the second round re-bins into a workspace the first round used
        torch.cuda.synchronize()
        ws = da.da_backward_bin(feat, ss, ls, loc, w, workspace=ws, deterministic=True, stream=side)
        done = torch.cuda.Event()
        done.record(side)
        da.da_forward(feat, ss, ls, loc, w, stream=main)
        main.wait_event(done)
        gf, gl, gw = da.da_backward(feat, ss, ls, loc, w, go, path="binned", workspace=ws, binned_ready=True,
                                    stream=main)
        torch.cuda.synchronize()
        _same_bits(ref, dict(zip(NAMES, (to_np(t) for t in (gf, gl, gw)))))
