"""GPU parity of the host pipeline (da_pipeline_*), through the C ABI.

Several different input draws are submitted back to back from pinned host
tensors, more draws than the pipeline has buffer sets, so buffer sets are
reused while earlier steps are still copying. Every host output is compared
with the oracle run on the same draw, with the tolerances of the other parity
tests. Cases: the Sparse4D training shape cut to a few anchors (binned
backward), a width the binned backward does not take (the scatter path), a
bf16 forward-only pipeline, depth 1, and an empty batch.
"""
import numpy as np
import pytest
import torch

import da_inputs
import oracle
from parity_util import TOL, conditioning_atol, violations, widened_violations

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def da():
    import deformable_view_feature_gb300 as m
    m.build.build()
    m.load_library()
    assert torch.cuda.is_available(), "the pipeline tests need a CUDA GPU"
    return m


def _draw(wl, seed):
    return da_inputs.make_inputs(wl, seed=seed)


def _host_outputs(pipe, backward):
    out = {}
    for name in ("out",) + (("grad_feat", "grad_loc", "grad_weight") if backward else ()):
        shape, dt = pipe.shapes()[name]
        out[name] = torch.full(shape, float("nan"), dtype=dt).pin_memory()
    return out


def _run_pipeline(da, draws, backward, depth):
    inp0 = draws[0]
    dims = da._dims(inp0.feat, da._host_i32(inp0.spatial_shape), inp0.loc, inp0.weights)
    results = []
    with da.HostPipeline(dims, inp0.spatial_shape, inp0.level_start_index, backward=backward,
                         depth=depth) as pipe:
        staged = []
        for inp in draws:
            h = [t.pin_memory() for t in (inp.feat, inp.loc, inp.weights, inp.grad_out)]
            o = _host_outputs(pipe, backward)
            pipe.submit(h[0], h[1], h[2], o["out"], grad_out=h[3], grad_feat=o.get("grad_feat"),
                        grad_loc=o.get("grad_loc"), grad_weight=o.get("grad_weight"))
            staged.append(o)
        pipe.sync()
        for o in staged:
            results.append({k: v.numpy().copy() for k, v in o.items()})
    return results


def _check(inp, got, ref):
    kind = inp.wl.feat_dtype
    extra = conditioning_atol(inp) if "grad_loc" in ref else {}
    msgs = []
    for name, r in ref.items():
        rtol, atol = TOL[kind][name]
        msgs += widened_violations(got[name], r, rtol, atol, extra.get(name), f"{inp.wl.name} {name}")
    assert not msgs, " | ".join(msgs)


@pytest.mark.parametrize("depth", [2, 1])
def test_pipeline_training_shape_binned(da, depth):
    wl = da_inputs.small_variant("sp4d_train", batch=2, num_anchors=20)
    draws = [_draw(wl, seed) for seed in (11, 12, 13)]
    got = _run_pipeline(da, draws, backward=True, depth=depth)
    for inp, g in zip(draws, got):
        _check(inp, g, oracle.run_inputs(inp, backward_pass=True))
    # Different draws give different outputs: no step read another's slot.
    assert not np.array_equal(got[0]["out"], got[1]["out"])


def test_pipeline_scatter_fallback_width(da):
    # C = 24 is not a power of two, so the pipeline's backward takes the
    # scatter path.
    wl = da_inputs.WORKLOADS["tiny"].replace(name="tiny_c24", num_embeds=24, num_groups=3, num_anchors=9)
    draws = [_draw(wl, seed) for seed in (21, 22, 23)]
    got = _run_pipeline(da, draws, backward=True, depth=2)
    for inp, g in zip(draws, got):
        _check(inp, g, oracle.run_inputs(inp, backward_pass=True))


def test_pipeline_forward_only_bf16(da):
    wl = da_inputs.small_variant("large_bf16", batch=1, num_anchors=30)
    draws = [_draw(wl, seed) for seed in (31, 32, 33, 34)]
    got = _run_pipeline(da, draws, backward=False, depth=3)
    for inp, g in zip(draws, got):
        assert set(g) == {"out"}
        _check(inp, g, oracle.run_inputs(inp, backward_pass=False))


def test_pipeline_matches_device_forward_bits(da):
    # The forward is deterministic, so the pipeline's host result equals the
    # device entry point's bit for bit.
    wl = da_inputs.small_variant("sp4d_inf", batch=1, num_anchors=40)
    inp = _draw(wl, 41)
    got = _run_pipeline(da, [inp, inp], backward=False, depth=2)
    dev = torch.device("cuda")
    ref = da.da_forward(inp.feat.to(dev), inp.spatial_shape, inp.level_start_index, inp.loc.to(dev),
                        inp.weights.to(dev)).cpu().numpy()
    for g in got:
        assert np.array_equal(g["out"], ref)


def test_pipeline_empty_batch(da):
    wl = da_inputs.WORKLOADS["tiny"].replace(name="tiny_b0", batch=0)
    inp = _draw(wl, 51)
    got = _run_pipeline(da, [inp, inp], backward=True, depth=2)
    for g in got:
        assert all(v.size == 0 for v in g.values())


def test_pipeline_rejects_device_tensors_and_wrong_shapes(da):
    wl = da_inputs.WORKLOADS["tiny"]
    inp = _draw(wl, 61)
    dims = da._dims(inp.feat, da._host_i32(inp.spatial_shape), inp.loc, inp.weights)
    with da.HostPipeline(dims, inp.spatial_shape, inp.level_start_index, backward=False) as pipe:
        out = torch.empty(1, wl.num_anchors, wl.num_embeds)
        with pytest.raises(ValueError):
            pipe.submit(inp.feat.cuda(), inp.loc, inp.weights, out)
        with pytest.raises(ValueError):
            pipe.submit(inp.feat, inp.loc[:, :1].contiguous(), inp.weights, out)
        pipe.submit(inp.feat, inp.loc, inp.weights, out)  # pageable memory works too
        pipe.sync()
        ref = oracle.run_inputs(inp, backward_pass=False)["out"]
        n, msg = violations(out.numpy(), ref, *TOL["f32"]["out"], "out")
        assert n == 0, msg
