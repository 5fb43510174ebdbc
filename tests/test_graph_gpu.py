"""CUDA graph capture of the hot path.

The C ABI enqueues work on the caller's stream, never synchronises and
allocates nothing, so a whole step can be captured in a CUDA graph and
replayed:
  * the binning of the binned backward on a second stream (da_backward_bin),
    forked from and joined back to the capturing stream;
  * the forward;
  * the pull and epilogue of the backward (DA_BACKWARD_BINNED_READY).
Replays must give the eager results bit for bit (deterministic mode), also
after the inputs are overwritten in place between replays. The scatter
backward is captured too; its grad_feat and grad_loc sums use atomics, so
those are compared within tolerance.
"""
import numpy as np
import pytest
import torch

import da_inputs
from parity_util import conditioning_atol

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def da():
    import deformable_view_feature_gb300 as m
    m.build.build()
    m.load_library()
    assert torch.cuda.is_available(), "the graph tests need a CUDA GPU"
    return m


class _Step:
    """One fwd+bwd step on static device buffers."""

    def __init__(self, da, inp, path):
        self.da, self.path = da, path
        dev = torch.device("cuda")
        self.feat, self.loc, self.w, self.go = (t.to(dev) for t in (inp.feat, inp.loc, inp.weights, inp.grad_out))
        self.ss, self.ls = inp.spatial_shape, inp.level_start_index
        self.out = torch.empty(self.go.shape, device=dev)
        self.gf = torch.empty(self.feat.shape, device=dev)
        self.gl = torch.empty(self.loc.shape, device=dev)
        self.gw = torch.empty(self.w.shape, device=dev)
        self.side = torch.cuda.Stream()
        self.ws = None
        if path == "binned":
            d = da._dims(self.feat, da._host_i32(self.ss), self.loc, self.w)
            self.ws = torch.empty(max(da.backward_workspace_size(d), 256), dtype=torch.uint8, device=dev)

    def __call__(self):
        da, s = self.da, torch.cuda.current_stream()
        if self.path == "binned":
            self.side.wait_stream(s)
            da.da_backward_bin(self.feat, self.ss, self.ls, self.loc, self.w, workspace=self.ws,
                               deterministic=True, stream=self.side)
        da.da_forward(self.feat, self.ss, self.ls, self.loc, self.w, out=self.out, stream=s)
        if self.path == "binned":
            s.wait_stream(self.side)
            da.da_backward(self.feat, self.ss, self.ls, self.loc, self.w, self.go, grad_feat=self.gf,
                           grad_loc=self.gl, grad_weight=self.gw, stream=s, path="binned", workspace=self.ws,
                           deterministic=True, binned_ready=True)
        else:
            da.da_backward(self.feat, self.ss, self.ls, self.loc, self.w, self.go, grad_feat=self.gf,
                           grad_loc=self.gl, grad_weight=self.gw, stream=s, path="scatter")

    def outputs(self):
        return [t.clone() for t in (self.out, self.gf, self.gl, self.gw)]

    def load(self, inp):
        for dst, src in ((self.feat, inp.feat), (self.loc, inp.loc), (self.w, inp.weights),
                         (self.go, inp.grad_out)):
            dst.copy_(src)


def _capture(step):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        for _ in range(2):  # warm up off the default stream before capture
            step()
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    return g


def _inputs(seed):
    wl = da_inputs.small_variant("sp4d_train", batch=2, num_anchors=96)
    return da_inputs.make_inputs(wl.replace(seed=seed))


def test_binned_step_replays_eager_bits(da):
    a, b = _inputs(70), _inputs(71)
    step = _Step(da, a, "binned")
    with torch.cuda.stream(torch.cuda.Stream()):
        step()
    torch.cuda.synchronize()
    eager_a = step.outputs()
    g = _capture(step)
    g.replay()
    torch.cuda.synchronize()
    for x, y in zip(step.outputs(), eager_a):
        assert torch.equal(x, y)
    # New inputs written into the captured buffers: the replay reads them.
    step.load(b)
    g.replay()
    torch.cuda.synchronize()
    replay_b = step.outputs()
    with torch.cuda.stream(torch.cuda.Stream()):
        step()
    torch.cuda.synchronize()
    for x, y in zip(replay_b, step.outputs()):
        assert torch.equal(x, y)
    assert not torch.equal(replay_b[0], eager_a[0])


def test_scatter_step_replays_eager(da):
    a = _inputs(72)
    step = _Step(da, a, "scatter")
    with torch.cuda.stream(torch.cuda.Stream()):
        step()
    torch.cuda.synchronize()
    eager = step.outputs()
    g = _capture(step)
    for x in (step.out, step.gf, step.gl, step.gw):
        x.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    got = step.outputs()
    assert torch.equal(got[0], eager[0])  # the forward has no atomics
    assert torch.equal(got[3], eager[3])  # grad_weight: plain stores of shuffle sums
    # grad_feat and grad_loc are summed with atomics in a run-dependent order.
    # Two such runs differ by at most twice the fp32 bound of each sum
    # (kappa*u*M, as in the parity tests): cancelling grad_loc sums can be
    # far smaller than their terms.
    extra = conditioning_atol(a, kind_names=("grad_loc", "grad_feat"))
    for name, x, y in (("grad_feat", got[1], eager[1]), ("grad_loc", got[2], eager[2])):
        atol = 1e-6 + 2 * extra[name].reshape(tuple(x.shape))
        diff = np.abs(x.cpu().numpy().astype(np.float64) - y.cpu().numpy())
        bound = 2e-4 * np.abs(y.cpu().numpy()) + atol
        assert np.all(diff <= bound), f"{name}: {int(np.sum(diff > bound))} elements differ"
