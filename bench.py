"""Benchmark: fwd+bwd bilinear samples/s of the deformable-aggregation op.

The default workload is the 6-camera, 4-scale Sparse4D training shape:
  * B=6, maps 64x176, 32x88, 16x44, 8x22;
  * C=256, G=8, 900 anchors, 13 points;
  * fp32 features.
One step is one pass of the whole path: da_forward, then da_backward (the
binding's choice of path for the shape; the binned path's binning runs on a
side stream while the forward runs). Inputs are synthetic and seeded
(da_inputs), and resident in HBM when the timed region starts. The feature
tensor alone (551 MB) is larger than L2, so no L2 flush is done between
steps. Other workloads (--workload) whose feature map is under twice the L2
size get an L2 flush before every step by default (--l2 auto): a write of
twice the L2 size, outside the step's own events, which then give the step
time (the side-stream binning starts after the step's first event).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload NAME] [--l2 auto|flush|none]

Prints ONE JSON line on rank 0. It holds:
  * value: samples/s over all ranks;
  * roofline: the step's algorithmic bytes (every tensor of the forward and
    backward read or written once) divided by the step's CUDA-event time,
    against the measured HBM copy bandwidth; with the forward's and the
    backward's own figures under "parts";
  * e2e: the same metric with host buffers and host<->device copies inside
    the timed region;
  * cpu_baseline: the CPU oracle timed on a bounded sample of anchors;
  * clocks: nvidia-smi samples taken during the timed region.

--impl reference times the CPU oracle (the only reference this project has)
on the same workload, one bounded sample of anchors per step.

With N > 1 (torchrun), each rank runs an independent replica of the workload
on its own GPU: the op does not shard, so there is no collective on the data
path ("scaling": "weak").
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import da_inputs  # noqa: E402

METRIC = "fwd+bwd bilinear samples/sec at 6-cam Sparse4D shape; GB/s vs HBM peak"

# DRAM bytes per call (dram__bytes_read.sum + dram__bytes_write.sum, summed over
# the call's kernels), from one ncu capture of this bench at sp4d_train. They
# describe the kernels whose sources hash to "digest", and are reported as null
# once the sources change.
NCU_TRAFFIC = {
    "digest": "abff704e3fdf1bcd",
    "workload": "sp4d_train",
    "da_forward": 727_568_128,
    "da_backward[binned]": 1_713_505_280,
}


def kernel_digest() -> str:
    """Hash (names and bytes) of the CUDA sources that define or share device
    code: the headers and every .cu file with a __global__ kernel. Host-only
    sources (the C ABI, the host pipeline) do not change the kernels' traffic."""
    import glob
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "deformable_view_feature_gb300", "csrc")
    files = sorted(glob.glob(os.path.join(csrc, "*.cu")) + glob.glob(os.path.join(csrc, "*.cuh"))
                   + glob.glob(os.path.join(csrc, "*.h")))
    for p in files:
        with open(p, "rb") as f:
            data = f.read()
        if p.endswith(".cu") and b"__global__" not in data:
            continue
        h.update(os.path.basename(p).encode())
        h.update(data)
    return h.hexdigest()[:16]


def ncu_traffic(workload: str, call: str):
    if workload != NCU_TRAFFIC["workload"] or kernel_digest() != NCU_TRAFFIC["digest"]:
        return None
    return NCU_TRAFFIC.get(call)
# Kernels da_backward launches: binned = row-count zero-fill, count, 3 scan
# steps, fill, pull, epilogue; scatter = grad_feat zero-fill, gather-scatter.
# binned-det adds the four kernels of the per-row sort (DA_BACKWARD_DETERMINISTIC).
# Where the pull takes fine maps in pixel runs it is two launches (the pull,
# then its leftover rows): see pull_launches.
BWD_LAUNCHES = {"binned": 8, "binned-det": 12, "scatter": 2}


def pull_launches(wl) -> int:
    """Kernels of the binned path's pull: 2 when the library pulls fine maps
    in pixel runs (standard layout, 256 channels, packed maps, and a map whose
    rows average fewer than 24 records: 4*A*P/(H*W) < 24), else 1. The rule
    is the one the library applies to choose its pull."""
    if wl.num_embeds != 256:
        return 1
    ap = wl.num_anchors * wl.num_pts
    return 2 if any(4.0 * ap / (h * w) < 24.0 for h, w in wl.shapes) else 1


def bwd_launches(path: str, wl) -> int:
    n = BWD_LAUNCHES[path]
    return n + pull_launches(wl) - 1 if path != "scatter" else n
FALLBACK_HBM_GBS = 6800.0


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def tensor_bytes(*ts):
    return sum(t.numel() * t.element_size() for t in ts if t is not None)


def algorithmic_bytes(inp: da_inputs.Inputs):
    """Compulsory DRAM bytes per call: every tensor read or written once.
    grad_feat counts twice in the backward (a zero-fill and a write-back)."""
    feat, loc, w, go = inp.feat, inp.loc, inp.weights, inp.grad_out
    out_b = go.numel() * 4
    gf_b = feat.numel() * 4
    fwd = tensor_bytes(feat, loc, w) + out_b
    grad_loc_b, grad_w_b = loc.numel() * 4, w.numel() * 4
    bwd = tensor_bytes(feat, loc, w, go) + 2 * gf_b + grad_loc_b + grad_w_b
    return fwd, bwd


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi sampling in the background; keeps samples by wall time."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.thread = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, ValueError):
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        if self.thread is not None:
            self.thread.join(timeout=5)

    def summary(self, t0: float, t1: float):
        sm, smax, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ts, line in self.lines:
            if not (t0 <= ts <= t1 + 0.05):
                continue
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                sm.append(float(parts[2]))
                smax = float(parts[3])
            except ValueError:
                continue
            for n, v in zip(names, parts[6:10]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": smax,
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------------------- dist

def dist_setup(n_gpus: int):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """Largest x over all ranks (a CUDA tensor under NCCL, a CPU one under gloo)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], device=dev, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(samples_per_rank_step: int, steps: int, world: int, ms_max: float) -> float:
    """Whole-job samples/s: every rank runs its own replica of the workload,
    and the job's time is the slowest rank's."""
    return samples_per_rank_step * steps * world / (ms_max / 1e3)


# ----------------------------------------------------------------------------- CPU oracle legs

def oracle_sample(inp: da_inputs.Inputs, n_anchors: int, start: int = 0):
    """Time the CPU oracle (fwd + bwd) on anchors [start, start+n) of the flat
    b*A+a index. Returns (samples, seconds)."""
    import oracle  # test infrastructure: only this leg and --impl reference use it
    wl = inp.wl
    args = (inp.feat_numpy(), inp.spatial_shape.numpy(), inp.level_start_index.numpy(),
            inp.loc.numpy(), inp.weights.numpy())
    rng = (start, start + n_anchors)
    t0 = time.perf_counter()
    oracle.forward(*args, ba_range=rng)
    if wl.backward:
        oracle.backward(*args, inp.grad_out.numpy(), ba_range=rng)
    dt = time.perf_counter() - t0
    per_anchor = wl.num_pts * wl.num_cams * wl.num_scales * wl.num_groups
    return n_anchors * per_anchor, dt


def cpu_baseline(inp, n_anchors: int):
    samples, dt = oracle_sample(inp, n_anchors)
    return {"value": samples / dt, "unit": "samples/s", "cores": 1, "kind": "oracle",
            "sample": (f"single-threaded C oracle, fwd+bwd over anchors 0..{n_anchors - 1} "
                       f"of {inp.wl.batch * inp.wl.num_anchors} ({samples} samples, {dt:.1f} s); "
                       f"host has {os.cpu_count()} cores")}


def run_reference(a, wl):
    rank, world, _ = int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")), 0
    if rank != 0:
        return
    inp = da_inputs.make_inputs(wl)
    n = max(1, min(a.ref_anchors, wl.batch * wl.num_anchors))
    nba = wl.batch * wl.num_anchors
    for i in range(a.warmup):
        oracle_sample(inp, n, (i * n) % max(1, nba - n + 1))
    tot_s, tot_t = 0, 0.0
    for i in range(a.steps):
        s, dt = oracle_sample(inp, n, (i * n) % max(1, nba - n + 1))
        tot_s += s
        tot_t += dt
    v = tot_s / tot_t
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": "samples/s", "n_gpus": a.gpus,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": 1e3 * tot_t / a.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded da_inputs draw; no dataset)",
        "config": config_of(wl, "CPU oracle; each step a bounded sample of "
                                f"{n} anchors"),
        "cpu_baseline": {"value": v, "unit": "samples/s", "cores": 1, "kind": "oracle",
                         "sample": f"{n} anchors (fwd+bwd) per step of the single-threaded C "
                                   f"oracle; host has {os.cpu_count()} cores"},
        "e2e": {"value": v, "unit": "samples/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def config_of(wl, l2):
    return {"workload": f"{wl.name}: B{wl.batch} K{wl.num_cams} S{wl.num_scales} maps "
                        + "/".join(f"{h}x{w}" for h, w in wl.shapes)
                        + f" C{wl.num_embeds} G{wl.num_groups} A{wl.num_anchors} P{wl.num_pts} "
                        + f"{wl.feat_dtype} features",
            "samples_per_step": wl.num_samples, "passes": "fwd+bwd" if wl.backward else "fwd",
            "l2": l2, "parallelism": "replicas (one independent workload per GPU)"}


# ----------------------------------------------------------------------------- our arm

def run_e2e(a, wl, inp, dev, world, dev_tensors, ss, ls):
    """End to end through the public API: pinned host tensors and the library's
    host pipeline (da_pipeline_*), whose copies in both directions and kernels
    overlap across consecutive steps. The timed region holds every step's
    host->device input copies, kernels and device->host output copies."""
    import deformable_view_feature_gb300 as da
    feat, loc, w, go, out, gf, gl, gw = dev_tensors
    h_in = [t.pin_memory() for t in (inp.feat, inp.loc, inp.weights, inp.grad_out)]
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in (out, gf, gl, gw)]
    if not wl.backward:
        h_in, h_out = h_in[:3], h_out[:1]
    e2e_steps = max(1, min(a.steps, a.e2e_steps))
    pipe = da.HostPipeline(da._dims(feat, da._host_i32(ss), loc, w), ss, ls, backward=wl.backward,
                           depth=2, device=dev)

    def e2e_step():
        hf, hl, hw = h_in[:3]
        if wl.backward:
            pipe.submit(hf, hl, hw, h_out[0], grad_out=h_in[3], grad_feat=h_out[1], grad_loc=h_out[2],
                        grad_weight=h_out[3])
        else:
            pipe.submit(hf, hl, hw, h_out[0])

    for _ in range(3):
        e2e_step()
    pipe.sync()
    barrier(world)
    t0 = time.perf_counter()
    for _ in range(e2e_steps):
        e2e_step()
    pipe.sync()
    e2e_ms = max_over_ranks((time.perf_counter() - t0) * 1e3, world)
    pipe.close()
    barrier(world)
    h2d = tensor_bytes(*h_in)
    d2h = tensor_bytes(*h_out)
    e2e = {"value": wl.num_samples * e2e_steps * world / (e2e_ms / 1e3), "unit": "samples/s",
           "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "steps": e2e_steps,
           "api": "HostPipeline (da_pipeline_submit, depth 2), pinned host tensors, wall clock"}

    return e2e


def run_ours(a, wl):
    import deformable_view_feature_gb300 as da
    da.load_library()
    rank, world, local = dist_setup(a.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    inp = da_inputs.make_inputs(wl)
    feat = inp.feat.to(dev)
    loc = inp.loc.to(dev)
    w = inp.weights.to(dev)
    go = inp.grad_out.to(dev)
    ss, ls = inp.spatial_shape, inp.level_start_index
    out = torch.empty(go.shape, device=dev)
    gf = torch.empty(feat.shape, device=dev)
    gl = torch.empty(loc.shape, device=dev)
    gw = torch.empty(w.shape, device=dev)
    stream = torch.cuda.Stream(device=dev)
    fwd_bytes, bwd_bytes = algorithmic_bytes(inp)
    ws = None
    dims = da._dims(feat, da._host_i32(ss), loc, w)
    if a.bwd_path == "auto":
        # The binding's choice for these sizes (the one autograd users get).
        a.bwd_path = da.backward_path(dims)
    path = "scatter" if a.bwd_path == "scatter" else "binned"
    if path == "binned":
        ws = torch.empty(max(da.backward_workspace_size(dims), 256), dtype=torch.uint8, device=dev)

    # The binning half of the binned backward needs the locations only: it runs
    # on a side stream while the forward runs (da_backward_bin), after the
    # previous step's backward has released the workspace.
    # L2 policy: flush before every step when the maps would otherwise stay
    # in L2 between steps.
    l2_bytes = torch.cuda.get_device_properties(dev).L2_cache_size
    feat_bytes = inp.feat.numel() * inp.feat.element_size()
    flush = a.l2 == "flush" or (a.l2 == "auto" and feat_bytes < 2 * l2_bytes)
    flush_buf = torch.empty(2 * l2_bytes // 4, dtype=torch.float32, device=dev) if flush else None
    # In flush mode the step time is the sum of each step's own events; the
    # side stream then waits for the step's first event, so the binning
    # overlaps the forward but never the flush before it.
    overlap = wl.backward and path == "binned" and not a.no_bin_overlap
    # Default priority: a high-priority side stream interleaves the binning
    # with the forward's blocks, but the forward then slows by as much as the
    # backward gains (measured); at equal priority the binning fills the
    # forward's tail and the step is 1 % shorter.
    side = torch.cuda.Stream(device=dev)
    bin_done, bwd_done, step_start = torch.cuda.Event(), torch.cuda.Event(), torch.cuda.Event()
    det = a.bwd_path == "binned-det"

    def step(ev=None):
        if flush:
            with torch.cuda.stream(stream):
                flush_buf.fill_(float(ev is not None))
        t0 = ev[0] if ev is not None else step_start
        t0.record(stream)
        if overlap:
            side.wait_event(bwd_done)
            if flush:
                side.wait_event(t0)
            da.da_backward_bin(feat, ss, ls, loc, w, workspace=ws, deterministic=det, stream=side)
            bin_done.record(side)
        da.da_forward(feat, ss, ls, loc, w, out=out, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if wl.backward:
            if overlap:
                stream.wait_event(bin_done)
            da.da_backward(feat, ss, ls, loc, w, go, grad_feat=gf, grad_loc=gl, grad_weight=gw,
                           stream=stream, path=path, workspace=ws, deterministic=det, binned_ready=overlap)
            if ev is not None:
                ev[2].record(stream)
            bwd_done.record(stream)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            step()
    torch.cuda.synchronize(dev)

    clocks = ClockSampler(local if world > 1 else 0)
    clocks.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(a.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    barrier(world)
    time.sleep(0.1)
    clocks.stop()
    fwd_ms = [evs[i][0].elapsed_time(evs[i][1]) for i in range(a.steps)]
    bwd_ms = [evs[i][1].elapsed_time(evs[i][2]) for i in range(a.steps)] if wl.backward else []
    # Without a flush the steps run back to back and the whole region counts;
    # with one, only each step's own events (the flush between them does not).
    ms = start.elapsed_time(end) if not flush else sum(fwd_ms) + sum(bwd_ms)
    ms_max = max_over_ranks(ms, world)

    value = job_throughput(wl.num_samples, a.steps, world, ms_max)

    # The same step captured once in a CUDA graph (the binning forked to the
    # side stream and joined inside the capture) and replayed.
    graph = None
    if a.graph and not flush:
        def graph_step():
            if wl.backward and path == "binned":
                side.wait_stream(stream)
                da.da_backward_bin(feat, ss, ls, loc, w, workspace=ws, deterministic=det, stream=side)
            da.da_forward(feat, ss, ls, loc, w, out=out, stream=stream)
            if wl.backward:
                if path == "binned":
                    stream.wait_stream(side)
                da.da_backward(feat, ss, ls, loc, w, go, grad_feat=gf, grad_loc=gl, grad_weight=gw, stream=stream,
                               path=path, workspace=ws, deterministic=det, binned_ready=path == "binned")
        torch.cuda.synchronize(dev)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=stream):
            graph_step()
        for _ in range(a.warmup):
            g.replay()
        g0, g1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        g0.record(stream)
        with torch.cuda.stream(stream):
            for _ in range(a.steps):
                g.replay()
        g1.record(stream)
        torch.cuda.synchronize(dev)
        gms = max_over_ranks(g0.elapsed_time(g1), world)
        graph = {"ms_per_step": gms / a.steps, "value": job_throughput(wl.num_samples, a.steps, world, gms),
                 "unit": "samples/s", "note": "one step captured in a CUDA graph, replayed back to back"}

    # End to end through the public API: pinned host tensors and the library's
    # host pipeline (da_pipeline_*), whose copies in both directions and
    # kernels overlap across consecutive steps. The timed region holds every
    # step's host->device input copies, kernels and device->host output copies.
    e2e = None
    if a.e2e_steps > 0:
        e2e = run_e2e(a, wl, inp, dev, world, (feat, loc, w, go, out, gf, gl, gw), ss, ls)

    if rank != 0:
        return
    peak, peak_kind = peaks()

    # The roofline is the whole step's: every kernel of da_forward and
    # da_backward (the side-stream binning included, since the step's events
    # cover it), against the step's compulsory bytes.
    step_ms = ms_max / a.steps
    step_bytes = fwd_bytes + (bwd_bytes if wl.backward else 0)
    achieved = step_bytes / (step_ms / 1e3) / 1e9
    if wl.backward:
        t_f, t_b = ncu_traffic(wl.name, "da_forward"), ncu_traffic(wl.name, f"da_backward[{a.bwd_path}]")
        traffic = t_f + t_b if t_f is not None and t_b is not None else None
        step_kernel = (f"one step: da_forward + da_backward ({a.bwd_path} path), every kernel of both"
                       + (", the binning on a side stream during the forward" if overlap else ""))
    else:
        traffic = ncu_traffic(wl.name, "da_forward")
        step_kernel = "one step: da_forward"
    fwd_mean = statistics.mean(fwd_ms)
    parts = {"da_forward": {"ms": fwd_mean, "algorithmic_bytes": fwd_bytes,
                            "frac": fwd_bytes / (fwd_mean / 1e3) / 1e9 / peak}}
    if wl.backward:
        bwd_mean = statistics.mean(bwd_ms)
        # The binned path writes every grad_feat row once: no zero-fill.
        bwd_own = bwd_bytes - (inp.feat.numel() * 4 if a.bwd_path != "scatter" else 0)
        parts["da_backward"] = {
            "ms": bwd_mean, "algorithmic_bytes": bwd_bytes, "frac": bwd_bytes / (bwd_mean / 1e3) / 1e9 / peak,
            "algorithmic_bytes_own_path": bwd_own, "frac_own_path": bwd_own / (bwd_mean / 1e3) / 1e9 / peak,
            "span": "from the end of the forward to the end of the backward"
                    + ("; includes the part of the side-stream binning the forward did not hide" if overlap else "")}
    line = {
        "metric": METRIC, "value": value, "unit": "samples/s", "n_gpus": world,
        "steps": a.steps, "warmup": a.warmup, "ms_per_step": step_ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32"
        if wl.feat_dtype == "f32" else "bf16-features/f32",
        "data": "synthetic (seeded da_inputs draw with the workload's shapes and distributions)",
        "config": config_of(wl, (f"L2 flushed before every step (a {2 * l2_bytes / 1e6:.0f} MB write outside "
                                 "the step's events; feature map "
                                 f"{feat_bytes / 1e6:.0f} MB)") if flush else
                            (f"no flush: feature map {feat_bytes / 1e6:.0f} MB"
                             + (" larger than L2" if feat_bytes >= 2 * l2_bytes else " (warm L2)"))),
        "channel_samples_per_s": value * (wl.num_embeds // wl.num_groups),
        # Effective gather bandwidth: every sample reads its four corner rows
        # (D channels each) once per pass when nothing is reused.
        "gather_gbs": (2 if wl.backward else 1) * wl.num_samples * 4 * (wl.num_embeds // wl.num_groups)
        * inp.feat.element_size() / (step_ms / 1e3) / 1e9,
        "gbs_step": (fwd_bytes + (bwd_bytes if wl.backward else 0)) / (step_ms / 1e3) / 1e9,
        "fwd_ms": statistics.mean(fwd_ms), "bwd_ms": statistics.mean(bwd_ms) if bwd_ms else None,
        "roofline": {"bound": "hbm", "kernel": step_kernel,
                     "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "algorithmic_bytes": step_bytes, "traffic": traffic,
                     "parts": parts},
        "e2e": e2e,
        "gpu_launches": a.steps * (1 + (bwd_launches(a.bwd_path, wl) if wl.backward else 0)),
        "bwd_path": a.bwd_path,
        "binning": "on a side stream during the forward (da_backward_bin)" if overlap else "inside da_backward",
        "workspace_bytes": int(ws.numel()) if ws is not None else 0,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    if graph is not None:
        line["graph"] = graph
    if world == 1 and not a.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(inp, a.cpu_anchors)
    print(json.dumps(line), flush=True)


def run_fused(a, wl):
    """The DCNv4 form (da_forward_fused + da_backward_fused, per-group points
    fused with their weights) on one GPU. Default workload: the DCNv4 page's
    kernel benchmark (its Table 10 excerpt: 56x56x128, batch 64, 4 groups,
    3x3 points), whose A100 kernel times the line quotes as context."""
    import deformable_view_feature_gb300 as da
    da.load_library()
    dev = torch.device("cuda", 0)
    inp = da_inputs.make_fused_inputs(wl)
    feat, lw, go = inp.feat.to(dev), inp.loc_weight.to(dev), inp.grad_out.to(dev)
    ss, ls = inp.spatial_shape, inp.level_start_index
    out = torch.empty(go.shape, device=dev)
    gf = torch.empty(feat.shape, device=dev)
    glw = torch.empty_like(lw)
    stream = torch.cuda.Stream(device=dev)
    fwd_bytes = tensor_bytes(feat, lw) + out.numel() * 4
    bwd_bytes = tensor_bytes(feat, lw, go) + 2 * gf.numel() * 4 + glw.numel() * 4
    # Default scatter: the binned rewrite measured slower on the DCNv4 shapes
    # (its 56x56 maps times 4 groups exceed the shared-memory binning).
    bwd_path = a.bwd_path if a.bwd_path in ("binned", "scatter") else "scatter"

    def step(ev=None):
        if ev is not None:
            ev[0].record(stream)
        da.da_forward_fused(feat, ss, ls, lw, out=out, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        if wl.backward:
            da.da_backward_fused(feat, ss, ls, lw, go, grad_feat=gf, grad_loc_weight=glw, stream=stream,
                                 path=bwd_path)
            if ev is not None:
                ev[2].record(stream)

    with torch.cuda.stream(stream):
        for _ in range(a.warmup):
            step()
    torch.cuda.synchronize(dev)
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(a.steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall0 = time.time()
    start.record(stream)
    for i in range(a.steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize(dev)
    t_wall1 = time.time()
    time.sleep(0.1)
    clocks.stop()
    ms = start.elapsed_time(end) / a.steps
    fwd_ms = statistics.mean(evs[i][0].elapsed_time(evs[i][1]) for i in range(a.steps))
    bwd_ms = statistics.mean(evs[i][1].elapsed_time(evs[i][2]) for i in range(a.steps)) if wl.backward else None
    peak, peak_kind = peaks()
    dom_ms, dom_bytes, dom = (bwd_ms, bwd_bytes, f"da_backward_fused ({bwd_path} path)") if wl.backward else \
        (fwd_ms, fwd_bytes, "da_forward_fused")
    achieved = dom_bytes / (dom_ms / 1e3) / 1e9
    line = {
        "metric": "fwd+bwd bilinear samples/sec, DCNv4 form (per-group points fused with weights)",
        "value": wl.num_samples / (ms / 1e3), "unit": "samples/s", "n_gpus": 1, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if wl.feat_dtype == "f32" else f"{wl.feat_dtype}-features/f32",
        "data": "synthetic (seeded da_inputs draw, per-group 3x3 grid points plus N(0, 1.5 px) offsets)",
        "config": {"workload": f"{wl.name}: B{wl.batch} {wl.shapes[0][0]}x{wl.shapes[0][1]} C{wl.num_embeds} "
                               f"G{wl.num_groups} P{wl.num_pts}, {wl.feat_dtype} features",
                   "samples_per_step": wl.num_samples,
                   "l2": "inputs and outputs larger than L2" if fwd_bytes > 129e6 else "fits in L2, no flush"},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "roofline": {"bound": "hbm", "kernel": dom, "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "algorithmic_bytes": dom_bytes, "traffic": None},
        "page_context": {"what": "DCNv4 page, Table 10 excerpt: DCNv4 CUDA kernel on A100 for this workload "
                                 "(another machine; context, not a target)",
                         "a100_kernel_ms": {"f32": 0.606, "f16": 0.404}.get(wl.feat_dtype),
                         "ours_fwd_ms": fwd_ms} if wl.name.startswith("dcnv4_table10") else None,
        "gpu_launches": a.steps * (1 + ((BWD_LAUNCHES[bwd_path]) if wl.backward else 0)),
        "bwd_path": bwd_path,
        "clocks": clocks.summary(t_wall0, t_wall1),
    }
    print(json.dumps(line), flush=True)


def _timed(step, stream, steps: int, warmup: int, phases: int):
    """Run warmup + timed steps of step(ev) on stream; step records ev[0..phases]
    around its phases. Returns (ms per step, [mean ms of each phase], clocks)."""
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            step(None)
    torch.cuda.synchronize()
    clocks = ClockSampler(0)
    clocks.start()
    time.sleep(0.3)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(phases + 1)] for _ in range(steps)]
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0 = time.time()
    start.record(stream)
    for i in range(steps):
        step(evs[i])
    end.record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    time.sleep(0.1)
    clocks.stop()
    per = [statistics.mean(evs[i][k].elapsed_time(evs[i][k + 1]) for i in range(steps)) for k in range(phases)]
    return start.elapsed_time(end) / steps, per, clocks.summary(t0, t1)


def run_projected(a, wl):
    """The projected layout at the training shape: da_forward_projected (key
    points projected into the cameras, softmax weights) + da_backward_projected
    (binned backward, chain rule to key points and logits)."""
    import deformable_view_feature_gb300 as da
    da.load_library()
    dev = torch.device("cuda", 0)
    inp = da_inputs.make_projected_inputs(wl)
    feat, kp, pr, z, go = (t.to(dev) for t in (inp.feat, inp.keypoints, inp.projection, inp.logits, inp.grad_out))
    ss, ls = inp.spatial_shape, inp.level_start_index
    stream = torch.cuda.Stream(device=dev)
    state = {}

    def step(ev):
        if ev is not None:
            ev[0].record(stream)
        out, loc, w = da.da_forward_projected(feat, ss, ls, kp, pr, inp.image_w, inp.image_h, z, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        state["g"] = da.da_backward_projected(feat, ss, ls, kp, pr, inp.image_w, inp.image_h, loc, w, go,
                                              stream=stream)
        if ev is not None:
            ev[2].record(stream)

    ms, (fwd_ms, bwd_ms), clocks = _timed(step, stream, a.steps, a.warmup, 2)
    # Compulsory bytes: every input read once, every output written once
    # (grad_feat counted twice, as in the headline line).
    n_w = z.numel() * 4  # logits, weights, grad_weight, grad_logits: one size
    n_loc = kp.numel() // 3 * inp.wl.num_cams * 2 * 4  # locations, grad_loc
    # backward reads feat, key points, cameras, locations, weights, grad_out;
    # writes grad_feat (zero-fill + write-back), grad_loc, grad_weight,
    # grad_keypoints, grad_logits.
    bwd_b = (tensor_bytes(feat, kp, pr, go) + n_loc + n_w + 2 * feat.numel() * 4 + n_loc + n_w
             + kp.numel() * 4 + n_w)
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": "fwd+bwd bilinear samples/sec, key points projected and weights normalised inside the forward",
        "value": wl.num_samples / (ms / 1e3), "unit": "samples/s", "n_gpus": 1, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic (anchors around the ego car, six-camera ring, N(0,1) logits)",
        "config": {"workload": f"{wl.name}: B{wl.batch} K{wl.num_cams} S{wl.num_scales} C{wl.num_embeds} "
                               f"G{wl.num_groups} A{wl.num_anchors} P{wl.num_pts}",
                   "samples_per_step": wl.num_samples, "l2": "inputs larger than L2, no flush"},
        "fwd_ms": fwd_ms, "bwd_ms": bwd_ms,
        "roofline": {"bound": "hbm", "kernel": "da_backward_projected (all its kernels)",
                     "achieved": bwd_b / (bwd_ms / 1e3) / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": bwd_b / (bwd_ms / 1e3) / 1e9 / peak, "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "algorithmic_bytes": bwd_b, "traffic": None},
        "gpu_launches": a.steps * (1 + bwd_launches("binned", wl) + 2),
        "clocks": clocks,
    }), flush=True)


def run_warpaffine(a):
    """The warpaffine preprocessing of the warpaffine page's benchmark
    (1920x1080 frames to 640x640, its §4.3), 64 frames per step: wa_preprocess
    (warp, BGR -> RGB, normalise, CHW) and wa_warpaffine_u8."""
    import deformable_view_feature_gb300 as da
    da.load_library()
    dev = torch.device("cuda", 0)
    inp = da_inputs.make_warpaffine_inputs(batch=64)
    src, d2i = inp.src.to(dev), inp.d2i.to(dev)
    stream = torch.cuda.Stream(device=dev)

    def step(ev):
        if ev is not None:
            ev[0].record(stream)
        da.warpaffine_preprocess(src, d2i, inp.dst_hw, inp.fill, stream=stream)
        if ev is not None:
            ev[1].record(stream)
        da.warpaffine_u8(src, d2i, inp.dst_hw, inp.fill, stream=stream)
        if ev is not None:
            ev[2].record(stream)

    ms, (pre_ms, u8_ms), clocks = _timed(step, stream, a.steps, a.warmup, 2)
    B = src.shape[0]
    npx = B * inp.dst_hw[0] * inp.dst_hw[1]
    pre_b = src.numel() + npx * 3 * 4
    peak, peak_kind = peaks()
    print(json.dumps({
        "metric": "frames/sec, 1920x1080 -> 640x640 warpaffine preprocessing (warp + RGB + normalise + CHW)",
        "value": B / (pre_ms / 1e3), "unit": "frames/s", "n_gpus": 1, "steps": a.steps, "warmup": a.warmup,
        "ms_per_step": ms, "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "u8->f32",
        "data": "synthetic (uniform random bytes, letterbox with random rotation and zoom)",
        "config": {"workload": f"warpaffine: {B} frames 1080x1920x3 uint8 -> 3x640x640 f32",
                   "l2": "inputs larger than L2 (398 MB of frames), no flush"},
        "preprocess_ms": pre_ms, "u8_ms": u8_ms, "u8_frames_per_s": B / (u8_ms / 1e3),
        "roofline": {"bound": "hbm", "kernel": "wa_preprocess", "achieved": pre_b / (pre_ms / 1e3) / 1e9,
                     "peak": peak, "unit": "GB/s", "frac": pre_b / (pre_ms / 1e3) / 1e9 / peak,
                     "peak_source": f"{peak_kind} hbm_gbs (copy)",
                     "algorithmic_bytes": pre_b, "traffic": None},
        "page_context": {"what": "warpaffine page §4.3: one 1080p frame to 640x640 on an RTX 3080 (another machine; "
                                 "context, not a target)", "fused_kernel_ms_per_frame": 0.8,
                         "ours_ms_per_frame": pre_ms / B},
        "gpu_launches": a.steps * 2,
        "clocks": clocks,
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="sp4d_train", choices=list(da_inputs.WORKLOADS))
    ap.add_argument("--e2e-steps", type=int, default=20,
                    help="steps of the end-to-end (host tensors) measurement; 0 skips it (profiling runs)")
    ap.add_argument("--cpu-anchors", type=int, default=1800,
                    help="anchors in the CPU-baseline sample")
    ap.add_argument("--ref-anchors", type=int, default=300,
                    help="anchors per step of --impl reference")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="also time the step captured in a CUDA graph (without an L2 flush)")
    ap.add_argument("--l2", choices=["auto", "flush", "none"], default="auto",
                    help="L2 flush before every step: auto = when the feature map is under twice the L2 size")
    ap.add_argument("--no-bin-overlap", action="store_true",
                    help="run the binned backward's binning inside da_backward instead of on a side stream "
                         "during the forward")
    ap.add_argument("--op", choices=["da", "fused", "projected", "warpaffine"], default="da",
                    help="da: the Sparse4D operator (the headline); fused: the DCNv4 form (default workload "
                         "dcnv4_table10); projected: projection and softmax fused in (sp4d_proj); "
                         "warpaffine: the frame preprocessing")
    ap.add_argument("--feat-dtype", choices=["f32", "bf16", "f16"], default=None,
                    help="override the workload's feature type (--op fused)")
    ap.add_argument("--batch", type=int, default=None,
                    help="override the workload's batch size (smaller cases for profiler captures; "
                         "the headline uses the workload's own)")
    ap.add_argument("--bwd-path", choices=["auto", "binned", "binned-det", "scatter"], default=None,
                    help="backward algorithm (binned needs a device workspace; binned-det is its "
                         "deterministic mode; auto is da_backward's default choice for the sizes). "
                         "Default: auto for --op da, scatter for --op fused")
    a = ap.parse_args()
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    if a.bwd_path is None and a.op == "da":
        a.bwd_path = "auto"
    if a.op in ("projected", "warpaffine"):
        if a.impl == "reference" or a.gpus != 1:
            ap.error(f"--op {a.op} runs our implementation on one GPU")
        if a.op == "projected":
            wl = da_inputs.WORKLOADS["sp4d_proj"]
            if a.batch is not None:
                wl = wl.replace(name=f"{wl.name}_b{a.batch}", batch=a.batch)
            run_projected(a, wl)
        else:
            run_warpaffine(a)
        return
    if a.op == "fused":
        wl = da_inputs.WORKLOADS["dcnv4_table10" if a.workload == "sp4d_train" else a.workload]
        if a.feat_dtype:
            wl = wl.replace(feat_dtype=a.feat_dtype)
        if a.impl == "reference" or a.gpus != 1:
            ap.error("--op fused runs our implementation on one GPU")
        run_fused(a, wl)
        return
    wl = da_inputs.WORKLOADS[a.workload]
    if a.batch is not None:
        wl = wl.replace(name=f"{wl.name}_b{a.batch}", batch=a.batch)
    if a.impl == "reference":
        run_reference(a, wl)
    else:
        run_ours(a, wl)
    if int(os.environ.get("WORLD_SIZE", "1")) > 1 and a.impl == "ours":
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
