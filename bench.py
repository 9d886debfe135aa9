"""Benchmark: batch-invariant RMSNorm fwd+bwd on GB300, reported as achieved HBM GB/s.

Workload (one step): rmsnorm_residual forward + backward at T=32768 rows,
D=4096, bf16 activations, fp32 gamma ~1+N(0,0.05), x/g/g_res ~N(0,1), eps=1e-6
— the configuration the metric is quoted on (the residual op's published
benchmark shape, RL-Kernel pull request 414 "[DSv4][P1-5] rmsnorm_residual",
Benchmarks). A step is three launches on one stream: the forward, backward
pass 1 (dx plus weight-gradient chunk partials) and pass 2 (fixed-order sum).

value = algorithmic bytes of the step (14*D + 8 bytes per row: x read, y and
x_copy written, rstd written; g, x, g_res and rstd read, dx written) / device
time of the step, summed over ranks (each rank runs its own replica: rows are
independent, so N GPUs process N batches with no exchange). Inputs are 1.9 GB
per step, far larger than the 129 MB L2, so no flush is needed between steps.

--impl reference times the float64 CPU oracle (the only reference: the pages
hold no runnable code) on bounded row samples of the same workload.
--workload gated times the Qwen3-Next gated step (262144 x 128) instead, as a
side line; it also serves as the fixed driver of the gated kernels' profile.
"""
from __future__ import annotations

import argparse
import hashlib
import re
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

T_ROWS, D_COLS, EPS = 32768, 4096, 1e-6
METRIC = "RMSNorm fwd+bwd HBM GB/s (% of GB300 peak) at T=32768, D=4096, bf16"
PAGES_H100_CUDA_MS = 10.043916  # residual fwd+bwd, T=32768, D=4096, H100 PCIe (context only)


def residual_config(world):
    """The benchmark's workload, the same for both arms."""
    return {"workload": "rmsnorm_residual fwd+bwd", "T": T_ROWS, "D": D_COLS,
            "io": "bf16 activations, fp32 gamma/rstd/dgamma", "eps": EPS, "zero_centered_gamma": False,
            "parallelism": f"replicas x{world}", "l2": "inputs 1.88 GB per step, larger than L2; no flush"}


def step_bytes(T, D):
    return T * (14 * D + 8)


def bwd_pass1_bytes(T, D):
    return T * (8 * D + 4)


def fwd_bytes(T, D):
    return T * (6 * D + 4)


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


# The files that build backward pass 1 at D=4096 and choose its launch shape;
# host-only conveniences of the library (noalloc.cu, host_step.cu) and the
# other activation format's instantiations are not among them.
KERNEL_SOURCES = ("api.cu", "common.cuh", "kernels.h", "reduce.cu", "wide.cu", "wide_impl.cuh")


def code_text(src: str) -> str:
    """C/C++ source without its comments and blank lines: what the compiler sees,
    so that an edit to a comment leaves the hash below unchanged."""
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    src = re.sub(r"//[^\n]*", "", src)
    return "\n".join(line.rstrip() for line in src.splitlines() if line.strip())


def source_hash(read=None):
    """Hash of the code (not the comments) of KERNEL_SOURCES; `read(name)` gives a
    file's text (default: the working tree)."""
    csrc = os.path.join(ROOT, "invariant_rmsnorm_gb300", "csrc")
    read = read or (lambda name: open(os.path.join(csrc, name)).read())
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        h.update(name.encode() + code_text(read(name)).encode())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per launch of backward pass 1, from the committed ncu summary —
    only while the kernel sources are the ones that were profiled."""
    p = os.path.join(ROOT, "profiles", "bwd_residual_T32768_D4096_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    if d.get("source_hash") != source_hash():
        return None
    return d.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []
        self.first = 0

    def mark(self):
        """Readings from here on are the ones reported (the GPU under load)."""
        self.first = len(self.lines)

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", self.gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._t = threading.Thread(target=self._read, daemon=True)
            self._t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self._t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in (self.lines[self.first:] or self.lines):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 8:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for nm, val in zip(names, parts[4:8]):
                if val.lower() == "active":
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU; replicas, no data exchange)
# ---------------------------------------------------------------------------
def dist_setup(n_gpus):
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    return rank, world, local


def dist_max(v):
    import torch
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        t = torch.tensor([float(v)], device="cuda" if torch.cuda.is_available() else "cpu")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        return float(t.item())
    return float(v)


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def run_ours(args):
    import torch

    import invariant_rmsnorm_gb300 as rn
    from invariant_rmsnorm_gb300 import synth

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    rn.load()
    T, D = T_ROWS, D_COLS
    wl = synth.residual(dev, seed=rank)
    y = torch.empty_like(wl.x)
    xc = torch.empty_like(wl.x)
    dx = torch.empty_like(wl.x)
    rstd = torch.empty(T, device=dev)
    dg = torch.empty(D, device=dev)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        rn.rmsnorm_residual_fwd(wl.x, wl.w, y, rstd, xc, EPS, False, stream=stream)
        if ev:
            ev[1].record(stream)
        rn.rmsnorm_residual_bwd(wl.g, wl.x, wl.w, rstd, wl.g_res, dx, None, ws, False, stream=stream)
        if ev:
            ev[2].record(stream)
        rn.rmsnorm_dgamma_reduce(ws, T, D, dg, stream=stream)
        if ev:
            ev[3].record(stream)

    # The clock sampler starts before the warm-up, so that its first reading
    # is taken while the GPU is idle and the warm-up then brings the clocks up
    # to their working level before the timed steps (a pause right before them
    # would let the GPU clock down and slow the first timed steps).
    gpu_id = "0"
    try:
        gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:
        gpu_id = str(dev.index or 0)
    sampler = ClockSampler(gpu_id)
    sampler.start()
    time.sleep(0.25)  # let the sampler take its first reading
    sampler.mark()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()

    # Per-kernel events bracket every 16th step only (from the 9th): an event recorded between
    # two kernels adds a small gap and stops the second from launching while
    # the first drains (programmatic dependent launch), so the sampled steps
    # run a little slower. The step time comes from the events around the loop.
    sampled = list(range(min(8, args.steps - 1), args.steps, 16))  # not the first step, which starts from an idle pipeline
    evs = {k: [torch.cuda.Event(enable_timing=True) for _ in range(4)] for k in sampled}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        step(evs.get(k))
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    total_ms = dist_max(start.elapsed_time(stop))
    fwd_ms = sum(e[0].elapsed_time(e[1]) for e in evs.values()) / len(evs)
    bwd_ms = sum(e[1].elapsed_time(e[2]) for e in evs.values()) / len(evs)
    red_ms = sum(e[2].elapsed_time(e[3]) for e in evs.values()) / len(evs)
    ms_per_step = total_ms / args.steps
    value = world * step_bytes(T, D) / (ms_per_step * 1e-3) / 1e9

    e2e = None
    extra = {}
    if not args.main_only:
        # End to end through the public API: every step copies its inputs from
        # pinned host memory, runs the step, and copies every output back.
        e2e_ms_serial, e2e_ms, h2d, d2h, e2e_same_bits = run_e2e(rn, wl, y, xc, dx, rstd, dg, ws, T, D, stream,
                                                                 max(3, min(20, args.steps)))
        e2e_value = world * step_bytes(T, D) / (e2e_ms * 1e-3) / 1e9
        e2e_serial_value = world * step_bytes(T, D) / (e2e_ms_serial * 1e-3) / 1e9
        e2e = {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
               "how": "rmsnorm_residual_step_host: 4096-row slabs, copies overlapped with the kernels inside the library",
               "bitwise_equal_to_unsliced_step": e2e_same_bits,
               "serial_value": round(e2e_serial_value, 2), "serial_ms_per_step": round(e2e_ms_serial, 4)}
        # side measurements (not part of `value`): other variants and shapes
        extra = side_measurements(rn, synth, dev, stream) if rank == 0 else {}
    # The dominant kernel launched back to back on its own (each launch chained
    # to the previous one by programmatic dependent launch, as in the step):
    # the sampled events above cost it its early launch, this does not.
    b2b = _time_gbs(lambda: rn.rmsnorm_residual_bwd(wl.g, wl.x, wl.w, rstd, wl.g_res, dx, None, ws, False,
                                                    stream=stream),
                    bwd_pass1_bytes(T, D), 200, stream)
    # The forward the same way: its roofline figure comes from this run, not
    # from the sampled steps' events (which cost it its early launch too).
    f2f = _time_gbs(lambda: rn.rmsnorm_residual_fwd(wl.x, wl.w, y, rstd, xc, EPS, False, stream=stream),
                    fwd_bytes(T, D), 200, stream)

    with_cpu = rank == 0 and world == 1 and not args.no_cpu_baseline and not args.main_only
    cpu = cpu_baseline_sample(gpu={"x": wl.x, "w": wl.w, "g": wl.g, "g_res": wl.g_res, "y": y, "x_copy": xc,
                                   "dx": dx, "rstd": rstd}) if with_cpu else None
    if with_cpu:
        extra["gated_262144x128_cpu_baseline"] = cpu_gated_sample()
        extra["tiny_16x128_cpu_baseline"] = cpu_tiny_sample()
    peak, peak_kind = peaks()
    bwd_gbs = bwd_pass1_bytes(T, D) / (bwd_ms * 1e-3) / 1e9
    traffic = recorded_traffic()
    if rank == 0:
        out = {
            "metric": METRIC, "value": round(value, 2), "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak",
            "vs_baseline": round((PAGES_H100_CUDA_MS / ms_per_step) * world, 3),
            "vs_baseline_basis": "pages' H100 PCIe residual fwd+bwd at the same shape (10.043916 ms); context only",
            "dtype": "f32", "data": "synthetic",
            "config": residual_config(world),
            "pct_of_peak": round(100.0 * value / (world * peak), 2),
            "rows_per_s": round(world * T / (ms_per_step * 1e-3)),
            "kernels_ms": {"fwd": round(fwd_ms, 5), "bwd_pass1": round(bwd_ms, 5), "dgamma_pass2": round(red_ms, 5),
                           "sampled_steps": len(evs),
                           "note": "events between the kernels of every 16th step; they delay each kernel's "
                                   "early launch, so these read slower than the back-to-back figures"},
            "roofline": {"kernel": "wide_bwd_kernel (residual, pass 1)", "bound": "hbm",
                         "achieved": round(bwd_gbs, 2), "peak": peak, "unit": "GB/s",
                         "frac": round(bwd_gbs / peak, 4), "peak_kind": peak_kind,
                         "traffic": traffic, "algorithmic_bytes_per_launch": bwd_pass1_bytes(T, D)},
            "fwd_roofline": {"kernel": "wide_fwd_kernel (residual)", "achieved": f2f["gbs"], "peak": peak,
                             "frac": round(f2f["gbs"] / peak, 4), "us": round(f2f["ms"] * 1e3, 2),
                             "how": "200 launches back to back on the stream, CUDA events around the run",
                             "sampled_steps_gbs": round(fwd_bytes(T, D) / (fwd_ms * 1e-3) / 1e9, 2)},
            "e2e": e2e,
            "gpu_launches": 3 * args.steps,
            "clocks": clocks,
            "bwd_pass1_back_to_back": {"us": round(b2b["ms"] * 1e3, 2), "gbs": b2b["gbs"],
                                       "frac": round(b2b["gbs"] / peak, 4), "launches": 200},
            "cpu_baseline": cpu,
            "extra": extra,
        }
        print(json.dumps(out))
    barrier()


def run_gated(args):
    """`--workload gated`: the Qwen3-Next gated norm step (forward, backward
    pass 1 with dx and dz, weight-gradient pass 2) over 8192 tokens x 32 heads
    = 262144 rows of head_v_dim 128, zero-centred weight, silu gate. Device
    timing only (the same protocol as the default workload); this is a side
    line and the fixed driver of the gated kernels' ncu profile."""
    import torch

    import invariant_rmsnorm_gb300 as rn
    from invariant_rmsnorm_gb300 import synth

    rank, world, local = dist_setup(args.gpus)
    dev = torch.device("cuda", local if world > 1 else 0)
    torch.cuda.set_device(dev)
    rn.load()
    g = synth.gated(dev, seed=rank)
    T, D = g.T, g.D
    y, dx, dz = torch.empty_like(g.x), torch.empty_like(g.x), torch.empty_like(g.x)
    rstd, dw = torch.empty(T, device=dev), torch.empty(D, device=dev)
    ws = torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        rn.rmsnorm_gated_fwd(g.x, g.z, g.w, y, rstd, EPS, True, stream=stream)
        if ev:
            ev[1].record(stream)
        rn.rmsnorm_gated_bwd(g.g, g.x, g.z, g.w, rstd, dx, dz, None, ws, True, stream=stream)
        if ev:
            ev[2].record(stream)
        rn.rmsnorm_dgamma_reduce(ws, T, D, dw, stream=stream)
        if ev:
            ev[3].record(stream)

    sampler = ClockSampler(str(dev.index or 0))
    sampler.start()
    time.sleep(0.25)  # first reading while idle; the warm-up then brings the clocks up
    sampler.mark()
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    sampled = list(range(min(8, args.steps - 1), args.steps, 16))  # not the first step, which starts from an idle pipeline
    evs = {k: [torch.cuda.Event(enable_timing=True) for _ in range(4)] for k in sampled}
    start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    start.record(stream)
    for k in range(args.steps):
        step(evs.get(k))
    stop.record(stream)
    torch.cuda.synchronize()
    clocks = sampler.stop()
    barrier()
    ms_per_step = dist_max(start.elapsed_time(stop)) / args.steps
    kms = [sum(e[i].elapsed_time(e[i + 1]) for e in evs.values()) / len(evs) for i in range(3)]
    nbytes = T * (16 * D + 8)  # fwd 6D+4 (x, z in; y, rstd out) + bwd 10D+4 (g, x, z, rstd in; dx, dz out)
    value = world * nbytes / (ms_per_step * 1e-3) / 1e9
    peak, peak_kind = peaks()
    bwd_bytes = T * (10 * D + 4)
    # each kernel launched back to back on its own (no events between kernels)
    b2b = _time_gbs(lambda: rn.rmsnorm_gated_bwd(g.g, g.x, g.z, g.w, rstd, dx, dz, None, ws, True, stream=stream),
                    bwd_bytes, 200, stream)
    f2f = _time_gbs(lambda: rn.rmsnorm_gated_fwd(g.x, g.z, g.w, y, rstd, EPS, True, stream=stream),
                    T * (6 * D + 4), 200, stream)
    if rank == 0:
        print(json.dumps({
            "metric": "gated RMSNorm fwd+bwd HBM GB/s at 262144 x 128, bf16", "value": round(value, 2),
            "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(ms_per_step, 5), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32", "data": "synthetic",
            "config": {"workload": "gated zero-centred RMSNorm fwd+bwd (Qwen3-Next)", "T": T, "D": D,
                       "gate": "silu", "eps": EPS, "parallelism": f"replicas x{world}",
                       "l2": "inputs 0.54 GB per step, larger than L2; no flush"},
            "pct_of_peak": round(100.0 * value / (world * peak), 2),
            "rows_per_s": round(world * T / (ms_per_step * 1e-3)),
            "kernels_ms": {"fwd": round(kms[0], 5), "bwd_pass1": round(kms[1], 5), "dgamma_pass2": round(kms[2], 5),
                           "sampled_steps": len(evs)},
            "roofline": {"kernel": "narrow_bwd_kernel (gated, pass 1)", "bound": "hbm",
                         "achieved": b2b["gbs"], "peak": peak, "unit": "GB/s",
                         "frac": round(b2b["gbs"] / peak, 4), "peak_kind": peak_kind, "us": round(b2b["ms"] * 1e3, 2),
                         "how": "200 launches back to back on the stream, CUDA events around the run",
                         "traffic": None, "algorithmic_bytes_per_launch": bwd_bytes},
            "fwd_roofline": {"kernel": "narrow_fwd_kernel (gated)", "achieved": f2f["gbs"], "peak": peak,
                             "frac": round(f2f["gbs"] / peak, 4), "us": round(f2f["ms"] * 1e3, 2)},
            "gpu_launches": 3 * args.steps, "clocks": clocks}))
    barrier()


def run_e2e(rn, wl, y, xc, dx, rstd, dg, ws, T, D, stream, steps, slab=4096):
    """Time the residual step end to end through the C ABI with pinned host
    buffers, twice: serially on one stream (copies in, the two device entry
    points, copies out), and through rmsnorm_residual_step_host, which
    pipelines row slabs inside the library (copies of slab k+1 in and slab k-1
    out overlap the kernels of slab k). Its outputs are checked bitwise
    against the serial step's.
    Returns (serial ms, pipelined ms, H2D bytes, D2H bytes, bits equal)."""
    import torch
    dev = wl.x.device
    h_in = [t.cpu().pin_memory() for t in (wl.x, wl.g, wl.g_res)]
    h_w = wl.w.cpu().pin_memory()
    d_in = [torch.empty_like(t) for t in (wl.x, wl.g, wl.g_res)]
    d_w = torch.empty_like(wl.w)
    outs = (y, xc, dx, rstd, dg)
    h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = sum(t.numel() * t.element_size() for t in h_in) + h_w.numel() * 4
    d2h = sum(t.numel() * t.element_size() for t in h_out)

    def serial_step():
        for h, d in zip(h_in, d_in):
            d.copy_(h, non_blocking=True)
        d_w.copy_(h_w, non_blocking=True)
        rn.rmsnorm_residual_fwd(d_in[0], d_w, y, rstd, xc, EPS, False, stream=stream)
        rn.rmsnorm_residual_bwd(d_in[1], d_in[0], d_w, rstd, d_in[2], dx, dg, ws, False, stream=stream)
        for h, d in zip(h_out, outs):
            h.copy_(d, non_blocking=True)

    # The pipelined step is one library call: rmsnorm_residual_step_host cuts
    # the rows into slabs and overlaps each slab's copies with the kernels of
    # its neighbours on the library's own copy streams.
    work = torch.empty(rn.rmsnorm_residual_step_host_work_bytes(T, D, slab), dtype=torch.uint8, device=dev)

    def pipelined_step():
        rn.rmsnorm_residual_step_host(h_in[0], h_in[1], h_in[2], h_w, h_out[0], h_out[1], h_out[3], h_out[2],
                                      h_out[4], work, EPS, False, slab_rows=slab, stream=stream)

    def timed(fn):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(steps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize()
        return dist_max(e0.elapsed_time(e1)) / steps

    ms_serial = timed(serial_step)
    ref = [h.clone() for h in h_out]
    ms_pipe = timed(pipelined_step)
    same = all(torch.equal(a.view(torch.uint8), b.view(torch.uint8)) for a, b in zip(ref, h_out))
    return ms_serial, ms_pipe, h2d, d2h, same


def side_measurements(rn, synth, dev, stream, reps=50):
    """Side lines (not part of `value`): other variants and the pages' other
    shapes, each timed back to back on the stream with inputs resident. Every
    entry gives ms per call, GB/s of algorithmic bytes, the fraction of the
    measured HBM peak and rows/s."""
    import torch
    peak, _ = peaks()
    res = {}

    def rec(name, fn, T, per_row):
        r = _time_gbs(fn, T * per_row, reps, stream)
        r["frac"] = round(r["gbs"] / peak, 4)
        r["rows_per_s"] = round(T / (r["ms"] * 1e-3))
        r["T"], r["bytes_per_row"] = T, per_row
        res[name] = r

    def buffers(T, D):
        return (torch.empty(T, device=dev), torch.empty(D, device=dev),
                torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=dev))

    # plain fwd+bwd, same shape (the metric's literal op): 10*D + 8 bytes per row
    T, D = T_ROWS, D_COLS
    wl = synth.tiny_plain(dev, seed=3, T=T, D=D)
    y, dx = torch.empty_like(wl.x), torch.empty_like(wl.x)
    r, dg, ws = buffers(T, D)

    def plain():
        rn.rmsnorm_fwd(wl.x, wl.w, y, r, EPS, False, stream=stream)
        rn.rmsnorm_bwd(wl.g, wl.x, wl.w, r, dx, dg, ws, False, stream=stream)
    rec("plain_fwd_bwd_gbs", plain, T, 10 * D + 8)
    del wl, y, dx, r, dg, ws
    # the tiny problem (T=16, D=128, zero-centred gamma off and on): launch-bound, reported per step
    for zc in (False, True):
        wl = synth.tiny_plain(dev, seed=0, zero_centered_gamma=zc)
        y, dx = torch.empty_like(wl.x), torch.empty_like(wl.x)
        r, dg, ws = buffers(wl.T, wl.D)

        def tiny():
            rn.rmsnorm_fwd(wl.x, wl.w, y, r, EPS, zc, stream=stream)
            rn.rmsnorm_bwd(wl.g, wl.x, wl.w, r, dx, dg, ws, zc, stream=stream)
        rec(f"tiny_16x128_zc{int(zc)}_fwd_bwd", tiny, wl.T, 10 * wl.D + 8)
        del wl, y, dx, r, dg, ws
    # the large sweep: plain fwd+bwd with 0.1 % outlier entries, 10*D + 8 bytes per row
    for T, D in ((131072, 2048), (131072, 4096), (131072, 7168), (131072, 8192), (262144, 4096)):
        wl = synth.large(dev, seed=1, T=T, D=D)
        y, dx = torch.empty_like(wl.x), torch.empty_like(wl.x)
        r, dg, ws = buffers(T, D)

        def large():
            rn.rmsnorm_fwd(wl.x, wl.w, y, r, EPS, False, stream=stream)
            rn.rmsnorm_bwd(wl.g, wl.x, wl.w, r, dx, dg, ws, False, stream=stream)
        rec(f"large_{T}x{D}_fwd_bwd_gbs", large, T, 10 * D + 8)
        del wl, y, dx, r, dg, ws
    # the residual step at the pages' two larger row counts (D = 4096): 14*D + 8 bytes per row
    for T in (131072, 262144):
        wl = synth.residual(dev, seed=11, T=T, D=D)
        y, xc, dx = torch.empty_like(wl.x), torch.empty_like(wl.x), torch.empty_like(wl.x)
        r, dg, ws = buffers(T, D)

        def step():
            rn.rmsnorm_residual_fwd(wl.x, wl.w, y, r, xc, EPS, False, stream=stream)
            rn.rmsnorm_residual_bwd(wl.g, wl.x, wl.w, r, wl.g_res, dx, dg, ws, False, stream=stream)
        rec(f"residual_{T}x{D}_fwd_bwd_gbs", step, T, 14 * D + 8)
        del wl, y, xc, dx, r, dg, ws
    # gated: Qwen3-Next 262144 x 128, and wide rows: 16*D + 8 bytes per row
    for T, D in ((262144, 128), (32768, 7168), (32768, 8192)):
        g = synth.gated(dev, seed=4, T=T, D=D)
        y, dx, dz = torch.empty_like(g.x), torch.empty_like(g.x), torch.empty_like(g.x)
        r, dw, ws = buffers(T, D)

        def gated():
            rn.rmsnorm_gated_fwd(g.x, g.z, g.w, y, r, EPS, True, stream=stream)
            rn.rmsnorm_gated_bwd(g.g, g.x, g.z, g.w, r, dx, dz, dw, ws, True, stream=stream)
        rec(f"gated_{T}x{D}_fwd_bwd_gbs", gated, T, 16 * D + 8)
        if D == 128:
            res[f"gated_{T}x{D}_fwd_bwd_gbs"]["note"] = (
                "buffers carved from memory freed by the earlier side lines, a placement that runs this "
                "step faster than freshly allocated buffers do (--workload gated times those)")
        del g, y, dx, dz, r, dw, ws
    # fused add + norm: 18*D + 8 bytes per row (x, res in; y, res_out, rstd out;
    # g, x, res, g_res, rstd in; dh out); the decoder shape 32768 x 2048 and wide rows
    for T, D in ((32768, 2048), (32768, 7168), (32768, 8192)):
        x = synth.normal_bf16((T, D), 5, dev)
        rs = synth.normal_bf16((T, D), 6, dev, std=4.0)
        gg = synth.normal_bf16((T, D), 7, dev)
        gr = synth.normal_bf16((T, D), 8, dev)
        w = synth.gamma_f32(D, 9, dev)
        y, ro, dh = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
        r, dw, ws = buffers(T, D)

        def fused():
            rn.rmsnorm_fused_add_fwd(x, rs, w, y, r, ro, EPS, False, stream=stream)
            rn.rmsnorm_fused_add_bwd(gg, x, rs, w, r, gr, dh, dw, ws, False, stream=stream)
        rec(f"fused_add_{T}x{D}_fwd_bwd_gbs", fused, T, 18 * D + 8)
        del x, rs, gg, gr, w, y, ro, dh, r, dw, ws
    # the widest rows: plain backward (pass 1 and 2) at 32768 x 16384, 6*D + 4 bytes per row
    T, D = 32768, 16384
    wl = synth.tiny_plain(dev, seed=12, T=T, D=D)
    y, dx = torch.empty_like(wl.x), torch.empty_like(wl.x)
    r, dg, ws = buffers(T, D)
    rn.rmsnorm_fwd(wl.x, wl.w, y, r, EPS, False, stream=stream)
    rec(f"plain_bwd_{T}x{D}_gbs", lambda: rn.rmsnorm_bwd(wl.g, wl.x, wl.w, r, dx, dg, ws, False, stream=stream),
        T, 6 * D + 4)
    rec(f"plain_fwd_{T}x{D}_gbs", lambda: rn.rmsnorm_fwd(wl.x, wl.w, y, r, EPS, False, stream=stream), T, 4 * D + 4)
    del wl, y, dx, r, dg, ws
    # the widest rows in the modes that stream three or four operands a row (CTA
    # pairs): residual (8*D + 4 bytes per row), gated and fused add (10*D + 4)
    x = synth.normal_bf16((T, D), 13, dev)
    z = synth.normal_bf16((T, D), 14, dev)
    gg = synth.normal_bf16((T, D), 15, dev)
    gr = synth.normal_bf16((T, D), 16, dev)
    w = synth.gamma_f32(D, 17, dev)
    y, dx, dz = torch.empty_like(x), torch.empty_like(x), torch.empty_like(x)
    r, dg, ws = buffers(T, D)
    rn.rmsnorm_fwd(x, w, y, r, EPS, False, stream=stream)
    rec(f"residual_bwd_{T}x{D}_gbs",
        lambda: rn.rmsnorm_residual_bwd(gg, x, w, r, gr, dx, dg, ws, False, stream=stream), T, 8 * D + 4)
    rec(f"gated_bwd_{T}x{D}_gbs",
        lambda: rn.rmsnorm_gated_bwd(gg, x, z, w, r, dx, dz, dg, ws, True, stream=stream), T, 10 * D + 4)
    rec(f"fused_add_bwd_{T}x{D}_gbs",
        lambda: rn.rmsnorm_fused_add_bwd(gg, x, z, w, r, gr, dx, dg, ws, False, stream=stream), T, 10 * D + 4)
    del x, z, gg, gr, w, y, dx, dz, r, dg, ws
    return res


def _time_gbs(fn, nbytes, reps, stream):
    import torch
    for _ in range(5):
        fn()
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    a.record(stream)
    for _ in range(reps):
        fn()
    b.record(stream)
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / reps
    return {"gbs": round(nbytes / (ms * 1e-3) / 1e9, 2), "ms": round(ms, 5)}


# ---------------------------------------------------------------------------
# CPU baseline / reference arm: the float64 oracle, as it stands
# ---------------------------------------------------------------------------
def _oracle_sample(rows, seed=0):
    import numpy as np

    from invariant_rmsnorm_gb300 import synth
    wl = synth.residual("cpu", seed=seed, T=rows, D=D_COLS)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    return f(wl.x), f(wl.w), f(wl.g), f(wl.g_res)


def _oracle_step(arrs):
    import oracle
    x, w, g, gr = arrs
    y, r, xc = oracle.residual_fwd(x, w, EPS, False)
    oracle.residual_bwd(g, x, w, r, gr, False)


def _bf16_ulp(v):
    """One bf16 ulp at each value (normal range; the subnormal quantum below it)."""
    import numpy as np
    _, e = np.frexp(np.abs(v))
    return np.ldexp(1.0, np.maximum(e - 8, -133))


def _ulp_histogram(got, ref, pre=None, scale=None):
    """Distance of the GPU's bf16 outputs from the oracle's correctly rounded ones:
    how many are equal, one bf16 ulp away, further but within the cancellation
    clause (|got - unrounded| <= ulp/2 + 96 * 2^-24 * scale), and beyond."""
    import numpy as np
    d = np.abs(got - ref) / _bf16_ulp(ref)
    h = {"0": int(np.sum(d == 0)), "1": int(np.sum((d > 0) & (d <= 1)))}
    beyond = d > 1
    if pre is not None:
        canc = beyond & (np.abs(got - pre) <= 0.5 * _bf16_ulp(ref) + 96 * 2.0**-24 * scale)
        h["cancellation"] = int(np.sum(canc))
        beyond &= ~canc
    h["beyond"] = int(np.sum(beyond))
    return h


def cpu_baseline_sample(target_s=10.0, gpu=None, rows=2048):
    """The float64 oracle timed on repeated row samples of the workload. With
    `gpu` (the benchmark's input and output tensors), the sample is the first
    `rows` rows of the benchmark's own workload, and the oracle's results on it
    are also compared with the GPU's outputs for those rows (bf16 ulp
    histograms of y and dx, rstd's largest relative error, the copy bitwise)."""
    import numpy as np

    import oracle
    acc = None
    if gpu is not None:
        f = lambda t: t[:rows].float().cpu().numpy().astype(np.float64)  # noqa: E731
        arrs = (f(gpu["x"]), gpu["w"].float().cpu().numpy().astype(np.float64), f(gpu["g"]), f(gpu["g_res"]))
        x, w, g, gr = arrs
        y_ref, r_ref, _ = oracle.residual_fwd(x, w, EPS, False)
        r_gpu = gpu["rstd"][:rows].cpu().numpy().astype(np.float64)
        dx_ref, _, diag = oracle.residual_bwd(g, x, w, r_gpu, gr, False, diagnostics=True)
        acc = {"rows": rows, "of": int(gpu["x"].shape[0]),
               "y_ulp": _ulp_histogram(f(gpu["y"]), y_ref),
               "dx_ulp": _ulp_histogram(f(gpu["dx"]), dx_ref, diag["dx_pre"], diag["dx_scale"]),
               "rstd_max_rel_err": float(np.max(np.abs(r_gpu - r_ref) / r_ref)),
               "x_copy_bitwise": bool(np.array_equal(f(gpu["x_copy"]), x)),
               "bar": "y, dx within 1 bf16 ulp of the oracle's correctly rounded value (dx: or the "
                      "cancellation clause); rstd within 1e-5 relative"}
    else:
        arrs = _oracle_sample(rows)
    _oracle_step(arrs)
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < target_s:
        _oracle_step(arrs)
        n += 1
    dt = time.perf_counter() - t0
    out = {"value": round(n * step_bytes(rows, D_COLS) / dt / 1e9, 4), "unit": "GB/s",
           "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"{n} repetitions of {rows} rows x {D_COLS} (residual fwd+bwd, float64 C oracle), {dt:.1f} s"}
    if acc is not None:
        out["accuracy_of_the_gpu_outputs_on_the_sample"] = acc
    return out


def cpu_gated_sample(target_s=5.0, rows=8192):
    """The oracle on the gated step (forward, backward with dx, dz and the weight
    gradient) on repeated row samples of the 262144 x 128 Qwen3-Next workload."""
    import numpy as np

    import oracle
    from invariant_rmsnorm_gb300 import synth
    g = synth.gated("cpu", seed=0, T=rows)
    f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    x, z, w, gg = f(g.x), f(g.z), f(g.w), f(g.g)

    def step():
        _, r = oracle.gated_fwd(x, z, w, EPS, True)
        oracle.gated_bwd(gg, x, z, w, r, True)
    step()
    t0 = time.perf_counter()
    n = 0
    while time.perf_counter() - t0 < target_s:
        step()
        n += 1
    dt = time.perf_counter() - t0
    D = g.D
    return {"value": round(n * rows * (16 * D + 8) / dt / 1e9, 4), "unit": "GB/s",
            "rows_per_s": round(n * rows / dt), "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{n} repetitions of {rows} rows x {D} (gated fwd+bwd, float64 C oracle), {dt:.1f} s"}


def cpu_tiny_sample(reps=200):
    """The oracle on the tiny plain fwd+bwd (T=16, D=128, zero-centred gamma
    off and on): wall clock per call, best of 3 runs of `reps` calls."""
    import numpy as np

    import oracle
    from invariant_rmsnorm_gb300 import synth
    res = {}
    for zc in (False, True):
        wl = synth.tiny_plain("cpu", seed=0, zero_centered_gamma=zc)
        f = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
        x, w, g = f(wl.x), f(wl.w), f(wl.g)
        best = float("inf")
        for _ in range(3):
            t0 = time.perf_counter()
            for _ in range(reps):
                _, r = oracle.rmsnorm_fwd(x, w, EPS, zc)
                oracle.rmsnorm_bwd(g, x, w, r, zc)
            best = min(best, (time.perf_counter() - t0) / reps)
        res[f"zero_centered_gamma={zc}"] = {"us_per_step": round(best * 1e6, 2),
                                             "rows_per_s": round(wl.T / best)}
    res.update({"cores": oracle.num_threads(), "kind": "oracle",
                "sample": f"best of 3 runs of {reps} fwd+bwd calls on the whole 16 x 128 problem"})
    return res


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return
    import oracle
    # size each step so that warmup + steps take about two minutes at most
    probe_rows = 64
    arrs = _oracle_sample(probe_rows, seed=1)
    t0 = time.perf_counter()
    _oracle_step(arrs)
    per_row = (time.perf_counter() - t0) / probe_rows
    budget = 120.0 / max(1, args.steps + args.warmup)
    rows = int(max(8, min(4096, budget / max(per_row, 1e-9))))
    arrs = _oracle_sample(rows, seed=2)
    for _ in range(args.warmup):
        _oracle_step(arrs)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        _oracle_step(arrs)
    dt = time.perf_counter() - t0
    value = args.steps * step_bytes(rows, D_COLS) / dt / 1e9
    out = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(1e3 * dt / args.steps, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": residual_config(world),
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": f"{rows} of {T_ROWS} rows per step, float64 C oracle"},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(out))


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true", help="skip the timed CPU-oracle sample")
    ap.add_argument("--main-only", action="store_true",
                    help="the timed steps and the back-to-back kernel runs only: no end-to-end run, side lines or "
                         "CPU samples (a small, fixed driver for profiler captures; the line then has no e2e)")
    ap.add_argument("--workload", choices=("residual", "gated"), default="residual",
                    help="residual: the benchmark line (default); gated: the 262144 x 128 gated step, device "
                         "timing only")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.impl == "reference":
        run_reference(args)
    elif args.workload == "gated":
        run_gated(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
