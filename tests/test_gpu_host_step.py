"""The rmsnorm_residual step on host buffers (rmsnorm_residual_step_host).

One call copies the host inputs in, runs the residual forward and backward and
copies every output back, pipelined in row slabs inside the library. Its
outputs must be bitwise those of the device entry points on the same inputs
(unsliced), whatever the slab size: the row outputs because every row is
reduced on its own, the weight gradient because slabs are whole chunks and
pass 2 runs once over all of them. Slab sizes down to one chunk exercise the
ring of three slots many times over; ragged T leaves a short last slab.
"""
from __future__ import annotations

import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV, check_bwd, check_fwd, run_bwd, run_fwd

pytestmark = pytest.mark.gpu

EPS = 1e-6


def _inputs(T, D, seed, dtype, zc, with_gres=True):
    x = synth.normal16((T, D), seed, DEV, dtype=dtype)
    g = synth.normal16((T, D), seed + 1, DEV, dtype=dtype)
    gr = synth.normal16((T, D), seed + 2, DEV, dtype=dtype) if with_gres else None
    w = synth.gamma_f32(D, seed + 3, DEV, mean=0.0 if zc else 1.0, std=0.1)
    return x, g, gr, w


def _host_step(x, g, gr, w, zc, slab_rows=0, pin=True, stream=None):
    """Host copies of the inputs, one call, host outputs (after a sync)."""
    T, D = x.shape
    h = (lambda t: t.cpu().pin_memory()) if pin else (lambda t: t.cpu())
    hx, hg, hw = h(x), h(g), h(w)
    hgr = h(gr) if gr is not None else None
    mk = (lambda *s, dt: torch.empty(s, dtype=dt, pin_memory=True)) if pin else \
        (lambda *s, dt: torch.empty(s, dtype=dt))
    out = {"y": mk(T, D, dt=x.dtype), "x_copy": mk(T, D, dt=x.dtype), "rstd": mk(T, dt=torch.float32),
           "dx": mk(T, D, dt=x.dtype), "dgamma": mk(D, dt=torch.float32)}
    work = torch.empty(rn.rmsnorm_residual_step_host_work_bytes(T, D, slab_rows), dtype=torch.uint8, device=DEV)
    rn.rmsnorm_residual_step_host(hx, hg, hgr, hw, out["y"], out["x_copy"], out["rstd"], out["dx"], out["dgamma"],
                                  work, EPS, zc, slab_rows=slab_rows, stream=stream)
    torch.cuda.synchronize()
    return out


def _device_step(x, g, gr, w, zc):
    fo = run_fwd("residual", x, w, EPS, zc, ex=True)
    bo = run_bwd("residual", g, x, w, fo["rstd"], zc, g_res=gr, ex=True)
    torch.cuda.synchronize()
    return {"y": fo["y"], "x_copy": fo["x_copy"], "rstd": fo["rstd"], "dx": bo["dx"], "dgamma": bo["dgamma"]}


def _bits(t):
    t = t.contiguous().cpu()
    return t.view(torch.int16) if t.element_size() == 2 else t.view(torch.int32)


def _assert_same(host, dev, name):
    for k in ("y", "x_copy", "rstd", "dx", "dgamma"):
        assert torch.equal(_bits(host[k]), _bits(dev[k])), f"{name}: {k} differs from the device entry points"


@pytest.mark.parametrize("T,D,slab,dtype", [
    (1, 8, 0, torch.bfloat16),
    (100, 64, 0, torch.bfloat16),          # narrow rows, one slab
    (1000, 128, 64, torch.float16),        # narrow, many slabs (ring reused)
    (777, 264, 32, torch.bfloat16),        # wide, one chunk per slab, ragged tail
    (4097, 4096, 0, torch.bfloat16),       # default slab, one-row last slab
    (3000, 4096, 512, torch.float16),
    (10000, 4096, 1000, torch.bfloat16),   # 17-row chunks: slabs of 1003 rows
    (257, 16384, 96, torch.bfloat16),      # widest rows
])
def test_host_step_matches_device_entry_points(T, D, slab, dtype):
    zc = (T % 2) == 1
    x, g, gr, w = _inputs(T, D, T + D, dtype, zc)
    host = _host_step(x, g, gr, w, zc, slab_rows=slab)
    dev = _device_step(x, g, gr, w, zc)
    _assert_same(host, dev, f"T={T} D={D} slab={slab} {dtype}")


def test_host_step_parity_with_oracle():
    """A small case against the oracle directly (outputs within one ulp, rstd
    1e-5 relative, weight gradient 1e-4 relative or the tree's bound)."""
    T, D = 203, 384
    x, g, gr, w = _inputs(T, D, 11, torch.bfloat16, True)
    host = _host_step(x, g, gr, w, True, slab_rows=64)
    fo = {k: host[k].to(DEV) for k in ("y", "x_copy", "rstd")}
    bo = {k: host[k].to(DEV) for k in ("dx", "dgamma")}
    check_fwd("residual", x, w, EPS, True, fo, name="host step")
    check_bwd("residual", g, x, w, fo["rstd"], True, bo, g_res=gr, name="host step")


def test_host_step_without_residual_gradient_and_pageable():
    """g_res = NULL means zero; pageable host memory gives the same bits."""
    T, D = 600, 2048
    x, g, _, w = _inputs(T, D, 5, torch.bfloat16, False, with_gres=False)
    dev = _device_step(x, g, None, w, False)
    _assert_same(_host_step(x, g, None, w, False, slab_rows=128), dev, "no g_res, pinned")
    _assert_same(_host_step(x, g, None, w, False, slab_rows=128, pin=False), dev, "no g_res, pageable")


def test_host_step_back_to_back_on_one_stream():
    """Two calls on one side stream share one work buffer with different inputs
    and no host sync between them: the second waits for the first."""
    T, D = 2048, 1024
    s = torch.cuda.Stream()
    cases = [_inputs(T, D, 40 + i, torch.bfloat16, False) for i in range(2)]
    work = torch.empty(rn.rmsnorm_residual_step_host_work_bytes(T, D, 256), dtype=torch.uint8, device=DEV)
    outs = []
    for x, g, gr, w in cases:
        hx, hg, hgr, hw = (t.cpu().pin_memory() for t in (x, g, gr, w))
        o = {"y": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
             "x_copy": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
             "rstd": torch.empty(T, pin_memory=True), "dx": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
             "dgamma": torch.empty(D, pin_memory=True)}
        rn.rmsnorm_residual_step_host(hx, hg, hgr, hw, o["y"], o["x_copy"], o["rstd"], o["dx"], o["dgamma"], work,
                                      EPS, False, slab_rows=256, stream=s)
        outs.append((o, (hx, hg, hgr, hw)))
    s.synchronize()
    for i, ((x, g, gr, w), (o, _)) in enumerate(zip(cases, outs)):
        _assert_same(o, _device_step(x, g, gr, w, False), f"call {i}")


def test_host_step_in_a_cuda_graph():
    """Captured in a CUDA graph, after one call outside capture has created the
    library's copy streams: the copy streams fork from and join the captured
    stream, and every replay gives the device entry points' bits."""
    T, D = 1000, 512
    x, g, gr, w = _inputs(T, D, 77, torch.bfloat16, False)
    dev = _device_step(x, g, gr, w, False)
    hx, hg, hgr, hw = (t.cpu().pin_memory() for t in (x, g, gr, w))
    o = {"y": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
         "x_copy": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
         "rstd": torch.empty(T, pin_memory=True), "dx": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
         "dgamma": torch.empty(D, pin_memory=True)}
    work = torch.empty(rn.rmsnorm_residual_step_host_work_bytes(T, D, 128), dtype=torch.uint8, device=DEV)
    s = torch.cuda.Stream()

    def call():
        rn.rmsnorm_residual_step_host(hx, hg, hgr, hw, o["y"], o["x_copy"], o["rstd"], o["dx"], o["dgamma"], work,
                                      EPS, False, slab_rows=128, stream=s)

    call()
    s.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=s):
        call()
    for rep in range(3):
        for t in o.values():
            t.zero_()
        graph.replay()
        torch.cuda.synchronize()
        _assert_same(o, dev, f"graph replay {rep}")


def test_host_step_from_two_host_threads():
    """Two host threads, each with its own stream, work buffer and inputs, call
    the step three times each at the same time (the binding releases the GIL
    in the call): the library serialises their enqueueing on its shared copy
    streams, and every result is the device entry points'."""
    import threading
    T, D = 1500, 1024
    cases = [_inputs(T, D, 90 + i, torch.bfloat16, i == 1) for i in range(2)]
    refs = [_device_step(x, g, gr, w, i == 1) for i, (x, g, gr, w) in enumerate(cases)]
    results, errors = [[], []], []

    def worker(i):
        try:
            x, g, gr, w = cases[i]
            hx, hg, hgr, hw = (t.cpu().pin_memory() for t in (x, g, gr, w))
            s = torch.cuda.Stream()
            work = torch.empty(rn.rmsnorm_residual_step_host_work_bytes(T, D, 256), dtype=torch.uint8, device=DEV)
            for _ in range(3):
                o = {"y": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
                     "x_copy": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
                     "rstd": torch.empty(T, pin_memory=True),
                     "dx": torch.empty((T, D), dtype=x.dtype, pin_memory=True),
                     "dgamma": torch.empty(D, pin_memory=True)}
                rn.rmsnorm_residual_step_host(hx, hg, hgr, hw, o["y"], o["x_copy"], o["rstd"], o["dx"], o["dgamma"],
                                              work, EPS, i == 1, slab_rows=256, stream=s)
                results[i].append(o)
            s.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(2)]
    for t in threads:
        t.start()
    for t in threads:
        t.join(timeout=120)
    assert not errors, errors
    for i in range(2):
        assert len(results[i]) == 3
        for k, o in enumerate(results[i]):
            _assert_same(o, refs[i], f"thread {i} call {k}")
