"""The library's calls inside a captured CUDA graph.

Every kernel is launched with programmatic stream serialization, so in a
captured graph consecutive kernels are joined by programmatic edges. A graph
of forward + backward + weight-gradient reduction, replayed, must give the
eager calls' bits exactly (both row paths, wide and narrow, and the backward
of rows wider than 8192, launched on two-CTA clusters), and replaying it on
new inputs copied into the captured buffers must match eager calls on those
inputs.
"""
from __future__ import annotations

import pytest
import torch

import invariant_rmsnorm_gb300 as rn
from invariant_rmsnorm_gb300 import synth
from tests.gpu_common import DEV

pytestmark = pytest.mark.gpu


def _bits(t):
    return t.view(torch.int32) if t.dtype == torch.float32 else t.view(torch.int16)


def _residual_step(b):
    rn.rmsnorm_residual_fwd(b["x"], b["w"], b["y"], b["rstd"], b["xc"], 1e-6, False)
    rn.rmsnorm_residual_bwd(b["g"], b["x"], b["w"], b["rstd"], b["gr"], b["dx"], b["dw"], b["ws"], False)


def _gated_step(b):
    rn.rmsnorm_gated_fwd(b["x"], b["z"], b["w"], b["y"], b["rstd"], 1e-6, True)
    rn.rmsnorm_gated_bwd(b["g"], b["x"], b["z"], b["w"], b["rstd"], b["dx"], b["dz"], b["dw"], b["ws"], True)


def _buffers(kind, T, D, seed):
    b = dict(x=synth.normal_bf16((T, D), seed, DEV), g=synth.normal_bf16((T, D), seed + 1, DEV),
             w=synth.gamma_f32(D, seed + 2, DEV, mean=0.0 if kind == "gated" else 1.0, std=0.1))
    if kind == "gated":
        b["z"] = synth.normal_bf16((T, D), seed + 3, DEV)
        b["dz"] = torch.empty_like(b["x"])
    else:
        b["gr"] = synth.normal_bf16((T, D), seed + 4, DEV)
        b["xc"] = torch.empty_like(b["x"])
    b.update(y=torch.empty_like(b["x"]), dx=torch.empty_like(b["x"]), rstd=torch.empty(T, device=DEV),
             dw=torch.empty(D, device=DEV),
             ws=torch.empty(rn.workspace_bytes(T, D), dtype=torch.uint8, device=DEV))
    return b


OUTS = {"residual": ("y", "xc", "rstd", "dx", "dw"), "gated": ("y", "rstd", "dx", "dz", "dw")}


@pytest.mark.parametrize("kind,T,D", [("residual", 4096, 4096), ("residual", 1000, 768), ("gated", 20000, 128),
                                      ("residual", 700, 16384), ("gated", 300, 12296)])  # CTA-pair backwards
def test_graph_replay_matches_eager(kind, T, D):
    step = _residual_step if kind == "residual" else _gated_step
    b = _buffers(kind, T, D, seed=3)
    # Eager reference (also fills the library's per-device launch caches, so that
    # capture records launches only).
    step(b)
    torch.cuda.synchronize()
    ref = {k: b[k].clone() for k in OUTS[kind]}
    for k in OUTS[kind]:
        b[k].fill_(0)
    s = torch.cuda.Stream(DEV)
    s.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            step(b)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(2):
        graph.replay()
        torch.cuda.synchronize()
        for k in OUTS[kind]:
            assert torch.equal(_bits(b[k]), _bits(ref[k])), k
    # New inputs copied into the captured buffers: the replay follows them.
    nb = _buffers(kind, T, D, seed=11)
    for k in ("x", "g", "w") + (("z",) if kind == "gated" else ("gr",)):
        b[k].copy_(nb[k])
    graph.replay()
    step(nb)
    torch.cuda.synchronize()
    for k in OUTS[kind]:
        assert torch.equal(_bits(b[k]), _bits(nb[k])), k
