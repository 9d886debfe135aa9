"""Seeded synthetic inputs for the RMSNorm workloads.

This module only draws random numbers and arranges rows; it holds none of the
normalisation arithmetic, so both the CUDA library's tests and the CPU oracle
can consume the same tensors without sharing any code of the method.

Distributions follow the workloads the pages describe (RL-Kernel pull request
414 "[DSv4][P1-5] rmsnorm_residual", Implementation and Benchmarks: bf16
activations, fp32 gamma, D=4096 in production and D=128 fixtures; RL-Kernel
pull request 467 "...zero-centred RMSNorm references and CUDA kernel": Qwen3-Next
gated norm over head_v_dim=128 rows, zero-centred weights ~ randn x 0.1).
No public dataset is involved.

All generators are deterministic functions of (seed, device). The same seed on
CPU and on CUDA gives different numbers (different generators); a test draws
once and hands copies of the same tensors to both sides.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Dict, List, Optional

import torch

EPS = 1e-6


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def normal_bf16(shape, seed: int, device="cpu", std: float = 1.0) -> torch.Tensor:
    """bf16 tensor of N(0, std^2) draws (drawn in fp32, rounded by torch to bf16)."""
    return normal16(shape, seed, device, std, torch.bfloat16)


def normal16(shape, seed: int, device="cpu", std: float = 1.0, dtype=torch.bfloat16) -> torch.Tensor:
    """16-bit (bf16 or fp16) tensor of N(0, std^2) draws: the same fp32 draws
    for either format, rounded by torch."""
    x = torch.randn(shape, generator=_gen(seed, device), device=device, dtype=torch.float32)
    if std != 1.0:
        x = x * std
    return x.to(dtype)


def gamma_f32(D: int, seed: int, device="cpu", mean: float = 1.0, std: float = 0.1) -> torch.Tensor:
    """fp32 weight of mean + N(0, std^2) draws."""
    w = torch.randn((D,), generator=_gen(seed, device), device=device, dtype=torch.float32)
    return w * std + mean


def with_outliers(x: torch.Tensor, seed: int, frac: float = 1e-3, scale: float = 100.0) -> torch.Tensor:
    """Copy of ``x`` with a random ``frac`` of its entries multiplied by ``scale``
    (outlier channels); the product is rounded to bf16 by torch."""
    u = torch.rand(x.shape, generator=_gen(seed, x.device), device=x.device, dtype=torch.float32)
    out = x.clone()
    mask = u < frac
    out[mask] = (out[mask].float() * scale).to(x.dtype)
    return out


def strided(t: torch.Tensor, ld: int) -> torch.Tensor:
    """A [T, D] view of ``t``'s values whose rows sit ``ld`` elements apart (ld >= D).

    The padding columns hold a fixed non-finite-free junk pattern, so a kernel
    that read past D would be caught by a value mismatch."""
    T, D = t.shape
    assert ld >= D
    base = torch.full((max(T, 1), ld), -7.0, dtype=t.dtype, device=t.device)
    base[:T, :D] = t
    return base[:T, :D]


# --------------------------------------------------------------------------
# Named workloads
# --------------------------------------------------------------------------

@dataclass
class Workload:
    """One problem instance: tensors on ``device`` plus its scalar settings."""
    name: str
    T: int
    D: int
    eps: float
    zero_centered_gamma: bool
    x: torch.Tensor
    w: torch.Tensor
    g: torch.Tensor
    z: Optional[torch.Tensor] = None
    g_res: Optional[torch.Tensor] = None
    extra: Dict[str, object] = field(default_factory=dict)


def tiny_plain(device="cpu", seed: int = 0, zero_centered_gamma: bool = False,
               T: int = 16, D: int = 128) -> Workload:
    """T=16, D=128 plain fwd+bwd; gamma ~1+N(0,0.1), or ~N(0,0.1) when zero-centred."""
    w = gamma_f32(D, seed + 1, device, mean=0.0 if zero_centered_gamma else 1.0, std=0.1)
    return Workload("tiny_plain", T, D, EPS, zero_centered_gamma,
                    x=normal_bf16((T, D), seed, device), w=w,
                    g=normal_bf16((T, D), seed + 2, device))


def residual(device="cpu", seed: int = 0, T: int = 32768, D: int = 4096) -> Workload:
    """rmsnorm_residual fwd+bwd: x, g, g_res ~N(0,1) bf16, gamma ~1+N(0,0.05) fp32."""
    return Workload("residual", T, D, EPS, False,
                    x=normal_bf16((T, D), seed, device),
                    w=gamma_f32(D, seed + 1, device, mean=1.0, std=0.05),
                    g=normal_bf16((T, D), seed + 2, device),
                    g_res=normal_bf16((T, D), seed + 3, device))


def gated(device="cpu", seed: int = 0, T: int = 8192 * 32, D: int = 128) -> Workload:
    """Qwen3-Next gated, zero-centred: 8192 tokens x 32 heads rows of head_v_dim=128;
    x, z, g ~N(0,1) bf16; weight ~N(0,0.1) fp32 (the +1 is the kernel's)."""
    return Workload("gated", T, D, EPS, True,
                    x=normal_bf16((T, D), seed, device),
                    w=gamma_f32(D, seed + 1, device, mean=0.0, std=0.1),
                    g=normal_bf16((T, D), seed + 2, device),
                    z=normal_bf16((T, D), seed + 4, device))


def large(device="cpu", seed: int = 0, T: int = 131072, D: int = 4096) -> Workload:
    """Large sweep: x ~N(0,1) with 0.1% of entries x100, gamma ~1+N(0,0.2), g ~N(0,1)."""
    x = with_outliers(normal_bf16((T, D), seed, device), seed + 5)
    return Workload("large", T, D, EPS, False, x=x,
                    w=gamma_f32(D, seed + 1, device, mean=1.0, std=0.2),
                    g=normal_bf16((T, D), seed + 2, device))


INVARIANCE_T: List[int] = [1, 2, 17, 33, 128, 257, 1000, 1024]
INVARIANCE_POSITIONS = ("first", "middle", "last", "shuffled")


def invariance_batch(anchor_x: torch.Tensor, anchor_g: torch.Tensor, T: int, position: str,
                     seed: int, pad_frac: float = 0.25):
    """Place one fixed anchor row in a batch of T rows.

    The other rows are fresh N(0,1) rows, except that the last ``pad_frac`` of
    them are zero padding rows. ``position`` is first / middle / last, or
    shuffled (the whole batch, anchor included, is permuted at random).
    Returns ``(x [T,D], g [T,D], anchor_index)``.
    """
    D = anchor_x.shape[-1]
    dev = anchor_x.device
    x = normal_bf16((T, D), seed, dev)
    g = normal_bf16((T, D), seed + 1, dev)
    n_pad = int(T * pad_frac) if T >= 4 else 0
    if n_pad:
        x[T - n_pad:] = 0
        g[T - n_pad:] = 0
    if position == "first":
        idx = 0
    elif position == "middle":
        idx = T // 2
    elif position == "last":
        idx = T - 1
    elif position == "shuffled":
        perm = torch.randperm(T, generator=_gen(seed + 2, "cpu")).to(dev)
        x = x[perm].contiguous()
        g = g[perm].contiguous()
        idx = int(torch.randint(0, T, (1,), generator=_gen(seed + 3, "cpu")).item())
    else:
        raise ValueError(position)
    x[idx] = anchor_x
    g[idx] = anchor_g
    return x, g, idx
