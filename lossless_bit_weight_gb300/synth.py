"""Seeded synthetic inputs shaped like the 27B-class projection and LM-head workloads.

This module holds no W12 arithmetic: it only draws weights and activations and rounds them to
bf16. The tests, the smoke check and the benchmark feed the same tensors to the CUDA path and to
the CPU oracle.

Recipe (per workload, seed = base_seed + 1000 * workload_id + layer):
  weights  w[n, k] ~ N(0, (sigma * s_n)^2), s_n = exp(U[ln 0.5, ln 2]) per output channel;
           a fraction ``f_out`` of entries is multiplied by 2^+12 or 2^-12 (fair coin);
           a fraction ``f_zero`` of the remaining entries is set to +0; then rounded to bf16 (RNE).
  activations x[m, k] ~ N(0, 1), rounded to bf16 (RNE).
"""
from __future__ import annotations

import math
from dataclasses import dataclass

import numpy as np
import torch


@dataclass(frozen=True)
class WeightRecipe:
    sigma: float
    f_out: float
    f_zero: float


# tiny round trip + GEMM (K=256, N=512, M=1)
TINY = WeightRecipe(sigma=0.02, f_out=1e-4, f_zero=1e-3)
# projections of a 27B-class dense layer, drawn like the tiny case with the smaller outlier
# fraction: 7e-5 outliers and 0.1% exact zeros. The zeros dominate the escapes (about 1.1e-3 of
# the weights, 9 per 128x64 record): ten times the fraction SpecPilot reports for real models.
PROJ = WeightRecipe(sigma=0.02, f_out=7e-5, f_zero=1e-3)
# the same without the zeros: the Gaussian tails and the 2^+-12 outliers alone give about
# 1.1e-4 escapes, inside the range SpecPilot reports for real models (7.3e-5 on its 27B model,
# under 1.3e-4 on every model: Fig. 5, App. E)
LIGHT = WeightRecipe(sigma=0.02, f_out=7e-5, f_zero=0.0)
# LM head (vocabulary 151936 x hidden 5120)
HEAD = WeightRecipe(sigma=0.01, f_out=7e-5, f_zero=0.0)

HIDDEN = 5120
MLP = 17408
VOCAB = 151936
# one synthetic decoder layer: (name, K, N)
LAYER_LINEARS = (
    ("q", HIDDEN, 6144), ("k", HIDDEN, 1024), ("v", HIDDEN, 1024), ("o", 6144, HIDDEN),
    ("gate", HIDDEN, MLP), ("up", HIDDEN, MLP), ("down", MLP, HIDDEN),
)


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def weights(N: int, K: int, recipe: WeightRecipe, seed: int, device="cpu",
            row_block: int = 16384) -> torch.Tensor:
    """bf16 [N, K] weights drawn by ``recipe``; generated in row blocks to bound temporaries."""
    device = torch.device(device)
    out = torch.empty((N, K), dtype=torch.bfloat16, device=device)
    g = _gen(seed, device)
    lo, hi = math.log(0.5), math.log(2.0)
    scale = torch.exp(torch.empty(N, device=device).uniform_(lo, hi, generator=g)) * recipe.sigma
    for r0 in range(0, N, row_block):
        r1 = min(N, r0 + row_block)
        w = torch.randn((r1 - r0, K), generator=g, device=device) * scale[r0:r1, None]
        u = torch.rand((r1 - r0, K), generator=g, device=device)
        coin = torch.rand((r1 - r0, K), generator=g, device=device) < 0.5
        outlier = u < recipe.f_out
        zero = (u >= recipe.f_out) & (u < recipe.f_out + recipe.f_zero)
        factor = torch.where(coin, torch.full_like(w, 4096.0), torch.full_like(w, 1.0 / 4096.0))
        w = torch.where(outlier, w * factor, w)
        w = torch.where(zero, torch.zeros_like(w), w)
        out[r0:r1] = w.to(torch.bfloat16)
        del w, u, coin, outlier, zero, factor
    return out


def activations(M: int, K: int, seed: int, device="cpu") -> torch.Tensor:
    g = _gen(seed, torch.device(device))
    return torch.randn((M, K), generator=g, device=device).to(torch.bfloat16)


def seed_for(workload: int, layer: int = 0, base: int = 0) -> int:
    return base + 1000 * workload + layer


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a tensor as a host uint16 array."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_bits(a: np.ndarray, device="cpu") -> torch.Tensor:
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16)).view(torch.bfloat16).to(device)


def all_bf16_patterns(K: int = 256) -> np.ndarray:
    """Every 16-bit pattern once, as a [65536 / K, K] uint16 array (row n holds n*K .. n*K+K-1)."""
    return np.arange(65536, dtype=np.uint32).astype(np.uint16).reshape(-1, K)
