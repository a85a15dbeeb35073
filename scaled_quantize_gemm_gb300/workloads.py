"""Seeded synthetic inputs for the five FP8 scaled-linear workloads.

This module only draws random numbers: it holds none of the quantisation,
scaling or GEMM arithmetic, so both the CUDA path's tests/bench and the CPU
oracle can take their inputs from it.  Every tensor is drawn in fp32 from a
``torch.Generator`` seeded with ``1000 * workload + 10 * step + role`` on the
requested device, then rounded to bf16 by torch (round-to-nearest-even) where
the workload is bf16.  The same call on the same device and torch build gives
the same bits.

Workloads (shapes from the pages: the Transformer Engine tutorial's MiniGPT
uses hidden 768, FFN 3072, sequence 256; the week-14 page's DeepSeek-V3 1x128
/ 128x128 granularity and MX 32-element blocks):
  1  per-tensor current scaling, A, B 256x256 fp32 N(0,1) with 4 outliers of
     magnitude 30 at seeded positions;
  2  MiniGPT-shaped linears, M = 2048 tokens, 768->2304, 768->3072, 3072->768,
     20 steps, activation std drifting linearly from 1 to 8;
  3  fine-grained current scaling, X 4096x4096 Student-t(3), W 4096x4096
     N(0, 0.02^2);
  4  MX blocks, A, B 8192x8192 N(0,1) with 0.1% of entries scaled by 100;
  5  large FFN step, M = 16384 tokens, 4096->14336 and 14336->4096, 10 steps.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import torch

ROLE_X, ROLE_W, ROLE_DY, ROLE_A, ROLE_B = 0, 1, 2, 3, 4


def seed_of(workload: int, step: int, role: int, layer: int = 0) -> int:
    return 1000 * workload + 10 * step + role + 100000 * layer


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal(shape, std: float, seed: int, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(dtype)


def student_t3(shape, seed: int, device="cpu", dtype=torch.bfloat16) -> torch.Tensor:
    """Student-t with 3 degrees of freedom: z / sqrt(chi2_3 / 3), chi2_3 the
    sum of three squared standard normals."""
    g = _gen(device, seed)
    z = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    chi = torch.zeros(shape, device=device, dtype=torch.float32)
    for _ in range(3):
        w = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
        chi.addcmul_(w, w)
    return (z / torch.sqrt(chi / 3.0)).to(dtype)


def with_outliers(shape, count: int, magnitude: float, seed: int, device="cpu",
                  dtype=torch.float32) -> torch.Tensor:
    """N(0,1) with `count` entries (seeded positions, without replacement)
    set to +-magnitude (seeded signs)."""
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    n = x.numel()
    idx = torch.randperm(n, generator=g, device=device)[:count]
    sign = torch.randint(0, 2, (count,), generator=g, device=device).to(torch.float32) * 2 - 1
    x.view(-1)[idx] = sign * magnitude
    return x.to(dtype)


def with_scaled_fraction(shape, fraction: float, factor: float, seed: int, device="cpu",
                         dtype=torch.bfloat16) -> torch.Tensor:
    """N(0,1) with round(fraction * n) entries (seeded, without replacement)
    multiplied by `factor`."""
    g = _gen(device, seed)
    x = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    n = x.numel()
    k = int(round(fraction * n))
    idx = torch.randperm(n, generator=g, device=device)[:k]
    x.view(-1)[idx] *= factor
    return x.to(dtype)


@dataclass
class Linear:
    in_features: int   # K
    out_features: int  # N


@dataclass
class Workload:
    ident: int
    name: str
    tokens: int = 0
    linears: list = field(default_factory=list)
    steps: int = 1
    history_len: int = 16


WORKLOADS = {
    1: Workload(1, "per-tensor current-scaled FP8 linear, A 256x256, B 256x256, fp32 out"),
    2: Workload(2, "MiniGPT-shaped HYBRID delayed-scaling linears, M=2048, 768->2304/768->3072/3072->768",
                tokens=2048, linears=[Linear(768, 2304), Linear(768, 3072), Linear(3072, 768)],
                steps=20, history_len=16),
    3: Workload(3, "fine-grained current scaling, X 4096x4096 Student-t(3) 1x128 tiles, "
                   "W 4096x4096 128x128 blocks, bf16 out"),
    4: Workload(4, "MXFP8 32-element E8M0 blocks, A, B 8192x8192, bf16 out"),
    5: Workload(5, "large FFN training step, HYBRID per-tensor delayed scaling, M=16384, 4096->14336->4096",
                tokens=16384, linears=[Linear(4096, 14336), Linear(14336, 4096)],
                steps=10, history_len=16),
}


# ---------------------------------------------------------------- per-workload tensors
def w1_operands(device="cpu", size: int = 256):
    a = with_outliers((size, size), 4, 30.0, seed_of(1, 0, ROLE_A), device)
    b = with_outliers((size, size), 4, 30.0, seed_of(1, 0, ROLE_B), device)
    return a, b


def w2_sigma(step: int, steps: int = 20) -> float:
    """activation std drifting linearly from 1 (first step) to 8 (last)."""
    return 1.0 + 7.0 * step / (steps - 1)


def linear_x(workload: int, layer: int, step: int, M: int, K: int, device="cpu", std: float = 1.0):
    return normal((M, K), std, seed_of(workload, step, ROLE_X, layer), device)


def linear_w(workload: int, layer: int, N: int, K: int, device="cpu"):
    return normal((N, K), 0.02, seed_of(workload, 0, ROLE_W, layer), device)


def linear_dy(workload: int, layer: int, step: int, M: int, N: int, device="cpu"):
    return normal((M, N), 1e-3, seed_of(workload, step, ROLE_DY, layer), device)


def w3_operands(device="cpu", size: int = 4096):
    x = student_t3((size, size), seed_of(3, 0, ROLE_X), device)
    w = normal((size, size), 0.02, seed_of(3, 0, ROLE_W), device)
    return x, w


def w4_operands(device="cpu", size: int = 8192):
    a = with_scaled_fraction((size, size), 1e-3, 100.0, seed_of(4, 0, ROLE_A), device)
    b = with_scaled_fraction((size, size), 1e-3, 100.0, seed_of(4, 0, ROLE_B), device)
    return a, b
