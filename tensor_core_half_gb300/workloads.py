"""Seeded synthetic inputs for the half-precision GEMM, and the workload table.

This module draws numbers and nothing else: it holds none of the product's
arithmetic, so both the CUDA path and the CPU oracle can be fed from it.

Recipe (the pages give no generator, so this is the plain reading):
  * a CPU ``torch.Generator`` seeded with the workload's seed;
  * A is drawn first, then B, each in its STORAGE shape: A [M,K]; B [N,K] for
    TN (B column-major, "HGEMM: WMMA and MMA PTX study notes", kernel header
    comment) or [K,N] for NN;
  * draws are fp32: uniform[a,b] = a + (b-a)*rand, normal(0,s) = s*randn,
    small integers = randint(lo, hi+1);
  * an optional fp32 scale multiplies BOTH operands (the 1/sqrt(K) sweep);
  * the fp32 values are rounded to the input dtype with round-to-nearest-even
    (``Tensor.to``).
The oracle reads exactly the resulting bytes.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import numpy as np
import torch

DTYPES = {"f16": torch.float16, "bf16": torch.bfloat16}


@dataclass(frozen=True)
class Workload:
    name: str
    M: int
    N: int
    K: int
    layout: str          # "TN" or "NN"
    in_dtype: str        # "f16" | "bf16"
    acc_dtype: str       # "f32" | "f16"
    out_dtype: str       # "f16" | "bf16"
    dist: tuple          # ("uniform", lo, hi) | ("normal", sigma) | ("int", lo, hi)
    seed: int
    scale_inv_sqrt_k: bool = False
    note: str = field(default="", compare=False)

    @property
    def flops(self) -> int:
        return 2 * self.M * self.N * self.K

    @property
    def compulsory_bytes(self) -> int:
        return 2 * (self.M * self.K + self.K * self.N + self.M * self.N)


def _sweep(size: int, acc: str) -> Workload:
    return Workload(f"sweep{size}_f16_acc{acc}", size, size, size, "TN", "f16", acc, "f16",
                    ("uniform", -1.0, 1.0), 2, scale_inv_sqrt_k=True,
                    note="square fp16 sweep, uniform[-1,1]/sqrt(K) on A and B")


WORKLOADS = {w.name: w for w in [
    Workload("square256_f16", 256, 256, 256, "TN", "f16", "f32", "f16", ("uniform", -1.0, 1.0), 0,
             note="small parity case"),
    Workload("square4096_bf16", 4096, 4096, 4096, "TN", "bf16", "f32", "bf16", ("normal", 1.0), 1,
             note="headline: 4096^3 bf16, fp32 accumulate"),
    *[_sweep(s, acc) for s in (2048, 4096, 8192, 12288, 16384) for acc in ("f32", "f16")],
    Workload("square8192_bf16", 8192, 8192, 8192, "TN", "bf16", "f32", "bf16", ("normal", 1.0), 1,
             note="8192^3 in bf16 with the headline's distribution"),
    Workload("nn8192x8192x16384_f16", 8192, 8192, 16384, "NN", "f16", "f32", "f16",
             ("uniform", -0.5, 0.5), 3, note="all row-major, B not pre-transposed"),
    Workload("ragged1000x3000x4104_bf16", 1000, 3000, 4104, "TN", "bf16", "f32", "bf16",
             ("normal", 0.02), 4, note="tile tails in M, N and K"),
    Workload("skinny16x16384x8192_bf16", 16, 16384, 8192, "TN", "bf16", "f32", "bf16",
             ("normal", 0.02), 4, note="HBM-bound, split-K"),
]}

HEADLINE = "square4096_bf16"


def _draw(gen: torch.Generator, shape, dist) -> torch.Tensor:
    kind = dist[0]
    if kind == "uniform":
        lo, hi = float(dist[1]), float(dist[2])
        return lo + (hi - lo) * torch.rand(shape, generator=gen, dtype=torch.float32)
    if kind == "normal":
        return float(dist[1]) * torch.randn(shape, generator=gen, dtype=torch.float32)
    if kind == "int":
        lo, hi = int(dist[1]), int(dist[2])
        return torch.randint(lo, hi + 1, shape, generator=gen, dtype=torch.int64).to(torch.float32)
    raise ValueError("unknown distribution %r" % (dist,))


def b_storage_shape(M: int, N: int, K: int, layout: str):
    if layout == "TN":
        return (N, K)
    if layout == "NN":
        return (K, N)
    raise ValueError("layout must be TN or NN")


def generate(M: int, N: int, K: int, layout: str, in_dtype: str, dist, seed: int,
             scale_inv_sqrt_k: bool = False):
    """Returns CPU tensors (A [M,K], B in storage shape) of the input dtype."""
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    a = _draw(gen, (M, K), dist)
    b = _draw(gen, b_storage_shape(M, N, K, layout), dist)
    if scale_inv_sqrt_k and K > 0:
        s = torch.tensor(1.0 / math.sqrt(K), dtype=torch.float32)
        a = a * s
        b = b * s
    dt = DTYPES[in_dtype]
    return a.to(dt).contiguous(), b.to(dt).contiguous()


def generate_workload(w: Workload):
    return generate(w.M, w.N, w.K, w.layout, w.in_dtype, w.dist, w.seed, w.scale_inv_sqrt_k)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a CPU fp16/bf16 tensor as numpy uint16."""
    if t.dtype not in (torch.float16, torch.bfloat16):
        raise TypeError("expected an fp16 or bf16 tensor")
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


def from_bits(b: np.ndarray, dtype: str) -> torch.Tensor:
    """numpy uint16 bit patterns -> CPU tensor of the given 16-bit dtype."""
    return torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(DTYPES[dtype])
