"""Seeded synthetic operands and the workload list shared by the tests, the
benchmark and the oracle checks.

This module draws random numbers and nothing else: it holds none of the
GEMM's arithmetic, so both the CUDA path's callers and the CPU oracle can take
their inputs from it without sharing any part of the method.

Recipe (one CPU ``torch.Generator`` per shape, seeded with the workload's
seed; A is drawn first, then B; values are drawn in fp32 and cast to the
input dtype by torch with round-to-nearest-even; FP8 inputs are E4M3 or E5M2):
  * ``uniform``: iid U[-1, 1) as ``rand * 2 - 1``;
  * ``normal``:  iid N(0, 1/K) as ``randn * K**-0.5`` (the standard deviation
    is read as 1/sqrt(K)).
The shapes are the Llama-3-70B projection sizes used as GEMM workloads in
"A Blackwell GEMM by Hand in CuTe DSL" (section 1, gemm_math.py shape table);
only their sizes are used, no model weights.
"""
from __future__ import annotations

from dataclasses import dataclass

import torch

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
TORCH_DTYPE = {F16: torch.float16, BF16: torch.bfloat16, F32: torch.float32,
               E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
DTYPE_NAME = {F16: "f16", BF16: "bf16", F32: "f32", E4M3: "e4m3", E5M2: "e5m2"}


@dataclass(frozen=True)
class Shape:
    M: int
    N: int
    K: int


@dataclass(frozen=True)
class Workload:
    name: str
    shapes: tuple
    dtype_in: int
    dtype_out: int
    dist: str
    seed: int


WORKLOADS = {
    "small_256": Workload("small_256", (Shape(256, 256, 256),), F16, F32, "uniform", 0),
    "square_4096": Workload("square_4096", (Shape(4096, 4096, 4096),), F16, F16, "uniform", 1),
    "prefill": Workload("prefill", (Shape(8192, 8192, 8192), Shape(8192, 28672, 8192)),
                        BF16, BF16, "normal", 2),
    "decode_m256": Workload("decode_m256", (Shape(256, 28672, 8192), Shape(256, 8192, 28672),
                                            Shape(256, 10240, 8192), Shape(256, 8192, 8192)),
                            F16, F16, "uniform", 3),
    "decode_small_m": Workload("decode_small_m", tuple(
        Shape(m, n, k) for m in (1, 8, 32, 64, 128)
        for n, k in ((8192, 8192), (28672, 8192), (8192, 28672))), F16, F16, "uniform", 5),
    # decode shapes on which the library takes the swapped tiling (17..128 rows of A where
    # the plain one-CTA tiles leave SMs idle)
    "decode_swapped": Workload("decode_swapped", (Shape(128, 14336, 8192), Shape(48, 14336, 8192),
                                                  Shape(128, 14336, 16384), Shape(32, 14336, 28672)),
                               F16, F16, "uniform", 7),
    "fp8": Workload("fp8", (Shape(4096, 4096, 4096), Shape(8192, 8192, 8192)),
                    E4M3, BF16, "uniform", 6),
    "sweep_bf16_f32": Workload("sweep_bf16_f32", (
        Shape(1024, 1024, 1024), Shape(2048, 2048, 2048), Shape(8192, 8192, 8192),
        Shape(16384, 16384, 16384), Shape(4095, 4097, 4096), Shape(1000, 3000, 2000)),
        BF16, F32, "uniform", 4),
}


def make_operands(M: int, N: int, K: int, dtype_in: int, dist: str = "uniform",
                  seed: int = 0):
    """Return (A, B): CPU tensors of shape (M, K) and (N, K) in the input dtype."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    td = TORCH_DTYPE[dtype_in]
    if dist == "uniform":
        A = (torch.rand(M, K, generator=g) * 2 - 1).to(td)
        B = (torch.rand(N, K, generator=g) * 2 - 1).to(td)
    elif dist == "normal":
        s = float(K) ** -0.5 if K > 0 else 1.0
        A = (torch.randn(M, K, generator=g) * s).to(td)
        B = (torch.randn(N, K, generator=g) * s).to(td)
    else:
        raise ValueError(f"unknown distribution {dist!r}")
    return A, B


def make_small_int_operands(M: int, N: int, K: int, dtype_in: int, seed: int = 0, lo: int = -3,
                            hi: int = 3):
    """iid integers in [lo, hi], stored in the input dtype (exact in fp16/bf16)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    td = TORCH_DTYPE[dtype_in]
    A = torch.randint(lo, hi + 1, (M, K), generator=g).to(td)
    B = torch.randint(lo, hi + 1, (N, K), generator=g).to(td)
    return A, B


@dataclass(frozen=True)
class MoeWorkload:
    """A Mixture-of-Experts projection as a grouped GEMM: `rows` routed token rows
    spread over `experts` experts, each expert a K x N weight (B_e, N x K) applied to
    its rows (A_e, M_e x K)."""
    name: str
    experts: int
    rows: int
    N: int
    K: int
    dtype_in: int
    dtype_out: int
    seed: int


# Expert counts and widths of two MoE layer families (8 large experts, 64 small ones),
# sizes only; the token-to-expert assignment is drawn by moe_counts.
MOE_WORKLOADS = {
    "moe_8x14336x4096": MoeWorkload("moe_8x14336x4096", 8, 8192, 14336, 4096, BF16, BF16, 20),
    "moe_64x2048x7168": MoeWorkload("moe_64x2048x7168", 64, 8192, 2048, 7168, BF16, BF16, 21),
    "moe_64x7168x2048": MoeWorkload("moe_64x7168x2048", 64, 8192, 7168, 2048, BF16, BF16, 22),
}


# A group whose problems differ in K, so that its tiles differ in cost: `problems` GEMMs of
# M x N with K drawn log-uniformly from {256, 512, ..., 16384} (seeded).
@dataclass(frozen=True)
class MixedKWorkload:
    name: str
    problems: int
    M: int
    N: int
    dtype_in: int
    dtype_out: int
    seed: int


MIXED_K_WORKLOADS = {
    "mixed_k_24x512x2048": MixedKWorkload("mixed_k_24x512x2048", 24, 512, 2048, F16, F16, 23),
}


def mixed_k_values(problems: int, seed: int) -> list:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return [256 << int(e) for e in torch.randint(0, 7, (problems,), generator=g)]


def moe_counts(experts: int, rows: int, seed: int) -> list:
    """Rows per expert: expert loads drawn from a flat Dirichlet (normalised iid
    exponentials), then `rows` tokens assigned by a multinomial draw -- an imbalanced
    routing, some experts possibly empty."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    w = -torch.log(torch.rand(experts, generator=g).clamp_min(1e-12))
    w = w / w.sum()
    return torch.multinomial(w, rows, replacement=True, generator=g).bincount(
        minlength=experts).tolist()


def make_block_scales(rows: int, cols: int, seed: int = 0, lo: float = -3.0, hi: float = 3.0):
    """A rows x cols float32 array of positive scales 2**u, u iid uniform in [lo, hi)
    (one per (row block, k block), as blockwise-scaled operands carry)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return torch.exp2(torch.rand(rows, cols, generator=g) * (hi - lo) + lo).float()


def sample_indices(n: int, count: int, seed: int, must=()):
    """Sorted unique indices in [0, n): `count` seeded draws plus the listed
    ones that fall inside the range (tile edges, the last row/column)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    pick = torch.randint(0, max(n, 1), (count,), generator=g).tolist() if n > 0 else []
    idx = {i for i in pick} | {i if i >= 0 else n + i for i in must}
    return sorted(i for i in idx if 0 <= i < n)


def rademacher(n: int, seed: int):
    """A seeded +-1 vector (float64), for Freivalds-style checks."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return (torch.randint(0, 2, (n,), generator=g).to(torch.float64) * 2 - 1)
