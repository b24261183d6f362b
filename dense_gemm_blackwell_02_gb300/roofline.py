"""Roofline, shared-memory budget and latency arithmetic for C = A . B^T.

Host-side analysis used by the benchmark and the tile heuristics.  The same
quantities are tabulated for a B200 in "A Blackwell GEMM by Hand in CuTe DSL"
(section 1, gemm_math.py parts 1-4; section 7 on the stage budget); the unit
tests reproduce those printed tables from these functions.

Algorithmic work of one GEMM (the minimum the method must move):
  FLOPs = 2 M N K
  bytes = in_bytes (M K + N K) + out_bytes M N     (A, B read once, C written once)
"""
from __future__ import annotations

import math


def gemm_flops(M: int, N: int, K: int) -> int:
    return 2 * M * N * K


def gemm_bytes(M: int, N: int, K: int, in_bytes: int = 2, out_bytes: int = 2) -> int:
    return in_bytes * (M * K + N * K) + out_bytes * M * N


def arithmetic_intensity(M, N, K, in_bytes=2, out_bytes=2) -> float:
    return gemm_flops(M, N, K) / gemm_bytes(M, N, K, in_bytes, out_bytes)


def roofline_floor_us(M, N, K, peak_tflops: float, bw_tbs: float, in_bytes=2, out_bytes=2):
    """(floor time in microseconds, "compute" | "memory") for the given peaks."""
    t_compute = gemm_flops(M, N, K) / (peak_tflops * 1e6)
    t_memory = gemm_bytes(M, N, K, in_bytes, out_bytes) / (bw_tbs * 1e6)
    return (t_compute, "compute") if t_compute > t_memory else (t_memory, "memory")


def ridge_flop_per_byte(peak_tflops: float, bw_tbs: float) -> float:
    return peak_tflops / bw_tbs


def tflops(M, N, K, us: float) -> float:
    return gemm_flops(M, N, K) / (us * 1e6)


def tbs(M, N, K, us: float, in_bytes=2, out_bytes=2) -> float:
    return gemm_bytes(M, N, K, in_bytes, out_bytes) / (us * 1e6)


def tile_count(M: int, N: int, bm: int, bn: int) -> int:
    return math.ceil(M / bm) * math.ceil(N / bn)


def waves(tiles: int, sms: int) -> float:
    return tiles / sms


def stage_bytes(a_rows: int, b_rows: int, tile_k: int, elem_bytes: int = 2) -> int:
    """Shared memory of one pipeline stage: an A slice and a B slice, tile_k deep."""
    return (a_rows + b_rows) * tile_k * elem_bytes


def max_stages(per_stage: int, smem_limit: int = 227 * 1024, reserved: int = 0) -> int:
    return (smem_limit - reserved) // per_stage


def flop_per_smem_byte(bm: int, bn: int, tile_k: int, per_stage: int) -> float:
    return 2 * bm * bn * tile_k / per_stage


def kstep_us(bm: int, bn: int, tile_k: int, peak_tflops: float, sms: int) -> float:
    """Time one SM needs at peak for one bm x bn x tile_k step."""
    return 2 * bm * bn * tile_k / (peak_tflops * 1e12 / sms) * 1e6


def stages_for_latency(latency_us: float, step_us: float) -> float:
    """Little's law: stages in flight needed to hide `latency_us` of load
    latency when one stage is consumed every `step_us`."""
    return 1 + latency_us / step_us


def tensor_peak_tflops(sms: int, sm_mhz: float, flop_per_sm_cycle: int = 8192) -> float:
    """Dense fp16/bf16 tensor peak from the per-SM rate (8192 FLOP per SM per
    cycle is the figure given for the sm_103 part in "Optimizing GEMMs using
    tcgen05 - Part 1", B300 details)."""
    return sms * flop_per_sm_cycle * sm_mhz * 1e6 / 1e12
