"""Exact-rational helpers for pinning the oracle (tests only).

These work in Python ``fractions.Fraction`` arithmetic, a number system
independent of the oracle's binary64 C code, so agreement between the two is
evidence rather than a restatement.
"""
from __future__ import annotations

from fractions import Fraction

import numpy as np
import torch

# (fraction bits, minimum normal exponent, maximum exponent) per IEEE format.
FORMATS = {0: (10, -14, 15), 1: (7, -126, 127), 2: (23, -126, 127)}
INF = float("inf")


def exact_values(t) -> list:
    """Exact rational values of a CPU fp16/bf16 tensor (via an exact widening
    to float64 by torch) as a nested list of Fractions."""
    d = t.to(torch.float64).numpy()
    return [[Fraction(float(x)) for x in row] for row in d]


def _binade(a: Fraction) -> int:
    """e such that 2**e <= a < 2**(e+1), for a > 0."""
    e = a.numerator.bit_length() - a.denominator.bit_length()
    two = Fraction(2)
    while two ** e > a:
        e -= 1
    while two ** (e + 1) <= a:
        e += 1
    return e


def round_exact(q: Fraction, fmt: int):
    """Nearest value of the format to the rational q, ties to even.
    Returns a Fraction, or +-inf on overflow."""
    frac_bits, emin, emax = FORMATS[fmt]
    if q == 0:
        return Fraction(0)
    sign = -1 if q < 0 else 1
    a = abs(q)
    e = max(_binade(a), emin)
    quantum = Fraction(2) ** (e - frac_bits)
    n = a / quantum
    fl = n.numerator // n.denominator
    rem = n - fl
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    val = fl * quantum
    max_finite = (2 - Fraction(2) ** (-frac_bits)) * Fraction(2) ** emax
    if val > max_finite:
        return sign * INF
    return sign * val


def as_float(x) -> float:
    return float(x) if not isinstance(x, float) else x


def exact_gemm(A, B) -> list:
    """Exact rational C = A . B^T for small CPU tensors."""
    a, b = exact_values(A), exact_values(B)
    return [[sum((x * y for x, y in zip(ra, rb)), Fraction(0)) for rb in b] for ra in a]


def abs_gemm_bound(A, B) -> np.ndarray:
    """sum_k |A_ik B_jk| in float64 (a bound helper, not a result)."""
    a = A.to(torch.float64).abs().numpy()
    b = B.to(torch.float64).abs().numpy()
    return a @ b.T
