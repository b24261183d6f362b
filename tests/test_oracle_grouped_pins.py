"""Pins for the oracle's grouped product ("CUTLASS Deep Dive: From CuTe Layouts to
Blackwell tcgen05", Part 6, Grouped GEMM): a list of independent problems of different
shapes, each C_g = A_g . B_g^T.  Checked against exact rationals per problem, against
problems whose answers are fixed in closed form, and for independence (each output
depends on its own operands only, whatever the order or the company)."""
from fractions import Fraction

import numpy as np
import torch

import seeded_inputs as si
from tests import exact

F16, BF16, F32 = 0, 1, 2


def _problems(shapes, dt, seed):
    return [si.make_operands(M, N, K, dt, "uniform", seed + t) for t, (M, N, K) in enumerate(shapes)]


def test_grouped_exact_rational_per_problem(oracle_lib):
    shapes = [(3, 5, 16), (1, 7, 8), (6, 2, 40), (4, 4, 24)]
    # small integers scaled by a power of two per problem: every sum is exact, so each
    # output must be the exact rational, rounded once
    probs = [(A * 2.0 ** -t, B) for t, (A, B) in enumerate(
        si.make_small_int_operands(M, N, K, F16, seed=500 + t) for t, (M, N, K) in enumerate(shapes))]
    outs = oracle_lib.gemm_grouped(probs, F16, F32)
    assert len(outs) == len(shapes)
    for (A, B), C, (M, N, K) in zip(probs, outs, shapes):
        assert C.shape == (M, N)
        ex = exact.exact_gemm(A, B)
        got = oracle_lib.decode(C, F32)
        for i in range(M):
            for j in range(N):
                assert Fraction(float(got[i, j])) == exact.round_exact(ex[i][j], F32)


def test_grouped_closed_forms(oracle_lib):
    # all-ones problems of different K give K; a K = 0 problem gives zeros; an identity
    # B gives A back
    A1 = torch.ones(2, 33, dtype=torch.bfloat16)
    A0 = torch.empty(3, 0, dtype=torch.bfloat16)
    B0 = torch.empty(4, 0, dtype=torch.bfloat16)
    Ai, _ = si.make_operands(5, 1, 16, BF16, "uniform", 501)
    outs = oracle_lib.gemm_grouped([(A1, torch.ones(3, 33, dtype=torch.bfloat16)), (A0, B0),
                                    (Ai, torch.eye(16, dtype=torch.bfloat16))], BF16, F32)
    assert np.all(oracle_lib.decode(outs[0], F32) == 33)
    assert outs[1].shape == (3, 4) and np.all(outs[1] == 0)
    assert np.array_equal(oracle_lib.decode(outs[2], F32), Ai.to(torch.float64).numpy())


def test_grouped_problems_are_independent(oracle_lib):
    shapes = [(7, 9, 64), (3, 12, 32), (10, 5, 48)]
    probs = _problems(shapes, BF16, 510)
    outs = oracle_lib.gemm_grouped(probs, BF16, BF16)
    # reversed order, and each problem alone, give the same outputs
    rev = oracle_lib.gemm_grouped(probs[::-1], BF16, BF16)[::-1]
    for g, (A, B) in enumerate(probs):
        alone = oracle_lib.gemm_grouped([(A, B)], BF16, BF16)[0]
        assert np.array_equal(outs[g], rev[g]) and np.array_equal(outs[g], alone)
    # changing one problem's operands changes only that problem's output
    A0, B0 = probs[0]
    changed = oracle_lib.gemm_grouped([(A0 * 2, B0)] + probs[1:], BF16, BF16)
    assert not np.array_equal(changed[0], outs[0])
    assert all(np.array_equal(changed[g], outs[g]) for g in (1, 2))
