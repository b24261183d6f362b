"""The oracle's pins must catch plausible mistakes in the oracle itself.

Each case plants one mistake in a copy of oracle.c (a dropped term, a wrong
sign, a wrong index, a transposed operand, a wrong tie rule, truncation, a
mis-scaled subnormal), compiles the copy on the CPU into a temporary library,
and asserts that at least one pin check rejects it.  The committed oracle is
never modified.
"""
import os
import subprocess
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import exact

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
TD = {F16: torch.float16, BF16: torch.bfloat16}
SRC = os.path.join(os.path.dirname(oracle.__file__), "oracle.c")

MUTANTS = {
    "drop_last_term": ("for (int64_t k = k0; k < k1; ++k) s += lut[a16[k]]",
                       "for (int64_t k = k0; k < k1 - 1; ++k) s += lut[a16[k]]"),
    "wrong_sign": ("s += lut[a16[k]] * lut[b16[k]];", "s -= lut[a16[k]] * lut[b16[k]];"),
    "reversed_index": ("s += lut[a16[k]] * lut[b16[k]];",
                       "s += lut[a16[k]] * lut[b16[k1 - 1 - (k - k0)]];"),
    # B walked with unit stride across j, as if it were stored transposed
    "transposed_B": ("const char* b_row = (const char*)jb->B + j * jb->K * jb->in_bytes;",
                     "const char* b_row = (const char*)jb->B + j * jb->in_bytes;"),
    "A_for_B": ("const char* b_row = (const char*)jb->B + j * jb->K * jb->in_bytes;",
                "const char* b_row = (const char*)jb->A + j * jb->K * jb->in_bytes;"),
    "ties_away": ("(rem == 0.5 && fmod(n, 2.0) != 0.0)", "(rem == 0.5)"),
    "truncate": ("if (rem > 0.5 ||", "if (rem > 2.0 ||"),
    "subnormal_scale": ("v = ldexp((double)frac, f->emin - f->frac_bits);",
                        "v = ldexp((double)frac, f->emin - f->frac_bits - 1);"),
    "no_overflow": ("if (ee > f->emax) return inf_bits;", "if (ee > f->emax + 1) return inf_bits;"),
    "bf16_as_f16_in": ("g_lut[ORACLE_BF16][b] = decode_bits(b, &FMT_BF16);",
                       "g_lut[ORACLE_BF16][b] = decode_bits(b, &FMT_F16);"),
    # fused epilogue
    "epi_alpha_dropped": ("v = jb->alpha * v;", "v = v;"),
    "epi_beta_as_one": ("v += jb->beta * decode_bits(bits, f);", "v += decode_bits(bits, f);"),
    "epi_bias_by_row": ("if (jb->bias) v += (double)jb->bias[j];",
                        "if (jb->bias) v += (double)jb->bias[i];"),
    # FP8 operands
    "e4m3_bias_8": ("else v = ldexp((double)(8u + frac), (int)e - 7 - 3);",
                    "else v = ldexp((double)(8u + frac), (int)e - 8 - 3);"),
    "e4m3_top_binade_as_nan": ("if (e == 15u && frac == 7u) return NAN;",
                               "if (e == 15u) return NAN;"),
    "e4m3_subnormal_scale": ("if (e == 0) v = ldexp((double)frac, 1 - 7 - 3);",
                             "if (e == 0) v = ldexp((double)frac, 0 - 7 - 3);"),
    "e5m2_as_e4m3": ("g_lut8[1][b] = decode_bits(b, &FMT_E5M2);", "g_lut8[1][b] = decode_e4m3(b);"),
    "fp8_wrong_index": ("s += lut[a8[k]] * lut[b8[k]];", "s += lut[a8[k]] * lut[b8[k1 - 1 - (k - k0)]];"),
    # blockwise scales
    "bw_sfb_by_row_block": ("(double)jb->sfb[(j / jb->bn) * jb->nkb + kb];",
                            "(double)jb->sfb[(i / jb->bn) * jb->nkb + kb];"),
    "bw_first_scale_only": ("const double scale = (double)jb->sfa[(i / jb->bm) * jb->nkb + kb] *",
                            "const double scale = (double)jb->sfa[(i / jb->bm) * jb->nkb + 0] *"),
    "bw_short_block": ("const int64_t k1 = k0 + jb->bk < jb->K ? k0 + jb->bk : jb->K;",
                       "const int64_t k1 = k0 + jb->bk - 1 < jb->K ? k0 + jb->bk - 1 : jb->K;"),
    "bw_sfa_by_col_block": ("const double scale = (double)jb->sfa[(i / jb->bm) * jb->nkb + kb] *",
                            "const double scale = (double)jb->sfa[(j / jb->bm) * jb->nkb + kb] *"),
    "epi_relu_before_bias": ("if (jb->bias) v += (double)jb->bias[j];\n        if (jb->relu && !(v > 0.0)) v = 0.0;",
                             "if (jb->relu && !(v > 0.0)) v = 0.0;\n        if (jb->bias) v += (double)jb->bias[j];"),
}


def _build_mutant(tmp_path, name):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / f"{name}.c"
    path.write_text(src.replace(old, new))
    lib = tmp_path / f"lib{name}.so"
    subprocess.run(["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
                    str(path), "-o", str(lib), "-lm"], check=True)
    return oracle.load_library(str(lib))


def _pins_pass(lib) -> bool:
    """A compact run of the pin families; False as soon as one rejects."""
    # all-ones -> K, both input formats
    for dt in (F16, BF16):
        for K in (1, 130, 2000):
            A = torch.ones(2, K, dtype=TD[dt])
            got = oracle.decode(oracle.gemm(A, A, dt, F32, lib=lib), F32, lib=lib)
            if not np.all(got == K):
                return False
    # identity B -> A (includes subnormal fp16 inputs)
    A = torch.tensor([[2.0**-24, 3 * 2.0**-24, 0.5, -1.5, 2.0**-20, -7.0]], dtype=torch.float16)
    I = torch.eye(6, dtype=torch.float16)
    if not np.array_equal(oracle.gemm(A, I, F16, F16, lib=lib),
                          A.view(torch.int16).numpy().view(np.uint16)):
        return False
    # small integers, non-square, bf16 inputs
    A, B = si.make_small_int_operands(5, 3, 37, BF16, seed=1)
    ints = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    got = oracle.decode(oracle.gemm(A, B, BF16, F32, lib=lib), F32, lib=lib)
    if not np.array_equal(got, ints.astype(np.float64)):
        return False
    # exact-rational brute force, fp16 output (ties, rounding)
    A, B = si.make_operands(4, 3, 24, F16, "uniform", seed=2)
    ex = exact.exact_gemm(A, B)
    got = oracle.decode(oracle.gemm(A, B, F16, F16, lib=lib), F16, lib=lib)
    for i in range(4):
        for j in range(3):
            if Fraction(float(got[i, j])) != exact.round_exact(ex[i][j], F16):
                return False
    # fused epilogue, exact rational: alpha, beta, per-column bias, ReLU
    M, N, K = 3, 5, 16
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=3)
    bias = np.array([0.75, -1.5, 0.25, -0.125, 2.0], dtype=np.float32)
    prev = oracle.round_to(np.linspace(-2, 2, M * N).reshape(M, N), F32, lib=lib)
    S = exact.exact_gemm(A, B)
    prev_exact = oracle.decode(prev, F32, lib=lib)
    for relu in (False, True):
        got = oracle.decode(oracle.gemm_epilogue(A, B, F16, F32, alpha=-1.5, beta=0.75, cprev=prev,
                                                 bias=bias, relu=relu, lib=lib), F32, lib=lib)
        for i in range(M):
            for j in range(N):
                q = (Fraction(-3, 2) * S[i][j] + Fraction(3, 4) * Fraction(float(prev_exact[i, j]))
                     + Fraction(float(bias[j])))
                if relu and q < 0:
                    q = Fraction(0)
                if Fraction(float(got[i, j])) != exact.round_exact(q, F32):
                    return False
    # FP8 decoders against torch's widening, all 256 patterns
    for dt, td in ((E4M3, torch.float8_e4m3fn), (E5M2, torch.float8_e5m2)):
        bits = np.arange(256, dtype=np.uint8)
        got = oracle.decode(bits, dt, lib=lib)
        want = torch.from_numpy(bits.copy()).view(td).to(torch.float64).numpy()
        nan = np.isnan(want)
        if not (np.array_equal(np.isnan(got), nan) and np.array_equal(got[~nan], want[~nan])):
            return False
    # FP8 product, exact rational (non-square, non-symmetric)
    for dt in (E4M3, E5M2):
        A, B = si.make_operands(4, 3, 24, dt, "uniform", seed=4)
        ex = exact.exact_gemm(A, B)
        got = oracle.decode(oracle.gemm(A, B, dt, F32, lib=lib), F32, lib=lib)
        for i in range(4):
            for j in range(3):
                if Fraction(float(got[i, j])) != exact.round_exact(ex[i][j], F32):
                    return False
    # blockwise scales, exact rational: M == N keeps a mis-indexed scale in bounds
    M = N = 5
    K, bm, bn, bk = 13, 2, 3, 4
    A, B = si.make_small_int_operands(M, N, K, E4M3, seed=5)
    g = torch.Generator().manual_seed(6)
    sfa = torch.exp2(torch.randint(-3, 4, (3, 4), generator=g).float()).numpy()
    sfb = torch.exp2(torch.randint(-3, 4, (2, 4), generator=g).float()).numpy()
    av, bv = exact.exact_values(A), exact.exact_values(B)
    got = oracle.decode(oracle.gemm_blockwise(A, B, sfa, sfb, bm, bn, bk, E4M3, F32, lib=lib),
                        F32, lib=lib)
    for i in range(M):
        for j in range(N):
            q = sum((Fraction(float(sfa[i // bm, k // bk])) * Fraction(float(sfb[j // bn, k // bk]))
                     * av[i][k] * bv[j][k] for k in range(K)), Fraction(0))
            if Fraction(float(got[i, j])) != exact.round_exact(q, F32):
                return False
    # rounding routine against numpy on ties and overflow
    x = np.array([1.0 + 2.0**-11, 1.0 + 3 * 2.0**-11, 65520.0, 70000.0, 2.0**-25 * 3])
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    if not np.array_equal(oracle.round_to(x, F16, lib=lib), want):
        return False
    return True


def test_committed_oracle_passes(tmp_path):
    assert _pins_pass(oracle.load_library(oracle.build()))


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(tmp_path, name):
    lib = _build_mutant(tmp_path, name)
    assert not _pins_pass(lib), f"planted mistake {name!r} slipped past the pins"
