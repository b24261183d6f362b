"""Pins for the oracle's FP8 operands and its blockwise-scaled product
("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05", Part 6, FP8 and
Blockwise Scaling), checked against things other than the oracle itself:

* E4M3 / E5M2 decoders -> torch's float8_e4m3fn / float8_e5m2 widening over all 256
  patterns, and values fixed by the OCP format definitions (largest finite, the NaN
  and infinity patterns, the smallest subnormal);
* the FP8 product      -> exact-rational brute force on tiny shapes, all-ones (C = K),
  identity B (C = A), small integers (exact integer products);
* the blockwise sum    -> exact rationals with per-block scales (independent Fraction
  arithmetic), all scales 1 (the plain product), one non-zero block (the plain product
  over that block's K range, scaled), and per-row-block scales that factor out.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import exact

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
TD = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}


# ---------------------------------------------------------------- decoders --

@pytest.mark.parametrize("dt", [E4M3, E5M2])
def test_decode_fp8_all_patterns(oracle_lib, dt):
    bits = np.arange(256, dtype=np.uint8)
    got = oracle_lib.decode(bits, dt)
    want = torch.from_numpy(bits.copy()).view(TD[dt]).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    assert np.signbit(got[0x80]) and not np.signbit(got[0])


def test_decode_fp8_definition_values(oracle_lib):
    e4 = oracle_lib.decode(np.array([0x7E, 0x7F, 0xFF, 0x01, 0x08, 0x07, 0x38, 0x78],
                                    dtype=np.uint8), E4M3)
    # largest finite 1.75 * 2^8; S.1111.111 is NaN (no infinity); smallest subnormal
    # 2^-9; smallest normal 2^-6; largest subnormal 7 * 2^-9; one; 2^8
    assert e4[0] == 448.0 and np.isnan(e4[1]) and np.isnan(e4[2])
    assert e4[3] == 2.0 ** -9 and e4[4] == 2.0 ** -6 and e4[5] == 7 * 2.0 ** -9
    assert e4[6] == 1.0 and e4[7] == 256.0
    e5 = oracle_lib.decode(np.array([0x7B, 0x7C, 0xFC, 0x7D, 0x01, 0x04, 0x3C],
                                    dtype=np.uint8), E5M2)
    # largest finite 1.75 * 2^15; +-infinity; NaN; smallest subnormal 2^-16; smallest
    # normal 2^-14; one
    assert e5[0] == 57344.0 and e5[1] == np.inf and e5[2] == -np.inf and np.isnan(e5[3])
    assert e5[4] == 2.0 ** -16 and e5[5] == 2.0 ** -14 and e5[6] == 1.0


# ------------------------------------------------------------- FP8 product --

def _exact_rounded(q, dtype_out):
    return float(exact.round_exact(q, dtype_out))


@pytest.mark.parametrize("dt", [E4M3, E5M2])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_fp8_brute_force_tiny(oracle_lib, dt, dtype_out):
    # With FP8 operands every product has at most 8 significant bits and these sums
    # stay far inside binary64's 53 bits, so the oracle's sum is exact and its one
    # rounding must equal the exact rational's.
    for t, (M, N, K) in enumerate([(1, 1, 1), (3, 5, 7), (5, 3, 16), (4, 6, 33), (2, 7, 130)]):
        A, B = si.make_operands(M, N, K, dt, "uniform", seed=200 + t)
        A = (A.float() * 8).to(TD[dt])        # more binades, up to |8|
        ex = exact.exact_gemm(A, B)
        got = oracle_lib.decode(oracle_lib.gemm(A, B, dt, dtype_out), dtype_out)
        for i in range(M):
            for j in range(N):
                assert got[i, j] == _exact_rounded(ex[i][j], dtype_out), (M, N, K, i, j)


@pytest.mark.parametrize("dt", [E4M3, E5M2])
@pytest.mark.parametrize("K", [1, 128, 257, 4096])
def test_fp8_all_ones_gives_K(oracle_lib, dt, K):
    A = torch.ones(3, K).to(TD[dt])
    B = torch.ones(4, K).to(TD[dt])
    for dtype_out in (F16, BF16, F32):
        got = oracle_lib.decode(oracle_lib.gemm(A, B, dt, dtype_out), dtype_out)
        assert np.all(got == _exact_rounded(Fraction(K), dtype_out))


@pytest.mark.parametrize("dt", [E4M3, E5M2])
def test_fp8_identity_and_small_integers(oracle_lib, dt):
    A, _ = si.make_operands(7, 1, 48, dt, "uniform", seed=210)
    B = torch.eye(48).to(TD[dt])
    got = oracle_lib.decode(oracle_lib.gemm(A, B, dt, F32), F32)
    assert np.array_equal(got, A.to(torch.float64).numpy())      # every FP8 value fits F32
    A, B = si.make_small_int_operands(11, 9, 300, dt, seed=211)
    ints = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T
    got = oracle_lib.decode(oracle_lib.gemm(A, B, dt, F32), F32)
    assert np.array_equal(got, ints.astype(np.float64))


def test_fp8_rejects_a_16_bit_operand(oracle_lib):
    A = torch.ones(2, 8, dtype=torch.float16)
    with pytest.raises(TypeError):
        oracle_lib.gemm(A, A, E4M3, F32)


# --------------------------------------------------------------- blockwise --

def _exact_blockwise(A, B, sfa, sfb, bm, bn, bk):
    a, b = exact.exact_values(A), exact.exact_values(B)
    K = len(a[0]) if a else 0
    nkb = -(-K // bk)
    out = []
    for i, ra in enumerate(a):
        row = []
        for j, rb in enumerate(b):
            s = Fraction(0)
            for kb in range(nkb):
                part = sum((x * y for x, y in zip(ra[kb * bk:(kb + 1) * bk], rb[kb * bk:(kb + 1) * bk])),
                           Fraction(0))
                s += Fraction(float(sfa[i // bm, kb])) * Fraction(float(sfb[j // bn, kb])) * part
            row.append(s)
        out.append(row)
    return out


@pytest.mark.parametrize("dt", [E4M3, E5M2, F16])
@pytest.mark.parametrize("M,N,K,bm,bn,bk", [(5, 5, 13, 2, 3, 4), (7, 4, 20, 3, 2, 5),
                                            (3, 6, 9, 128, 128, 128), (6, 6, 32, 1, 4, 8)])
def test_blockwise_exact_rational(oracle_lib, dt, M, N, K, bm, bn, bk):
    # small-integer operands and power-of-two scales: every step is exact in binary64,
    # so the oracle must return the exact rational rounded once
    A, B = si.make_small_int_operands(M, N, K, dt, seed=220 + K)
    nkb = -(-K // bk)
    g = torch.Generator().manual_seed(221 + K)
    sfa = torch.exp2(torch.randint(-3, 4, (-(-M // bm), nkb), generator=g).float()).numpy()
    sfb = torch.exp2(torch.randint(-3, 4, (-(-N // bn), nkb), generator=g).float()).numpy()
    ex = _exact_blockwise(A, B, sfa, sfb, bm, bn, bk)
    for dtype_out in (F32, BF16):
        got = oracle_lib.decode(oracle_lib.gemm_blockwise(A, B, sfa, sfb, bm, bn, bk, dt, dtype_out),
                                dtype_out)
        for i in range(M):
            for j in range(N):
                assert got[i, j] == _exact_rounded(ex[i][j], dtype_out), (i, j, dtype_out)


def test_blockwise_general_scales_exact_rational(oracle_lib):
    # scales that are not powers of two: the exact value, rounded, wherever binary64's
    # error (a few units of 2^-53 of the sum of |terms|) cannot cross a rounding edge
    M, N, K, bm, bn, bk = 6, 5, 40, 2, 3, 16
    A, B = si.make_operands(M, N, K, E4M3, "uniform", seed=230)
    sfa = si.make_block_scales(3, 3, seed=231).numpy()
    sfb = si.make_block_scales(2, 3, seed=232).numpy()
    ex = _exact_blockwise(A, B, sfa, sfb, bm, bn, bk)
    got = oracle_lib.decode(oracle_lib.gemm_blockwise(A, B, sfa, sfb, bm, bn, bk, E4M3, F32), F32)
    a, b = A.to(torch.float64).abs().numpy(), B.to(torch.float64).abs().numpy()
    checked = 0
    for i in range(M):
        for j in range(N):
            mag = sum(float(sfa[i // bm, kb] * sfb[j // bn, kb])
                      * float(a[i, kb * bk:(kb + 1) * bk] @ b[j, kb * bk:(kb + 1) * bk]) for kb in range(3))
            bound = Fraction(mag) * (K + 8) * Fraction(1, 2 ** 53)
            r = exact.round_exact(ex[i][j], F32)
            if exact.round_exact(ex[i][j] - bound, F32) != r or exact.round_exact(ex[i][j] + bound, F32) != r:
                continue
            checked += 1
            assert got[i, j] == float(r), (i, j)
    assert checked >= 25


@pytest.mark.parametrize("dt", [E4M3, BF16])
def test_blockwise_unit_scales_are_the_plain_product(oracle_lib, dt):
    M, N, K = 9, 11, 300
    A, B = si.make_operands(M, N, K, dt, "uniform", seed=240)
    for bm, bn, bk in ((128, 128, 128), (4, 3, 64), (1, 1, 7)):
        nkb = -(-K // bk)
        sfa = np.ones((-(-M // bm), nkb), np.float32)
        sfb = np.ones((-(-N // bn), nkb), np.float32)
        _, v = oracle_lib.gemm_blockwise(A, B, sfa, sfb, bm, bn, bk, dt, F32, want_f64=True)
        # blocks summed separately differ from one running sum only by binary64 rounding
        want = oracle_lib.decode(oracle_lib.gemm(A, B, dt, F32), F32)
        assert np.allclose(v, want, rtol=1e-6, atol=1e-6)
    # one block covering all of K is the plain product, bit for bit
    sfa = np.ones((1, 1), np.float32)
    sfb = np.ones((1, 1), np.float32)
    got = oracle_lib.gemm_blockwise(A, B, sfa, sfb, 128, 128, 512, dt, F16)
    assert np.array_equal(got, oracle_lib.gemm(A, B, dt, F16))


def test_blockwise_one_live_block(oracle_lib):
    # zero scales everywhere except k block 2 (of A's row block 0 and every B block):
    # rows of A's first row block are 0.25 * the plain product over that block's K range
    M, N, K, bm, bn, bk = 8, 6, 100, 4, 2, 24
    A, B = si.make_operands(M, N, K, E5M2, "uniform", seed=250)
    nkb = -(-K // bk)
    sfa = np.zeros((2, nkb), np.float32)
    sfb = np.zeros((3, nkb), np.float32)
    sfa[0, 2] = 0.5
    sfb[:, 2] = 0.5
    got = oracle_lib.decode(oracle_lib.gemm_blockwise(A, B, sfa, sfb, bm, bn, bk, E5M2, F32), F32)
    part = oracle_lib.decode(oracle_lib.gemm(A[:, 48:72].contiguous(), B[:, 48:72].contiguous(),
                                             E5M2, F32), F32)
    assert np.array_equal(got[:4], 0.25 * part[:4])
    assert np.all(got[4:] == 0)


def test_blockwise_row_scales_factor_out(oracle_lib):
    # a scale that depends only on A's row block (the same in every k block) and unit
    # B scales multiply whole rows of the plain product (powers of two: exact)
    M, N, K, bm = 12, 7, 256, 4
    A, B = si.make_operands(M, N, K, E4M3, "uniform", seed=260)
    r = np.array([0.5, 4.0, 0.125], np.float32)
    sfa = np.repeat(r[:, None], 2, axis=1)
    sfb = np.ones((1, 2), np.float32)
    _, v = oracle_lib.gemm_blockwise(A, B, sfa, sfb, bm, 128, 128, E4M3, F32, want_f64=True)
    _, plain = oracle_lib.gemm_select(A, B, None, None, E4M3, F32, want_f64=True)
    scale = np.repeat(r, bm)[:, None].astype(np.float64)
    assert np.allclose(v, scale * plain, rtol=1e-12, atol=0)


def test_blockwise_rejects_bad_scale_shapes(oracle_lib):
    A = torch.ones(4, 16).to(torch.float8_e4m3fn)
    with pytest.raises(ValueError):
        oracle_lib.gemm_blockwise(A, A, np.ones((1, 1), np.float32), np.ones((1, 2), np.float32),
                                  4, 4, 8, E4M3, F32)
