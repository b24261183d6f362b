"""Pins for the CPU oracle: it is checked against things other than itself.

* format decoders   -> numpy/torch widening casts over every 16-bit pattern;
* RNE encoder       -> numpy's float64->float16/float32 casts, torch's
                       float32->bfloat16 cast, and exact-rational rounding;
* the GEMM          -> exact-rational brute force on tiny shapes, and the
                       closed forms named for the method: all-ones (C = K),
                       identity B (C = A), small-integer operands (exact integer
                       products), rank-1 operands (C_ij = u_i v_j (a.b)).
A dropped term, a wrong sign or index, or a transposed operand in the oracle
fails the brute-force and rank-1 checks (non-square, non-symmetric inputs).
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import seeded_inputs as si
from tests import exact

F16, BF16, F32 = 0, 1, 2
TD = {F16: torch.float16, BF16: torch.bfloat16}


# ---------------------------------------------------------------- decoders --

def test_decode_f16_all_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_lib.decode(bits, F16)
    want = bits.view(np.float16).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])
    # signed zero
    assert np.signbit(got[0x8000]) and not np.signbit(got[0])


def test_decode_bf16_all_patterns(oracle_lib):
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    got = oracle_lib.decode(bits, BF16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_decode_f32_sample(oracle_lib):
    rng = np.random.default_rng(5)
    bits = rng.integers(0, 2**32, 200000, dtype=np.uint64).astype(np.uint32)
    bits[:4] = [0, 0x80000000, 0x00000001, 0x7F7FFFFF]
    got = oracle_lib.decode(bits, F32)
    want = bits.view(np.float32).astype(np.float64)
    nan = np.isnan(want)
    assert np.array_equal(got[~nan], want[~nan])


# ----------------------------------------------------------------- rounding --

def _hard_doubles(seed, n):
    """Doubles spread over the f16/bf16/f32 ranges, including subnormals,
    exact ties between neighbours, overflow and values near zero."""
    rng = np.random.default_rng(seed)
    mags = [np.exp2(rng.uniform(-30, 20, n)), np.exp2(rng.uniform(-140, 130, n))]
    x = np.concatenate(mags) * rng.choice([-1.0, 1.0], 2 * n)
    # exact midpoints between consecutive fp16 values (ties)
    h = rng.integers(0, 0x7BFF, n, dtype=np.uint16)
    lo = h.view(np.float16).astype(np.float64)
    hi = (h + 1).view(np.float16).astype(np.float64)
    ties = (lo + hi) / 2
    extra = np.array([0.0, -0.0, 65504.0, 65519.99, 65520.0, 65536.0, 1e300, -1e300,
                      2.0**-24, 2.0**-25, 2.0**-25 * 1.0000001, 2.0**-26, 5.96e-8,
                      3.4028234663852886e38, 3.4028235677973366e38, 2.0**-149, 2.0**-150])
    return np.concatenate([x, ties, -ties, extra])


def test_round_f16_matches_numpy(oracle_lib):
    x = _hard_doubles(1, 20000)
    got = oracle_lib.round_to(x, F16)
    with np.errstate(over="ignore"):
        want = x.astype(np.float16).view(np.uint16)
    assert np.array_equal(got, want)


def test_round_f32_matches_numpy(oracle_lib):
    x = _hard_doubles(2, 20000)
    # exact f32 midpoints
    rng = np.random.default_rng(3)
    f = rng.integers(0x00800000, 0x7F000000, 5000, dtype=np.uint64).astype(np.uint32)
    lo = f.view(np.float32).astype(np.float64)
    hi = (f + 1).view(np.float32).astype(np.float64)
    x = np.concatenate([x, (lo + hi) / 2])
    got = oracle_lib.round_to(x, F32)
    with np.errstate(over="ignore"):
        want = x.astype(np.float32).view(np.uint32)
    assert np.array_equal(got, want)


def test_round_bf16_matches_torch_on_f32_values(oracle_lib):
    # values exactly representable in fp32: torch's fp32 -> bf16 cast is then
    # a single RNE step, the same operation the oracle performs.
    rng = np.random.default_rng(4)
    f = rng.integers(0, 0x7F7FFFFF, 50000, dtype=np.uint64).astype(np.uint32)
    f[:1000] = (f[:1000] & 0xFFFF0000) | 0x8000        # exact bf16 ties
    x32 = f.view(np.float32)
    x = np.concatenate([x32, -x32]).astype(np.float64)
    got = oracle_lib.round_to(x, BF16)
    want = torch.from_numpy(x.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(got, want.numpy().view(np.uint16))


@pytest.mark.parametrize("fmt", [F16, BF16, F32])
def test_round_matches_exact_rational(oracle_lib, fmt):
    x = _hard_doubles(10 + fmt, 3000)
    got = oracle_lib.decode(oracle_lib.round_to(x, fmt), fmt)
    for xi, gi in zip(x, got):
        want = exact.round_exact(Fraction(float(xi)), fmt)
        if want in (exact.INF, -exact.INF):
            assert gi == float(want), (xi, gi)
        else:
            assert Fraction(float(gi)) == want, (xi, gi, want)


# -------------------------------------------------------- brute-force GEMM --

def _rounding_is_stable(value: Fraction, bound: Fraction, fmt: int) -> bool:
    """True when every number within `bound` of `value` rounds the same way,
    i.e. the binary64 sum cannot land on the other side of a tie."""
    r = exact.round_exact(value, fmt)
    return exact.round_exact(value - bound, fmt) == r == exact.round_exact(value + bound, fmt)


def _binary64_sum_is_exact(a_row, b_row) -> bool:
    """True when every partial sum of the sequential dot product is a binary64
    number, so the oracle's sum carries no rounding error at all (then even an
    exact tie of the output format must be resolved to even)."""
    s = Fraction(0)
    for x, y in zip(a_row, b_row):
        s += x * y
        if Fraction(float(s)) != s:
            return False
    return True


@pytest.mark.parametrize("dtype_in", [F16, BF16])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_brute_force_tiny(oracle_lib, dtype_in, dtype_out):
    shapes = [(1, 1, 1), (3, 5, 7), (5, 3, 16), (4, 6, 33), (2, 7, 64), (6, 2, 130),
              (7, 4, 129)]
    checked = skipped = ties = 0
    for t, (M, N, K) in enumerate(shapes):
        A, B = si.make_operands(M, N, K, dtype_in, "uniform", seed=100 + t)
        A = A * 3           # push some products past 1 to exercise more binades
        A = A.to(TD[dtype_in])
        ex = exact.exact_gemm(A, B)
        absb = exact.abs_gemm_bound(A, B)
        av, bv = exact.exact_values(A), exact.exact_values(B)
        got = oracle_lib.decode(oracle_lib.gemm(A, B, dtype_in, dtype_out), dtype_out)
        for i in range(M):
            for j in range(N):
                # binary64 sequential-sum error bound: K * 2^-53 * sum|a b|
                bound = Fraction(float(absb[i, j])) * K * Fraction(1, 2**53)
                if not (_binary64_sum_is_exact(av[i], bv[j])
                        or _rounding_is_stable(ex[i][j], bound, dtype_out)):
                    skipped += 1
                    continue
                if not _rounding_is_stable(ex[i][j], bound, dtype_out):
                    ties += 1
                checked += 1
                want = exact.round_exact(ex[i][j], dtype_out)
                assert Fraction(float(got[i, j])) == want, (M, N, K, i, j)
    assert checked > 20 * skipped
    if dtype_out == F32:
        assert ties > 0      # exact fp32 ties do occur here and were resolved to even


def test_oracle_select_matches_full(oracle_lib):
    M, N, K = 37, 41, 96
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=7)
    full = oracle_lib.gemm(A, B, F16, F32)
    rows, cols = [0, 5, 36], [40, 1, 7, 0]
    sub = oracle_lib.gemm_select(A, B, rows, cols, F16, F32)
    assert np.array_equal(sub, full[np.ix_(rows, cols)])
    rsub, r64 = oracle_lib.gemm_select(A, B, rows, None, F16, F32, want_f64=True)
    assert np.array_equal(rsub, full[rows])
    assert np.array_equal(oracle_lib.round_to(r64, F32), rsub)
    csub = oracle_lib.gemm_select(A, B, None, cols, F16, F32)
    assert np.array_equal(csub, full[:, cols])


# ---------------------------------------------------------- closed forms --

@pytest.mark.parametrize("dtype_in", [F16, BF16])
@pytest.mark.parametrize("K", [1, 16, 130, 256, 257, 2000, 4096, 28672])
def test_all_ones_gives_K(oracle_lib, dtype_in, K):
    M, N = 3, 5
    A = torch.ones(M, K, dtype=TD[dtype_in])
    B = torch.ones(N, K, dtype=TD[dtype_in])
    for dtype_out in (F16, BF16, F32):
        got = oracle_lib.decode(oracle_lib.gemm(A, B, dtype_in, dtype_out), dtype_out)
        want = float(exact.round_exact(Fraction(K), dtype_out))
        assert np.all(got == want), (K, dtype_out, got[0, 0], want)
    # K = 257 is a bf16 tie (256 and 258 are neighbours): ties-to-even gives 256
    if K == 257:
        got = oracle_lib.decode(oracle_lib.gemm(A, B, dtype_in, BF16), BF16)
        assert np.all(got == 256.0)


@pytest.mark.parametrize("dtype_in", [F16, BF16])
def test_identity_B_gives_A(oracle_lib, dtype_in):
    M, K = 19, 48
    A, _ = si.make_operands(M, 1, K, dtype_in, "uniform", seed=11)
    B = torch.eye(K, dtype=TD[dtype_in])
    same = oracle_lib.gemm(A, B, dtype_in, dtype_in)
    assert np.array_equal(same, A.view(torch.int16).numpy().view(np.uint16))
    f32 = oracle_lib.decode(oracle_lib.gemm(A, B, dtype_in, F32), F32)
    assert np.array_equal(f32, A.to(torch.float64).numpy())


@pytest.mark.parametrize("dtype_in", [F16, BF16])
def test_small_integers_exact(oracle_lib, dtype_in):
    M, N, K = 23, 17, 515
    A, B = si.make_small_int_operands(M, N, K, dtype_in, seed=12)
    ints = A.to(torch.int64).numpy() @ B.to(torch.int64).numpy().T   # exact integers
    f32 = oracle_lib.decode(oracle_lib.gemm(A, B, dtype_in, F32), F32)
    assert np.array_equal(f32, ints.astype(np.float64))
    f16 = oracle_lib.gemm(A, B, dtype_in, F16)
    assert np.array_equal(f16, ints.astype(np.float64).astype(np.float16).view(np.uint16))
    bf16 = oracle_lib.gemm(A, B, dtype_in, BF16)
    want = torch.from_numpy(ints.astype(np.float32)).to(torch.bfloat16).view(torch.int16)
    assert np.array_equal(bf16, want.numpy().view(np.uint16))


@pytest.mark.parametrize("dtype_in", [F16, BF16])
def test_rank1_operands(oracle_lib, dtype_in):
    M, N, K = 9, 13, 200
    g = torch.Generator().manual_seed(13)
    u = torch.tensor([2.0 ** int(e) for e in torch.randint(-3, 4, (M,), generator=g)])
    v = torch.tensor([2.0 ** int(e) for e in torch.randint(-3, 4, (N,), generator=g)])
    u = u * torch.where(torch.rand(M, generator=g) < 0.5, -1.0, 1.0)
    a = torch.randint(-3, 4, (K,), generator=g).to(torch.float64)
    b = torch.randint(-3, 4, (K,), generator=g).to(torch.float64)
    A = (u[:, None] * a[None, :]).to(TD[dtype_in])
    B = (v[:, None] * b[None, :]).to(TD[dtype_in])
    dot = float((a * b).sum())
    want = (u[:, None] * v[None, :]).numpy() * dot
    got = oracle_lib.decode(oracle_lib.gemm(A, B, dtype_in, F32), F32)
    assert np.array_equal(got, want)
    assert not np.array_equal(got, got.T[:M, :N]) if M == N else True


def test_empty_K_gives_zero(oracle_lib):
    A = torch.empty(4, 0, dtype=torch.float16)
    B = torch.empty(3, 0, dtype=torch.float16)
    got = oracle_lib.gemm(A, B, F16, F32)
    assert got.shape == (4, 3) and np.all(got == 0)


def test_threads_do_not_change_result(oracle_lib):
    A, B = si.make_operands(64, 48, 320, BF16, "normal", seed=14)
    one = oracle_lib.gemm(A, B, BF16, F32, nthreads=1)
    many = oracle_lib.gemm(A, B, BF16, F32, nthreads=7)
    assert np.array_equal(one, many)


def test_rejects_bad_dtype(oracle_lib):
    A = torch.zeros(2, 2, dtype=torch.float16)
    with pytest.raises(ValueError):
        oracle_lib.gemm(A, A, 2, 0)


# ---------------------------------------------------------------------------------------
# Fused epilogue: D = act(alpha * S + beta * Cprev + bias[j])  ("CUTLASS Deep Dive: From
# CuTe Layouts to Blackwell tcgen05", Part 6: Epilogue Visitor Trees; Classic Fused
# Epilogue: Bias + ReLU).
# ---------------------------------------------------------------------------------------

@pytest.mark.parametrize("dtype_in", [F16, BF16])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_epilogue_identity_is_the_plain_product(oracle_lib, dtype_in, dtype_out):
    A, B = si.make_operands(9, 11, 40, dtype_in, "uniform", seed=60)
    assert np.array_equal(oracle_lib.gemm_epilogue(A, B, dtype_in, dtype_out),
                          oracle_lib.gemm(A, B, dtype_in, dtype_out))


def _f32(x):
    return np.float32(x)


@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
@pytest.mark.parametrize("relu", [False, True])
def test_epilogue_exact_rational(oracle_lib, dtype_out, relu):
    # every term exact in rational arithmetic (alpha, beta, bias are binary32 values,
    # Cprev the decoded output patterns), ReLU applied, then one round-to-nearest-even
    g = torch.Generator().manual_seed(61 + dtype_out + 3 * relu)
    M, N, K = 4, 5, 24
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=62)
    alpha, beta = _f32(-0.7109375), _f32(1.3125)
    bias = (torch.rand(N, generator=g) * 4 - 2).numpy().astype(np.float32)
    prev_vals = (torch.rand(M, N, generator=g) * 6 - 3)
    prev = oracle_lib.round_to(prev_vals.numpy().astype(np.float64), dtype_out)
    got = oracle_lib.decode(oracle_lib.gemm_epilogue(A, B, F16, dtype_out, alpha, beta, prev, bias,
                                                     relu), dtype_out)
    S = exact.exact_gemm(A, B)
    prev_exact = oracle_lib.decode(prev, dtype_out)
    for i in range(M):
        for j in range(N):
            q = (Fraction(float(alpha)) * S[i][j] + Fraction(float(beta)) * Fraction(float(prev_exact[i, j]))
                 + Fraction(float(bias[j])))
            if relu and q < 0:
                q = Fraction(0)
            assert Fraction(float(got[i, j])) == exact.round_exact(q, dtype_out), (i, j)


def test_epilogue_closed_forms(oracle_lib):
    M, N = 3, 6
    # K = 0: D = round(beta * Cprev + bias); numpy's float64 -> float16 cast rounds to even
    A = torch.empty(M, 0, dtype=torch.float16)
    B = torch.empty(N, 0, dtype=torch.float16)
    prev = np.arange(M * N, dtype=np.float16).reshape(M, N).view(np.uint16)
    bias = np.linspace(-1.0, 1.0, N).astype(np.float32)
    got = oracle_lib.gemm_epilogue(A, B, F16, F16, beta=0.5, cprev=prev, bias=bias)
    want = (0.5 * prev.view(np.float16).astype(np.float64) + bias.astype(np.float64)).astype(np.float16)
    assert np.array_equal(got, want.view(np.uint16))
    # alpha a power of two scales the plain result exactly (no overflow or subnormals here)
    A, B = si.make_operands(M, N, 64, F16, "uniform", seed=63)
    plain = oracle_lib.decode(oracle_lib.gemm(A, B, F16, F32), F32)
    got = oracle_lib.decode(oracle_lib.gemm_epilogue(A, B, F16, F32, alpha=4.0), F32)
    assert np.array_equal(got, 4.0 * plain)
    # ReLU: negatives become +0, the rest is untouched
    got = oracle_lib.gemm_epilogue(A, B, F16, F32, relu=True)
    want = np.where(plain > 0, plain, 0.0)
    assert np.array_equal(oracle_lib.decode(got, F32), want)
    assert np.all(got[plain <= 0] == 0)                        # +0, not -0
    # the bias is per column: a bias on column 2 only changes column 2
    bias = np.zeros(N, dtype=np.float32)
    bias[2] = 1024.0
    got = oracle_lib.decode(oracle_lib.gemm_epilogue(A, B, F16, F32, bias=bias), F32)
    assert np.array_equal(got[:, [0, 1, 3, 4, 5]], plain[:, [0, 1, 3, 4, 5]])
    assert np.all(got[:, 2] != plain[:, 2])


def test_epilogue_rejects_beta_without_prev(oracle_lib):
    A, B = si.make_operands(2, 2, 8, F16, "uniform", seed=64)
    with pytest.raises(ValueError):
        oracle_lib.gemm_epilogue(A, B, F16, F16, beta=1.0, cprev=None)
