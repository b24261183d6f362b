"""Blockwise-scaled FP8 products through the C ABI (gemm_run_blockwise) against the
oracle's gemm_blockwise, element by element ("CUTLASS Deep Dive: From CuTe Layouts to
Blackwell tcgen05", Part 6, FP8 and Blockwise Scaling):
    C[i, j] = sum_kb sfa[i // block_m, kb] * sfb[j // 128, kb] * P_kb[i, j]
with P_kb the product over the kb-th 128 elements of K.

Tolerance.  The kernel accumulates each K block in fp32 in Tensor Memory, rounds the
scale product sfa * sfb to binary32 and adds with one fma per block.  The accumulation
bound tau uses sigma over the scaled terms (sfa sfb a_ik b_jk); the scale-product and
fma roundings add at most 2 * 2^-24 * sum_kb |s_kb P_kb|, folded into an effective
sigma.  Integer operands with power-of-two scales are exact at every step: bit-exact.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
TD = si.TORCH_DTYPE


@pytest.fixture(scope="module")
def g():
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    h = Gemm()
    yield h
    h.close()


def _scales(M, N, K, bm, seed, pow2=False):
    nkb = -(-K // 128)
    if pow2:
        gen = torch.Generator().manual_seed(seed)
        sfa = torch.exp2(torch.randint(-3, 4, (-(-M // bm), nkb), generator=gen).float())
        sfb = torch.exp2(torch.randint(-3, 4, (-(-N // 128), nkb), generator=gen).float())
        return sfa, sfb
    return (si.make_block_scales(-(-M // bm), nkb, seed=seed),
            si.make_block_scales(-(-N // 128), nkb, seed=seed + 1))


def _kmajor(scales):
    """The library's scale layout: K-block-major (ceil(K/128) x blocks), on the device."""
    return scales.T.contiguous().cuda()


def _effective_sigma(A, B, sfa, sfb, bm, bn=128):
    """sigma over the scaled terms, plus the scale-product and fma roundings (see the
    module docstring); sfa rows are taken per block of bm rows of A, sfb per bn of B."""
    M, K = A.shape
    N = B.shape[0]
    a = A.to(torch.float64).numpy()
    b = B.to(torch.float64).numpy()
    fa = sfa.double().numpy()[np.arange(M) // bm]      # M x nkb
    fb = sfb.double().numpy()[np.arange(N) // bn]      # N x nkb
    kb = np.arange(K) // 128
    sigma = np.sqrt(np.square(a * fa[:, kb]) @ np.square(b * fb[:, kb]).T)
    absum = np.zeros((M, N))
    for t in range(-(-K // 128)):
        blk = slice(128 * t, 128 * t + 128)
        absum += np.abs(np.outer(fa[:, t], fb[:, t]) * (a[:, blk] @ b[:, blk].T))
    return sigma + absum / (2.0 * np.sqrt(max(K, 1)))


def _case(g, M, N, K, dt, dtype_out, bm, seed, cfg=None, ints=False):
    if ints:
        A, B = si.make_small_int_operands(M, N, K, dt, seed=seed)
    else:
        gen = torch.Generator().manual_seed(seed)
        A = ((torch.rand(M, K, generator=gen) * 2 - 1) * 4).to(TD[dt])
        B = ((torch.rand(N, K, generator=gen) * 2 - 1) * 4).to(TD[dt])
    sfa, sfb = _scales(M, N, K, bm, seed + 7, pow2=ints)
    C = torch.empty(M, N, dtype=TD[dtype_out], device="cuda")
    try:
        if cfg:
            g.set_config(**cfg)
        g.run_blockwise(A.cuda(), B.cuda(), C, _kmajor(sfa), _kmajor(sfb), bm)
        torch.cuda.synchronize()
        st = g.device_status()
        used = g.last_config()
    finally:
        g.reset_config()
    assert st[0] == 0, f"device status {st}"
    want, c64 = oracle.gemm_blockwise(A, B, sfa.numpy(), sfb.numpy(), bm, 128, 128, dt, dtype_out,
                                      want_f64=True)
    what = f"blockwise {dt} bm={bm} M={M} N={N} K={K} out={dtype_out} {used}"
    if ints:
        parity.check(parity.bits_of(C), want, dtype_out, exact=True, what=what)
    else:
        parity.check(parity.bits_of(C), want, dtype_out, what=what, c64=c64,
                     sigma=_effective_sigma(A, B, sfa, sfb, bm), K=K)
    return used


@pytest.mark.parametrize("dt", [E4M3, E5M2])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
@pytest.mark.parametrize("bm", [1, 128, 37])
def test_blockwise_against_oracle(g, dt, dtype_out, bm):
    used = _case(g, 300, 700, 1040, dt, dtype_out, bm, seed=400)   # ragged M, N, K tails
    assert used["chain_kblocks"] == 1 and used["epilogue"] == 1, used
    # one CTA per 128 x 128 tile (four accumulator slots)
    assert used["variant"] == 1 and used["block_n"] == 128, used


@pytest.mark.parametrize("cfg,M,N,K", [
    ({"variant": 2, "block_n": 256}, 512, 768, 4096),
    ({"variant": 2, "block_n": 256, "splits": 2}, 256, 1024, 4096),       # split-K
    ({"variant": 1, "block_n": 256, "splits": 3}, 300, 1100, 2048),
    ({"variant": 1, "block_n": 128}, 131, 1001, 1024),                    # direct stores
    ({"variant": 2, "block_n": 128, "splits": -1, "max_ctas": 38}, 300, 1100, 2048),  # stream-K
    ({"variant": 2, "block_n": 256, "max_ctas": 10}, 640, 1024, 1408),    # half-tile tail
    ({"variant": 1, "block_n": 256, "max_ctas": 5}, 5, 3000, 640),        # M-row A box, halves
    ({"variant": 2, "block_n": 128, "max_ctas": 4, "group_m": 3}, 640, 1280, 768),  # persistent
])
@pytest.mark.parametrize("bm", [1, 128])
def test_blockwise_schedules(g, cfg, M, N, K, bm):
    _case(g, M, N, K, E4M3, BF16, bm, seed=401, cfg=cfg)
    _case(g, M, N, K, E5M2, F32, bm, seed=402, cfg=cfg, ints=True)


def test_blockwise_unit_scales_match_the_plain_product(g):
    # with every scale 1 the result is the plain FP8 product, up to accumulation order
    M, N, K = 256, 512, 2048
    gen = torch.Generator().manual_seed(403)
    A = (torch.rand(M, K, generator=gen) * 2 - 1).to(torch.float8_e4m3fn)
    B = (torch.rand(N, K, generator=gen) * 2 - 1).to(torch.float8_e4m3fn)
    ones_a = torch.ones(K // 128, M, device="cuda")
    ones_b = torch.ones(K // 128, N // 128, device="cuda")
    C1 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    C2 = torch.empty_like(C1)
    g.run_blockwise(A.cuda(), B.cuda(), C1, ones_a, ones_b, 1)
    g.run(A.cuda(), B.cuda(), C2)
    torch.cuda.synchronize()
    _, c64 = oracle.gemm_select(A, B, None, None, E4M3, F32, want_f64=True)
    parity.check_pair(parity.bits_of(C1), parity.bits_of(C2), F32, c64, parity.sigma_of(A, B), K,
                      what="unit block scales")


def test_blockwise_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmBlockScales, GemmError, lib
    import ctypes
    A = torch.zeros(128, 256, dtype=torch.float8_e4m3fn, device="cuda")
    C = torch.zeros(128, 128, dtype=torch.float32, device="cuda")
    sfa = torch.ones(2, 128, device="cuda")     # K-block-major: 2 K blocks x 128 rows
    sfb = torch.ones(2, 1, device="cuda")
    A16 = torch.zeros(128, 256, dtype=torch.float16, device="cuda")
    with pytest.raises(GemmError) as e:                    # not FP8
        g.run_blockwise(A16, A16, C, sfa, sfb, 1)
    assert e.value.code == 2
    with pytest.raises(GemmError) as e:                    # B blocks of 64 rows
        g.run_blockwise(A, A, C, sfa, torch.ones(2, 2, device="cuda"), 1, block_n=64)
    assert e.value.code == 2
    for cfg in ({"chain_kblocks": 2}, {"epilogue": 2}):
        g.set_config(**cfg)
        try:
            with pytest.raises(GemmError) as e:
                g.run_blockwise(A, A, C, sfa, sfb, 1)
            assert e.value.code == 2
        finally:
            g.reset_config()
    h = g._h
    for sc, code in ((GemmBlockScales(None, sfb.data_ptr(), 1, 128), 1),       # no sfa
                     (GemmBlockScales(sfa.data_ptr(), sfb.data_ptr(), 0, 128), 1),  # block_m 0
                     (GemmBlockScales(sfa.data_ptr() + 2, sfb.data_ptr(), 1, 128), 2)):  # misaligned
        rc = lib().gemm_run_blockwise(h, A.data_ptr(), A.data_ptr(), C.data_ptr(), 128, 128, 256,
                                      E4M3, F32, ctypes.byref(sc), None)
        assert rc == code
    assert lib().gemm_run_blockwise(h, A.data_ptr(), A.data_ptr(), C.data_ptr(), 128, 128, 256,
                                    E4M3, F32, None, None) == 1


@pytest.mark.parametrize("n,bm", [(4096, 1), (8192, 1), (8192, 128)])
def test_blockwise_full_size(g, n, bm):
    # the sizes the bench times (E4M3 -> bf16), in the configuration the library
    # chooses: seeded rows and columns, tile edges included, against the oracle
    M = N = K = n
    A, B = si.make_operands(M, N, K, E4M3, "uniform", seed=6)
    sfa, sfb = _scales(M, N, K, bm, seed=410)
    C = torch.empty(M, N, dtype=torch.bfloat16, device="cuda")
    g.reset_config()
    g.run_blockwise(A.cuda(), B.cuda(), C, _kmajor(sfa), _kmajor(sfb), bm)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    Cc = C.cpu()
    rows = si.sample_indices(M, 12, seed=411, must=(0, 127, 128, 255, 256, M // 2, -129, -1))
    cols = si.sample_indices(N, 12, seed=412, must=(0, 127, 128, 255, 256, N // 2, -257, -1))
    for sel_rows, sel_cols in ((rows, None), (None, cols)):
        got = Cc[rows] if sel_rows is not None else Cc[:, cols]
        want, c64 = oracle.gemm_blockwise(A, B, sfa.numpy(), sfb.numpy(), bm, 128, 128, E4M3, BF16,
                                          rows=sel_rows, cols=sel_cols, want_f64=True)
        # a selected row (column) keeps its own scale row: block size 1 for that side
        if sel_rows is not None:
            As, fa, a_bm = parity.take_rows(A, rows), sfa[[r // bm for r in rows]], 1
            Bs, fb, b_bn = B, sfb, 128
        else:
            As, fa, a_bm = A, sfa, bm
            Bs, fb, b_bn = parity.take_rows(B, cols), sfb[[c // 128 for c in cols]], 1
        parity.check(parity.bits_of(got.contiguous()), want, BF16, c64=c64, K=K,
                     sigma=_effective_sigma(As, Bs, fa, fb, a_bm, bn=b_bn),
                     what=f"blockwise full size {n} bm={bm}")
