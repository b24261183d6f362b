"""Fused epilogue through the C ABI (gemm_run_epilogue) against the oracle's
gemm_epilogue, element by element:
    C = act(alpha * A . B^T + beta * C_prev + bias[j])
("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05", Part 6: Epilogue Visitor
Trees; Classic Fused Epilogue: Bias + ReLU).

Tolerance.  The kernel evaluates the expression in binary32 on its fp32 accumulator:
alpha * acc rounds once, fma(beta, c, .) once, + bias once.  So, next to the
accumulation bound tau (scaled by |alpha|), the pre-rounding value may be off by
4 * 2^-24 * (|alpha S| + |beta c| + |bias|).  That is folded into an effective sigma
for parity.check, whose bound is ulp/2 + 8 * 2^-24 * sqrt(K) * sigma.  ReLU is
1-Lipschitz, so the same bound holds after it.  Everything else (1 ulp for fp16/bf16,
relative Frobenius 1e-5 for fp32) is unchanged.
"""
import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

F16, BF16, F32 = 0, 1, 2
TD = si.TORCH_DTYPE


@pytest.fixture(scope="module")
def g():
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    h = Gemm()
    yield h
    h.close()


def _prev_values(M, N, dtype_out, seed):
    gen = torch.Generator().manual_seed(seed)
    return ((torch.rand(M, N, generator=gen) * 4 - 2)).to(TD[dtype_out])


def _check_case(g, M, N, K, dtype_in, dtype_out, alpha, beta, use_bias, relu, seed, cfg=None):
    A, B = si.make_operands(M, N, K, dtype_in, "uniform", seed)
    prev = _prev_values(M, N, dtype_out, seed + 1)
    bias = None
    if use_bias:
        gen = torch.Generator().manual_seed(seed + 2)
        bias = (torch.rand(N, generator=gen) * 2 - 1).float()
    C = prev.cuda().clone()
    try:
        if cfg:
            g.set_config(**cfg)
        g.run_epilogue(A.cuda(), B.cuda(), C, alpha=alpha, beta=beta,
                       bias=None if bias is None else bias.cuda(), relu=relu)
        torch.cuda.synchronize()
        assert g.device_status()[0] == 0
        used = g.last_config()
    finally:
        g.reset_config()
    prev_bits = parity.bits_of(prev)
    want = oracle.gemm_epilogue(A, B, dtype_in, dtype_out, alpha=alpha, beta=beta,
                                cprev=prev_bits, bias=None if bias is None else bias.numpy(),
                                relu=relu)
    # unrounded reference for the cancellation bound: the oracle's binary64 sums, then the
    # epilogue in binary64 (a bound helper only; the rounded reference is the oracle's)
    _, S = oracle.gemm_select(A, B, None, None, dtype_in, dtype_out, want_f64=True)
    c_prev = oracle.decode(prev_bits, dtype_out)
    b = np.zeros(N) if bias is None else bias.numpy().astype(np.float64)
    pre = alpha * S + beta * c_prev + b[None, :]
    c64 = np.where(pre > 0, pre, 0.0) if relu else pre
    sigma = parity.sigma_of(A, B)
    sig_eff = abs(alpha) * sigma + (np.abs(alpha * S) + np.abs(beta * c_prev)
                                    + np.abs(b)[None, :]) / (2.0 * np.sqrt(max(K, 1)))
    what = (f"epilogue alpha={alpha} beta={beta} bias={use_bias} relu={relu} {M}x{N}x{K} "
            f"in={dtype_in} out={dtype_out} {used}")
    return parity.check(parity.bits_of(C), want, dtype_out, what=what, c64=c64, sigma=sig_eff, K=K)


@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
@pytest.mark.parametrize("alpha,beta,use_bias,relu", [
    (1.0, 0.0, True, False),      # bias
    (1.0, 0.0, False, True),      # ReLU
    (0.5, 1.0, False, False),     # alpha and beta
    (-1.25, 0.75, True, True),    # everything
])
def test_epilogue_against_oracle(g, dtype_out, alpha, beta, use_bias, relu):
    _check_case(g, 384, 640, 512, F16, dtype_out, alpha, beta, use_bias, relu, seed=70)


@pytest.mark.parametrize("cfg,M,N,K", [
    ({"variant": 2, "block_n": 256}, 512, 768, 6144),                   # two chains, general epilogue
    ({"variant": 2, "block_n": 256, "splits": 2}, 256, 1024, 4096),     # split-K: applied once
    ({"variant": 1, "block_n": 256, "splits": 3}, 300, 1100, 2000),
    ({"variant": 2, "block_n": 128, "splits": -1, "max_ctas": 38}, 300, 1100, 2000),  # stream-K
    ({"variant": 2, "block_n": 256, "max_ctas": 10}, 640, 1024, 704),   # half-tile tail
    ({"variant": 2, "block_n": 256}, 129, 4097, 512),                   # ragged, direct stores
    ({"variant": 1, "block_n": 128}, 131, 1001, 1024),                  # ragged, direct, one CTA
])
def test_epilogue_schedules(g, cfg, M, N, K):
    _check_case(g, M, N, K, BF16, F16, -0.5, 1.5, True, True, seed=71, cfg=cfg)
    _check_case(g, M, N, K, F16, F32, 2.0, -1.0, True, False, seed=72, cfg=cfg)


def test_identity_epilogue_is_gemm_run(g):
    A, B = si.make_operands(256, 512, 1024, F16, "uniform", 73)
    Ad, Bd = A.cuda(), B.cuda()
    C1 = torch.empty(256, 512, dtype=torch.float16, device="cuda")
    C2 = torch.full_like(C1, 7.0)
    g.run(Ad, Bd, C1)
    g.run_epilogue(Ad, Bd, C2)              # alpha 1, beta 0: C2's old contents unused
    torch.cuda.synchronize()
    assert torch.equal(C1, C2)


def test_small_integers_exact(g):
    # integer operands, integer bias, beta and alpha small powers of two: every step exact
    A, B = si.make_small_int_operands(200, 300, 512, F16, seed=74)
    prev = torch.randint(-8, 9, (200, 300), generator=torch.Generator().manual_seed(75)).float()
    bias = torch.randint(-5, 6, (300,), generator=torch.Generator().manual_seed(76)).float()
    C = prev.cuda().clone()
    g.run_epilogue(A.cuda(), B.cuda(), C, alpha=2.0, beta=-0.5, bias=bias.cuda(), relu=True)
    torch.cuda.synchronize()
    want = oracle.gemm_epilogue(A, B, F16, F32, alpha=2.0, beta=-0.5,
                                cprev=parity.bits_of(prev), bias=bias.numpy(), relu=True)
    parity.check(parity.bits_of(C), want, F32, exact=True, what="integer epilogue")


def test_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.ones(64, 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    base = torch.zeros(68, dtype=torch.float32, device="cuda")
    with pytest.raises(GemmError) as e:                 # bias not 16-byte aligned
        g.run_epilogue(A, A, C, bias=base[1:65])
    assert e.value.code == 2
    K0 = torch.empty(64, 0, dtype=torch.float16, device="cuda")
    with pytest.raises(GemmError) as e:                 # K = 0 with a non-trivial epilogue
        g.run_epilogue(K0, K0, C, alpha=2.0)
    assert e.value.code == 2
