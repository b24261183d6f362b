"""FP8 operands through the C ABI (tcgen05.mma kind::f8f6f4) against the oracle,
element by element: E4M3 and E5M2 inputs, every output type, every schedule, the
per-tensor scale pair as the fused epilogue's alpha ("CUTLASS Deep Dive: From CuTe
Layouts to Blackwell tcgen05", Part 6: FP8 and Blockwise Scaling).

The tolerance is the GEMM's: 1 ulp for fp16/bf16 C (or ulp/2 + tau where the sum
cancels), relative Frobenius 1e-5 and max abs 1e-2 for fp32 C; integer-valued
operands bit-exact.  Every product of two FP8 values is exact in fp32, so the only
rounding is the fp32 accumulation, as for fp16/bf16 operands.
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


def _operands(M, N, K, dt, seed, scale=4.0):
    # U[-scale, scale) drawn in fp32 and cast by torch: several binades of each format
    gen = torch.Generator().manual_seed(seed)
    A = ((torch.rand(M, K, generator=gen) * 2 - 1) * scale).to(TD[dt])
    B = ((torch.rand(N, K, generator=gen) * 2 - 1) * scale).to(TD[dt])
    return A, B


def _case(g, M, N, K, dt, dtype_out, seed, cfg=None, ints=False):
    if ints:
        A, B = si.make_small_int_operands(M, N, K, dt, seed=seed)
    else:
        A, B = _operands(M, N, K, dt, seed)
    try:
        if cfg:
            g.set_config(**cfg)
        C = parity.run_gpu(g, A, B, dtype_out)
        st = g.device_status()
        used = g.last_config()
    finally:
        g.reset_config()
    assert st[0] == 0, f"device status {st}"
    what = f"fp8 {dt} M={M} N={N} K={K} out={dtype_out} {used}"
    parity.oracle_check(parity.bits_of(C), A, B, dt, dtype_out, what=what, exact=ints)
    return used


@pytest.mark.parametrize("dt", [E4M3, E5M2])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_fp8_against_oracle(g, dt, dtype_out):
    _case(g, 300, 700, 1040, dt, dtype_out, seed=300)     # ragged M, N and K tails


@pytest.mark.parametrize("dt", [E4M3, E5M2])
def test_fp8_small_integers_exact(g, dt):
    for dtype_out in (F16, BF16, F32):
        _case(g, 257, 383, 2048, dt, dtype_out, seed=301, ints=True)


@pytest.mark.parametrize("cfg,M,N,K", [
    ({"variant": 2, "block_n": 256}, 512, 768, 8192),                     # two chains of 32
    ({"variant": 2, "block_n": 256, "splits": 2}, 256, 1024, 4096),       # split-K
    ({"variant": 1, "block_n": 256, "splits": 3}, 300, 1100, 2048),
    ({"variant": 1, "block_n": 128}, 131, 1001, 1024),                    # direct stores
    ({"variant": 2, "block_n": 128, "splits": -1, "max_ctas": 38}, 300, 1100, 2048),  # stream-K
    ({"variant": 2, "block_n": 256, "max_ctas": 10}, 640, 1024, 1408),    # half-tile tail
    ({"variant": 1, "block_n": 256, "max_ctas": 5}, 5, 3000, 640),        # M-row A box, halves
    ({"variant": 2, "block_n": 256, "chain_kblocks": 3}, 256, 512, 2048), # short chains
    ({"variant": 1, "block_n": 128, "epilogue": 1}, 200, 384, 512),       # general epilogue
    ({"variant": 2, "block_n": 256, "splits": 2, "epilogue": 2}, 256, 1024, 4096),  # single chain
    ({"variant": 2, "block_n": 256, "max_ctas": 10, "epilogue": 2}, 640, 1024, 1408),  # its tail
    ({"variant": 2, "block_n": 128, "max_ctas": 4, "group_m": 3}, 640, 1280, 768),  # persistent
])
@pytest.mark.parametrize("dt", [E4M3, E5M2])
def test_fp8_schedules(g, cfg, M, N, K, dt):
    _case(g, M, N, K, dt, BF16, seed=302, cfg=cfg)
    _case(g, M, N, K, dt, F32, seed=303, cfg=cfg, ints=True)


def test_fp8_auto_takes_the_general_epilogue(g):
    # one-chain FP8 units take the general epilogue unless the single-chain one is
    # forced; both give the same bits (the same additions in the same order)
    A, B = _operands(640, 1024, 1408, E4M3, seed=305)
    out = {}
    try:
        for epi in (0, 2):
            g.set_config(epilogue=epi, variant=2, block_n=256, max_ctas=10)
            out[epi] = parity.run_gpu(g, A, B, BF16)
            assert g.device_status()[0] == 0
            assert g.last_config()["epilogue"] == (1 if epi == 0 else 2), g.last_config()
    finally:
        g.reset_config()
    assert np.array_equal(parity.bits_of(out[0]), parity.bits_of(out[2]))
    parity.oracle_check(parity.bits_of(out[0]), A, B, E4M3, BF16, what="fp8 general epilogue")


def test_fp8_auto_chain_is_4096_elements(g):
    used = _case(g, 256, 512, 8192, E4M3, F32, seed=304)
    assert used["chain_kblocks"] == 32, used


@pytest.mark.parametrize("dt", [E4M3, E5M2])
def test_fp8_per_tensor_scales_as_alpha(g, dt):
    # C = act(scale_a * scale_b * A.B^T + beta * C_prev + bias): the scale pair is the
    # epilogue's alpha
    M, N, K = 384, 640, 1024
    A, B = _operands(M, N, K, dt, seed=305)
    sa, sb = 0.37, 2.5
    gen = torch.Generator().manual_seed(306)
    prev = (torch.rand(M, N, generator=gen) * 4 - 2).to(torch.bfloat16)
    bias = (torch.rand(N, generator=gen) * 2 - 1).float()
    C = prev.cuda().clone()
    g.run_epilogue(A.cuda(), B.cuda(), C, alpha=sa * sb, beta=0.5, bias=bias.cuda(), relu=True)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    alpha = float(np.float32(sa * sb))
    prev_bits = parity.bits_of(prev)
    want = oracle.gemm_epilogue(A, B, dt, BF16, alpha=alpha, beta=0.5, cprev=prev_bits,
                                bias=bias.numpy(), relu=True)
    _, S = oracle.gemm_select(A, B, None, None, dt, BF16, want_f64=True)
    pre = alpha * S + 0.5 * oracle.decode(prev_bits, BF16) + bias.numpy().astype(np.float64)[None, :]
    c64 = np.where(pre > 0, pre, 0.0)
    sigma = parity.sigma_of(A, B)
    sig_eff = abs(alpha) * sigma + (np.abs(alpha * S) + 0.5 * np.abs(oracle.decode(prev_bits, BF16))
                                    + np.abs(bias.numpy())[None, :]) / (2.0 * np.sqrt(K))
    parity.check(parity.bits_of(C), want, BF16, what="fp8 scaled epilogue", c64=c64,
                 sigma=sig_eff, K=K)


def test_fp8_e5m2_is_not_read_as_e4m3(g):
    # the same bytes as E4M3 and as E5M2 give different products: each run must match
    # the oracle of its own format (pins the instruction descriptor's format code)
    A, B = _operands(128, 256, 512, E4M3, seed=307, scale=2.0)
    a8, b8 = A.view(torch.uint8), B.view(torch.uint8)
    outs = {}
    for dt in (E4M3, E5M2):
        Ad, Bd = a8.view(TD[dt]).cuda(), b8.view(TD[dt]).cuda()
        valid = torch.isfinite(Ad.float()).all() and torch.isfinite(Bd.float()).all()
        if not valid:
            continue
        C = torch.empty(128, 256, dtype=torch.float32, device="cuda")
        g.run(Ad, Bd, C)
        torch.cuda.synchronize()
        parity.oracle_check(parity.bits_of(C), a8.view(TD[dt]), b8.view(TD[dt]), dt, F32,
                            what=f"format {dt}")
        outs[dt] = C.cpu()
    assert E4M3 in outs


def test_fp8_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError, lib
    A = torch.zeros(64, 40, dtype=torch.float8_e4m3fn, device="cuda")   # K = 40: 40 bytes
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(GemmError) as e:
        g.run(A, A, C)
    assert e.value.code == 2
    A = torch.zeros(64, 64, dtype=torch.float8_e4m3fn, device="cuda")
    C8 = torch.zeros(64, 64, dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(GemmError) as e:                                  # FP8 output
        g.run(A, A, C8)
    assert e.value.code == 2
    rc = lib().gemm_run_noalloc(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64,
                                E4M3, F32, None)
    assert rc == 2


def test_fp8_k_zero_and_host_buffers(g):
    A = torch.empty(64, 0, dtype=torch.float8_e5m2, device="cuda")
    C = torch.full((64, 32), 7.0, dtype=torch.float16, device="cuda")
    g.run(A, A[:32], C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    A, B = si.make_small_int_operands(96, 160, 256, E4M3, seed=308)
    C = torch.empty(96, 160, dtype=torch.float32).pin_memory()
    g.run_host(A.pin_memory(), B.pin_memory(), C, E4M3, F32)
    want = A.to(torch.int64) @ B.to(torch.int64).T
    assert torch.equal(C, want.float())
