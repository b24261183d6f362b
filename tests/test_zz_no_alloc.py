"""gemm_run_noalloc: the GEMM entry point for callers that cannot allocate.

Some callers may not call cudaMalloc (a custom device allocator or pool that
needs a GEMM, a plug-in whose framework owns all device memory, a process that
reserved its memory up front).  gemm_run_noalloc keeps its scratch in a fixed
static device array instead.  These tests call it through the C ABI and check
that it gives the same answer as gemm_run, within the tolerance the other
parity tests use, on two calls in a row (the second reuses the array the first
left behind), and that a product whose K slices would overflow the fixed scratch
is cut into fewer slices rather than refused.

This file is named so that pytest collects it last.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

F16, BF16, F32 = 0, 1, 2


def _noalloc(A, B, C, din, dout):
    from dense_gemm_blackwell_02_gb300 import binding
    M, K = A.shape
    N = B.shape[0]
    stream = torch.cuda.current_stream().cuda_stream
    return binding.lib().gemm_run_noalloc(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                          din, dout, ctypes.c_void_p(stream))


# Shapes with fewer tiles than half the SMs, so K is sliced and the scratch is used.
CASES = [(256, 512, 4096, F16, F32), (300, 700, 2048, BF16, BF16), (128, 256, 8192, F16, F16)]


@pytest.mark.parametrize("M,N,K,din,dout", CASES)
def test_noalloc_matches_gemm_run_on_two_calls(M, N, K, din, dout):
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    assert torch.cuda.is_available()
    A, B = si.make_operands(M, N, K, din, "uniform", seed=77)
    Ad, Bd = A.cuda(), B.cuda()
    td = si.TORCH_DTYPE[dout]
    with Gemm() as g:
        ref = torch.empty(M, N, dtype=td, device="cuda")
        g.run(Ad, Bd, ref)
        code, word = g.device_status()
        assert code == 0, word
        # fewer 128x256 tiles than half the SMs: gemm_run_noalloc slices K (scratch in use)
        assert 2 * (-(-M // 128)) * (-(-N // 256)) <= g.sm_count, "case does not use the scratch"
    ref_bits = parity.bits_of(ref)
    _, c64 = oracle.gemm_select(A, B, None, None, din, dout, want_f64=True)
    sigma = parity.sigma_of(A, B)
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=td, device="cuda")
        assert _noalloc(Ad, Bd, C, din, dout) == 0
        torch.cuda.synchronize()
        got = parity.bits_of(C)
        # against gemm_run's result (the two may slice K differently, so they agree
        # within the sum of the tolerances each has against the exact product) ...
        parity.check_pair(got, ref_bits, dout, c64, sigma, K,
                          what=f"noalloc vs gemm_run, call {call}")
        if dout == F32:
            parity.check(got, ref_bits, F32, what=f"noalloc vs gemm_run, call {call}")
        # ... and against the oracle
        parity.oracle_check(got, A, B, din, dout, what=f"noalloc vs oracle, call {call}")


def test_noalloc_caps_its_k_slices_at_the_scratch():
    # 16 tiles with long K: 9 slices would need 16 x 9 x 128 x 256 x 4 B = 18.9 MB of
    # partial tiles, more than the 16 MiB the fixed scratch holds, so the call takes 8
    # slices instead (two calls in a row, against the oracle and gemm_run)
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    M, N, K = 256, 2048, 16384
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=78)
    Ad, Bd = A.cuda(), B.cuda()
    with Gemm() as g:
        ref = torch.empty(M, N, dtype=torch.float32, device="cuda")
        g.run(Ad, Bd, ref)
        assert g.device_status()[0] == 0
    ref_bits = parity.bits_of(ref)
    rows = si.sample_indices(M, 24, seed=5, must=(0, 127, 128, 255))
    cols = si.sample_indices(N, 24, seed=6, must=(0, 255, 256, N - 1))
    for call in range(2):
        C = torch.full((M, N), float("nan"), dtype=torch.float32, device="cuda")
        assert _noalloc(Ad, Bd, C, F16, F32) == 0
        torch.cuda.synchronize()
        got = parity.bits_of(C)
        parity.check(got, ref_bits, F32, what=f"long-K noalloc vs gemm_run, call {call}")
        parity.oracle_check(got[np.ix_(rows, cols)], A, B, F16, F32, rows=rows, cols=cols,
                            what=f"long-K noalloc vs oracle, call {call}")


def test_noalloc_argument_errors():
    A = torch.zeros(256, 1024, dtype=torch.float16, device="cuda")
    B = torch.zeros(512, 1024, dtype=torch.float16, device="cuda")
    C = torch.zeros(256, 512, dtype=torch.float32, device="cuda")
    assert _noalloc(A, B, C, F16, 7) == 1            # bad dtype: GEMM_ERR_INVALID_ARG
    assert _noalloc(A, B, C, 3, F32) == 2            # FP8 inputs: GEMM_ERR_UNSUPPORTED
    assert _noalloc(A[:, :1020], B[:, :1020], C, F16, F32) != 0  # K % 8 != 0 / misaligned
