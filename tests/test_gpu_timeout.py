"""Failure detection without a GPU fault: every wait inside the kernels is bounded.

The test hook makes the MMA-issuing thread wait on a barrier that nothing ever
arrives on, with a short wait limit.  The kernel must give up, record the site in
the device status word, drain its own copies, free Tensor Memory and return; the
host then reads GEMM_ERR_TIMEOUT from gemm_device_status, and the next ordinary
call on the same handle and context computes the right answer.
"""
import pytest
import torch

import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

TIMEOUT, SITE_TEST_STALL = 5, 5


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("splits", [1, 3])
def test_stalled_wait_times_out_and_the_context_survives(variant, splits):
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    M, N, K = 512, 768, 1024
    A, B = si.make_operands(M, N, K, si.F16, "uniform", seed=61)
    Ad, Bd = A.cuda(), B.cuda()
    with Gemm() as g:
        g.set_config(variant=variant, splits=splits)
        g.set_wait_limit(50_000_000)          # 50 ms
        g.set_test_stall(True)
        C = torch.zeros(M, N, dtype=torch.float32, device="cuda")
        g.run(Ad, Bd, C)
        code, word = g.device_status()
        assert code == TIMEOUT, (code, hex(word))
        assert word >> 24 == 1                      # timeout
        sites = {(word >> 16) & 0xFF}
        assert sites & {SITE_TEST_STALL, 3, 4, 1}, hex(word)   # the stall or a wait it starved
        # the status word was cleared by the read
        assert g.device_status() == (0, 0)
        # same handle, same context: an ordinary run is correct again
        g.set_test_stall(False)
        g.set_wait_limit(2_000_000_000)
        C2 = torch.empty(M, N, dtype=torch.float32, device="cuda")
        g.run(Ad, Bd, C2)
        assert g.device_status()[0] == 0
        parity.oracle_check(parity.bits_of(C2), A, B, si.F16, si.F32, what="after timeout")
        torch.cuda.synchronize()


@pytest.mark.parametrize("case", ["cluster_split_pair", "cluster_split_one", "grouped",
                                  "grouped_clc", "fp8", "blockwise"])
def test_stalled_wait_times_out_in_every_kernel_family(case):
    # the same stall in the other kernel families: the cluster K split (whose slices also
    # wait on each other), a grouped launch, FP8 and blockwise FP8; each run must return
    # a timeout and leave the handle and context usable
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    M, N, K = 256, 1024, 4096
    din = si.E4M3 if case in ("fp8", "blockwise") else si.F16
    A, B = si.make_operands(M, N, K, din, "uniform", seed=62)
    Ad, Bd = A.cuda(), B.cuda()
    sfa = torch.ones(K // 128, M, device="cuda")
    sfb = torch.ones(K // 128, N // 128, device="cuda")
    C = torch.zeros(M, N, dtype=torch.float32, device="cuda")

    def run(g):
        if case in ("grouped", "grouped_clc"):
            g.run_grouped([(Ad, Bd, C), (Ad[:100], Bd[:300], C[:100, :300].contiguous())])
        elif case == "blockwise":
            g.run_blockwise(Ad, Bd, C, sfa, sfb, 1)
        else:
            g.run(Ad, Bd, C)

    with Gemm() as g:
        if case == "cluster_split_pair":
            g.set_config(variant=2, block_n=256, splits=2, epilogue=3)
        elif case == "cluster_split_one":
            g.set_config(variant=1, block_n=128, splits=2, epilogue=3)
        elif case == "grouped_clc":
            g.set_config(variant=2, scheduler=2)   # the answer ring's waits and drain
        g.set_wait_limit(50_000_000)
        g.set_test_stall(True)
        run(g)
        code, word = g.device_status()
        assert code == TIMEOUT, (code, hex(word))
        assert word >> 24 == 1
        g.set_test_stall(False)
        g.set_wait_limit(2_000_000_000)
        C.zero_()
        run(g)
        assert g.device_status()[0] == 0
        if case in ("cluster_split_pair", "cluster_split_one"):
            assert g.last_config()["epilogue"] == 3
        if case == "grouped_clc":
            assert g.last_config()["scheduler"] == 2
        if case in ("grouped", "grouped_clc"):
            return
        # unit block scales: the blockwise product is the plain one, up to the order of
        # the fp32 additions, so the plain oracle and tolerance apply
        parity.oracle_check(parity.bits_of(C), A, B, din, si.F32, what=f"after timeout ({case})")
