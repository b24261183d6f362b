"""Parity at the full configured sizes, in the launch configuration the library
chooses (the one bench.py times): seeded rows and columns (including the first
and last rows/columns of every tile edge class) against the oracle element by
element, plus a Freivalds check of the whole product."""
import pytest
import torch

import seeded_inputs as si
from tests import parity

pytestmark = pytest.mark.gpu

CASES = [(name, i) for name, wl in si.WORKLOADS.items() for i in range(len(wl.shapes))]


@pytest.fixture(scope="module")
def g():
    from dense_gemm_blackwell_02_gb300.binding import Gemm
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    h = Gemm()
    yield h
    h.close()


@pytest.mark.parametrize("name,idx", CASES, ids=[f"{n}-{i}" for n, i in CASES])
def test_full_size_workload(g, name, idx):
    wl = si.WORKLOADS[name]
    s = wl.shapes[idx]
    M, N, K = s.M, s.N, s.K
    A, B = si.make_operands(M, N, K, wl.dtype_in, wl.dist, wl.seed)
    C = torch.empty(M, N, dtype=si.TORCH_DTYPE[wl.dtype_out], device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    code, word = g.device_status()
    assert code == 0, f"device status {code} ({word:#x})"
    cfg = g.last_config()
    what = f"{name}[{idx}] {M}x{N}x{K} {cfg}"

    small = M * N * K <= 2 ** 31
    if small:
        parity.oracle_check(parity.bits_of(C), A, B, wl.dtype_in, wl.dtype_out, what=what)
        return
    rows = si.sample_indices(M, 16, seed=wl.seed + 100,
                             must=(0, 127, 128, 255, 256, M // 2, -129, -128, -1))
    cols = si.sample_indices(N, 16, seed=wl.seed + 200,
                             must=(0, 127, 128, 255, 256, N // 2, -257, -256, -1))
    Cc = C.cpu()
    parity.oracle_check(parity.bits_of(Cc[rows]), A, B, wl.dtype_in, wl.dtype_out, rows=rows,
                        what=what + " rows")
    parity.oracle_check(parity.bits_of(Cc[:, cols].contiguous()), A, B, wl.dtype_in,
                        wl.dtype_out, cols=cols, what=what + " cols")
    parity.freivalds(A, B, Cc, wl.dtype_out)


def test_freivalds_catches_a_skipped_tile(g):
    """The Freivalds bound is sharp enough to see one missing 128x256 tile."""
    M, N, K = 1024, 2048, 4096
    A, B = si.make_operands(M, N, K, si.F16, "uniform", 5)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    Cc = C.cpu()
    parity.freivalds(A, B, Cc, si.F16)
    Cc[256:384, 512:768] = 0
    with pytest.raises(AssertionError):
        parity.freivalds(A, B, Cc, si.F16)


MOE = sorted(si.MOE_WORKLOADS)


@pytest.mark.parametrize("name", MOE)
def test_grouped_moe_full_size(g, name):
    """The grouped MoE workloads the bench times, in the configuration the library
    chooses: per expert, seeded rows (first and last included) and two columns against
    the oracle."""
    wl = si.MOE_WORKLOADS[name]
    counts = si.moe_counts(wl.experts, wl.rows, wl.seed)
    probs = []
    for e, m in enumerate(counts):
        A, B = si.make_operands(m, wl.N, wl.K, wl.dtype_in, "uniform", wl.seed * 1000 + e)
        probs.append((A, B))
    dev = [(A.cuda(), B.cuda(), torch.empty(A.shape[0], wl.N, dtype=si.TORCH_DTYPE[wl.dtype_out],
                                            device="cuda")) for A, B in probs]
    g.reset_config()
    g.run_grouped(dev)
    code, word = g.device_status()
    assert code == 0, f"device status {code} ({word:#x})"
    cfg = g.last_config()
    for e, ((A, B), (_, _, C)) in enumerate(zip(probs, dev)):
        M = A.shape[0]
        if M == 0:
            continue
        Cc = C.cpu()
        rows = si.sample_indices(M, 3, seed=e, must=(0, -1))
        cols = si.sample_indices(wl.N, 2, seed=e + 7, must=(-1,))
        what = f"{name} expert {e} ({M} rows) {cfg}"
        parity.oracle_check(parity.bits_of(Cc[rows]), A, B, wl.dtype_in, wl.dtype_out, rows=rows,
                            what=what + " rows")
        parity.oracle_check(parity.bits_of(Cc[:, cols].contiguous()), A, B, wl.dtype_in,
                            wl.dtype_out, cols=cols, what=what + " cols")
