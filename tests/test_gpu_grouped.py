"""Grouped launches through the C ABI (gemm_run_grouped) against the oracle's grouped
product, problem by problem and element by element ("CUTLASS Deep Dive: From CuTe
Layouts to Blackwell tcgen05", Part 6, Grouped GEMM).  Tolerances are the GEMM's (1 ulp
for fp16/bf16, relative Frobenius 1e-5 for fp32, ulp/2 + tau where a sum cancels);
integer operands bit-exact."""
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


def _make(shapes, dt, seed, ints=False):
    probs = []
    for t, (M, N, K) in enumerate(shapes):
        if ints:
            A, B = si.make_small_int_operands(M, N, K, dt, seed=seed + t)
        else:
            A, B = si.make_operands(M, N, K, dt, "uniform", seed + t)
        probs.append((A, B))
    return probs


def _run_and_check(g, shapes, dt, dtype_out, seed, cfg=None, ints=False):
    probs = _make(shapes, dt, seed, ints)
    dev = [(A.cuda(), B.cuda(), torch.full((A.shape[0], B.shape[0]), 3.0, dtype=TD[dtype_out],
                                           device="cuda")) for A, B in probs]
    try:
        if cfg:
            g.set_config(**cfg)
        g.run_grouped(dev)
        torch.cuda.synchronize()
        st = g.device_status()
        used = g.last_config()
    finally:
        g.reset_config()
    assert st[0] == 0, f"device status {st}"
    for i, ((A, B), (_, _, C)) in enumerate(zip(probs, dev)):
        what = f"grouped problem {i} {tuple(A.shape)}x{tuple(B.shape)} out={dtype_out} {used}"
        if A.shape[1] == 0:
            assert torch.all(C == 0), what
            continue
        parity.oracle_check(parity.bits_of(C), A, B, dt, dtype_out, what=what, exact=ints)
    return used


MOE = [(384, 512, 1024), (128, 512, 1024), (0, 512, 1024), (17, 512, 1024), (700, 512, 1024),
       (1, 512, 1024), (256, 512, 1024)]
RAGGED = [(100, 300, 256), (257, 129, 520), (5, 1000, 64), (300, 77, 136), (64, 64, 2048)]


@pytest.mark.parametrize("dt", [F16, BF16])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_grouped_moe_like(g, dt, dtype_out):
    # one expert matrix shape, imbalanced token counts (one expert empty)
    _run_and_check(g, MOE, dt, dtype_out, seed=600)


def test_grouped_ragged_shapes_and_small_integers(g):
    _run_and_check(g, RAGGED, F16, F32, seed=601)
    _run_and_check(g, RAGGED, BF16, BF16, seed=602, ints=True)


@pytest.mark.parametrize("cfg", [{"variant": 1, "block_n": 128}, {"variant": 1, "block_n": 256},
                                 {"variant": 2, "block_n": 128}, {"variant": 2, "block_n": 256},
                                 {"variant": 2, "max_ctas": 6, "group_m": 2},
                                 {"variant": 1, "max_ctas": 3}, {"chain_kblocks": 3}])
def test_grouped_forced_configs(g, cfg):
    used = _run_and_check(g, MOE + RAGGED, F16, F16, seed=603, cfg=cfg)
    for k in ("variant", "block_n", "group_m", "chain_kblocks"):
        if k in cfg:
            assert used[k] == cfg[k], used
    _run_and_check(g, RAGGED, BF16, F32, seed=604, cfg=cfg, ints=True)


def test_grouped_empty_and_degenerate(g):
    # K = 0 writes zeros; M = 0 / N = 0 touch nothing; an all-degenerate group is a no-op
    shapes = [(5, 7, 0), (0, 9, 64), (9, 0, 64), (33, 65, 64)]
    _run_and_check(g, shapes, BF16, F32, seed=605)
    A = torch.empty(0, 64, dtype=torch.float16, device="cuda")
    C = torch.empty(0, 3, dtype=torch.float16, device="cuda")
    g.run_grouped([(A, torch.zeros(3, 64, dtype=torch.float16, device="cuda"), C)])
    torch.cuda.synchronize()


def test_grouped_many_problems_and_the_table_ring(g):
    # 64 experts with multinomial token counts, then six groups queued back to back
    # without synchronising (the problem-table ring holds four)
    gen = torch.Generator().manual_seed(606)
    counts = torch.multinomial(torch.ones(64), 2048, replacement=True, generator=gen).bincount(
        minlength=64).tolist()
    shapes = [(c, 256, 512) for c in counts]
    _run_and_check(g, shapes, BF16, BF16, seed=607)
    groups = []
    for r in range(6):
        probs = _make([(40 + 30 * r, 128 + 64 * (r % 3), 256), (200, 96, 256 + 128 * r)], F16, 610 + 10 * r)
        dev = [(A.cuda(), B.cuda(), torch.empty(A.shape[0], B.shape[0], dtype=torch.float32,
                                                device="cuda")) for A, B in probs]
        groups.append((probs, dev))
        g.run_grouped(dev)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    for probs, dev in groups:
        for (A, B), (_, _, C) in zip(probs, dev):
            parity.oracle_check(parity.bits_of(C), A, B, F16, F32, what="ring")


def test_grouped_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError, GemmProblem, lib
    A8 = torch.zeros(64, 64, dtype=torch.float8_e4m3fn, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    with pytest.raises(GemmError) as e:                      # FP8 inputs
        g.run_grouped([(A8, A8, C)])
    assert e.value.code == 2
    A = torch.zeros(64, 60, dtype=torch.float16, device="cuda")   # K % 8 != 0
    with pytest.raises(GemmError) as e:
        g.run_grouped([(A, A, C)])
    assert e.value.code == 2
    A = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    g.set_config(splits=2)
    try:
        with pytest.raises(GemmError) as e:
            g.run_grouped([(A, A, C)])
        assert e.value.code == 2
    finally:
        g.reset_config()
    bad = (GemmProblem * 2)(GemmProblem(A.data_ptr(), A.data_ptr(), C.data_ptr(), 64, 64, 64),
                            GemmProblem(A.data_ptr(), A.data_ptr(), None, 64, 64, 64))
    assert lib().gemm_run_grouped(g._h, bad, 2, F16, F32, None) == 1      # a NULL C
    bad[1] = GemmProblem(A.data_ptr(), A.data_ptr(), C.data_ptr(), -1, 64, 64)
    assert lib().gemm_run_grouped(g._h, bad, 2, F16, F32, None) == 1      # negative M
    assert lib().gemm_run_grouped(g._h, None, 1, F16, F32, None) == 1     # no table
    assert lib().gemm_run_grouped(g._h, None, 0, F16, F32, None) == 0     # nothing to do


# Cluster launch control ("A Blackwell GEMM by Hand in CuTe DSL", section 8): a CTA (pair)
# per tile in the grid; running ones cancel the launches of the rest and take their tiles.
MANY = [(1000, 2048, 512), (3, 2048, 512), (600, 2048, 512), (0, 2048, 512), (2100, 2048, 512),
        (130, 2048, 512)]   # 3833 rows: more tiles than resident CTAs, so tiles are stolen


@pytest.mark.parametrize("cfg", [{"variant": 1, "block_n": 128}, {"variant": 1, "block_n": 256},
                                 {"variant": 2, "block_n": 128}, {"variant": 2, "block_n": 256}])
def test_grouped_cluster_launch_control(g, cfg):
    cfg = dict(cfg, scheduler=2)
    used = _run_and_check(g, MOE + RAGGED, F16, F16, seed=620, cfg=cfg)
    assert used["scheduler"] == 2 and used["variant"] == cfg["variant"], used
    cg = cfg["variant"]
    assert used["max_ctas"] == used["dp_tiles"] * cg, used   # a CTA (pair) per tile
    _run_and_check(g, RAGGED, BF16, F32, seed=621, cfg=cfg, ints=True)
    used = _run_and_check(g, MANY, BF16, BF16, seed=622, cfg=cfg)
    assert used["dp_tiles"] > g.sm_count // cg, used


def test_grouped_cluster_launch_control_matches_round_robin(g):
    # integer operands: every schedule gives the same bits; repeated launches too
    probs = _make(MANY, F16, 623, ints=True)
    got = {}
    for sched in (1, 2, 2):
        dev = [(A.cuda(), B.cuda(), torch.empty(A.shape[0], B.shape[0], dtype=torch.float32,
                                                device="cuda")) for A, B in probs]
        g.set_config(scheduler=sched, variant=2)
        try:
            g.run_grouped(dev)
            torch.cuda.synchronize()
            assert g.device_status()[0] == 0
            assert g.last_config()["scheduler"] == sched
        finally:
            g.reset_config()
        bits = [parity.bits_of(C) for _, _, C in dev]
        if sched in got:
            assert all(np.array_equal(a, b) for a, b in zip(got[sched], bits)), "CLC rerun differs"
        got[sched] = bits
    assert all(np.array_equal(a, b) for a, b in zip(got[1], got[2]))


def test_grouped_cluster_launch_control_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.zeros(64, 64, dtype=torch.float16, device="cuda")
    C = torch.zeros(64, 64, dtype=torch.float32, device="cuda")
    for cfg, call in (({"scheduler": 2}, lambda: g.run(A, A, C)),                 # not grouped
                      ({"scheduler": 2, "max_ctas": 8}, lambda: g.run_grouped([(A, A, C)]))):
        g.set_config(**cfg)
        try:
            with pytest.raises(GemmError) as e:
                call()
            assert e.value.code == 2, cfg
        finally:
            g.reset_config()


def test_grouped_unequal_k_takes_cluster_launch_control(g):
    # problems whose K differ by 2x or more: tiles of unequal cost, scheduled by cluster
    # launch control automatically, handed out longest K first (the result does not
    # depend on the order); equal K: round-robin
    mixed = [(300, 512, 256), (200, 512, 4096), (64, 300, 1024), (512, 512, 8192), (7, 100, 512)]
    used = _run_and_check(g, mixed, F16, F32, seed=630)
    assert used["scheduler"] == 2, used
    used = _run_and_check(g, mixed, BF16, BF16, seed=631, ints=True)
    assert used["scheduler"] == 2, used
    used = _run_and_check(g, [(300, 512, 1024), (200, 512, 1024)], F16, F16, seed=632)
    assert used["scheduler"] == 1, used
