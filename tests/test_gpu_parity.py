"""Parity of the CUDA path (through the C ABI) with the CPU oracle, element by
element, at sizes the oracle finishes in seconds: several tiles, ragged tails,
ring wrap-around, split-K, persistent scheduling, every dtype pair."""
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


def _case(g, M, N, K, dtype_in, dtype_out, dist="uniform", seed=0, exact=False, ints=False):
    if ints:
        A, B = si.make_small_int_operands(M, N, K, dtype_in, seed=seed)
    else:
        A, B = si.make_operands(M, N, K, dtype_in, dist, seed)
    C = parity.run_gpu(g, A, B, dtype_out)
    st = g.device_status()
    assert st[0] == 0, f"device status {st}"
    return parity.oracle_check(parity.bits_of(C), A, B, dtype_in, dtype_out, exact=exact,
                               what=f"M={M} N={N} K={K} in={dtype_in} out={dtype_out} "
                                    f"{g.last_config()}")


def test_small_256_config(g):
    # 256^3, fp16 in, fp32 out, U[-1,1] from seed 0 (the small workload)
    wl = si.WORKLOADS["small_256"]
    s = wl.shapes[0]
    _case(g, s.M, s.N, s.K, wl.dtype_in, wl.dtype_out, wl.dist, wl.seed)


@pytest.mark.parametrize("dtype_in", [F16, BF16])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_dtype_pairs(g, dtype_in, dtype_out):
    g.reset_config()
    _case(g, 384, 640, 512, dtype_in, dtype_out, "uniform", seed=21)


@pytest.mark.parametrize("dtype_in", [F16, BF16])
@pytest.mark.parametrize("dtype_out", [F16, BF16, F32])
def test_small_integers_bit_exact(g, dtype_in, dtype_out):
    g.reset_config()
    _case(g, 300, 520, 1000, dtype_in, dtype_out, seed=22, exact=True, ints=True)


# K around the ring depth S = 4 (BN 256) and 6 (BN 128): K = 64 S - 64 never recycles a
# stage, 64 S exactly fills the ring once, 64 S + 64 recycles; plus K tails < 64.
@pytest.mark.parametrize("K", [8, 56, 64, 72, 192, 256, 320, 384, 448, 1000, 2048])
def test_k_edges(g, K):
    g.reset_config()
    _case(g, 256, 512, K, F16, F32, seed=23)


@pytest.mark.parametrize("M,N", [(1, 1), (1, 256), (127, 255), (129, 257), (200, 300),
                                 (1000, 3000), (130, 4097), (513, 8)])
def test_ragged_shapes(g, M, N):
    g.reset_config()
    _case(g, M, N, 128, BF16, F32, seed=24)
    _case(g, M, N, 136, F16, F16, seed=25)


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("bn", [128, 256])
@pytest.mark.parametrize("splits", [1, 2, 3, 7])
def test_forced_tiles_and_splits(g, variant, bn, splits):
    g.set_config(variant=variant, block_n=bn, splits=splits)
    try:
        _case(g, 300, 700, 1024, F16, F32, seed=26)
        _case(g, 256, 512, 960, BF16, BF16, seed=27)
        cfg = g.last_config()
        kb = 960 // 64                       # k-blocks of the last case
        per = -(-kb // splits)
        assert cfg["variant"] == variant and cfg["block_n"] == bn
        assert cfg["splits"] == -(-kb // per)
    finally:
        g.reset_config()


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("max_ctas", [2, 4, 10, 38])
def test_persistent_loops_many_units_per_cta(g, variant, max_ctas):
    # few CTAs: each walks many tiles, so both accumulator slots and the operand
    # ring go through many phases
    g.set_config(variant=variant, max_ctas=max_ctas, group_m=3)
    try:
        _case(g, 640, 1280, 704, F16, F16, seed=28)
    finally:
        g.reset_config()


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("block_n", [256, 128])
@pytest.mark.parametrize("max_ctas,M,N,K", [(10, 640, 1024, 704), (6, 512, 1280, 2048),
                                             (14, 300, 2100, 1000), (10, 640, 1100, 704),
                                             (16, 1000, 1000, 512)])
def test_partial_last_wave_is_spread(g, variant, block_n, max_ctas, M, N, K):
    # more tiles than resident units, not a whole number of waves: the tiles of the
    # last wave run as two half-width units (256-column tiles) or as K slices reduced
    # in the kernel; the others run whole.  N = 1100 leaves the last half tile
    # entirely outside C.
    g.set_config(variant=variant, block_n=block_n, max_ctas=max_ctas)
    try:
        _case(g, M, N, K, F16, F16, seed=38)
        _case(g, M, N, K, BF16, F32, seed=39, exact=True, ints=True)
        cfg = g.last_config()
        tiles = -(-M // (128 * variant)) * -(-N // block_n)
        units = max_ctas // variant
        rem, kb = tiles % units, -(-K // 64)
        if tiles > units and rem and block_n == 256 and 2 * rem <= units:
            assert cfg["splits"] == 1 and cfg["dp_tiles"] == tiles - rem, cfg   # halves
        elif tiles > units and rem and min(units // rem, kb // 4, 8) >= 2:
            assert cfg["splits"] > 1 and cfg["dp_tiles"] == tiles - rem, cfg   # K slices
        else:
            assert cfg["splits"] == 1 and cfg["dp_tiles"] == tiles, cfg
    finally:
        g.reset_config()


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("block_n", [128, 256])
@pytest.mark.parametrize("max_ctas,M,N,K", [(152, 256, 512, 8192), (38, 300, 1100, 2000),
                                             (20, 256, 2048, 1000), (8, 129, 300, 4096),
                                             (152, 256, 8192, 512)])
def test_stream_k(g, variant, block_n, max_ctas, M, N, K):
    # fewer tiles than resident units: each unit takes an equal share of the
    # (tile, k-block) iterations, crossing tile boundaries; the segments of a tile are
    # reduced in K order by whichever arrives last
    g.set_config(variant=variant, block_n=block_n, max_ctas=max_ctas, splits=-1)
    try:
        _case(g, M, N, K, F16, F16, seed=40)
        _case(g, M, N, K, BF16, F32, seed=41, exact=True, ints=True)
        cfg = g.last_config()
        assert cfg["splits"] < 0 and cfg["dp_tiles"] == 0, cfg
        # deterministic: the same bits on a second run
        A, B = si.make_operands(M, N, K, F16, "uniform", 42)
        C1 = parity.run_gpu(g, A, B, F32)
        C2 = parity.run_gpu(g, A, B, F32)
        assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
    finally:
        g.reset_config()


@pytest.mark.parametrize("variant,block_n", [(1, 128), (1, 256), (2, 128), (2, 256)])
@pytest.mark.parametrize("max_ctas,M,N,K", [(38, 256, 2560, 8192), (24, 256, 1024, 2048),
                                             (40, 200, 1800, 1504), (30, 256, 4096, 1024)])
def test_stream_k_staged_fix_up_matches_the_direct_one(g, variant, block_n, max_ctas, M, N, K):
    # segments of two and three per tile: the plain kernel's last segment stages the
    # others' partials in its idle operand ring (and may skip publishing its own), the
    # fused kernel with the identity epilogue reads them straight into registers; both sum
    # in K order, so the bits agree
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=43)
    Ad, Bd = A.cuda(), B.cuda()
    C1 = torch.empty(M, N, dtype=torch.float32, device="cuda")
    C2 = torch.empty_like(C1)
    # chains of 4 K blocks: the launch takes the general epilogue
    g.set_config(variant=variant, block_n=block_n, max_ctas=max_ctas, splits=-1, chain_kblocks=4)
    try:
        g.run(Ad, Bd, C1)
        g.run_epilogue(Ad, Bd, C2, alpha=1.0, beta=0.0)
        torch.cuda.synchronize()
        assert g.device_status()[0] == 0
        cfg = g.last_config()
    finally:
        g.reset_config()
    assert cfg["splits"] < 0 and cfg["epilogue"] == 1, cfg
    assert torch.equal(C1, C2)
    parity.oracle_check(parity.bits_of(C1), A, B, F16, F32, what=f"staged stream-K {cfg}")


@pytest.mark.parametrize("dtype_out", [F16, F32])
def test_between_one_and_two_waves_takes_stream_k(g, dtype_out):
    # more tiles than resident pairs but fewer than twice as many, each of several
    # accumulation chains: the library spreads them over every pair by stream-K
    pairs = g.sm_count // 2
    M, N, K = 256, 256 * (pairs + pairs // 4), 4160
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=44)
    C = torch.empty(M, N, dtype=TD[dtype_out], device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    cfg = g.last_config()
    assert cfg["splits"] == -pairs and cfg["dp_tiles"] == 0 and cfg["epilogue"] == 1, cfg
    rows = si.sample_indices(M, 12, seed=45, must=(0, 127, 128, 255))
    parity.oracle_check(parity.bits_of(C.cpu()[rows]), A, B, F16, dtype_out, rows=rows,
                        what=f"auto stream-K {cfg}")


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("chain", [1, 3, 5, 64])
@pytest.mark.parametrize("splits", [1, 3])
def test_accumulation_chains(g, variant, chain, splits):
    # K split into several TMEM accumulation chains summed by the epilogue in fp32
    # registers; with split-K on top, and with the chain not dividing the slice
    g.set_config(variant=variant, chain_kblocks=chain, splits=splits)
    try:
        _case(g, 300, 520, 1280, BF16, F32, seed=34)
        _case(g, 256, 512, 1000, F16, F16, seed=35, exact=True, ints=True)
        assert g.last_config()["chain_kblocks"] == chain
    finally:
        g.reset_config()


@pytest.mark.parametrize("variant", [1, 2])
@pytest.mark.parametrize("M,N", [(1, 257), (129, 4097), (383, 136), (256, 264)])
def test_pair_and_single_on_ragged_edges(g, variant, M, N):
    # N = 4097 and N = 257 (fp16) are not 16-byte row pitches: direct stores; the
    # others go through the TMA store, which must clip rows >= M and columns >= N
    g.set_config(variant=variant)
    try:
        _case(g, M, N, 192, F16, F16, seed=36)
        _case(g, M, N, 200, BF16, F32, seed=37)
    finally:
        g.reset_config()


def test_split_k_small_ints_exact_and_deterministic(g):
    g.set_config(splits=5)
    try:
        A, B = si.make_small_int_operands(256, 768, 2048, BF16, seed=29)
        C1 = parity.run_gpu(g, A, B, F32)
        C2 = parity.run_gpu(g, A, B, F32)
        want = oracle.gemm(A, B, BF16, F32)
        parity.check(parity.bits_of(C1), want, F32, exact=True, what="split-K ints")
        assert torch.equal(C1.view(torch.int32), C2.view(torch.int32))
        # non-integer inputs: run to run identical bits (fixed slice order)
        A, B = si.make_operands(256, 768, 2048, F16, "uniform", 30)
        C3 = parity.run_gpu(g, A, B, F32)
        C4 = parity.run_gpu(g, A, B, F32)
        assert torch.equal(C3.view(torch.int32), C4.view(torch.int32))
    finally:
        g.reset_config()


def test_all_ones_and_identity(g):
    for dt in (F16, BF16):
        K = 4096
        A = torch.ones(130, K, dtype=TD[dt])
        B = torch.ones(260, K, dtype=TD[dt])
        C = parity.run_gpu(g, A, B, F32)
        assert torch.all(C == K)
        C = parity.run_gpu(g, A, B, dt)
        assert torch.all(C.float() == K)
        A, _ = si.make_operands(200, 1, 512, dt, "uniform", 31)
        I = torch.eye(512, dtype=TD[dt])
        C = parity.run_gpu(g, A, I, dt)
        assert torch.equal(C.cpu().view(torch.int16), A.view(torch.int16))


def test_rank1_exact(g):
    M, N, K = 192, 320, 512
    gen = torch.Generator().manual_seed(32)
    u = 2.0 ** torch.randint(-3, 4, (M,), generator=gen).double()
    v = 2.0 ** torch.randint(-3, 4, (N,), generator=gen).double()
    a = torch.randint(-3, 4, (K,), generator=gen).double()
    b = torch.randint(-3, 4, (K,), generator=gen).double()
    A = (u[:, None] * a[None]).to(torch.bfloat16)
    B = (v[:, None] * b[None]).to(torch.bfloat16)
    C = parity.run_gpu(g, A, B, F32).cpu().double()
    assert torch.equal(C, u[:, None] * v[None] * float((a * b).sum()))


def test_k_zero_and_empty(g):
    C = torch.full((5, 7), 3.0, device="cuda")
    A = torch.empty(5, 0, dtype=torch.float16, device="cuda")
    B = torch.empty(7, 0, dtype=torch.float16, device="cuda")
    g.run(A, B, C)
    torch.cuda.synchronize()
    assert torch.all(C == 0)
    A = torch.empty(0, 64, dtype=torch.float16, device="cuda")
    B = torch.ones(7, 64, dtype=torch.float16, device="cuda")
    C = torch.empty(0, 7, device="cuda")
    g.run(A, B, C)


def test_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.ones(64, 60, dtype=torch.float16, device="cuda")
    B = torch.ones(64, 60, dtype=torch.float16, device="cuda")
    C = torch.empty(64, 64, device="cuda")
    with pytest.raises(GemmError) as e:        # K % 8 != 0
        g.run(A, B, C)
    assert e.value.code == 2
    base = torch.ones(64 * 64 + 8, dtype=torch.float16, device="cuda")
    A = base[4:4 + 64 * 64].view(64, 64)       # 8-byte aligned only
    B = torch.ones(64, 64, dtype=torch.float16, device="cuda")
    with pytest.raises(GemmError) as e:
        g.run(A, B, C)
    assert e.value.code == 2
    assert g.run_ptr(0, B.data_ptr(), C.data_ptr(), 64, 64, 64, 0, 2, 0) == 1
    assert g.run_ptr(B.data_ptr(), B.data_ptr(), C.data_ptr(), -1, 64, 64, 0, 2, 0) == 1
    assert g.run_ptr(B.data_ptr(), B.data_ptr(), C.data_ptr(), 64, 64, 64, 2, 2, 0) == 2
    assert g.run_ptr(B.data_ptr(), B.data_ptr(), C.data_ptr(), 64, 64, 64, 0, 7, 0) == 1


def test_run_host_matches_device(g):
    A, B = si.make_operands(300, 500, 256, F16, "uniform", 33)
    Cd = parity.run_gpu(g, A, B, F16)
    Ch = torch.empty(300, 500, dtype=torch.float16).pin_memory()
    g.run_host(A.pin_memory(), B.pin_memory(), Ch, F16, F16)
    assert torch.equal(Ch.view(torch.int16), Cd.cpu().view(torch.int16))


@pytest.mark.parametrize("M,N,K,din,dout", [(2048, 512, 512, F16, F32), (3000, 700, 1024, BF16, BF16),
                                            (5000, 300, 256, si.E4M3, F16), (2100, 96, 64, F16, F16)])
def test_run_host_row_chunk_pipeline(g, M, N, K, din, dout):
    # from 2048 rows on, A and C cross in row chunks (the last one ragged) on copy streams
    # overlapped with the GEMMs; each element is checked against the oracle, and the
    # call is repeated back to back (the handle's staging buffers and events are reused)
    A, B = si.make_operands(M, N, K, din, "uniform", 34)
    Ah, Bh = A.pin_memory(), B.pin_memory()
    outs = []
    for _ in range(3):
        Ch = torch.full((M, N), 5.0, dtype=TD[dout]).pin_memory()
        g.run_host(Ah, Bh, Ch, din, dout)
        outs.append(Ch)
    parity.oracle_check(parity.bits_of(outs[0]), A, B, din, dout, what="run_host chunks")
    assert all(torch.equal(o, outs[0]) for o in outs[1:])


@pytest.mark.parametrize("cfg,M,N,K,dtype_out", [
    ({"variant": 2, "block_n": 256}, 512, 768, 1024, F16),                  # whole tiles
    ({"variant": 2, "block_n": 256, "splits": 2}, 256, 1024, 4096, BF16),   # two K slices
    ({"variant": 1, "block_n": 256, "splits": 3}, 300, 1100, 2000, F32),    # three K slices
    ({"variant": 2, "block_n": 128, "splits": -1, "max_ctas": 38}, 300, 1100, 2000, F16),  # stream-K
    ({"variant": 2, "block_n": 256, "max_ctas": 10}, 640, 1024, 704, F16),  # half-tile tail
    ({"variant": 1, "block_n": 128, "max_ctas": 6}, 512, 1280, 2048, BF16),  # K-sliced tail
    ({"variant": 2, "block_n": 256}, 129, 4097, 512, F16),                  # direct stores
    ({"variant": 1, "block_n": 256, "splits": 2}, 131, 1001, 1024, F32),    # direct, split
])
def test_single_chain_epilogue_matches_general(g, cfg, M, N, K, dtype_out):
    # Every unit here is one accumulation chain, so the streaming epilogue applies; it
    # performs the same additions in the same order as the general one (the own slice's
    # partial is read from TMEM instead of the workspace, the same bits), so the two
    # must agree bit for bit, and both with the oracle.
    A, B = si.make_operands(M, N, K, F16, "uniform", 50)
    out = {}
    try:
        for epi in (1, 2):
            g.set_config(epilogue=epi, **cfg)
            out[epi] = parity.run_gpu(g, A, B, dtype_out)
            assert g.device_status()[0] == 0
            assert g.last_config()["epilogue"] == epi
        g.set_config(**cfg)
        auto = parity.run_gpu(g, A, B, dtype_out)
        assert g.last_config()["epilogue"] == 2        # chosen automatically
    finally:
        g.reset_config()
    assert np.array_equal(parity.bits_of(out[1]), parity.bits_of(out[2]))
    assert np.array_equal(parity.bits_of(out[2]), parity.bits_of(auto))
    parity.oracle_check(parity.bits_of(out[2]), A, B, F16, dtype_out,
                        what=f"single-chain epilogue {cfg} {M}x{N}x{K}")


def test_single_chain_epilogue_needs_single_chain_units(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A, B = si.make_operands(256, 256, 8192, F16, "uniform", 51)
    try:
        g.set_config(variant=2, splits=1, epilogue=2)          # 128 k-blocks in one unit
        with pytest.raises(GemmError) as e:
            parity.run_gpu(g, A, B, F32)
        assert e.value.code == 2
        g.set_config(variant=2, splits=1)
        C = parity.run_gpu(g, A, B, F32)
        assert g.last_config()["epilogue"] == 1
    finally:
        g.reset_config()
    parity.oracle_check(parity.bits_of(C), A, B, F16, F32, what="two chains, general epilogue")


@pytest.mark.parametrize("M", [1, 2, 3, 7, 8, 31, 33, 100])
@pytest.mark.parametrize("cfg,N,K", [
    ({}, 1000, 2048),                                                   # auto: K slices
    ({"variant": 1, "block_n": 256, "splits": 3}, 700, 1024),           # general epilogue, split
    ({"variant": 1, "block_n": 128, "splits": 2, "epilogue": 2}, 520, 4096),  # single chain, split
    ({"variant": 1, "block_n": 256, "max_ctas": 5}, 3000, 640),         # half-tile tail
    ({"variant": 1, "block_n": 128, "splits": -1, "max_ctas": 38}, 900, 1504),  # stream-K
])
def test_one_row_tile_of_few_rows(g, M, cfg, N, K):
    # M < 128 in one-CTA tiles: A is loaded as an M-row box (the stage's other rows are
    # never written) and epilogue warps whose 32 rows lie past M skip their partials
    if cfg:
        g.set_config(**cfg)
    try:
        _case(g, M, N, K, F16, F16, seed=90 + M)
        _case(g, M, N, K, BF16, F32, seed=91 + M, exact=True, ints=True)
        # one row of A without a forced configuration takes the matrix-vector path
        assert g.last_config()["variant"] == (3 if (M == 1 and not cfg) else 1)
    finally:
        g.reset_config()


@pytest.mark.parametrize("M", [2, 8, 64, 128])
def test_small_m_decode_takes_narrow_tiles(g, M):
    # M <= 128, N = 8192: 64 tiles of 128 columns in two K slices beat 32 tiles of 256
    # columns in four (fewer slices to reduce)
    _case(g, M, 8192, 1024, F16, F16, seed=95)
    cfg = g.last_config()
    assert cfg["variant"] == 1 and cfg["block_n"] == 128, cfg
    assert cfg["splits"] == min(g.sm_count // 64, 1024 // 64 // 4), cfg


@pytest.mark.parametrize("variant,block_n", [(1, 128), (1, 256), (2, 128), (2, 256)])
@pytest.mark.parametrize("M,N,K,dtype_out", [(256, 1024, 4096, F16), (200, 1000, 2048, F32),
                                             (96, 520, 1024, BF16), (256, 777, 4096, F16)])
def test_cluster_k_split_matches_the_workspace_split(g, variant, block_n, M, N, K, dtype_out):
    # the two K slices summed through distributed shared memory (epilogue 3) give the same
    # bits as the same slices summed through the global workspace (epilogue 2)
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=97)
    Ad, Bd = A.cuda(), B.cuda()
    outs = {}
    for epi in (2, 3):
        C = torch.empty(M, N, dtype=TD[dtype_out], device="cuda")
        g.set_config(variant=variant, block_n=block_n, splits=2, epilogue=epi)
        try:
            g.run(Ad, Bd, C)
            torch.cuda.synchronize()
            assert g.device_status()[0] == 0
            used = g.last_config()
        finally:
            g.reset_config()
        assert used["epilogue"] == epi and used["splits"] == 2, used
        outs[epi] = C
    assert torch.equal(outs[2], outs[3])
    parity.oracle_check(parity.bits_of(outs[3]), A, B, F16, dtype_out, what=f"cluster split {used}")
    Ai, Bi = si.make_small_int_operands(M, N, K, F16, seed=98)
    C = torch.empty(M, N, dtype=torch.float32, device="cuda")
    g.set_config(variant=variant, block_n=block_n, splits=2, epilogue=3)
    try:
        g.run(Ai.cuda(), Bi.cuda(), C)
        torch.cuda.synchronize()
    finally:
        g.reset_config()
    parity.oracle_check(parity.bits_of(C), Ai, Bi, F16, F32, exact=True, what="cluster split ints")


@pytest.mark.parametrize("variant,block_n", [(1, 128), (2, 256)])
@pytest.mark.parametrize("M,N,K,chain,dtype_out", [(256, 1024, 16384, 0, F16),
                                                   (200, 1000, 2048, 3, F32),
                                                   (96, 520, 4096, 5, BF16)])
def test_cluster_k_split_of_several_chains(g, variant, block_n, M, N, K, chain, dtype_out):
    # slices of several accumulation chains: the general epilogue sums each slice's chains
    # in registers, then the two slices meet in distributed shared memory (epilogue 3) or
    # in the workspace (epilogue 1); the bits agree
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=99)
    Ad, Bd = A.cuda(), B.cuda()
    outs = {}
    for epi in (1, 3):
        C = torch.empty(M, N, dtype=TD[dtype_out], device="cuda")
        g.set_config(variant=variant, block_n=block_n, splits=2, epilogue=epi, chain_kblocks=chain)
        try:
            g.run(Ad, Bd, C)
            torch.cuda.synchronize()
            assert g.device_status()[0] == 0
            used = g.last_config()
        finally:
            g.reset_config()
        assert used["epilogue"] == epi and used["splits"] == 2, used
        outs[epi] = C
    assert torch.equal(outs[1], outs[3])
    parity.oracle_check(parity.bits_of(outs[3]), A, B, F16, dtype_out, what=f"cluster split {used}")


@pytest.mark.parametrize("M,N,K,cfg", [(256, 2048, 4096, {}), (200, 1000, 2048, {"splits": -1}),
                                       (64, 4096, 1024, {}), (1000, 600, 512, {"variant": 2}),
                                       (96, 520, 1024, {"variant": 1, "splits": 3})])
def test_l2_policy_changes_no_bits(g, M, N, K, cfg):
    # the evict-first / evict-last hints on the operand loads only steer L2: every
    # policy gives the same bits, and the automatic choice takes the hints exactly
    # when the tiles form one row
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=101)
    Ad, Bd = A.cuda(), B.cuda()
    outs = {}
    for hint in (0, 1, 2):
        C = torch.empty(M, N, dtype=torch.float16, device="cuda")
        g.set_config(l2_hint=hint, **cfg)
        try:
            g.run(Ad, Bd, C)
            torch.cuda.synchronize()
            assert g.device_status()[0] == 0
            used = g.last_config()
        finally:
            g.reset_config()
        if hint:
            assert used["l2_hint"] == hint, used
        else:
            rows = 128 * used["variant"]
            assert used["l2_hint"] == (2 if M <= rows else 1), used
        outs[hint] = C
    assert torch.equal(outs[0], outs[1]) and torch.equal(outs[1], outs[2])
    parity.oracle_check(parity.bits_of(outs[2]), A, B, F16, F16, what=f"l2 hints {used}")


@pytest.mark.parametrize("M", [1, 3, 8, 16, 17])
@pytest.mark.parametrize("N,K,dtype_out", [(8192, 1024, F16), (1000, 8192, F32), (4096, 2048, BF16),
                                           (3000, 520, F16)])
def test_rows_of_at_most_16_take_the_deeper_ring(g, M, N, K, dtype_out):
    # one CTA per row tile of <= 16 rows: stages of 16 A rows (2 KiB), a deeper ring
    # (10 stages of 128 columns, 5 of 256; 12 and 6 under the cluster K split, whose
    # staging lies in the ring); the MMA's 128-row A operand runs on over the next stages'
    # bytes, which feed only accumulator rows that are never stored
    _case(g, M, N, K, F16, dtype_out, seed=48)
    cfg = g.last_config()
    if cfg["variant"] == 1:          # (one row of A may take the matrix-vector path)
        kx = cfg["epilogue"] == 3
        deep = {128: 12 if kx else 10, 256: 6 if kx else 5}[cfg["block_n"]]
        assert (cfg["stages"] == deep) == (M <= 16), cfg
    _case(g, M, N, K, BF16, F32, seed=49, exact=True, ints=True)


def test_deeper_ring_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.zeros(20, 1024, dtype=torch.float16, device="cuda")
    B = torch.zeros(512, 1024, dtype=torch.float16, device="cuda")
    C = torch.zeros(20, 512, dtype=torch.float16, device="cuda")
    g.set_config(variant=1, block_n=128, stages=10)
    try:
        with pytest.raises(GemmError) as e:                 # 20 rows do not fit 16-row stages
            g.run(A, B, C)
        assert e.value.code == 2
        with pytest.raises(GemmError) as e:                 # no fused kernel with that ring
            g.run_epilogue(A[:8], B, C[:8], alpha=2.0)
        assert e.value.code == 2
        g.run(A[:16], B, C[:16])                            # 16 rows: fine
        torch.cuda.synchronize()
    finally:
        g.reset_config()


@pytest.mark.parametrize("M,N,K,dtype_out", [(256, 1280, 4096, F16), (256, 1000, 2048, BF16),
                                             (200, 700, 8192, F32), (256, 3200, 1024, F16)])
def test_320_column_pair_tiles(g, M, N, K, dtype_out):
    # two MMAs per K step (N = 256 and N = 64) into one 320-column accumulator, each CTA
    # loading 128 + 32 B rows; two K slices in a 4-CTA cluster
    g.set_config(variant=2, block_n=320, splits=2, epilogue=3)
    try:
        _case(g, M, N, K, F16, dtype_out, seed=50)
        used = g.last_config()
        _case(g, M, N, K, BF16, F32, seed=51, exact=True, ints=True)
    finally:
        g.reset_config()
    assert used["block_n"] == 320 and used["epilogue"] == 3 and used["splits"] == 2, used


def test_320_column_tiles_taken_when_256_do_not_fit_the_split(g):
    # 40 tiles of 256 columns need 80 pairs for two K slices; 32 tiles of 320 need 64
    M, N, K = 256, 10240, 2048
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=52)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    cfg = g.last_config()
    assert cfg["block_n"] == 320 and cfg["epilogue"] == 3, cfg
    rows = si.sample_indices(M, 10, seed=53, must=(0, 127, 128, 255))
    parity.oracle_check(parity.bits_of(C.cpu()[rows]), A, B, F16, F16, rows=rows,
                        what=f"auto 320-column tiles {cfg}")


def test_short_wave_of_wide_tiles_takes_narrow_stream_k(g):
    # 40 tiles of 256 columns leave 36 of 76 pairs idle; 80 tiles of 128 columns fill one
    # wave and 5% of a second: with tiles of two accumulation chains, stream-K over every
    # pair with 128-column tiles (sampled rows and columns against the oracle)
    M, N, K = 256, 10240, 4608
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=53)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    cfg = g.last_config()
    if g.sm_count >= 152:
        assert cfg["block_n"] == 128 and cfg["splits"] < 0, cfg
    rows = si.sample_indices(M, 24, seed=7, must=(0, 127, 128, 255))
    cols = si.sample_indices(N, 48, seed=8, must=(0, 127, 128, N - 1))
    parity.oracle_check(parity.bits_of(C)[np.ix_(rows, cols)], A, B, F16, F16, rows=rows,
                        cols=cols, what=f"narrow stream-K {cfg}")


@pytest.mark.parametrize("M,N,K,swapped", [(128, 14336, 8192, True),   # plain tiles: 112 CTAs
                                           (24, 14336, 8192, True),    # a few rows of A
                                           (100, 14336, 16384, True),  # ragged rows of A
                                           (16, 14336, 8192, False),   # 16-row stages stay
                                           (128, 20480, 8192, False),  # a nearly empty 2nd wave
                                           (64, 28672, 8192, True),    # a 2nd wave 47% full
                                           (128, 14336, 4096, False),  # one chain of K
                                           (256, 8192, 4096, False),   # pair tiles stay
                                           (256, 8192, 8192, False)])  # the cluster split stays
def test_decode_takes_the_swapped_tiling_where_it_measured_faster(g, M, N, K, swapped):
    # the automatic choice weighs the swapped tiling against the plain one (sampled rows
    # and columns against the oracle whichever is taken)
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=54)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    cfg = g.last_config()
    if g.sm_count >= 152:
        assert (cfg["swap_ab"] == 2) == swapped, cfg
        if swapped:
            assert cfg["swap_rows"] >= 96 and cfg["l2_hint"] == 2 and cfg["splits"] == 1, cfg
    rows = si.sample_indices(M, 16, seed=9, must=(0, M // 2, M - 1))
    cols = si.sample_indices(N, 48, seed=10, must=(0, 111, 112, N - 1))
    parity.oracle_check(parity.bits_of(C)[np.ix_(rows, cols)], A, B, F16, F16, rows=rows,
                        cols=cols, what=f"automatic swapped tiling {cfg}")


@pytest.mark.parametrize("M,N,K,stream_k", [(384, 14336, 8192, False),  # half tiles fill the tail
                                            (1024, 8192, 8192, False),  # a second wave of whole tiles
                                            (384, 10240, 8192, True)])  # a nearly empty tail
def test_two_rows_of_tiles_take_half_tiles_over_stream_k(g, M, N, K, stream_k):
    # with two rows of 256-row tiles or more between one and two waves, stream-K gives way
    # to whole tiles (half tiles in the last wave where they fit) unless the last wave holds
    # at most a quarter of the units (sampled rows and columns against the oracle)
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=55)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    cfg = g.last_config()
    if g.sm_count >= 152:
        assert cfg["block_n"] == 256 and (cfg["splits"] < 0) == stream_k, cfg
        if not stream_k:
            assert cfg["splits"] == 1, cfg
    rows = si.sample_indices(M, 16, seed=11, must=(0, 255, 256, M - 1))
    cols = si.sample_indices(N, 48, seed=12, must=(0, 127, 128, N - 1))
    parity.oracle_check(parity.bits_of(C)[np.ix_(rows, cols)], A, B, F16, F16, rows=rows,
                        cols=cols, what=f"two rows of tiles {cfg}")


@pytest.mark.parametrize("M,N,K", [(384, 4096, 4096), (256, 8192, 2048)])
def test_unsplit_narrow_tiles_are_not_replaced_by_320_column_split_tiles(g, M, N, K):
    # 128-column pair tiles that fill one wave without a K split stay (the 320-column
    # cluster split is for 256-column tiles that do not fit a two-way split)
    A, B = si.make_operands(M, N, K, F16, "uniform", seed=56)
    C = torch.empty(M, N, dtype=torch.float16, device="cuda")
    g.reset_config()
    g.run(A.cuda(), B.cuda(), C)
    torch.cuda.synchronize()
    assert g.device_status()[0] == 0
    cfg = g.last_config()
    if g.sm_count >= 152:
        assert cfg["block_n"] == 128 and cfg["splits"] == 1 and cfg["swap_ab"] == 1, cfg
    rows = si.sample_indices(M, 16, seed=13, must=(0, 255, M - 1))
    cols = si.sample_indices(N, 48, seed=14, must=(0, 127, 128, N - 1))
    parity.oracle_check(parity.bits_of(C)[np.ix_(rows, cols)], A, B, F16, F16, rows=rows,
                        cols=cols, what=f"narrow tiles {cfg}")


def test_320_column_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.zeros(256, 16384, dtype=torch.float16, device="cuda")
    B = torch.zeros(640, 16384, dtype=torch.float16, device="cuda")
    C = torch.zeros(256, 640, dtype=torch.float16, device="cuda")
    for cfg in ({"variant": 2, "block_n": 320},                           # no K split
                {"variant": 2, "block_n": 320, "splits": 2, "epilogue": 3},  # slices of 2 chains
                {"variant": 1, "block_n": 320, "splits": 2, "epilogue": 3}):  # one CTA
        g.set_config(**cfg)
        try:
            with pytest.raises(GemmError) as e:
                g.run(A, B, C)
            assert e.value.code in (1, 2), cfg
        finally:
            g.reset_config()


def test_cluster_k_split_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.zeros(256, 4096, dtype=torch.float16, device="cuda")
    C = torch.zeros(256, 1024, dtype=torch.float16, device="cuda")
    B = torch.zeros(1024, 4096, dtype=torch.float16, device="cuda")
    g.set_config(variant=2, splits=2, epilogue=3)
    try:
        with pytest.raises(GemmError) as e:                     # with a fused epilogue
            g.run_epilogue(A, B, C, alpha=2.0)
        assert e.value.code == 2
        A8 = torch.zeros(256, 4096, dtype=torch.float8_e4m3fn, device="cuda")
        B8 = torch.zeros(1024, 4096, dtype=torch.float8_e4m3fn, device="cuda")
        with pytest.raises(GemmError) as e:                     # FP8 operands
            g.run(A8, B8, C)
        assert e.value.code == 2
    finally:
        g.reset_config()
    for cfg in ({"splits": 3, "epilogue": 3},):                   # not two slices
        g.set_config(**cfg)
        try:
            with pytest.raises(GemmError) as e:
                g.run(A, B, C)
            assert e.value.code == 2
        finally:
            g.reset_config()
    # more tiles than fit at once in clusters
    A = torch.zeros(4096, 4096, dtype=torch.float16, device="cuda")
    C = torch.zeros(4096, 4096, dtype=torch.float16, device="cuda")
    B = torch.zeros(4096, 4096, dtype=torch.float16, device="cuda")
    g.set_config(variant=2, splits=2, epilogue=3)
    try:
        with pytest.raises(GemmError) as e:
            g.run(A, B, C)
        assert e.value.code == 2
    finally:
        g.reset_config()


@pytest.mark.parametrize("M", [1, 2, 3, 4])
@pytest.mark.parametrize("N,K", [(1, 8), (7, 1000), (1000, 2048), (4097, 520), (300, 8192)])
def test_matrix_vector_path(g, M, N, K):
    # variant 3: the CUDA-core path for up to four rows of A
    g.set_config(variant=3)
    try:
        _case(g, M, N, K, F16, F32, seed=110 + M)
        _case(g, M, N, K, BF16, BF16, seed=111 + M)
        _case(g, M, N, K, F16, F16, seed=112 + M, exact=True, ints=True)
        assert g.last_config()["variant"] == 3
    finally:
        g.reset_config()


def test_one_row_takes_the_matrix_vector_path(g):
    _case(g, 1, 8192, 8192, F16, F16, seed=113)
    assert g.last_config()["variant"] == 3
    _case(g, 1, 8192, 28672, F16, F16, seed=114)      # long rows stay on the tensor cores
    assert g.last_config()["variant"] == 1
    _case(g, 2, 8192, 8192, F16, F16, seed=115)
    assert g.last_config()["variant"] == 1


def test_matrix_vector_path_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    g.set_config(variant=3)
    try:
        A = torch.zeros(5, 64, dtype=torch.float16, device="cuda")       # five rows
        B = torch.zeros(32, 64, dtype=torch.float16, device="cuda")
        C = torch.zeros(5, 32, dtype=torch.float32, device="cuda")
        with pytest.raises(GemmError) as e:
            g.run(A, B, C)
        assert e.value.code == 2
        with pytest.raises(GemmError) as e:                              # fused epilogue
            g.run_epilogue(A[:2], B, C[:2], alpha=2.0)
        assert e.value.code == 2
        A8 = torch.zeros(2, 64, dtype=torch.float8_e4m3fn, device="cuda")
        B8 = torch.zeros(32, 64, dtype=torch.float8_e4m3fn, device="cuda")
        with pytest.raises(GemmError) as e:                              # FP8 operands
            g.run(A8, B8, C[:2])
        assert e.value.code == 2
    finally:
        g.reset_config()


# The swapped tiling: B's rows are the MMA's row operand (swap_rows per CTA, a short box
# whose missing rows only feed accumulator lanes that are never stored), A's rows its
# columns; C is written transposed.  Ragged rows of A and of B, K tails, two accumulation
# chains, 256 rows of A per tile, a persistent loop of several tiles per pair.
@pytest.mark.parametrize("M,N,K,din,dout,extra", [
    (256, 8192, 1024, F16, F16, {}),                      # one wave, automatic rows
    (200, 3000, 2048, BF16, F32, {}),                     # ragged rows of A and of B
    (256, 1000, 520, F16, BF16, {"swap_rows": 40}),       # K tail, many tiles per pair
    (100, 777, 4096, F16, F16, {"block_n": 256}),         # 256 rows of A per tile
    (1, 4097, 512, BF16, F32, {}),                        # one row of A
    (256, 2048, 8192, F16, F32, {"swap_rows": 128}),      # two accumulation chains
    (129, 5000, 1024, F16, F16, {"swap_rows": 96, "max_ctas": 16}),  # persistent loop
])
def test_swapped_tiling(g, M, N, K, din, dout, extra):
    cfg = dict(swap_ab=2, **extra)
    g.set_config(**cfg)
    try:
        _case(g, M, N, K, din, dout, seed=61)
        used = g.last_config()
        _case(g, M, N, K, BF16, F32 if dout == F32 else dout, seed=62, exact=True, ints=True)
    finally:
        g.reset_config()
    assert used["swap_ab"] == 2 and used["variant"] == 2 and used["splits"] == 1, used
    w = used["swap_rows"]
    assert 1 <= w <= 128 and (extra.get("swap_rows", w) == w), used
    bn = extra.get("block_n", 128)
    assert used["block_n"] == bn and used["dp_tiles"] == -(-N // (2 * w)) * -(-M // bn), used


def test_swapped_tiling_matches_the_plain_tiling_on_integers(g):
    # the same integer-valued product both ways: bit-identical (every partial sum exact)
    M, N, K = 256, 4096, 2048
    A, B = si.make_small_int_operands(M, N, K, F16, seed=63)
    got = {}
    for swap in (1, 2):
        g.set_config(swap_ab=swap)
        try:
            C = parity.run_gpu(g, A, B, F32)
            assert g.device_status()[0] == 0
            assert g.last_config()["swap_ab"] == swap
        finally:
            g.reset_config()
        got[swap] = parity.bits_of(C)
    assert np.array_equal(got[1], got[2])


def test_swapped_tiling_rejections(g):
    from dense_gemm_blackwell_02_gb300.binding import GemmError
    A = torch.zeros(256, 1024, dtype=torch.float16, device="cuda")
    B = torch.zeros(512, 1024, dtype=torch.float16, device="cuda")
    C = torch.zeros(256, 512, dtype=torch.float16, device="cuda")
    for cfg in ({"swap_ab": 2, "variant": 1}, {"swap_ab": 2, "splits": 2},
                {"swap_ab": 2, "splits": -1}, {"swap_ab": 2, "epilogue": 2},
                {"swap_ab": 2, "block_n": 320}):
        g.set_config(**cfg)
        try:
            with pytest.raises(GemmError) as e:
                g.run(A, B, C)
            assert e.value.code == 2, cfg
        finally:
            g.reset_config()
    g.set_config(swap_ab=2)
    try:
        with pytest.raises(GemmError) as e:                       # a fused epilogue
            g.run_epilogue(A, B, C, alpha=2.0)
        assert e.value.code == 2
        A8 = A.to(torch.float8_e4m3fn)
        B8 = B.to(torch.float8_e4m3fn)
        with pytest.raises(GemmError) as e:                       # FP8 operands
            g.run(A8, B8, C)
        assert e.value.code == 2
    finally:
        g.reset_config()
    from dense_gemm_blackwell_02_gb300.binding import lib, GemmConfig
    import ctypes
    for bad in ({"swap_ab": 3}, {"swap_rows": 129}, {"swap_rows": -1}):
        cfg = GemmConfig(**{**{n: 0 for n, _ in GemmConfig._fields_}, **bad})
        assert lib().gemm_set_config(g._h, ctypes.byref(cfg)) == 1, bad
