"""Host-side analysis helpers reproduce the tables the pages print
(tests/golden/p1_*.txt, each citing its section)."""
import os

import pytest

from dense_gemm_blackwell_02_gb300 import roofline as rl
from dense_gemm_blackwell_02_gb300 import swizzle as sw

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name, tag=None):
    out = []
    for line in open(os.path.join(GOLDEN, name)):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        left, right = (s.split() for s in line.split("|"))
        if tag is not None:
            if left[0] != tag:
                continue
            left = left[1:]
        out.append((left, right))
    return out


# B200 constants the page's script used (section 1).
PEAK, BW, SMS, SMEM = 1500, 7.7, 148, 227 * 1024


def test_roofline_table_matches_page():
    rows = _rows("p1_gemm_math_roofline.txt")
    assert len(rows) == 7
    for left, right in rows:
        M, N, K = map(int, left[:3])
        t, tc = float(left[3]), float(left[4])
        fpb, bound, floor_us, tf, tb, ratio, ctas, wv = right
        assert f"{rl.arithmetic_intensity(M, N, K):.0f}" == fpb
        floor, b = rl.roofline_floor_us(M, N, K, PEAK, BW)
        assert b == bound and f"{floor:.1f}" == floor_us
        assert f"{rl.tflops(M, N, K, t):.0f}" == tf
        assert f"{rl.tbs(M, N, K, t):.2f}" == tb
        assert f"{tc / t:.2f}" == ratio
        tiles = rl.tile_count(M, N, 128, 256)
        assert str(tiles) == ctas
        assert f"{rl.waves(tiles, SMS):.2f}" == wv
    assert f"{rl.ridge_flop_per_byte(PEAK, BW):.0f}" == "195"


def test_stage_budget_matches_page():
    for left, right in _rows("p1_gemm_math_budget.txt", "stage"):
        _, a_rows, b_rows = left
        per = rl.stage_bytes(int(a_rows), int(b_rows), 64)
        kib, fpb, nmax = right
        assert str(per // 1024) == kib
        # each CTA accumulates 128x256 per k-step in both variants
        assert f"{rl.flop_per_smem_byte(128, 256, 64, per):.1f}" == fpb
        assert str(rl.max_stages(per, SMEM)) == nmax


def test_littles_law_matches_page():
    step = rl.kstep_us(128, 256, 64, PEAK, SMS)
    for left, right in _rows("p1_gemm_math_budget.txt", "little"):
        lat = float(left[0])
        assert f"{step:.2f}" == right[0]
        assert f"{rl.stages_for_latency(lat, step):.1f}" == right[1]


def test_ladder_matches_page():
    prev = None
    for left, right in _rows("p1_gemm_math_budget.txt", "ladder"):
        us = float(left[1])
        tf, frac, speed = right
        assert f"{rl.tflops(4096, 4096, 4096, us):.0f}" == tf
        assert f"{94.9 / us:.2f}" == frac
        if prev is None:
            assert speed == "-"
        else:
            assert f"{prev / us:.2f}" == speed
        prev = us


def test_swizzle_passes_match_page():
    for left, right in _rows("p1_swizzle_model.txt", "passes"):
        tile_k, pitch, layout = int(left[0]), int(left[1]), left[2]
        assert tile_k * 2 == pitch
        got = sw.column_passes(tile_k, 2, swizzled=(layout == "sw128"))
        assert got == [int(x) for x in right]
    assert sw.column_passes(16, 2, swizzled=True) is None


def test_swizzle_permutation_matches_page():
    rows = _rows("p1_swizzle_model.txt", "perm")
    assert len(rows) == 8
    for left, right in rows:
        assert sw.sw128_chunk_permutation(int(left[0])) == [int(x) for x in right]


@pytest.mark.parametrize("addr", [0, 16, 127, 128, 1023, 1024, 5000, 123456])
def test_swizzle_is_a_permutation_within_rows(addr):
    # stays inside its own 128-byte row and is an involution
    assert sw.sw128(addr) // 128 == addr // 128
    assert sw.sw128(sw.sw128(addr)) == addr


def test_gb300_peak_from_clock():
    # 152 SMs x 8192 FLOP/cycle at 2070 MHz ~ 2.58 PFLOP/s dense fp16
    assert abs(rl.tensor_peak_tflops(152, 2070) - 2577.4) < 0.5
