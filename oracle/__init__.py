"""CPU oracle for C = A . B^T -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The GEMM library under
``dense_gemm_blackwell_02_gb300`` never imports it, and this package imports
nothing from there: the two share no code.

The arithmetic lives in ``oracle.c`` (plain C, binary64 accumulation, its own
fp16/bf16/fp32 decoders and round-to-nearest-even encoder written from the
format definitions).  This module only builds and loads that library and
marshals numpy arrays through ctypes.

Definition followed ("A Blackwell GEMM by Hand in CuTe DSL", section 1;
"Speed-of-Light GEMM, Part 1", naive matmul listing):

    C[i, j] = round_out( sum_k double(A[i, k]) * double(B[j, k]) )

with A (M x K) and B (N x K) K-major, k summed in increasing order in
binary64, and round_out a single round-to-nearest-even step from binary64 to
the output format.

FP8 operands (codes E4M3 = 3, E5M2 = 4; OCP 8-bit formats) and the blockwise-scaled
product ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05", Part 6, FP8 and
Blockwise Scaling) are described at the top of oracle.c.

Pins (tests/test_oracle_pins.py): exact rational brute force on tiny shapes,
all-ones (C = K), identity B (C = A), small-integer operands (exact integer
products), rank-1 operands (C = u v^T (a.b)), and the converters against
numpy's IEEE casts and an exact-rational rounding written independently.
"""
from __future__ import annotations

import ctypes
import os
import platform
import subprocess

import numpy as np

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
FP8 = (E4M3, E5M2)
_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it (gcc, no GPU needed)."""
    stamp = _LIB_PATH + ".arch"
    same_arch = os.path.exists(stamp) and open(stamp).read().strip() == platform.machine()
    if (not force and same_arch and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-ffp-contract=off", "-fPIC", "-shared", "-pthread",
           _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    with open(stamp, "w") as f:
        f.write(platform.machine())
    return _LIB_PATH


def load_library(path: str):
    """Load an oracle shared library from `path` and declare its entry points."""
    lib = ctypes.CDLL(path)
    i64, i32, vp = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p
    lib.oracle_gemm.argtypes = [vp, vp, vp, i64, i64, i64, i32, i32, i32]
    lib.oracle_gemm.restype = i32
    lib.oracle_gemm_select.argtypes = [vp, vp, vp, vp, i64, vp, i64, vp, i64,
                                       i32, i32, i32]
    lib.oracle_gemm_select.restype = i32
    lib.oracle_decode.argtypes = [vp, vp, i64, i32]
    lib.oracle_decode.restype = i32
    lib.oracle_round.argtypes = [vp, vp, i64, i32]
    lib.oracle_round.restype = i32
    if hasattr(lib, "oracle_gemm_blockwise"):
        lib.oracle_gemm_blockwise.argtypes = [vp, vp, vp, vp, i64, i64, i64, vp, vp, i64, i64,
                                              vp, i64, vp, i64, i32, i32, i32]
        lib.oracle_gemm_blockwise.restype = i32
    if hasattr(lib, "oracle_gemm_epilogue"):
        lib.oracle_gemm_epilogue.argtypes = [vp, vp, vp, vp, ctypes.c_double, ctypes.c_double,
                                             i32, vp, i64, i64, i64, i32, i32, i32]
        lib.oracle_gemm_epilogue.restype = i32
    return lib


def _load(lib=None):
    global _lib
    if lib is not None:
        return lib
    if _lib is None:
        _lib = load_library(build())
    return _lib


def _bits16(x, dtype_in: int = F16) -> np.ndarray:
    """Accept a numpy array of bit patterns or a CPU torch tensor (fp16/bf16, or
    fp8 for the E4M3/E5M2 codes) and return a C-contiguous view of its bit
    patterns: uint16, or uint8 for fp8."""
    width = 1 if dtype_in in FP8 else 2
    if hasattr(x, "detach"):  # torch tensor (CPU); reinterpret without copying values
        import torch
        if x.element_size() != width:
            raise TypeError(f"oracle operands for dtype {dtype_in} must be {8 * width}-bit, "
                            f"got {x.dtype}")
        x = x.detach().contiguous().view(torch.uint8 if width == 1 else torch.int16).numpy()
    a = np.ascontiguousarray(x)
    if a.dtype.itemsize != width:
        raise TypeError(f"oracle operands for dtype {dtype_in} must be {8 * width}-bit "
                        f"patterns, got {a.dtype}")
    return a.view(np.uint8 if width == 1 else np.uint16)


def _out_array(shape, dtype_out):
    return np.empty(shape, dtype=np.uint32 if dtype_out == F32 else np.uint16)


def _check(rc):
    if rc < 0:
        raise ValueError("oracle rejected its arguments")
    return rc


def gemm(A, B, dtype_in: int, dtype_out: int, nthreads: int = 0, lib=None) -> np.ndarray:
    """Full C = A . B^T as output-format bit patterns (uint16 or uint32), M x N."""
    a, b = _bits16(A, dtype_in), _bits16(B, dtype_in)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    C = _out_array((M, N), dtype_out)
    _check(_load(lib).oracle_gemm(a.ctypes.data, b.ctypes.data, C.ctypes.data, M, N, K,
                               dtype_in, dtype_out, nthreads))
    return C


def gemm_grouped(problems, dtype_in: int, dtype_out: int, nthreads: int = 0, lib=None) -> list:
    """A group of independent products ("CUTLASS Deep Dive: From CuTe Layouts to
    Blackwell tcgen05", Part 6, Grouped GEMM: many GEMMs of different shapes, as the
    experts of a Mixture-of-Experts layer need): for each (A_g, B_g) in `problems`,
    C_g = A_g . B_g^T by the definition above (its own M_g, N_g, K_g; K_g = 0 gives
    zeros).  Returns the list of C_g bit patterns, in order."""
    return [gemm(A, B, dtype_in, dtype_out, nthreads=nthreads, lib=lib) for A, B in problems]


def gemm_select(A, B, rows, cols, dtype_in: int, dtype_out: int, nthreads: int = 0,
                want_f64: bool = False):
    """Outputs C[rows][:, cols] (len(rows) x len(cols)); rows/cols None = all.

    Returns the rounded bit patterns, or (bits, binary64 sums) if want_f64."""
    a, b = _bits16(A, dtype_in), _bits16(B, dtype_in)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else len(r)
    nc = N if c is None else len(c)
    if r is not None and len(r) and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    if c is not None and len(c) and (c.min() < 0 or c.max() >= N):
        raise IndexError("column index out of range")
    out = _out_array((nr, nc), dtype_out)
    f64 = np.empty((nr, nc), dtype=np.float64) if want_f64 else None
    _check(_load().oracle_gemm_select(
        a.ctypes.data, b.ctypes.data, out.ctypes.data,
        None if f64 is None else f64.ctypes.data, K,
        None if r is None else r.ctypes.data, nr,
        None if c is None else c.ctypes.data, nc, dtype_in, dtype_out, nthreads))
    return (out, f64) if want_f64 else out


def gemm_epilogue(A, B, dtype_in: int, dtype_out: int, alpha=1.0, beta=0.0, cprev=None,
                  bias=None, relu=False, nthreads: int = 0, lib=None) -> np.ndarray:
    """D = act(alpha * A . B^T + beta * cprev + bias[j]) as output-format bit patterns
    (M x N): cprev is M x N output-format bit patterns (needed when beta != 0), bias N
    binary32 values, act ReLU when relu.  Evaluated in binary64, rounded once."""
    a, b = _bits16(A, dtype_in), _bits16(B, dtype_in)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    cp = None
    if beta != 0.0:
        if cprev is None:
            raise ValueError("beta != 0 needs the previous output")
        want = np.uint32 if dtype_out == F32 else np.uint16
        cp = np.ascontiguousarray(np.asarray(cprev).view(want).reshape(M, N))
    bs = None if bias is None else np.ascontiguousarray(np.asarray(bias, dtype=np.float32).reshape(N))
    D = _out_array((M, N), dtype_out)
    _check(_load(lib).oracle_gemm_epilogue(
        a.ctypes.data, b.ctypes.data, None if cp is None else cp.ctypes.data,
        None if bs is None else bs.ctypes.data, float(alpha), float(beta), 1 if relu else 0,
        D.ctypes.data, M, N, K, dtype_in, dtype_out, nthreads))
    return D


def gemm_blockwise(A, B, sfa, sfb, bm: int, bn: int, bk: int, dtype_in: int, dtype_out: int,
                   rows=None, cols=None, nthreads: int = 0, want_f64: bool = False, lib=None):
    """Outputs C[rows][:, cols] of the blockwise-scaled product
        C[i, j] = sum_kb sfa[i // bm, kb] * sfb[j // bn, kb] * sum_{k in block kb} A[i, k] B[j, k]
    (blocks of bk along K), as output-format bit patterns; sfa is ceil(M/bm) x
    ceil(K/bk) and sfb ceil(N/bn) x ceil(K/bk) binary32 scales.  rows/cols None = all.
    Returns the bits, or (bits, binary64 values) if want_f64."""
    a, b = _bits16(A, dtype_in), _bits16(B, dtype_in)
    M, K = a.shape
    N, K2 = b.shape
    if K != K2:
        raise ValueError("A and B disagree on K")
    nkb = -(-K // bk) if bk > 0 else 0
    fa = np.ascontiguousarray(np.asarray(sfa, dtype=np.float32))
    fb = np.ascontiguousarray(np.asarray(sfb, dtype=np.float32))
    if fa.shape != (-(-M // bm), nkb) or fb.shape != (-(-N // bn), nkb):
        raise ValueError(f"scale shapes {fa.shape}, {fb.shape} do not match the blocks")
    r = None if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    c = None if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    nr = M if r is None else len(r)
    nc = N if c is None else len(c)
    if r is not None and len(r) and (r.min() < 0 or r.max() >= M):
        raise IndexError("row index out of range")
    if c is not None and len(c) and (c.min() < 0 or c.max() >= N):
        raise IndexError("column index out of range")
    out = _out_array((nr, nc), dtype_out)
    f64 = np.empty((nr, nc), dtype=np.float64) if want_f64 else None
    _check(_load(lib).oracle_gemm_blockwise(
        a.ctypes.data, b.ctypes.data, fa.ctypes.data, fb.ctypes.data, bm, bn, bk,
        out.ctypes.data, None if f64 is None else f64.ctypes.data, M, K,
        None if r is None else r.ctypes.data, nr, None if c is None else c.ctypes.data, nc,
        dtype_in, dtype_out, nthreads))
    return (out, f64) if want_f64 else out


def decode(bits: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Exact binary64 values of fp16/bf16 (uint16), fp32 (uint32) or fp8 E4M3/E5M2
    (uint8) patterns."""
    want = np.uint32 if dtype == F32 else np.uint8 if dtype in FP8 else np.uint16
    b = np.ascontiguousarray(bits).view(want)
    out = np.empty(b.shape, dtype=np.float64)
    _check(_load(lib).oracle_decode(b.ctypes.data, out.ctypes.data, b.size, dtype))
    return out


def round_to(x: np.ndarray, dtype: int, lib=None) -> np.ndarray:
    """Round binary64 values to dtype with ties-to-even; returns bit patterns."""
    v = np.ascontiguousarray(x, dtype=np.float64)
    out = _out_array(v.shape, dtype)
    _check(_load(lib).oracle_round(v.ctypes.data, out.ctypes.data, v.size, dtype))
    return out
