"""Comparison rules between the CUDA path and the CPU oracle (tests only).

Tolerances (the GEMM's stated bar):
  * fp16 / bf16 C: every element within 1 unit in the last place of the
    oracle's correctly rounded value, |ord(gpu) - ord(oracle)| <= 1, where ord
    maps a bit pattern to a monotone integer (+0 and -0 both map to 0).
    Reading for elements whose exact value nearly cancels: there an output ulp
    is smaller than any fp32 accumulator's rounding error, so such an element
    instead passes when |gpu - exact| <= ulp_out(exact)/2 + tau, with
    tau = 8 * 2^-24 * sqrt(K) * sigma,  sigma = sqrt(sum_k (a_ik b_jk)^2)
    (a random walk of K fp32 roundings of partial sums of size ~sigma, with a
    factor 8 of headroom).  For typical elements tau is far below half an
    output ulp, so the 1-ulp rule is what binds.
  * fp32 C: relative Frobenius error <= 1e-5 and max abs error <= 1e-2, and
    every element within ulp/2 + tau of the exact sum.
  * integer-valued inputs (every partial sum exact in fp32): bit-exact.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle
import seeded_inputs as si

F16, BF16, F32 = 0, 1, 2
FRO_TOL = 1e-5
ABS_TOL = 1e-2


def bits_of(t: torch.Tensor) -> np.ndarray:
    """Bit patterns of a (CPU or CUDA) fp16/bf16/fp32 tensor as uint16/uint32."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.float32:
        return t.view(torch.int32).numpy().view(np.uint32)
    return t.view(torch.int16).numpy().view(np.uint16)


def ordinal(bits: np.ndarray) -> np.ndarray:
    b = bits.astype(np.int64)
    sign = np.int64(1) << (8 * bits.dtype.itemsize - 1)
    mag = b & (sign - 1)
    return np.where(b & sign, -mag, mag)


def ulp_distance(got_bits: np.ndarray, want_bits: np.ndarray) -> np.ndarray:
    return np.abs(ordinal(got_bits) - ordinal(want_bits))


def _decode(bits: np.ndarray, dtype_out: int) -> np.ndarray:
    if dtype_out == F32:
        return bits.view(np.float32).astype(np.float64)
    t = torch.from_numpy(bits.view(np.int16).copy())
    return t.view(torch.float16 if dtype_out == F16 else torch.bfloat16).double().numpy()


def ulp_of(x: np.ndarray, dtype_out: int) -> np.ndarray:
    """Spacing of the output format at |x| (subnormal spacing below the normal range)."""
    frac, emin = {F16: (10, -14), BF16: (7, -126), F32: (23, -126)}[dtype_out]
    mag = np.maximum(np.abs(x), 2.0 ** emin)
    return np.exp2(np.floor(np.log2(mag)) - frac)


def take_rows(t: torch.Tensor, idx) -> torch.Tensor:
    """t[idx] for a list of row indices; FP8 tensors are gathered through their bytes
    (torch has no CPU index kernel for them)."""
    if t.element_size() == 1 and t.is_floating_point():
        return t.view(torch.uint8)[list(idx)].view(t.dtype)
    return t[list(idx)]


def sigma_of(A, B, rows=None) -> np.ndarray:
    """sqrt(sum_k (a_ik b_jk)^2) for the selected rows (float64 on the host)."""
    a = A if rows is None else take_rows(A, rows)
    a2 = a.to(torch.float64).square()
    out = torch.empty(a.shape[0], B.shape[0], dtype=torch.float64)
    for j0 in range(0, B.shape[0], 8192):
        out[:, j0:j0 + 8192] = a2 @ B[j0:j0 + 8192].to(torch.float64).square().T
    return out.sqrt().numpy()


def tau_of(sigma: np.ndarray, K: int) -> np.ndarray:
    return 8.0 * 2.0 ** -24 * np.sqrt(max(K, 1)) * sigma


def check(got_bits: np.ndarray, want_bits: np.ndarray, dtype_out: int, exact: bool = False,
          what: str = "", c64: np.ndarray = None, sigma: np.ndarray = None, K: int = None):
    """Assert the stated tolerance; returns a dict of error metrics.

    want_bits: the oracle's rounded output; c64: its unrounded binary64 sums;
    sigma/K: the accumulation scale for the cancellation reading above."""
    assert got_bits.shape == want_bits.shape, (got_bits.shape, want_bits.shape)
    if exact:
        bad = np.argwhere(got_bits != want_bits)
        assert bad.size == 0, f"{what}: {len(bad)} elements differ bitwise, first at {bad[:5]}"
        return {"max_ulp": 0}
    g = _decode(got_bits, dtype_out)
    assert np.all(np.isfinite(g)), f"{what}: non-finite output"
    out = {}
    if dtype_out == F32:
        w = _decode(want_bits, dtype_out)
        err = g - w
        fro = float(np.linalg.norm(err) / max(np.linalg.norm(w), 1e-300))
        mx = float(np.max(np.abs(err))) if err.size else 0.0
        assert fro <= FRO_TOL and mx <= ABS_TOL, f"{what}: rel fro {fro:.3g}, max abs {mx:.3g}"
        out.update({"rel_fro": fro, "max_abs": mx})
        d = None
    else:
        d = ulp_distance(got_bits, want_bits)
        out.update({"max_ulp": int(d.max()) if d.size else 0,
                    "frac_beyond_1ulp": float((d > 1).mean()) if d.size else 0.0})
    if c64 is not None and sigma is not None:
        bound = ulp_of(c64, dtype_out) / 2 + tau_of(sigma, K)
        err = np.abs(g - c64)
        ok = err <= bound
        if d is not None:
            ok |= d <= 1
        if not ok.all():
            idx = np.argwhere(~ok)[:5]
            detail = [(tuple(int(v) for v in ij), float(c64[tuple(ij)]), float(g[tuple(ij)]),
                       float(bound[tuple(ij)])) for ij in idx]
            raise AssertionError(f"{what}: {int((~ok).sum())} elements outside tolerance; "
                                 f"(index, exact, gpu, bound): {detail}")
        # how close the worst element came to its bound (<= 1 passes)
        rel = err / bound
        if d is not None:
            rel = np.where(d <= 1, 0.0, rel)
        out["max_err_over_bound"] = float(rel.max()) if rel.size else 0.0
    elif d is not None and out["max_ulp"] > 1:
        raise AssertionError(f"{what}: elements beyond 1 ulp and no cancellation data given")
    return out


def check_pair(got_bits, ref_bits, dtype_out, c64, sigma, K, what=""):
    """Two GPU results of the same product that may accumulate in different orders:
    each may lie within ulp/2 + tau of the exact sum (and within 1 ulp of its rounding),
    so they must agree within 2 ulps, or within ulp + 2 tau where the sum cancels."""
    g = _decode(got_bits, dtype_out)
    r = _decode(ref_bits, dtype_out)
    ok = np.abs(g - r) <= ulp_of(c64, dtype_out) + 2 * tau_of(sigma, K)
    if dtype_out != F32:
        ok |= ulp_distance(got_bits, ref_bits) <= 2
    if not ok.all():
        idx = np.argwhere(~ok)[:5]
        raise AssertionError(f"{what}: {int((~ok).sum())} elements differ beyond the tolerance; "
                             f"first at {idx.tolist()}")


def oracle_check(got_bits, A, B, dtype_in, dtype_out, rows=None, cols=None, what="",
                 exact=False):
    """Oracle on the same inputs (optionally selected rows/cols), then check()."""
    want, c64 = oracle.gemm_select(A, B, rows, cols, dtype_in, dtype_out, want_f64=True)
    if exact:
        return check(got_bits, want, dtype_out, exact=True, what=what)
    Bs = B if cols is None else take_rows(B, cols)
    sig = sigma_of(A, Bs, rows)
    return check(got_bits, want, dtype_out, what=what, c64=c64, sigma=sig, K=A.shape[1])


def oracle_full(A, B, dtype_in, dtype_out):
    return oracle.gemm(A, B, dtype_in, dtype_out)


def run_gpu(g, A, B, dtype_out, device="cuda"):
    """Copy the CPU operands to the device, run the library, return C's bits."""
    Ad, Bd = A.to(device), B.to(device)
    C = torch.empty(A.shape[0], B.shape[0], dtype=si.TORCH_DTYPE[dtype_out], device=device)
    g.run(Ad, Bd, C)
    torch.cuda.synchronize()
    return C


def freivalds(A, B, C_gpu, dtype_out, seeds=(0, 1, 2)):
    """Freivalds' check in float64 on the host: for x in {+-1}^N,
    |C x - A (B^T x)|_i <= sum_j (ulp_out(C_ij)/2 + gamma sum_k |A_ik B_jk|),
    gamma = K 2^-24 (worst-case fp32 accumulation).  Processes rows in chunks."""
    M, K = A.shape
    N = B.shape[0]
    gamma = K * 2.0 ** -24
    colsum_absB = torch.zeros(K, dtype=torch.float64)
    for j0 in range(0, N, 4096):
        colsum_absB += B[j0:j0 + 4096].to(torch.float64).abs().sum(0)
    xs = [si.rademacher(N, s) for s in seeds]
    btx = [torch.zeros(K, dtype=torch.float64) for _ in xs]
    for j0 in range(0, N, 4096):
        Bc = B[j0:j0 + 4096].to(torch.float64)
        for t, x in enumerate(xs):
            btx[t] += x[j0:j0 + 4096] @ Bc
    worst = 0.0
    Cc = C_gpu
    for i0 in range(0, M, 1024):
        Ac = A[i0:i0 + 1024].to(torch.float64)
        Cr = Cc[i0:i0 + 1024].cpu().to(torch.float64)
        assert torch.isfinite(Cr).all(), "non-finite output"
        mag = Cr.abs()
        if dtype_out == F32:
            half_ulp = torch.ldexp(torch.ones_like(mag), torch.floor(torch.log2(mag.clamp_min(2.0 ** -126))).to(torch.int32) - 24)
        else:
            frac = 10 if dtype_out == F16 else 7
            emin = -14 if dtype_out == F16 else -126
            e = torch.floor(torch.log2(mag.clamp_min(2.0 ** emin))).to(torch.int32)
            half_ulp = torch.ldexp(torch.ones_like(mag), e - frac - 1)
        bound = half_ulp.sum(1) + gamma * (Ac.abs() @ colsum_absB)
        for t, x in enumerate(xs):
            y = Cr @ x
            z = Ac @ btx[t]
            r = (y - z).abs() / bound
            worst = max(worst, float(r.max()))
            bad = torch.nonzero(r > 1.0)
            assert bad.numel() == 0, f"Freivalds failed at rows {(bad[:5].flatten() + i0).tolist()}"
    return worst
