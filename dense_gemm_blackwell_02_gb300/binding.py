"""ctypes binding of libgemm.so (include/gemm.h): argument marshalling only.

Every step of the GEMM runs inside the library's CUDA kernels; this module
passes pointers, sizes, dtype codes and the caller's CUDA stream.  If the
library is missing it raises instead of falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

F16, BF16, F32, E4M3, E5M2 = 0, 1, 2, 3, 4
STATUS_NAMES = {0: "GEMM_OK", 1: "GEMM_ERR_INVALID_ARG", 2: "GEMM_ERR_UNSUPPORTED",
                3: "GEMM_ERR_CUDA", 4: "GEMM_ERR_OOM", 5: "GEMM_ERR_TIMEOUT"}
LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgemm.so")

# Every function include/gemm.h declares (checked against the header by the tests).
EXPORTS = ("gemm_create", "gemm_destroy", "gemm_run", "gemm_run_epilogue", "gemm_run_blockwise",
           "gemm_run_grouped", "gemm_run_host",
           "gemm_set_config",
           "gemm_last_config", "gemm_device_status", "gemm_set_wait_limit",
           "gemm_set_test_stall", "gemm_sm_count", "gemm_status_string", "gemm_run_noalloc",
           "gemm_last_cuda_error", "gemm_plan")


class GemmConfig(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int32) for n in ("variant", "block_n", "splits", "stages",
                                                "group_m", "max_ctas", "chain_kblocks",
                                                "dp_tiles", "prefetch_kblocks", "epilogue",
                                                "l2_hint", "swap_ab", "swap_rows", "scheduler")]

    def as_dict(self):
        return {n: getattr(self, n) for n, _ in self._fields_}


ACT_NONE, ACT_RELU = 0, 1


class GemmEpilogue(ctypes.Structure):
    """gemm_epilogue_t: C = act(alpha * A . B^T + beta * C_prev + bias)."""
    _fields_ = [("alpha", ctypes.c_float), ("beta", ctypes.c_float), ("bias", ctypes.c_void_p),
                ("activation", ctypes.c_int32)]


class GemmBlockScales(ctypes.Structure):
    """gemm_block_scales_t: FP8 block scales, sfa per (block_m rows, 128 of K) of A and
    sfb per (128 rows, 128 of K) of B."""
    _fields_ = [("sfa", ctypes.c_void_p), ("sfb", ctypes.c_void_p), ("block_m", ctypes.c_int32),
                ("block_n", ctypes.c_int32)]


class GemmProblem(ctypes.Structure):
    """gemm_problem_t: one problem of a grouped launch, C = A . B^T."""
    _fields_ = [("A", ctypes.c_void_p), ("B", ctypes.c_void_p), ("C", ctypes.c_void_p),
                ("M", ctypes.c_int64), ("N", ctypes.c_int64), ("K", ctypes.c_int64)]


class GemmError(RuntimeError):
    def __init__(self, code: int, what: str = ""):
        self.code = code
        super().__init__(f"{STATUS_NAMES.get(code, code)}{': ' + what if what else ''}")


class GemmDeviceModel(ctypes.Structure):
    """gemm_device_model_t: a GPU described for gemm_plan (SMs, resident CTA pairs,
    resident clusters of four CTAs)."""
    _fields_ = [("sms", ctypes.c_int32), ("pairs", ctypes.c_int32), ("clusters4", ctypes.c_int32)]


GB300_MODEL = (152, 76, 36)  # a full GB300: 152 SMs, 76 pairs, 36 clusters of four


def plan(M, N, K, dtype_in=F16, dtype_out=F16, fused=False, blockwise=False, config=None,
         device=GB300_MODEL) -> dict:
    """The configuration the library would launch for this product on the described
    device (gemm_plan): the host's decisions only, no GPU needed.  Raises GemmError with
    the call's status when it refuses."""
    cfg = None
    if config:
        cfg = GemmConfig(**{**{n: 0 for n, _ in GemmConfig._fields_}, **config})
    dev = GemmDeviceModel(*device)
    out = GemmConfig()
    _check(lib().gemm_plan(ctypes.byref(dev), ctypes.byref(cfg) if cfg is not None else None,
                           M, N, K, dtype_in, dtype_out, 1 if fused else 0,
                           1 if blockwise else 0, ctypes.byref(out)), "gemm_plan")
    return out.as_dict()


_lib = None


def lib():
    """Load libgemm.so (built in-tree) and declare its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is not built; run "
                           "`python -m dense_gemm_blackwell_02_gb300.build` first")
    L = ctypes.CDLL(LIB_PATH)
    vp, i64, i32, u32, u64 = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32,
                              ctypes.c_uint64)
    L.gemm_create.argtypes = [ctypes.POINTER(vp)]
    L.gemm_destroy.argtypes = [vp]
    L.gemm_run.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp]
    L.gemm_run_host.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, vp]
    L.gemm_set_config.argtypes = [vp, ctypes.POINTER(GemmConfig)]
    L.gemm_last_config.argtypes = [vp, ctypes.POINTER(GemmConfig)]
    L.gemm_device_status.argtypes = [vp, vp, ctypes.POINTER(u32)]
    L.gemm_set_wait_limit.argtypes = [vp, u64]
    L.gemm_set_test_stall.argtypes = [vp, i32]
    L.gemm_sm_count.argtypes = [vp]
    L.gemm_sm_count.restype = i32
    L.gemm_run_noalloc.argtypes = [vp, vp, vp, i64, i64, i64, i32, i32, vp]
    L.gemm_run_epilogue.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32,
                                    ctypes.POINTER(GemmEpilogue), vp]
    L.gemm_run_blockwise.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32,
                                     ctypes.POINTER(GemmBlockScales), vp]
    L.gemm_run_grouped.argtypes = [vp, ctypes.POINTER(GemmProblem), i32, i32, i32, vp]
    L.gemm_status_string.argtypes = [i32]
    L.gemm_status_string.restype = ctypes.c_char_p
    L.gemm_plan.argtypes = [ctypes.POINTER(GemmDeviceModel), ctypes.POINTER(GemmConfig), i64, i64,
                            i64, i32, i32, i32, i32, ctypes.POINTER(GemmConfig)]
    L.gemm_last_cuda_error.argtypes = [vp]
    L.gemm_last_cuda_error.restype = ctypes.c_char_p
    for name in EXPORTS:
        if name not in ("gemm_sm_count", "gemm_status_string", "gemm_last_cuda_error"):
            getattr(L, name).restype = i32
    _lib = L
    return L


def _check(code: int, what: str = "", h=None):
    if code != 0:
        if code == 3 and h is not None:  # GEMM_ERR_CUDA: name the CUDA error behind it
            detail = lib().gemm_last_cuda_error(h).decode()
            if detail:
                what = f"{what} ({detail})" if what else detail
        raise GemmError(code, what)


def torch_float32():
    import torch
    return torch.float32


def torch_dtype_code(dt) -> int:
    import torch
    return {torch.float16: F16, torch.bfloat16: BF16, torch.float32: F32,
            torch.float8_e4m3fn: E4M3, torch.float8_e5m2: E5M2}[dt]


def _stream_ptr(stream, device):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


class Gemm:
    """One library handle (workspace, status word, tensor-map cache)."""

    def __init__(self):
        h = ctypes.c_void_p()
        _check(lib().gemm_create(ctypes.byref(h)), "gemm_create")
        self._h = h

    @property
    def handle(self):
        return self._h

    def close(self):
        if self._h:
            lib().gemm_destroy(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    @property
    def sm_count(self) -> int:
        return lib().gemm_sm_count(self._h)

    # ------------------------------------------------------------ raw pointers --
    def run_ptr(self, a_ptr, b_ptr, c_ptr, M, N, K, dtype_in, dtype_out, stream_ptr=0) -> int:
        """gemm_run on raw device pointers; returns the status code."""
        return lib().gemm_run(self._h, a_ptr, b_ptr, c_ptr, M, N, K, dtype_in, dtype_out,
                              stream_ptr)

    # ----------------------------------------------------------- torch tensors --
    def run(self, A, B, C, stream=None):
        """C = A @ B.T for CUDA tensors A (M,K), B (N,K), C (M,N), all contiguous."""
        if not (A.is_cuda and B.is_cuda and C.is_cuda):
            raise ValueError("A, B and C must be CUDA tensors")
        if not (A.is_contiguous() and B.is_contiguous() and C.is_contiguous()):
            raise ValueError("A, B and C must be contiguous (row-major, K-major operands)")
        if A.dim() != 2 or B.dim() != 2 or C.dim() != 2:
            raise ValueError("A, B and C must be 2-D")
        M, K = A.shape
        N, K2 = B.shape
        if K != K2 or tuple(C.shape) != (M, N):
            raise ValueError(f"shape mismatch: A {tuple(A.shape)}, B {tuple(B.shape)}, "
                             f"C {tuple(C.shape)}")
        if A.dtype != B.dtype:
            raise ValueError("A and B must share a dtype")
        code = self.run_ptr(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                            torch_dtype_code(A.dtype), torch_dtype_code(C.dtype),
                            _stream_ptr(stream, A.device))
        _check(code, f"gemm_run M={M} N={N} K={K}", self._h)
        return C

    def run_epilogue(self, A, B, C, alpha=1.0, beta=0.0, bias=None, relu=False, stream=None):
        """C = act(alpha * A @ B.T + beta * C + bias) in the GEMM's epilogue: bias a CUDA
        float32 tensor of N values (or None), act ReLU when relu."""
        M, K = A.shape
        N = B.shape[0]
        if bias is not None:
            if not (bias.is_cuda and bias.dtype == torch_float32() and bias.is_contiguous()
                    and bias.numel() == N):
                raise ValueError("bias must be a contiguous float32 CUDA tensor of N values")
        if not (A.is_cuda and B.is_cuda and C.is_cuda and A.is_contiguous() and B.is_contiguous()
                and C.is_contiguous() and B.shape[1] == K and tuple(C.shape) == (M, N)
                and A.dtype == B.dtype):
            raise ValueError("A (M,K), B (N,K), C (M,N): contiguous CUDA tensors, A and B of one dtype")
        epi = GemmEpilogue(float(alpha), float(beta), None if bias is None else bias.data_ptr(),
                           ACT_RELU if relu else ACT_NONE)
        code = lib().gemm_run_epilogue(self._h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                       torch_dtype_code(A.dtype), torch_dtype_code(C.dtype),
                                       ctypes.byref(epi), _stream_ptr(stream, A.device))
        _check(code, f"gemm_run_epilogue M={M} N={N} K={K}", self._h)
        return C

    def run_blockwise(self, A, B, C, sfa, sfb, block_m, block_n=128, stream=None):
        """C = sum_kb sfa[kb, i // block_m] * sfb[kb, j // block_n] * (A @ B.T over the kb-th
        128 columns of K), A and B FP8 CUDA tensors; sfa and sfb contiguous float32 CUDA
        tensors stored K-block-major, ceil(K / 128) x ceil(M / block_m) and
        ceil(K / 128) x ceil(N / block_n)."""
        M, K = A.shape
        N = B.shape[0]
        nkb = -(-K // 128)
        for t, rows, name in ((sfa, -(-M // max(block_m, 1)), "sfa"), (sfb, -(-N // max(block_n, 1)), "sfb")):
            if not (t.is_cuda and t.dtype == torch_float32() and t.is_contiguous()
                    and tuple(t.shape) == (nkb, rows)):
                raise ValueError(f"{name} must be a contiguous float32 CUDA tensor of {nkb} x {rows}")
        if not (A.is_cuda and B.is_cuda and C.is_cuda and A.is_contiguous() and B.is_contiguous()
                and C.is_contiguous() and B.shape[1] == K and tuple(C.shape) == (M, N)
                and A.dtype == B.dtype):
            raise ValueError("A (M,K), B (N,K), C (M,N): contiguous CUDA tensors, A and B of one dtype")
        sc = GemmBlockScales(sfa.data_ptr(), sfb.data_ptr(), int(block_m), int(block_n))
        code = lib().gemm_run_blockwise(self._h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                        torch_dtype_code(A.dtype), torch_dtype_code(C.dtype),
                                        ctypes.byref(sc), _stream_ptr(stream, A.device))
        _check(code, f"gemm_run_blockwise M={M} N={N} K={K}", self._h)
        return C

    def run_grouped(self, problems, stream=None):
        """C_g = A_g @ B_g.T for every (A_g, B_g, C_g) in `problems`, in one launch: CUDA
        tensors, contiguous, one input dtype and one output dtype for all."""
        if not problems:
            return
        din, dout = problems[0][0].dtype, problems[0][2].dtype
        arr = (GemmProblem * len(problems))()
        for i, (A, B, C) in enumerate(problems):
            M, K = A.shape
            N = B.shape[0]
            if not (A.is_cuda and B.is_cuda and C.is_cuda and A.is_contiguous()
                    and B.is_contiguous() and C.is_contiguous() and B.shape[1] == K
                    and tuple(C.shape) == (M, N) and A.dtype == din and B.dtype == din
                    and C.dtype == dout):
                raise ValueError(f"problem {i}: A (M,K), B (N,K), C (M,N) contiguous CUDA tensors "
                                 "with the group's dtypes")
            arr[i] = GemmProblem(A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K)
        code = lib().gemm_run_grouped(self._h, arr, len(problems), torch_dtype_code(din),
                                      torch_dtype_code(dout),
                                      _stream_ptr(stream, problems[0][0].device))
        _check(code, f"gemm_run_grouped count={len(problems)}", self._h)

    def run_host(self, A, B, C, dtype_in, dtype_out, stream=None):
        """gemm_run_host on CPU tensors (pinned for asynchronous copies)."""
        M, K = A.shape
        N = B.shape[0]
        sp = 0 if stream is None else _stream_ptr(stream, None)
        code = lib().gemm_run_host(self._h, A.data_ptr(), B.data_ptr(), C.data_ptr(), M, N, K,
                                   dtype_in, dtype_out, sp)
        _check(code, "gemm_run_host", self._h)
        return C

    # ----------------------------------------------------------------- control --
    def set_config(self, variant=0, block_n=0, splits=0, stages=0, group_m=0, max_ctas=0,
                   chain_kblocks=0, prefetch_kblocks=0, epilogue=0, l2_hint=0, swap_ab=0,
                   swap_rows=0, scheduler=0):
        cfg = GemmConfig(variant, block_n, splits, stages, group_m, max_ctas, chain_kblocks, 0,
                         prefetch_kblocks, epilogue, l2_hint, swap_ab, swap_rows, scheduler)
        _check(lib().gemm_set_config(self._h, ctypes.byref(cfg)), "gemm_set_config")

    def reset_config(self):
        _check(lib().gemm_set_config(self._h, None), "gemm_set_config")

    def last_config(self) -> dict:
        cfg = GemmConfig()
        _check(lib().gemm_last_config(self._h, ctypes.byref(cfg)), "gemm_last_config")
        return cfg.as_dict()

    def device_status(self, stream=None):
        """(status code, raw device word) after synchronising the stream."""
        import torch
        detail = ctypes.c_uint32(0)
        sp = _stream_ptr(stream, torch.cuda.current_device())
        code = lib().gemm_device_status(self._h, sp, ctypes.byref(detail))
        return code, detail.value

    def set_wait_limit(self, ns: int):
        _check(lib().gemm_set_wait_limit(self._h, int(ns)), "gemm_set_wait_limit")

    def set_test_stall(self, enable: bool):
        _check(lib().gemm_set_test_stall(self._h, 1 if enable else 0), "gemm_set_test_stall")


def status_string(code: int) -> str:
    return lib().gemm_status_string(code).decode()
