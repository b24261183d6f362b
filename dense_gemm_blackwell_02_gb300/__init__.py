"""GB300 (sm_103a) dense tensor-core GEMM  C = A . B^T  behind a C ABI.

The compute path is libgemm.so (hand-written CUDA in csrc/, interface in
include/gemm.h).  ``binding`` marshals torch tensors or raw pointers into its
entry points; importing this package does not load the library, so the host
tools (``roofline``, ``swizzle``) work on machines without a GPU.
"""

__all__ = ["binding", "roofline", "swizzle"]


def __getattr__(name):
    if name in ("Gemm", "GemmError", "lib", "F16", "BF16", "F32", "GemmConfig"):
        from . import binding
        return getattr(binding, name)
    raise AttributeError(name)
