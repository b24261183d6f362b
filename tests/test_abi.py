"""The C-ABI library builds, loads and exports every function include/gemm.h
declares; host-side argument handling works without a GPU (no kernel launches)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gemm.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w]+\**\s+\**(gemm_\w+)\s*\(", text, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    from dense_gemm_blackwell_02_gb300 import build, binding
    build.build()
    return binding.lib()


def test_header_declares_the_three_core_calls():
    names = _declared_functions()
    for core in ("gemm_create", "gemm_run", "gemm_destroy"):
        assert core in names


def test_every_declared_symbol_is_exported(lib):
    from dense_gemm_blackwell_02_gb300 import binding
    names = _declared_functions()
    assert set(names) == set(binding.EXPORTS), "binding and header disagree"
    for n in names:
        assert hasattr(lib, n), f"{n} missing from libgemm.so"


def test_status_strings(lib):
    for code in range(6):
        assert lib.gemm_status_string(code)
    assert lib.gemm_status_string(99) == b"unknown status"
    assert lib.gemm_last_cuda_error(None) == b""


def test_null_handle_is_rejected_without_touching_the_gpu(lib):
    assert lib.gemm_run(None, None, None, None, 1, 1, 8, 0, 0, None) == 1
    assert lib.gemm_set_config(None, None) == 1
    assert lib.gemm_device_status(None, None, None) == 1
    assert lib.gemm_set_wait_limit(None, 5) == 1
    assert lib.gemm_sm_count(None) == 0
    assert lib.gemm_destroy(None) == 0
    assert lib.gemm_create(None) == 1
    # the wider entry points reject a NULL handle (or table) before any device work
    assert lib.gemm_run_epilogue(None, None, None, None, 1, 1, 8, 0, 0, None, None) == 1
    assert lib.gemm_run_blockwise(None, None, None, None, 1, 1, 16, 3, 0, None, None) == 1
    assert lib.gemm_run_grouped(None, None, 0, 0, 0, None) == 1
    assert lib.gemm_run_host(None, None, None, None, 1, 1, 8, 0, 0, None) == 1


def test_library_is_built_for_sm_103a_only():
    from dense_gemm_blackwell_02_gb300 import build
    assert build.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]


def test_descriptor_packing_matches_the_documented_fields():
    # host-side restatement of the two descriptor layouts, checked field by field
    # against a CUDA translation unit compiled for the host (no GPU involved)
    import subprocess
    import tempfile
    src = r'''
#include <cstdio>
#include "umma.cuh"
int main() {
  using namespace gb300;
  std::printf("%llx %x %x\n", (unsigned long long)smem_desc_sw128_kmajor(0x12400u),
              idesc_f16_kmajor(128, 256, false), idesc_f16_kmajor(128, 128, true));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        cpp = os.path.join(d, "t.cu")
        exe = os.path.join(d, "t")
        open(cpp, "w").write(src)
        csrc = os.path.join(ROOT, "dense_gemm_blackwell_02_gb300", "csrc")
        subprocess.run(["nvcc", "-std=c++17", "-I", csrc, cpp, "-o", exe], check=True,
                       capture_output=True)
        desc, i1, i2 = subprocess.run([exe], capture_output=True, text=True).stdout.split()
    desc, i1, i2 = int(desc, 16), int(i1, 16), int(i2, 16)
    assert desc & 0x3FFF == 0x12400 >> 4            # start address >> 4
    assert (desc >> 16) & 0x3FFF == 1                # leading offset (unused) = 16 B
    assert (desc >> 32) & 0x3FFF == 1024 >> 4        # stride offset: 8 rows x 128 B
    assert (desc >> 46) & 0x7 == 1                   # fixed 0b001
    assert (desc >> 61) & 0x7 == 2                   # 128-byte swizzle
    for idesc, n, bf in ((i1, 256, 0), (i2, 128, 1)):
        assert (idesc >> 4) & 0x3 == 1               # fp32 accumulator
        assert (idesc >> 7) & 0x7 == bf and (idesc >> 10) & 0x7 == bf
        assert (idesc >> 15) & 0x3 == 0              # both K-major
        assert (idesc >> 17) & 0x3F == n >> 3
        assert (idesc >> 24) & 0x1F == 128 >> 4
