// Instantiations of the one-CTA (cta_group::1) kernel and its launcher.
#include "gemm_kernel.cuh"
#include "launch.h"

namespace gb300 {
namespace {

template <int BN, int STAGES, int OUT>
cudaError_t launch_impl(const LaunchSpec& s) {
  auto kernel = gemm_1cta_kernel<BN, STAGES, OUT>;
  constexpr uint32_t smem = SmemLayout1<BN, STAGES>::kDynamicBytes;
  cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.grid, 1, 1);
  cfg.blockDim = dim3(kThreads1, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s.stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kernel, s.tmA, s.tmB, s.p);
}

template <int BN, int STAGES>
cudaError_t by_out(const LaunchSpec& s) {
  switch (s.out) {
    case kOutF16: return launch_impl<BN, STAGES, kOutF16>(s);
    case kOutBF16: return launch_impl<BN, STAGES, kOutBF16>(s);
    case kOutF32: return launch_impl<BN, STAGES, kOutF32>(s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace

// Instantiated (BN, stages): 48 KiB stages x 4 at BN = 256, 32 KiB stages x 6 at 128
// ("A Blackwell GEMM by Hand in CuTe DSL", section 7: at most 4 such 1-CTA stages fit).
bool one_cta_supported(int bn, int stages) {
  return (bn == 256 && stages == 4) || (bn == 128 && stages == 6);
}

size_t one_cta_smem_bytes(int bn, int stages) {
  if (bn == 256 && stages == 4) return SmemLayout1<256, 4>::kDynamicBytes;
  if (bn == 128 && stages == 6) return SmemLayout1<128, 6>::kDynamicBytes;
  return 0;
}

cudaError_t launch_one_cta(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<256, 4>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<128, 6>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
