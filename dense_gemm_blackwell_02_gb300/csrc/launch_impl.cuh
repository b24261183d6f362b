// Template launcher shared by the per-cta_group instantiation files.
#pragma once
#include "gemm_kernel.cuh"
#include "launch.h"

namespace gb300 {

template <int CG, int BN, int STAGES, int OUT, bool ONE, bool FUSED, int KIND = 0,
          bool GROUPED = false, bool KX2 = false, bool STAGED = false, bool SWAP = false,
          bool CLC = false>
cudaError_t launch_one(const LaunchSpec& s) {
  auto kernel = gemm_kernel<CG, BN, STAGES, OUT, ONE, FUSED, KIND, GROUPED, KX2, STAGED, SWAP, CLC>;
  constexpr unsigned kCluster = CG * (KX2 ? 2 : 1);
  using L = Layout<CG, BN, STAGES, KX2, SWAP>;
  cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kDynamicBytes);
  if (e != cudaSuccess) return e;
  if (kCluster > 1) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(s.grid, 1, 1);
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kDynamicBytes;
  cfg.stream = s.stream;
  cudaLaunchAttribute attr[2];
  unsigned n = 0;
  // Programmatic dependent launch: the kernel's setup may overlap the preceding
  // kernel's tail; the kernel waits for it (griddepcontrol.wait) before touching
  // global memory.
  attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[n].val.programmaticStreamSerializationAllowed = 1;
  ++n;
  if (kCluster > 1) {
    attr[n].id = cudaLaunchAttributeClusterDimension;
    attr[n].val.clusterDim.x = kCluster;
    attr[n].val.clusterDim.y = 1;
    attr[n].val.clusterDim.z = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, s.tmA, s.tmB, s.tmB2, s.tmC, s.p);
}

template <int CG, int BN, int STAGES, int OUT, bool KX2 = false>
int resident_one() {
  auto kernel = gemm_kernel<CG, BN, STAGES, OUT, KX2, false, 0, false, KX2, false>;
  constexpr unsigned kCluster = CG * (KX2 ? 2 : 1);
  using L = Layout<CG, BN, STAGES, KX2>;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           L::kDynamicBytes) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2 * kCluster, 1, 1);
  cfg.blockDim = dim3(L::kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kDynamicBytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kCluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

template <int CG, int BN, int STAGES, bool ONE, bool FUSED, int KIND = 0, bool GROUPED = false,
          bool KX2 = false, bool STAGED = false, bool SWAP = false, bool CLC = false>
cudaError_t by_out(const LaunchSpec& s) {
  switch (s.out) {
    case kOutF16: return launch_one<CG, BN, STAGES, kOutF16, ONE, FUSED, KIND, GROUPED, KX2, STAGED, SWAP, CLC>(s);
    case kOutBF16: return launch_one<CG, BN, STAGES, kOutBF16, ONE, FUSED, KIND, GROUPED, KX2, STAGED, SWAP, CLC>(s);
    case kOutF32: return launch_one<CG, BN, STAGES, kOutF32, ONE, FUSED, KIND, GROUPED, KX2, STAGED, SWAP, CLC>(s);
    default: return cudaErrorInvalidValue;
  }
}

template <int CG, int BN, int STAGES, bool KX2 = false>
int resident_by_out(int out) {
  switch (out) {
    case kOutF16: return resident_one<CG, BN, STAGES, kOutF16, KX2>();
    case kOutBF16: return resident_one<CG, BN, STAGES, kOutBF16, KX2>();
    case kOutF32: return resident_one<CG, BN, STAGES, kOutF32, KX2>();
    default: return 0;
  }
}

}  // namespace gb300
