// Instantiations of the one-CTA (cta_group::1) kernel for FP8 operands (tcgen05.mma
// kind::f8f6f4) with the general epilogue and the fused epilogue, which applies
// the per-tensor scale product as alpha.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_fp8(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, true, 1>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, true, 1>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
