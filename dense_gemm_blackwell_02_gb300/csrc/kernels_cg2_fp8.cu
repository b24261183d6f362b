// Instantiations of the CTA-pair (cta_group::2) kernel for FP8 operands (tcgen05.mma
// kind::f8f6f4) with the general epilogue and the fused epilogue, which applies
// the per-tensor scale product as alpha.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_fp8(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, false, true, 1>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, false, true, 1>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
