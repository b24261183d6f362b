// Instantiations of the CTA-pair (cta_group::2) kernel for FP8 operands with blockwise
// scales (tcgen05.mma kind::f8f6f4, one accumulation chain per 128-element K block,
// scaled in the general epilogue).
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_fp8bw(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, false, false, 2>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, false, false, 2>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
