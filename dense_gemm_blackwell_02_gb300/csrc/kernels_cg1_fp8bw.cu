// Instantiations of the one-CTA (cta_group::1) kernel for FP8 operands with blockwise
// scales (tcgen05.mma kind::f8f6f4, one accumulation chain per 128-element K block,
// scaled in the general epilogue).
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_fp8bw(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, false, 2>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, false, 2>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
