// Instantiations of the one-CTA (cta_group::1) kernel with the general epilogue
// and the fused epilogue (alpha, beta * C, bias, ReLU) compiled in.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_fused(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, true>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
