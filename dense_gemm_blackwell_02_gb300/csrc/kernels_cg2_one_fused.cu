// Instantiations of the CTA-pair (cta_group::2) kernel with the single-chain epilogue
// and the fused epilogue (alpha, beta * C, bias, ReLU) compiled in.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_one_fused(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, true, true>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, true, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
