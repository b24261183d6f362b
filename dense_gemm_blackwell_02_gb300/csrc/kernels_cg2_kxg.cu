// Instantiations of the CTA-pair kernel for the cluster K split with the general
// epilogue (slices of several accumulation chains).
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_kxg(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 7) return by_out<2, 256, 7, false, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 9) return by_out<2, 128, 9, false, false, 0, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
