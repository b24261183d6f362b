// Instantiations of the one-CTA kernel for the cluster K split with the general
// epilogue (slices of several accumulation chains).
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_kxg(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 7) return by_out<1, 128, 7, false, false, 0, false, true>(s);
  if (s.bn == 256 && s.stages == 6) return by_out<1, 256, 6, false, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 12) return by_out<1, 128, 12, false, false, 0, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
