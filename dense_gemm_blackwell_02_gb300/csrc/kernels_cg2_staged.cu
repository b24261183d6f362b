// Instantiations of the cta_group::2 general-epilogue kernel for split launches (K
// slices or stream-K segments meeting in the workspace): the last slice to finish on a
// CTA's last unit stages the other slices' partials in the idle operand ring.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_staged(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, false, false, 0, false, false, true>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, false, false, 0, false, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
