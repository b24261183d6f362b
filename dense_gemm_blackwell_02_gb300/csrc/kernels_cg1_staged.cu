// Instantiations of the cta_group::1 general-epilogue kernel for split launches (K
// slices or stream-K segments meeting in the workspace): the last slice to finish on a
// CTA's last unit stages the other slices' partials in the idle operand ring.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_staged(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, false, 0, false, false, true>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, false, 0, false, false, true>(s);
  if (s.bn == 256 && s.stages == 5) return by_out<1, 256, 5, false, false, 0, false, false, true>(s);
  if (s.bn == 128 && s.stages == 10) return by_out<1, 128, 10, false, false, 0, false, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
