// Instantiations of the one-CTA kernel for grouped launches scheduled by cluster launch
// control: a CTA per tile in the grid, running CTAs taking over the tiles of launches that
// have not started.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_grouped_clc(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, false, 0, true, false, false, false, true>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, false, 0, true, false, false, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
