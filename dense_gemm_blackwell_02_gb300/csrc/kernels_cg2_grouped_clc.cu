// Instantiations of the CTA-pair kernel for grouped launches scheduled by cluster launch
// control: a pair per tile in the grid, running pairs taking over the tiles of pair
// launches that have not started.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_grouped_clc(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, false, false, 0, true, false, false, false, true>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, false, false, 0, true, false, false, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
