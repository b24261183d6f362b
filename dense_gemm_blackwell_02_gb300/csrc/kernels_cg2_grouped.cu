// Instantiations of the CTA-pair (cta_group::2) kernel for grouped launches: per-problem
// tensor maps and shapes from the launch's problem table, whole tiles, general epilogue.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_grouped(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, false, false, 0, true>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, false, false, 0, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
