// Instantiations of the one-CTA (cta_group::1) kernel for grouped launches: per-problem
// tensor maps and shapes from the launch's problem table, whole tiles, general epilogue.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_grouped(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, false, 0, true>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, false, 0, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
