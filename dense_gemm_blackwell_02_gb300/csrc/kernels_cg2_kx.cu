// Instantiations of the CTA-pair kernel for the cluster K split: two K slices of one
// tile in one cluster of 4 CTAs, reduced through distributed shared memory,
// single-chain and general epilogues.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_kx(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 7) return by_out<2, 256, 7, true, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 9) return by_out<2, 128, 9, true, false, 0, false, true>(s);
  if (s.bn == 320 && s.stages == 6) return by_out<2, 320, 6, true, false, 0, false, true>(s);
  return cudaErrorInvalidValue;
}

int resident_cg2_kx(int bn, int stages, int out) {
  if (bn == 256 && stages == 7) return resident_by_out<2, 256, 7, true>(out);
  if (bn == 128 && stages == 9) return resident_by_out<2, 128, 9, true>(out);
  if (bn == 320 && stages == 6) return resident_by_out<2, 320, 6, true>(out);
  return 0;
}

}  // namespace gb300
