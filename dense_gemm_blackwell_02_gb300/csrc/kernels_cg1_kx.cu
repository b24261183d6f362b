// Instantiations of the one-CTA kernel for the cluster K split: two K slices of one
// tile in one cluster of 2 CTAs, reduced through distributed shared memory,
// single-chain and general epilogues.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_kx(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, true, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 7) return by_out<1, 128, 7, true, false, 0, false, true>(s);
  if (s.bn == 256 && s.stages == 6) return by_out<1, 256, 6, true, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 12) return by_out<1, 128, 12, true, false, 0, false, true>(s);
  return cudaErrorInvalidValue;
}

int resident_cg1_kx(int bn, int stages, int out) {
  if (bn == 256 && stages == 4) return resident_by_out<1, 256, 4, true>(out);
  if (bn == 128 && stages == 7) return resident_by_out<1, 128, 7, true>(out);
  if (bn == 256 && stages == 6) return resident_by_out<1, 256, 6, true>(out);
  if (bn == 128 && stages == 12) return resident_by_out<1, 128, 12, true>(out);
  return 0;
}

}  // namespace gb300
