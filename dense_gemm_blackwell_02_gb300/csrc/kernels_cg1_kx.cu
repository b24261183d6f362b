// Instantiations of the one-CTA kernel for the cluster K split: two K slices of one
// tile in one cluster of 2 CTAs, reduced through distributed shared memory,
// single-chain and general epilogues.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_kx(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, true, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, true, false, 0, false, true>(s);
  if (s.bn == 256 && s.stages == 5) return by_out<1, 256, 5, true, false, 0, false, true>(s);
  if (s.bn == 128 && s.stages == 10) return by_out<1, 128, 10, true, false, 0, false, true>(s);
  return cudaErrorInvalidValue;
}

int resident_cg1_kx(int bn, int stages, int out) {
  if (bn == 256 && stages == 4) return resident_by_out<1, 256, 4, true>(out);
  if (bn == 128 && stages == 6) return resident_by_out<1, 128, 6, true>(out);
  if (bn == 256 && stages == 5) return resident_by_out<1, 256, 5, true>(out);
  if (bn == 128 && stages == 10) return resident_by_out<1, 128, 10, true>(out);
  return 0;
}

}  // namespace gb300
