// Instantiations of the CTA-pair kernel with A multicast across the two pairs of a
// 4-CTA cluster (two tiles of the same rows side by side, whole tiles): single-chain and
// general epilogues, BN 256 and 128.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_mca(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) {
    return s.one_chain ? by_out<2, 256, 6, true, false, 0, false, false, false, true>(s)
                       : by_out<2, 256, 6, false, false, 0, false, false, false, true>(s);
  }
  if (s.bn == 128 && s.stages == 8) {
    return s.one_chain ? by_out<2, 128, 8, true, false, 0, false, false, false, true>(s)
                       : by_out<2, 128, 8, false, false, 0, false, false, false, true>(s);
  }
  return cudaErrorInvalidValue;
}

int resident_cg2_mca(int bn, int stages, int out) {
  if (bn == 256 && stages == 6) return resident_by_out<2, 256, 6, false, true>(out);
  if (bn == 128 && stages == 8) return resident_by_out<2, 128, 8, false, true>(out);
  return 0;
}

}  // namespace gb300
