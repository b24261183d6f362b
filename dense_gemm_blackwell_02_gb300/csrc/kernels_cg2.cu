// Instantiations of the CTA-pair (cta_group::2) kernel: 256 x BN tiles, each CTA
// holding half of B per stage.  BN = 256: 32 KiB stages x 6; BN = 128: 24 KiB x 8.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, false, false>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, false, false>(s);
  return cudaErrorInvalidValue;
}

int resident_cg2(int bn, int stages, int out) {
  if (bn == 256 && stages == 6) return resident_by_out<2, 256, 6>(out);
  if (bn == 128 && stages == 8) return resident_by_out<2, 128, 8>(out);
  return 0;
}

}  // namespace gb300
