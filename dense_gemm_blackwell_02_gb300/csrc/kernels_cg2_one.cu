// Instantiations of the CTA-pair (cta_group::2) kernel with the single-chain epilogue:
// for products whose every work unit is one accumulation chain (K of at most 4096
// per unit), the accumulator is streamed out of TMEM in 32-column pieces.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_one(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 6) return by_out<2, 256, 6, true, false>(s);
  if (s.bn == 128 && s.stages == 8) return by_out<2, 128, 8, true, false>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
