// Instantiations of the one-CTA (cta_group::1) kernel with the single-chain epilogue:
// for products whose every work unit is one accumulation chain (K of at most 4096
// per unit), the accumulator is streamed out of TMEM in 32-column pieces.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1_one(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, true, false>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, true, false>(s);
  if (s.bn == 256 && s.stages == 5) return by_out<1, 256, 5, true, false>(s);
  if (s.bn == 128 && s.stages == 10) return by_out<1, 128, 10, true, false>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
