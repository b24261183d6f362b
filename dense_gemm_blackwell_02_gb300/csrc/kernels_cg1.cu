// Instantiations of the one-CTA (cta_group::1) kernel: 128 x BN tiles.
// BN = 256: 48 KiB stages x 4; BN = 128: 32 KiB stages x 6 (plus 32 KiB of epilogue
// staging), the budget of "A Blackwell GEMM by Hand in CuTe DSL", section 7.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg1(const LaunchSpec& s) {
  if (s.bn == 256 && s.stages == 4) return by_out<1, 256, 4, false, false>(s);
  if (s.bn == 128 && s.stages == 6) return by_out<1, 128, 6, false, false>(s);
  if (s.bn == 256 && s.stages == 5) return by_out<1, 256, 5, false, false>(s);
  if (s.bn == 128 && s.stages == 10) return by_out<1, 128, 10, false, false>(s);
  return cudaErrorInvalidValue;
}

int resident_cg1(int bn, int stages, int out) {
  if (bn == 256 && stages == 4) return resident_by_out<1, 256, 4>(out);
  if (bn == 128 && stages == 6) return resident_by_out<1, 128, 6>(out);
  if (bn == 256 && stages == 5) return resident_by_out<1, 256, 5>(out);
  if (bn == 128 && stages == 10) return resident_by_out<1, 128, 10>(out);
  return 0;
}

}  // namespace gb300
