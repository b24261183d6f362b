// Instantiations of the CTA-pair kernel with the operands' roles swapped (B the MMA's
// row operand, a few rows of A its columns; general epilogue, transposed store of C):
// 128 or 256 rows of A per tile.
#include "launch_impl.cuh"

namespace gb300 {

cudaError_t launch_cg2_swap(const LaunchSpec& s) {
  if (s.bn == 128 && s.stages == 9) return by_out<2, 128, 9, false, false, 0, false, false, false, true>(s);
  if (s.bn == 256 && s.stages == 7) return by_out<2, 256, 7, false, false, 0, false, false, false, true>(s);
  return cudaErrorInvalidValue;
}

}  // namespace gb300
