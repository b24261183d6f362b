// Internal launch interface between the C ABI (gemm_api.cu) and the translation units
// that instantiate the kernel templates.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace gb300 {

struct LaunchSpec {
  int bn;          // columns of C per tile
  int stages;      // operand ring depth
  int out;         // OutKind
  int grid;        // CTAs (a multiple of 2 for the pair kernel)
  CUtensorMap tmA; // A: box {64, rows of A per CTA}
  CUtensorMap tmB; // B: box {64, rows of B per CTA}
  GemmParams p;
  cudaStream_t stream;
};

// One CTA per 128-row tile (cta_group::1).
bool one_cta_supported(int bn, int stages);
size_t one_cta_smem_bytes(int bn, int stages);
cudaError_t launch_one_cta(const LaunchSpec& s);

}  // namespace gb300
