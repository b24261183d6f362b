// Dispatch over the instantiated kernel menu.
#include "gemm_kernel.cuh"
#include "launch.h"

namespace gb300 {

// The plain (unsplit or workspace-split) kernels' menu; the cluster K split has its own
// ring depths (kx_stages).  BN 320 exists only for the cluster K split.
bool kernel_supported(int cg, int bn, int stages) {
  if (cg == 1)
    return (bn == 256 && (stages == 4 || stages == 5)) || (bn == 128 && (stages == 6 || stages == 10));
  if (cg == 2) return (bn == 256 && stages == 6) || (bn == 128 && stages == 8) ||
                     (bn == 320 && stages == 6);
  return false;
}

int default_stages(int cg, int bn, bool small_a) {
  if (cg == 1) return bn == 256 ? (small_a ? 5 : 4) : (small_a ? 10 : 6);
  return bn == 320 ? 6 : bn == 256 ? 6 : 8;
}

// The cluster K split keeps its epilogue staging inside the idle ring, which leaves room
// for one more stage (two more of the 16-row A stages).
int kx_stages(int cg, int bn, bool small_a) {
  if (cg == 1) return bn == 256 ? (small_a ? 6 : 4) : (small_a ? 12 : 7);
  return bn == 320 ? 6 : bn == 256 ? 7 : 9;
}

// The swapped tiling writes C with direct stores and keeps no staging boxes, which also
// leaves room for one more stage.
int swap_stages(int bn) { return bn == 256 ? 7 : 9; }

// One-CTA kernels deeper than 7 stages of 128 columns or 4 of 256 hold 16 rows of A per
// stage (the Layout's rule).
int a_rows(int cg, int bn, int stages) {
  if (cg == 1 && ((bn == 128 && stages > 7) || (bn == 256 && stages > 4))) return 16;
  return kBlockM;
}

int max_resident_units(int cg, int bn, int stages, int out) {
  return cg == 1 ? resident_cg1(bn, stages, out) : resident_cg2(bn, stages, out);
}

int max_resident_kx_clusters(int cg, int bn, int stages, int out) {
  return cg == 1 ? resident_cg1_kx(bn, stages, out) : resident_cg2_kx(bn, stages, out);
}

cudaError_t launch_gemm(const LaunchSpec& s) {
  if (s.clc && !s.grouped) return cudaErrorInvalidValue;
  if (s.swap) {
    if (s.kind != 0 || s.fused || s.grouped || s.kx2 || s.staged || s.one_chain || s.cta_group != 2)
      return cudaErrorInvalidValue;
    return launch_cg2_swap(s);
  }
  if (s.kx2) {
    if (s.kind != 0 || s.fused || s.grouped) return cudaErrorInvalidValue;
    if (s.cta_group == 1) return s.one_chain ? launch_cg1_kx(s) : launch_cg1_kxg(s);
    if (s.cta_group == 2) return s.one_chain ? launch_cg2_kx(s) : launch_cg2_kxg(s);
    return cudaErrorInvalidValue;
  }
  if (s.grouped) {
    if (s.kind != 0 || s.fused || s.one_chain) return cudaErrorInvalidValue;
    if (s.cta_group == 1) return s.clc ? launch_cg1_grouped_clc(s) : launch_cg1_grouped(s);
    if (s.cta_group == 2) return s.clc ? launch_cg2_grouped_clc(s) : launch_cg2_grouped(s);
    return cudaErrorInvalidValue;
  }
  if (s.kind == 2) {
    if (s.fused || s.one_chain) return cudaErrorInvalidValue;
    if (s.cta_group == 1) return launch_cg1_fp8bw(s);
    if (s.cta_group == 2) return launch_cg2_fp8bw(s);
    return cudaErrorInvalidValue;
  }
  if (s.kind == 1) {
    if (!s.fused) return cudaErrorInvalidValue;
    if (s.cta_group == 1) return s.one_chain ? launch_cg1_one_fp8(s) : launch_cg1_fp8(s);
    if (s.cta_group == 2) return s.one_chain ? launch_cg2_one_fp8(s) : launch_cg2_fp8(s);
    return cudaErrorInvalidValue;
  }
  if (s.cta_group == 1) {
    if (s.fused) return s.one_chain ? launch_cg1_one_fused(s) : launch_cg1_fused(s);
    if (s.one_chain) return launch_cg1_one(s);
    return s.staged ? launch_cg1_staged(s) : launch_cg1(s);
  }
  if (s.cta_group == 2) {
    if (s.fused) return s.one_chain ? launch_cg2_one_fused(s) : launch_cg2_fused(s);
    if (s.one_chain) return launch_cg2_one(s);
    return s.staged ? launch_cg2_staged(s) : launch_cg2(s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace gb300
