// Internal launch interface between the C ABI (gemm_api.cu, gemm_noalloc.cu) and the
// translation units that instantiate the kernel templates.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>

#include "params.h"

namespace gb300 {

struct LaunchSpec {
  int cta_group;   // 1: one CTA per 128-row tile; 2: a CTA pair per 256-row tile
  int bn;          // columns of C per tile
  int stages;      // operand ring depth
  int out;         // OutKind
  int grid;        // CTAs (a multiple of cta_group)
  bool one_chain;  // every unit is one accumulation chain (streaming epilogue)
  bool fused;      // the fused epilogue (p.fused) is compiled in
  int kind;        // 0: fp16/bf16 operands (kind::f16); 1: FP8 (kind::f8f6f4, always fused);
                   // 2: FP8 with blockwise scales (general epilogue, not fused)
  bool grouped;    // a grouped launch: p.groups holds the problems (kind 0, general epilogue)
  bool kx2;        // two K slices per tile, one per CTA group of a cluster of 2 * cta_group
                   // (one unit per CTA group)
  bool staged;     // plain general epilogue, K slices or stream-K segments meeting in the
                   // workspace: the kernel with the staged fix-up
  bool swap;       // the swapped tiling: tmA maps B (box p.swap_rows rows), tmB maps A
                   // (box bn / 2 rows), C written transposed by direct stores
  bool clc;        // grouped launches: units handed out by cluster launch control (a CTA or
                   // pair per unit in the grid) instead of round-robin over resident ones
  CUtensorMap tmA; // A: box {128 bytes of K, 128 (or M < 128) rows}
  CUtensorMap tmB; // B: box {128 bytes of K, bn / cta_group}
  CUtensorMap tmB2; // B: box {128 bytes of K, bn / cta_group / 2} (half-tile units; else tmB);
                    // with bn 320, {128 bytes of K, 32 rows}
  CUtensorMap tmC; // C: box {128 bytes of columns, 32 rows} (used when p.tma_store)
  GemmParams p;
  cudaStream_t stream;
};

// The CUDA-core matrix-vector path (gemv_kernel.cu) for M <= kGemvMaxRows rows of A.
constexpr int kGemvMaxRows = 4;
struct GemvSpec {
  const void* A;   // M x K, fp16 or bf16, 16-byte aligned rows
  const void* B;   // N x K
  void* C;         // M x N in `out`
  int32_t M, N;
  int32_t chunks;  // K / 8: 16-byte chunks per row
  bool bf16;       // input type (else fp16)
  int out;         // OutKind
  int grid;        // CTAs (each takes rows blockIdx.x + j * grid of B)
  cudaStream_t stream;
};
cudaError_t launch_gemv(const GemvSpec& s);

// The instantiated (cta_group, bn, stages) menu.
bool kernel_supported(int cta_group, int bn, int stages);
// small_a: a one-CTA row tile of at most 16 rows (the ring then holds 16 rows of A per
// stage and is deeper)
int default_stages(int cta_group, int bn, bool small_a = false);
// the ring depth of the cluster-K-split kernels (their staging lies inside the ring)
int kx_stages(int cta_group, int bn, bool small_a = false);
int swap_stages(int bn);  // the swapped tiling's ring depth
int a_rows(int cta_group, int bn, int stages);  // A rows a stage of that kernel holds
// Clusters (CTAs for cta_group 1) of this configuration that can be resident at once
// on the current device; 0 if the query fails.
int max_resident_units(int cta_group, int bn, int stages, int out);
cudaError_t launch_gemm(const LaunchSpec& s);

// Per-translation-unit launchers (kernels_cg1.cu, kernels_cg2.cu: the general
// epilogue; kernels_cg1_one.cu, kernels_cg2_one.cu: single-chain units).
cudaError_t launch_cg1(const LaunchSpec& s);
cudaError_t launch_cg2(const LaunchSpec& s);
cudaError_t launch_cg1_one(const LaunchSpec& s);
cudaError_t launch_cg2_one(const LaunchSpec& s);
// ... and with the fused epilogue (kernels_cg*_fused.cu)
cudaError_t launch_cg1_fused(const LaunchSpec& s);
cudaError_t launch_cg2_fused(const LaunchSpec& s);
cudaError_t launch_cg1_one_fused(const LaunchSpec& s);
cudaError_t launch_cg2_one_fused(const LaunchSpec& s);
// ... and with FP8 operands (kernels_cg*_fp8.cu; the fused epilogue carries the scales)
cudaError_t launch_cg1_fp8(const LaunchSpec& s);
cudaError_t launch_cg2_fp8(const LaunchSpec& s);
cudaError_t launch_cg1_one_fp8(const LaunchSpec& s);
cudaError_t launch_cg2_one_fp8(const LaunchSpec& s);
// ... and FP8 with blockwise scales (kernels_cg*_fp8bw.cu)
cudaError_t launch_cg1_fp8bw(const LaunchSpec& s);
cudaError_t launch_cg2_fp8bw(const LaunchSpec& s);
// ... and grouped launches (kernels_cg*_grouped.cu)
cudaError_t launch_cg1_grouped(const LaunchSpec& s);
cudaError_t launch_cg2_grouped(const LaunchSpec& s);
cudaError_t launch_cg1_grouped_clc(const LaunchSpec& s);  // ... scheduled by cluster launch control
cudaError_t launch_cg2_grouped_clc(const LaunchSpec& s);
// ... and the cluster K split (kernels_cg*_kx.cu)
cudaError_t launch_cg1_kx(const LaunchSpec& s);
cudaError_t launch_cg2_kx(const LaunchSpec& s);
cudaError_t launch_cg1_kxg(const LaunchSpec& s);  // general epilogue
cudaError_t launch_cg1_staged(const LaunchSpec& s);  // general epilogue, staged fix-up
cudaError_t launch_cg2_staged(const LaunchSpec& s);
cudaError_t launch_cg2_swap(const LaunchSpec& s);  // the swapped tiling (kernels_cg2_swap.cu)
cudaError_t launch_cg2_kxg(const LaunchSpec& s);
int resident_cg1_kx(int bn, int stages, int out);
int resident_cg2_kx(int bn, int stages, int out);
// Clusters of 2 * cta_group CTAs of the cluster-K-split kernel that fit at once (0 if the
// query fails).
int max_resident_kx_clusters(int cta_group, int bn, int stages, int out);
int resident_cg1(int bn, int stages, int out);
int resident_cg2(int bn, int stages, int out);

}  // namespace gb300
