// Kernel parameter block and device status codes shared by the kernels and the
// host dispatcher (internal; the public interface is include/gemm.h).
#pragma once
#include <cuda.h>

#include <cstdint>

namespace gb300 {

// Tile edge along K of one pipeline stage: 64 x 16-bit = 128 bytes, the row of the
// 128-byte swizzle atom ("A Blackwell GEMM by Hand in CuTe DSL", section 6).
constexpr int kBlockK = 64;
// Rows of C per CTA (the M of a cta_group::1 MMA; half of a pair's 256).
constexpr int kBlockM = 128;
// Longest run of k-blocks accumulated in one TMEM accumulator before the epilogue
// folds it into its fp32 registers (64 x 64 = K 4096).  The tensor core's fp32
// accumulation error grows linearly with the length of one accumulation chain
// (measured: relative Frobenius error 4.0e-6 at K = 4096, 1.8e-5 at 16384, 3.2e-5
// at 28672 for U[-1,1] inputs); capping the chain keeps it near the K = 4096 value.
constexpr int kChainKBlocks = 64;

enum OutKind : int { kOutF16 = 0, kOutBF16 = 1, kOutF32 = 2 };

// Device status word: 0 = fine; otherwise (code << 24) | (site << 16) | blockIdx.x.
enum DeviceCode : uint32_t { kDevTimeout = 1u };
enum WaitSite : uint32_t {
  kSiteEmpty = 1,     // producer waiting for a free stage
  kSiteFull = 2,      // MMA issuer waiting for a loaded stage
  kSiteAccEmpty = 3,  // MMA issuer waiting for a drained accumulator slot
  kSiteAccFull = 4,   // epilogue waiting for a finished accumulator
  kSiteTestStall = 5, // deliberate wait on a barrier nothing arrives on (test only)
  kSiteDrain = 6,     // teardown: outstanding copies / MMAs
  kSiteKx = 7,        // two-slice exchange through distributed shared memory
  kSiteClc = 8,       // cluster launch control: a free answer slot, or the next answer
};

// One problem of a grouped launch ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell
// tcgen05", Part 6, Grouped GEMM: each tile fetches its problem's pointers and tensor
// maps).  Written by the host into device memory; aligned as its tensor maps require.
struct GroupDesc {
  CUtensorMap tmA;        // A_g: box {128 bytes of K, 128 (or M_g < 128) rows}
  CUtensorMap tmB;        // B_g: box {128 bytes of K, BN / CTA_GROUP rows}
  CUtensorMap tmC;        // C_g: box {128 bytes of columns, 32 rows} (when tma_store)
  void* C;
  int32_t M, N, K;
  int32_t k_blocks;       // ceil(K_g / K block)
  int32_t num_m, num_n;   // tiles of this problem along M and N
  uint32_t a_tx_short;    // as GemmParams::a_tx_short, for this problem
  int32_t vec_store;      // 16-byte vector stores of C_g are aligned
  int32_t tma_store;      // C_g is written through tmC
};

struct GemmParams {
  void* C;                 // M x N row-major output
  int32_t M, N, K;
  int32_t num_m_tiles;     // ceil(M / rows per tile); a tile is 128 * CTA_GROUP rows
  int32_t num_n_tiles;     // ceil(N / BN)
  int32_t tiles;           // num_m_tiles * num_n_tiles
  int32_t k_blocks;        // ceil(K / 64)
  int32_t dp_tiles;        // tiles [0, dp_tiles) run whole, one unit each
  int32_t half_tail;       // 1: each later tile runs as two BN/2-column halves (full K)
  int32_t splits;          // otherwise: K slices of each later tile (1 = no split)
  int32_t kb_per_split;    // k-blocks per slice (the last slice may be shorter)
  int32_t units;           // dp_tiles + (tiles - dp_tiles) * (half_tail ? 2 : splits)
  int32_t sk_workers;      // > 0: tiles after dp_tiles go to stream-K over this many units
  int32_t ws_slots;        // partial-tile slots per cut tile in the workspace
  int32_t group_m;         // grouped rasterisation: M-tiles per group
  int32_t chain_kb;        // k-blocks per TMEM accumulation chain
  int32_t prefetch_kb;     // L2 prefetch of B this many k-blocks ahead of the ring (0: off)
  int32_t l2_hint;         // 2: B's loads evict-first and A's evict-last in L2; else none
  uint32_t a_tx_short;     // bytes of A's 128-row box that A's tensor map does not load:
                           // (128 - M) * 128 when a one-CTA tile's A box is M < 128 rows
                           // (for the pair in the swapped tiling: 2 * (128 - swap_rows) * 128)
  int32_t swap_rows;       // swapped tiling (B is the MMA's row operand): B rows per CTA
  int32_t vec_store;       // 1 when 16-byte vector stores of C are aligned
  int32_t tma_store;       // 1 when C is written through the C tensor map
  uint32_t idesc;          // tcgen05 instruction descriptor (N = BN)
  uint32_t idesc_half;     // the same for N = BN / 2 (half-tile units)
  float* workspace;        // splits > 1: fp32 partial tiles
  uint32_t* counters;      // splits > 1: per (tile, CTA of the pair, quarter, half) counters
  uint32_t* status;        // device status word
  // fused epilogue, fused = 0: C = A . B^T; else C = act(alpha * A . B^T + beta * C + bias)
  int32_t fused;
  int32_t relu;            // act: ReLU when 1, the identity when 0
  float alpha, beta;
  const float* bias;       // N values (16-byte aligned), or nullptr
  // blockwise FP8 scales (KIND 2), K-block-major: sfa[kb * sf_lda + m / sf_bm],
  // sfb[kb * sf_ldb + n / 128]
  const float* sfa;
  const float* sfb;
  int32_t sf_bm, sf_lda, sf_ldb;
  // grouped launches (GROUPED kernels): problem g owns units [group_start[g],
  // group_start[g + 1]); units = group_start[num_groups]
  const GroupDesc* groups;
  const int32_t* group_start;
  int32_t num_groups;
  uint64_t wait_limit_ns;  // bound on every mbarrier wait
  int32_t test_stall;      // 1: the MMA issuer waits on a barrier that never completes
};

}  // namespace gb300
