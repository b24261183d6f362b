// Kernel parameter block and device status codes shared by the kernels and the
// host dispatcher (internal; the public interface is include/gemm.h).
#pragma once
#include <cstdint>

namespace gb300 {

// Tile edge along K of one pipeline stage: 64 x 16-bit = 128 bytes, the row of the
// 128-byte swizzle atom ("A Blackwell GEMM by Hand in CuTe DSL", section 6).
constexpr int kBlockK = 64;
// Rows of C per CTA (the M of a cta_group::1 MMA; half of a pair's 256).
constexpr int kBlockM = 128;

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
  kSitePairFull = 7,  // pair: follower signalling
};

struct GemmParams {
  void* C;                 // M x N row-major output
  int32_t M, N, K;
  int32_t num_m_tiles;     // ceil(M / rows per tile)
  int32_t num_n_tiles;     // ceil(N / BN)
  int32_t tiles;           // num_m_tiles * num_n_tiles
  int32_t k_blocks;        // ceil(K / 64)
  int32_t splits;          // K slices per tile (1 = no split)
  int32_t kb_per_split;    // k-blocks per slice (the last slice may be shorter)
  int32_t units;           // tiles * splits
  int32_t group_m;         // grouped rasterisation: M-tiles per group
  int32_t vec_store;       // 1 when 16-byte vector stores of C are aligned
  uint32_t idesc;          // tcgen05 instruction descriptor
  float* workspace;        // splits > 1: fp32 partial tiles
  uint32_t* counters;      // splits > 1: per (tile, row quarter) arrival counters
  uint32_t* status;        // device status word
  uint64_t wait_limit_ns;  // bound on every mbarrier wait
  int32_t test_stall;      // 1: the MMA issuer waits on a barrier that never completes
};

}  // namespace gb300
