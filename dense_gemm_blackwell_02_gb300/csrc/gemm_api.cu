// C ABI of libgemm.so (declared in include/gemm.h): argument validation, the
// shape -> kernel-configuration heuristic, TMA tensor-map encoding with a small
// cache, workspace management, launch, and the device status word.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "gemm.h"
#include "launch.h"
#include "umma.cuh"

using namespace gb300;

namespace {

constexpr int kTmapCacheSize = 16;
// A single row of A takes the matrix-vector path without being asked when K is at most
// this (measured back to back, M = 1: 8192 x 8192 27.5 us against 28.9 on the tensor
// cores, 28672 x 8192 74.5 against 81.4, 4096 x 4096 9.0 against 13.9, 14336 x 4096
// 22.1 against 25.7; but 8192 x 28672 85.0 against 83.9, and with two or more rows of
// A the tensor cores win: 2 x 8192 x 8192 30.4 against 28.7).
constexpr int64_t kGemvAutoMaxK = 16384;

struct TmapKey {
  const void* ptr;
  int64_t rows, cols;
  int32_t dtype, box_rows;
  bool operator==(const TmapKey& o) const {
    return ptr == o.ptr && rows == o.rows && cols == o.cols && dtype == o.dtype &&
           box_rows == o.box_rows;
  }
};

struct TmapEntry {
  TmapKey key;
  CUtensorMap map;
  bool valid;
};

}  // namespace

struct gemm_ctx {
  int device = 0;
  cudaError_t last_cuda = cudaSuccess;  // the CUDA error behind the last GEMM_ERR_CUDA launch
  int sms = 0;
  uint32_t* d_status = nullptr;
  float* d_ws = nullptr;
  size_t ws_bytes = 0;
  uint32_t* d_ctr = nullptr;
  size_t ctr_count = 0;
  void* d_stage[3] = {nullptr, nullptr, nullptr};  // gemm_run_host: A, B, C
  size_t stage_bytes[3] = {0, 0, 0};
  gemm_config_t forced = {};
  gemm_config_t last = {};
  uint64_t wait_limit_ns = 2000000000ull;
  int32_t test_stall = 0;
  TmapEntry cache[kTmapCacheSize] = {};
  int cache_next = 0;
  int resident[2][2][2][3] = {};  // [cta_group-1][bn==256][small A][out]: co-resident units (0: unknown)
  // gemm_plan: a device described instead of queried (resident CTA pairs, and clusters of
  // four CTAs for the pair's cluster K split); the GPU is never touched
  bool model = false;
  int model_pairs = 0, model_clusters4 = 0;
  // grouped launches: a ring of problem tables (pinned host copy, device copy and the
  // event that marks the host copy reusable)
  static constexpr int kGroupRing = 4;
  GroupDesc* h_groups[kGroupRing] = {};
  GroupDesc* d_groups[kGroupRing] = {};
  int32_t* h_gstart[kGroupRing] = {};
  int32_t* d_gstart[kGroupRing] = {};
  cudaEvent_t group_done[kGroupRing] = {};
  size_t group_cap[kGroupRing] = {};
  int group_next = 0;
  // gemm_run_host: copy streams and the events that order the chunks of the pipeline
  static constexpr int kHostChunks = 8;
  cudaStream_t copy_in = nullptr, copy_out = nullptr;
  cudaEvent_t host_ev[2 + 3 * kHostChunks] = {};
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  }
  return fn;
}

bool is_fp8(int d) { return d == GEMM_E4M3 || d == GEMM_E5M2; }

// 2-D tensor map over a row-major rows x cols matrix, 128-byte swizzle, box of 128
// bytes of columns x box_rows rows.  Loads read out-of-range elements as zero (M, N and
// K tails); stores skip them.
bool make_map(gemm_ctx* h, const void* ptr, int64_t rows, int64_t cols, int dtype,
              int box_rows, CUtensorMap* out) {
  const TmapKey key{ptr, rows, cols, dtype, box_rows};
  for (auto& e : h->cache)
    if (e.valid && e.key == key) {
      *out = e.map;
      return true;
    }
  auto fn = encode_fn();
  if (!fn) return false;
  CUtensorMap m;
  const cuuint64_t esz = dtype == GEMM_F32 ? 4 : is_fp8(dtype) ? 1 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = dtype == GEMM_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                 : is_fp8(dtype)     ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  CUresult r = fn(&m, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  TmapEntry& slot = h->cache[h->cache_next];
  h->cache_next = (h->cache_next + 1) % kTmapCacheSize;
  slot.key = key;
  slot.map = m;
  slot.valid = true;
  *out = m;
  return true;
}

int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

size_t out_size(gemm_dtype_t d) { return d == GEMM_F32 ? 4 : 2; }

bool valid_dtype(int d) { return d >= GEMM_F16 && d <= GEMM_E5M2; }

size_t in_size(gemm_dtype_t d) { return is_fp8(d) ? 1 : 2; }

struct Choice {
  int variant, bn, stages, splits, kb_per_split, group_m, grid, chain_kb, half_tail, prefetch_kb;
  int l2_hint;
  bool one_chain;
  bool kx2;  // the two K slices of a tile reduced inside a cluster (single chain)
  bool swap;      // the swapped tiling: B the MMA's row operand, swap_rows rows per CTA
  int swap_rows;
  int64_t tiles, dp_tiles, units, k_blocks, num_m, num_n;
  int64_t sk_workers, ws_slots;
};

int out_kind(gemm_dtype_t d) { return d == GEMM_F16 ? kOutF16 : d == GEMM_BF16 ? kOutBF16 : kOutF32; }

// Units of this configuration that can run at once: CTAs (variant 1) or CTA pairs
// (variant 2), from the occupancy query, at most one CTA per SM.
int resident_units(gemm_ctx* h, int cg, int bn, int stages, int out) {
  if (h->model) return cg == 1 ? h->sms : std::min(h->model_pairs, h->sms / 2);
  int& slot = h->resident[cg - 1][bn == 256 ? 1 : 0][a_rows(cg, bn, stages) < kBlockM ? 1 : 0][out];
  if (slot == 0) {
    int n = max_resident_units(cg, bn, stages, out);
    const int cap = h->sms / cg;
    slot = (n <= 0 || n > cap) ? cap : n;
  }
  return slot;
}

// Clusters of the cluster K split that can be resident at once (pairs: clusters of four
// CTAs; one CTA: clusters of two).
int kx_clusters(gemm_ctx* h, int cg, int bn, int stages, int out) {
  if (h->model) return cg == 1 ? h->sms / 2 : h->model_clusters4;
  return max_resident_kx_clusters(cg, bn, stages, out);
}

// The default accumulation chain: K 4096 elements, 64 blocks of fp16/bf16, 32 of FP8.
int64_t chain_kb_of(int kb_elems) { return kChainKBlocks * kBlockK / kb_elems; }

// kb_elems: K elements per 128-byte K block (64 fp16/bf16, 128 FP8).
// blockwise: one accumulation chain per K block (scaled in the general epilogue).
// allow_kx: the cluster K split and the staged stream-K fix-up have kernels for this call
// (fp16/bf16, plain epilogue).
// The swapped tiling for a few rows of A ("A Blackwell GEMM by Hand in CuTe DSL", section
// 9: decode shapes are decided by how many SMs the tiles occupy).  B's rows are the MMA's
// 128-row operand (swap_rows of them loaded per CTA), A's rows its columns (block_n per
// tile, half of them loaded by each CTA of the pair), so that a handful of token rows
// times thousands of weight rows fill every SM in one wave without cutting K.
gemm_status_t choose_swap(gemm_ctx* h, int64_t M, int64_t N, int64_t K, int out, int kb_elems,
                          Choice* c) {
  const gemm_config_t& f = h->forced;
  if ((f.variant && f.variant != 2) || (f.splits && f.splits != 1) || f.epilogue > 1 ||
      f.block_n == 320)
    return GEMM_ERR_UNSUPPORTED;
  c->variant = 2;
  c->bn = f.block_n ? f.block_n : 128;
  if (c->bn != 128 && c->bn != 256) return GEMM_ERR_INVALID_ARG;
  c->stages = f.stages ? f.stages : swap_stages(c->bn);
  if (c->stages != swap_stages(c->bn)) return GEMM_ERR_INVALID_ARG;
  c->k_blocks = ceil_div(K, (int64_t)kb_elems);
  // (one CTA per SM in pairs, like the plain pair kernel of this width, whose count stands in)
  int64_t pairs = resident_units(h, 2, c->bn, default_stages(2, c->bn), out);
  if (f.max_ctas) pairs = std::min<int64_t>(pairs, std::max<int64_t>(f.max_ctas / 2, 1));
  c->num_n = ceil_div(M, (int64_t)c->bn);  // tiles along A's rows
  int64_t w = f.swap_rows;
  if (!w) {
    // the fewest B rows per CTA that make one wave: as many blocks of B rows as pairs
    // are left per tile of A rows
    const int64_t blocks = std::max<int64_t>(1, pairs / c->num_n);
    w = std::min<int64_t>(128, ceil_div(ceil_div(N, 2 * blocks), (int64_t)8) * 8);
  }
  c->swap = true;
  c->swap_rows = (int)w;
  c->num_m = ceil_div(N, 2 * w);           // tiles along B's rows
  c->tiles = c->num_m * c->num_n;
  c->dp_tiles = c->tiles;
  c->units = c->tiles;
  c->splits = 1;
  c->kb_per_split = (int)c->k_blocks;
  c->half_tail = 0;
  c->sk_workers = 0;
  c->ws_slots = 1;
  c->group_m = f.group_m ? f.group_m : 16;
  c->chain_kb = f.chain_kblocks ? f.chain_kblocks : chain_kb_of(kb_elems);
  c->prefetch_kb = f.prefetch_kblocks > 0 ? f.prefetch_kblocks : 0;
  // One tile of A rows, or one wave: every B element is read once, or by every tile of A
  // rows at about the same time, and A by every tile, so B's lines are marked first to be
  // evicted and A's last (as for one row of tiles otherwise; 256 x 8192 x 8192, one wave
  // of two tiles of A rows: 31.9 us against 33.3 without the hints).
  c->l2_hint = f.l2_hint ? f.l2_hint : (c->num_n == 1 || c->tiles <= pairs ? 2 : 1);
  c->one_chain = false;
  c->kx2 = false;
  c->grid = (int)(std::min<int64_t>(c->units, pairs) * 2);
  if (c->units > INT32_MAX || c->tiles * 16 > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  return GEMM_OK;
}

gemm_status_t choose_plain(gemm_ctx* h, int64_t M, int64_t N, int64_t K, int out, int kb_elems,
                           bool blockwise, bool allow_kx, Choice* c) {
  const gemm_config_t& f = h->forced;
  c->swap = false;
  c->swap_rows = 0;
  // A CTA pair (256-row tiles, each CTA loading half of B) whenever M fills one.
  // Blockwise scales hand every K block's accumulator to the epilogue and back: one CTA
  // per 128 x 128 tile, whose kernel keeps four accumulator slots (so the MMAs run up to
  // three K blocks ahead of the scaling) where 256 columns leave room for two (measured,
  // E4M3 -> bf16, one GB300: 4096^3 106.0 us against 114.8 for 128 x 256 and 102.4 for a
  // pair's 256 x 128; 8192^3 687.9 against 679.9 and 827.5).
  c->variant = f.variant ? f.variant : (M > kBlockM && !blockwise ? 2 : 1);
  const int cg = c->variant;
  c->bn = f.block_n ? f.block_n : (N <= 128 || blockwise ? 128 : 256);
  // A row tile of at most 16 rows holds 16 rows of A per stage and a deeper ring (the
  // plain fp16/bf16 kernels)
  const bool small_a = cg == 1 && M <= 16 && allow_kx;
  c->stages = f.stages ? f.stages : default_stages(cg, c->bn, small_a);
  if (!kernel_supported(cg, c->bn, c->stages)) return GEMM_ERR_INVALID_ARG;
  c->k_blocks = ceil_div(K, (int64_t)kb_elems);
  c->num_m = ceil_div(M, (int64_t)kBlockM * cg);
  c->num_n = ceil_div(N, c->bn);
  c->tiles = c->num_m * c->num_n;
  int64_t slots = resident_units(h, cg, c->bn, c->stages, out);
  if (f.max_ctas) slots = std::min<int64_t>(slots, std::max<int64_t>(f.max_ctas / cg, 1));
  // Too few 256-column tiles for the SMs, but 128-column tiles fill more than half of
  // one wave:
  // with K of at most 8192 the narrower tiles without a K split beat splitting K
  // (measured, 256 x 8192 x 8192: 38.3 us against 40.5 us for two K slices, whose
  // hand-over of fp32 partials costs several microseconds at the end).  For longer K the
  // hand-over is amortised and split-K wins (256 x 8192 x 28672: 98 against 110 us).
  // With one CTA per 128-row tile (M <= 128), 128-column tiles are taken whenever they
  // need fewer K slices than 256-column ones, for any K (measured, M = 8..128,
  // N = 8192: K 8192, 32 against 38 us; K 28672, 84 against 91 us).
  if (!f.block_n && !f.splits && !f.stages && c->bn == 256 && c->tiles * 2 <= slots &&
      (c->k_blocks <= 128 || cg == 1)) {
    const int64_t tiles128 = c->num_m * ceil_div(N, (int64_t)128);
    const int64_t slots128 = [&] {
      int64_t n = resident_units(h, cg, 128, default_stages(cg, 128, small_a), out);
      if (f.max_ctas) n = std::min<int64_t>(n, std::max<int64_t>(f.max_ctas / cg, 1));
      return n;
    }();
    const auto slices = [&](int64_t tiles, int64_t sl) {
      return tiles * 2 <= sl ? std::min<int64_t>({sl / tiles, c->k_blocks / 4, 32}) : 1;
    };
    const bool fewer = cg == 1 ? slices(tiles128, slots128) < slices(c->tiles, slots)
                               : tiles128 * 2 > slots128;
    if (tiles128 <= slots128 && fewer) {
      c->bn = 128;
      c->stages = default_stages(cg, 128, small_a);
      c->num_n = ceil_div(N, (int64_t)128);
      c->tiles = tiles128;
      slots = slots128;
    }
  }
  // CTA pairs whose 256-column tiles fall short of one wave while 128-column tiles fill
  // one wave and at most 30% of a second, with tiles of several accumulation chains:
  // 128-column tiles, for the stream-K rule below to spread over every pair (measured
  // back to back: 256 x 10240 x 8192 37.7 us against 39.7 for 320-column cluster-split
  // tiles; 256 x 12288 x 8192 43.6 against 45.7 for a partial wave of whole 256-column
  // tiles; 256 x 10240 x 16384 66.5 against 78.8; equal at 256 x 11264 x 8192; at 1.47
  // waves, 256 x 14336 x 8192, whole 256-column tiles stay ahead: 48.7 against 49.6).
  bool sk_narrow = false;
  if (cg == 2 && allow_kx && !f.block_n && !f.splits && !f.stages && !f.epilogue &&
      !f.chain_kblocks && !f.max_ctas && c->bn == 256 && c->tiles < slots &&
      c->k_blocks > chain_kb_of(kb_elems)) {
    const int64_t tiles128 = c->num_m * ceil_div(N, (int64_t)128);
    const int64_t slots128 = resident_units(h, cg, 128, default_stages(cg, 128, small_a), out);
    if (tiles128 > slots128 && 10 * tiles128 <= 13 * slots128) {
      c->bn = 128;
      c->stages = default_stages(cg, 128, small_a);
      c->num_n = ceil_div(N, (int64_t)128);
      c->tiles = tiles128;
      slots = slots128;
      sk_narrow = true;
    }
  }
  // The cluster K split: when one of the two tile widths gives exactly two K slices of
  // single chains for a wave, those slices meet in distributed shared memory rather than
  // in the global workspace (measured, back to back: 256 x 4096 x 4096 16.7 us against
  // 22.2 for four slices of 256-column tiles; 256 x 8192 x 8192 34.9 us against 36.5 for
  // unsplit 128-column tiles; M <= 128, 8192 x 8192: 28-30 us against 30-32 for two
  // slices through the workspace; slices of several chains too: 256 x 8192 x 28672
  // 93.7 us against 96.2, M <= 128 x 8192 x 28672 82-84 against 84-86).  Unsplit
  // 128-column tiles stay when K is short (256 x 8192 x 4096: 21.9 us against 23.2).
  bool auto_kx = false;
  if (allow_kx && !f.block_n && !f.splits && !f.stages && !f.epilogue &&
      !f.chain_kblocks && !sk_narrow &&
      c->k_blocks >= 8) {
    // 320-column pair tiles (two MMAs per K step) have a cluster-K-split kernel for
    // single-chain slices only
    const bool try320 = cg == 2 && ceil_div(c->k_blocks, (int64_t)2) <= chain_kb_of(kb_elems);
    for (int bn : {128, 256, 320}) {
      if (bn == 320 && !try320) continue;
      const int st = kx_stages(cg, bn, small_a);
      int64_t sl = bn == 320 ? h->sms / cg
                             : resident_units(h, cg, bn, default_stages(cg, bn, small_a), out);
      if (f.max_ctas) sl = std::min<int64_t>(sl, std::max<int64_t>(f.max_ctas / cg, 1));
      const int64_t tl = c->num_m * ceil_div(N, (int64_t)bn);
      if (tl * 2 > sl || std::min<int64_t>({sl / tl, c->k_blocks / 4, 32}) != 2) continue;
      // keep unsplit narrow tiles (256 x 8192 x 4096: 19.5 us against 26.0 for 320-column
      // split tiles; 384 x 4096 x 4096: 18.4 against 25.3)
      if (bn != 128 && c->bn == 128 && c->k_blocks < 128) continue;
      const int clusters = kx_clusters(h, cg, bn, st, out);
      if (clusters <= 0 || tl > clusters) continue;
      c->bn = bn;
      c->stages = st;
      c->num_n = ceil_div(N, (int64_t)bn);
      c->tiles = tl;
      slots = sl;
      auto_kx = true;
      break;
    }
  }
  int64_t s = 1, dp = c->tiles;
  c->half_tail = 0;
  c->sk_workers = 0;
  if (f.splits < 0) {
    // forced stream-K: every resident unit takes an equal share of the (tile, k-block)
    // iterations ("A Blackwell GEMM by Hand in CuTe DSL", section 9; "CUTLASS Deep
    // Dive", StreamK).  Below one wave of tiles it lost to split-K on the M = 256 decode
    // shapes (the three-segment tiles cost more to reduce than the balance saves), so it
    // is chosen automatically only as below: between one and two waves of tiles.
    dp = 0;
    c->sk_workers = std::min<int64_t>(slots, c->tiles * c->k_blocks);
    // the kernel splits the iteration range in 32-bit arithmetic
    if (c->tiles * c->k_blocks * c->sk_workers >= (int64_t(1) << 32)) return GEMM_ERR_UNSUPPORTED;
  } else if (f.splits) {
    s = f.splits;  // forced: every tile is sliced
    dp = 0;
  } else if (c->tiles * 2 <= slots && c->k_blocks >= 8) {
    // Fewer tiles than half the resident units: slice every tile along K so all SMs
    // have work ("A Blackwell GEMM by Hand in CuTe DSL", section 9: decode shapes are
    // decided by waves).
    s = std::min<int64_t>({slots / c->tiles, c->k_blocks / 4, 32});
    dp = 0;
  } else if (allow_kx && !f.max_ctas && !f.block_n && !f.stages && !f.epilogue &&
             !f.chain_kblocks && c->tiles > slots && c->tiles < 2 * slots && c->k_blocks > chain_kb_of(kb_elems) &&
             c->tiles * c->k_blocks * slots < (int64_t(1) << 32) &&
             !(c->num_m > 1 && 4 * (c->tiles % slots) > slots)) {
    // Between one and two waves of tiles of several accumulation chains: stream-K over
    // every resident unit instead of a second, mostly idle wave (measured, back to back:
    // 256 x 28672 x 8192 88.9 us against 97.6 for whole tiles and half tiles; 512 x 10240 x
    // 8192 66.4 against 87.2).  Below one wave the segments' fix-up costs more than the
    // balance gains (512 x 8192 x 8192: 58.7 against 48.4 us).  With two rows of tiles or
    // more, the tiles that share B's columns reach the same K at far-apart times under
    // stream-K, so B comes from DRAM once per row of tiles: whole tiles (and half tiles in
    // the last wave where they fit) then win unless the last wave holds at most a quarter
    // of the units (320 .. 512 x 14336 x 8192: 75.3 to 77.8 us against 94.8 to 96.7;
    // 768 x 10240 x 8192 84 against 103; 1024 x 8192 x 8192 84 against 110; 2048 x 4096 x
    // 8192 83 against 99), and stream-K stays for a nearly empty one (384 and 512 x 10240
    // x 8192: 60.8 and 62.1 against 81.5 and 72.4).
    dp = 0;
    c->sk_workers = slots;
  } else if (c->tiles > slots && c->tiles % slots != 0) {
    // Whole waves run whole tiles; the tiles of the partial last wave are spread over
    // more units so that the last wave keeps (nearly) every unit busy: as two
    // 128-column halves when they fit (no reduction), else as K slices.
    const int64_t rem = c->tiles % slots;
    if (c->bn == 256 && 2 * rem <= slots) {
      c->half_tail = 1;
      dp = c->tiles - rem;
    } else if (c->k_blocks >= 8) {
      s = std::min<int64_t>({slots / rem, c->k_blocks / 4, 8});
      dp = s >= 2 ? c->tiles - rem : c->tiles;
    }
  }
  if (s < 1) s = 1;
  if (s > c->k_blocks) s = c->k_blocks;
  const int64_t per = ceil_div(c->k_blocks, s);
  s = ceil_div(c->k_blocks, per);  // no empty slice
  if (s == 1 && !c->half_tail && !c->sk_workers) dp = c->tiles;
  c->splits = (int)s;
  c->kb_per_split = (int)per;
  c->dp_tiles = dp;
  c->units = c->sk_workers ? dp : dp + (c->tiles - dp) * (c->half_tail ? 2 : s);
  c->ws_slots = s;
  if (c->sk_workers) {
    // A tile meets at most ceil(k_blocks / share) + 1 workers' ranges.
    const int64_t share = (c->tiles - dp) * c->k_blocks / c->sk_workers;
    c->ws_slots = ceil_div(c->k_blocks, std::max<int64_t>(share, 1)) + 1;
  }
  c->group_m = f.group_m ? f.group_m : 16;
  c->chain_kb = f.chain_kblocks ? f.chain_kblocks : chain_kb_of(kb_elems);
  if (blockwise) {
    if (f.chain_kblocks > 1 || f.epilogue >= 2) return GEMM_ERR_UNSUPPORTED;
    c->chain_kb = 1;
  }
  // Prefetching B into L2 ahead of the ring: off unless asked for (measured on the
  // M = 256 decode shapes and the square ones it did not help).
  c->prefetch_kb = f.prefetch_kblocks > 0 ? f.prefetch_kblocks : 0;
  // One row of tiles reads every B element once while every tile re-reads A: B's lines
  // go first out of L2, A's last.
  c->l2_hint = f.l2_hint ? f.l2_hint : (c->num_m == 1 ? 2 : 1);
  c->grid = (int)(std::min<int64_t>(std::max(c->units, c->sk_workers), slots) * cg);
  // The single-chain epilogue needs every unit to be one accumulation chain.
  int64_t longest = c->k_blocks;  // whole tiles and half-tile units
  if (c->sk_workers)
    longest = std::min<int64_t>(c->k_blocks,
                                ceil_div((c->tiles - dp) * c->k_blocks, c->sk_workers));
  else if (!c->half_tail && s > 1 && dp == 0)
    longest = c->kb_per_split;
  const bool one_ok = longest <= c->chain_kb;
  if (f.epilogue == 2 && !one_ok) return GEMM_ERR_UNSUPPORTED;
  // FP8 operands: the general epilogue unless the single-chain one is asked for.  An FP8
  // tile is half the stages of an fp16 tile of the same K, and the single-chain form
  // holds its accumulator slot through the stores, which then delays the MMAs of the
  // tile after next (E4M3 -> bf16, A/B on one GPU, flushed: 4096^3 53.2 -> 50.7 us,
  // 2048x8192x4096 55.3 -> 51.2, 4096x4096x1024 41.0 -> 34.1, 1024x1024x4096 37.2 ->
  // 30.7; within 1% at 8192x8192x2048 and 256x8192x4096).  fp16/bf16 keep it
  // (4096^3 79.4 against 82.0 us).
  const bool fp8 = kb_elems == 2 * kBlockK;
  c->one_chain = (f.epilogue == 1 || blockwise || (fp8 && f.epilogue == 0)) ? false : one_ok;
  // (epilogue 3: either form)
  // The cluster K split: every tile's two K slices run on the two CTA groups of one
  // cluster of 2 * cg CTAs, each group one unit, and meet in distributed shared memory.
  c->kx2 = false;
  if (f.epilogue == 3 || auto_kx) {
    bool valid = allow_kx && !c->sk_workers && !c->half_tail && dp == 0 && s == 2 &&
                 c->units <= slots;
    // its own ring depth (the staging inside the ring); a forced depth must be that one
    const int kst = kx_stages(cg, c->bn, a_rows(cg, c->bn, c->stages) < kBlockM);
    if (f.stages && f.stages != kst) valid = false;
    if (valid) {
      const int clusters = kx_clusters(h, cg, c->bn, kst, out);
      valid = clusters > 0 && c->tiles <= clusters;
    }
    if (valid) {
      c->kx2 = true;
      c->stages = kst;
      c->grid = (int)(c->units * cg);
    } else if (f.epilogue == 3) {
      return GEMM_ERR_UNSUPPORTED;
    }
  }
  if (c->bn == 320 && !(c->kx2 && c->one_chain)) return GEMM_ERR_UNSUPPORTED;
  // the deeper rings of 16-row A stages: plain fp16/bf16 kernels, row tiles of <= 16 rows
  if (a_rows(cg, c->bn, c->stages) < kBlockM && (M > a_rows(cg, c->bn, c->stages) || !allow_kx))
    return GEMM_ERR_UNSUPPORTED;
  if (c->units > INT32_MAX || c->tiles * cg * 8 > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  return GEMM_OK;
}

gemm_status_t choose(gemm_ctx* h, int64_t M, int64_t N, int64_t K, int out, int kb_elems,
                     bool blockwise, bool allow_kx, Choice* c) {
  const gemm_config_t& f = h->forced;
  if (f.swap_ab == 2) {
    if (!allow_kx) return GEMM_ERR_UNSUPPORTED;
    return choose_swap(h, M, N, K, out, kb_elems, c);
  }
  gemm_status_t st = choose_plain(h, M, N, K, out, kb_elems, blockwise, allow_kx, c);
  if (st != GEMM_OK || f.swap_ab == 1 || !allow_kx || f.variant || f.block_n || f.splits ||
      f.stages || f.max_ctas || f.chain_kblocks || f.dp_tiles || f.epilogue || f.swap_rows)
    return st;
  // The swapped tiling in place of plain one-CTA tiles (17..128 rows of A, K of two
  // accumulation chains or more) that leave a quarter of the SMs idle, with at least 96
  // rows of B per CTA, so that B's rows stay most of each stage next to the 64 rows of A,
  // when the swapped tiles form one wave, or with K of at most two chains a second wave
  // at least 40% full (measured back to back over cold operands, one GB300: 17 to 128 x
  // 14336 x 8192, one wave: 42.5 to 43.8 us against 44.3 to 46.3; 32 and 128 x 14336 x
  // 28672: 130.2 and 130.9 against 138.6; 32 to 128 x 28672 x 8192, a second wave 47%
  // full: 76.4 to 78.2 against 77.9 to 79.2; with K 16384 from 2% slower to 1.5% faster).
  // With 16 rows the plain kernel's 16-row stages are as fast (16 x 14336 x 8192: 42.6
  // both), and a nearly empty second wave costs more than the idle SMs (128 x 20480 x
  // 8192, 5% full: 75.5 against 65.0).  For 129..256
  // rows the plain pair tiles keep up with it (256 x 8192 x 4096, unsplit 128-column
  // tiles: 19.5 against 19.8; 256 x 8192 x 8192, the cluster K split: 31.1 against 32.2).
  Choice sw;
  if (M <= 16 || M > kBlockM || c->k_blocks < 2 * chain_kb_of(kb_elems) ||
      4 * (int64_t)c->grid > 3 * (int64_t)h->sms)
    return st;
  if (choose_swap(h, M, N, K, out, kb_elems, &sw) != GEMM_OK || sw.swap_rows < 96)
    return st;
  const int64_t pairs = sw.grid / 2, rest = sw.units % pairs;
  if (sw.units > pairs && (sw.units > 2 * pairs || c->k_blocks > 2 * chain_kb_of(kb_elems) ||
                           (rest != 0 && 5 * rest < 2 * pairs)))
    return st;
  *c = sw;
  return st;
}

gemm_status_t ensure_workspace(gemm_ctx* h, size_t ws_bytes, size_t ctr_count) {
  if (ws_bytes > h->ws_bytes) {
    if (h->d_ws) cudaFree(h->d_ws);
    h->d_ws = nullptr;
    h->ws_bytes = 0;
    if (cudaMalloc(&h->d_ws, ws_bytes) != cudaSuccess) return GEMM_ERR_OOM;
    h->ws_bytes = ws_bytes;
  }
  if (ctr_count > h->ctr_count) {
    if (h->d_ctr) cudaFree(h->d_ctr);
    h->d_ctr = nullptr;
    h->ctr_count = 0;
    if (cudaMalloc(&h->d_ctr, ctr_count * sizeof(uint32_t)) != cudaSuccess) return GEMM_ERR_OOM;
    if (cudaMemset(h->d_ctr, 0, ctr_count * sizeof(uint32_t)) != cudaSuccess) return GEMM_ERR_CUDA;
    h->ctr_count = ctr_count;
  }
  return GEMM_OK;
}

}  // namespace

extern "C" {

const char* gemm_last_cuda_error(gemm_handle_t h) {
  if (!h) return "";
  return h->last_cuda == cudaSuccess ? "" : cudaGetErrorName(h->last_cuda);
}

const char* gemm_status_string(gemm_status_t s) {
  switch (s) {
    case GEMM_OK: return "ok";
    case GEMM_ERR_INVALID_ARG: return "invalid argument";
    case GEMM_ERR_UNSUPPORTED: return "unsupported (dtype, alignment, K row pitch, or device)";
    case GEMM_ERR_CUDA: return "CUDA error";
    case GEMM_ERR_OOM: return "out of memory";
    case GEMM_ERR_TIMEOUT: return "kernel wait timed out";
    default: return "unknown status";
  }
}

gemm_status_t gemm_create(gemm_handle_t* out) {
  if (!out) return GEMM_ERR_INVALID_ARG;
  *out = nullptr;
  int dev = 0, major = 0, minor = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
  gemm_ctx* h = new (std::nothrow) gemm_ctx();
  if (!h) return GEMM_ERR_OOM;
  h->device = dev;
  h->sms = sms;
  if (cudaMalloc(&h->d_status, sizeof(uint32_t)) != cudaSuccess) {
    delete h;
    return GEMM_ERR_OOM;
  }
  if (cudaMemset(h->d_status, 0, sizeof(uint32_t)) != cudaSuccess) {
    cudaFree(h->d_status);
    delete h;
    return GEMM_ERR_CUDA;
  }
  *out = h;
  return GEMM_OK;
}

gemm_status_t gemm_destroy(gemm_handle_t h) {
  if (!h) return GEMM_OK;
  cudaDeviceSynchronize();
  cudaFree(h->d_status);
  if (h->d_ws) cudaFree(h->d_ws);
  if (h->d_ctr) cudaFree(h->d_ctr);
  for (auto* p : h->d_stage)
    if (p) cudaFree(p);
  if (h->copy_in) cudaStreamDestroy(h->copy_in);
  if (h->copy_out) cudaStreamDestroy(h->copy_out);
  for (auto e : h->host_ev)
    if (e) cudaEventDestroy(e);
  for (int i = 0; i < gemm_ctx::kGroupRing; ++i) {
    if (h->h_groups[i]) cudaFreeHost(h->h_groups[i]);
    if (h->h_gstart[i]) cudaFreeHost(h->h_gstart[i]);
    if (h->d_groups[i]) cudaFree(h->d_groups[i]);
    if (h->d_gstart[i]) cudaFree(h->d_gstart[i]);
    if (h->group_done[i]) cudaEventDestroy(h->group_done[i]);
  }
  delete h;
  return GEMM_OK;
}

gemm_status_t gemm_set_config(gemm_handle_t h, const gemm_config_t* cfg) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (!cfg) {
    h->forced = gemm_config_t{};
    return GEMM_OK;
  }
  const gemm_config_t& c = *cfg;
  if (c.variant < 0 || c.variant > 3) return GEMM_ERR_INVALID_ARG;
  if (c.block_n != 0 && c.block_n != 128 && c.block_n != 256 && c.block_n != 320)
    return GEMM_ERR_INVALID_ARG;
  if (c.splits < -1 || c.stages < 0 || c.group_m < 0 || c.max_ctas < 0 || c.chain_kblocks < 0 ||
      c.dp_tiles != 0 || c.prefetch_kblocks < -1 || c.epilogue < 0 || c.epilogue > 3 ||
      c.l2_hint < 0 || c.l2_hint > 2 || c.swap_ab < 0 || c.swap_ab > 2 || c.swap_rows < 0 ||
      c.swap_rows > 128 || c.scheduler < 0 || c.scheduler > 2)
    return GEMM_ERR_INVALID_ARG;
  if (c.stages) {
    const int bn = c.block_n ? c.block_n : 256;
    const bool any = kernel_supported(1, bn, c.stages) || kernel_supported(2, bn, c.stages);
    if (c.variant ? !kernel_supported(c.variant, bn, c.stages) : !any) return GEMM_ERR_INVALID_ARG;
  }
  h->forced = c;
  return GEMM_OK;
}

gemm_status_t gemm_last_config(gemm_handle_t h, gemm_config_t* out) {
  if (!h || !out) return GEMM_ERR_INVALID_ARG;
  *out = h->last;
  return GEMM_OK;
}

gemm_status_t gemm_set_wait_limit(gemm_handle_t h, uint64_t ns) {
  if (!h || ns == 0) return GEMM_ERR_INVALID_ARG;
  h->wait_limit_ns = ns;
  return GEMM_OK;
}

gemm_status_t gemm_set_test_stall(gemm_handle_t h, int32_t enable) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  h->test_stall = enable ? 1 : 0;
  return GEMM_OK;
}

int32_t gemm_sm_count(gemm_handle_t h) { return h ? h->sms : 0; }

namespace {

gemm_status_t run_impl(gemm_handle_t h, const void* A, const void* B, void* C, int64_t M,
                       int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                       const gemm_epilogue_t* epi, const gemm_block_scales_t* bs,
                       gemm_stream_t stream_) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (bs) {
    if (!bs->sfa || !bs->sfb || bs->block_m < 1) return GEMM_ERR_INVALID_ARG;
    if (!is_fp8(dtype_in) || bs->block_n != 128 ||
        reinterpret_cast<uintptr_t>(bs->sfa) % 4 || reinterpret_cast<uintptr_t>(bs->sfb) % 4)
      return GEMM_ERR_UNSUPPORTED;
  }
  const bool fused = epi && (epi->alpha != 1.0f || epi->beta != 0.0f || epi->bias ||
                             epi->activation != GEMM_ACT_NONE);
  if (epi && epi->activation != GEMM_ACT_NONE && epi->activation != GEMM_ACT_RELU)
    return GEMM_ERR_INVALID_ARG;
  if (fused && epi->bias && reinterpret_cast<uintptr_t>(epi->bias) % 16)
    return GEMM_ERR_UNSUPPORTED;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(dtype_in) || !valid_dtype(dtype_out)) return GEMM_ERR_INVALID_ARG;
  if (dtype_in == GEMM_F32 || is_fp8(dtype_out)) return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t osz = out_size(dtype_out);
  if (reinterpret_cast<uintptr_t>(C) % osz) return GEMM_ERR_UNSUPPORTED;
  if (K == 0) {  // the empty sum: C = 0 (all-zero bits in every output format)
    if (fused) return GEMM_ERR_UNSUPPORTED;
    if (cudaMemsetAsync(C, 0, (size_t)M * (size_t)N * osz, stream) != cudaSuccess)
      return GEMM_ERR_CUDA;
    return GEMM_OK;
  }
  if ((K * (int64_t)in_size(dtype_in)) % 16) return GEMM_ERR_UNSUPPORTED;  // TMA row pitch
  if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
    return GEMM_ERR_UNSUPPORTED;

  const int out = out_kind(dtype_out);
  const bool fp8_in = is_fp8(dtype_in);
  // A few rows of A: the CUDA-core matrix-vector path (variant 3), forced or automatic.
  const gemm_config_t& fc = h->forced;
  if (fc.variant == 3 || (!fc.variant && !fc.block_n && !fc.splits && !fc.stages && !fc.epilogue &&
                          !fc.chain_kblocks && fc.swap_ab != 2 && M == 1 && K <= kGemvAutoMaxK &&
                          !fused && !fp8_in && !bs)) {
    if (M > kGemvMaxRows || fused || fp8_in || bs) return GEMM_ERR_UNSUPPORTED;
    GemvSpec g;
    g.A = A;
    g.B = B;
    g.C = C;
    g.M = (int32_t)M;
    g.N = (int32_t)N;
    g.chunks = (int32_t)(K / 8);
    g.bf16 = dtype_in == GEMM_BF16;
    g.out = out;
    // 4 x 256 threads per SM, one warp per row of B at a time
    const int64_t cap = fc.max_ctas ? fc.max_ctas : (int64_t)h->sms * 4;
    g.grid = (int)std::min<int64_t>(ceil_div(N, (int64_t)8), cap);
    g.stream = stream;
    if ((h->last_cuda = launch_gemv(g)) != cudaSuccess) return GEMM_ERR_CUDA;
    h->last = gemm_config_t{3, 0, 1, 0, 0, g.grid, 0, (int32_t)N, -1, 1, 1, 1, 0, 1};
    return GEMM_OK;
  }
  if (fc.scheduler == 2) return GEMM_ERR_UNSUPPORTED;  // (cluster launch control: grouped launches)
  Choice ch;
  const bool fp8 = is_fp8(dtype_in);
  gemm_status_t st = choose(h, M, N, K, out, fp8 ? 2 * kBlockK : kBlockK, bs != nullptr,
                            !fp8 && !fused && !bs, &ch);
  if (st != GEMM_OK) return st;

  LaunchSpec s;
  std::memset(&s, 0, sizeof(s));
  s.cta_group = ch.variant;
  s.bn = ch.bn;
  s.stages = ch.stages;
  s.out = out;
  s.grid = ch.grid;
  s.one_chain = ch.one_chain;
  s.kx2 = ch.kx2;
  s.swap = ch.swap;
  // FP8 kernels always carry the epilogue: the per-tensor scales arrive as alpha
  s.fused = (fused || fp8) && !bs;
  s.kind = bs ? 2 : fp8 ? 1 : 0;
  s.staged = !ch.kx2 && !ch.swap && !s.fused && s.kind == 0 && !ch.one_chain &&
             ((ch.splits > 1 && !ch.half_tail) || ch.sk_workers);
  s.stream = stream;
  const bool c_tma = reinterpret_cast<uintptr_t>(C) % 16 == 0 && ((size_t)N * osz) % 16 == 0;
  // A single one-CTA row tile of M < 128 rows loads A as an M-row box: the stage's
  // rows M..127 are never written and only feed accumulator rows that are never
  // stored.  (A 128-row box over fewer than 8 rows of A ran up to 1.5x slower on the
  // decode shapes than over 8 or more, measured.)
  const int a_box = (ch.variant == 1 && M < kBlockM) ? (int)M : kBlockM;
  if (ch.swap) {
    // B is the MMA's row operand (swap_rows rows per CTA), A its columns (bn / 2 rows per
    // CTA); C is written transposed with direct stores
    if (!make_map(h, B, N, K, dtype_in, ch.swap_rows, &s.tmA) ||
        !make_map(h, A, M, K, dtype_in, ch.bn / 2, &s.tmB))
      return GEMM_ERR_CUDA;
    s.tmB2 = s.tmB;
    s.tmC = s.tmB;  // (not read: no TMA store)
  } else if (!make_map(h, A, M, K, dtype_in, a_box, &s.tmA) ||
      !make_map(h, B, N, K, dtype_in, ch.bn == 320 ? 128 : ch.bn / ch.variant, &s.tmB) ||
      (ch.half_tail && !make_map(h, B, N, K, dtype_in, ch.bn / ch.variant / 2, &s.tmB2)) ||
      (c_tma && !make_map(h, C, M, N, dtype_out, 32, &s.tmC)))
    return GEMM_ERR_CUDA;
  if (ch.swap) {
  } else if (ch.bn == 320) {
    // the last 32 of each CTA's 160 B rows
    if (!make_map(h, B, N, K, dtype_in, 32, &s.tmB2)) return GEMM_ERR_CUDA;
  } else if (!ch.half_tail) {
    s.tmB2 = s.tmB;
  }

  GemmParams& p = s.p;
  p.C = C;
  p.fused = s.fused ? 1 : 0;
  p.relu = fused && epi->activation == GEMM_ACT_RELU ? 1 : 0;
  p.alpha = fused ? epi->alpha : 1.0f;
  p.beta = fused ? epi->beta : 0.0f;
  p.bias = fused ? epi->bias : nullptr;
  p.M = (int32_t)M;
  p.N = (int32_t)N;
  p.K = (int32_t)K;
  p.num_m_tiles = (int32_t)ch.num_m;
  p.num_n_tiles = (int32_t)ch.num_n;
  p.tiles = (int32_t)ch.tiles;
  p.k_blocks = (int32_t)ch.k_blocks;
  p.dp_tiles = (int32_t)ch.dp_tiles;
  p.half_tail = ch.half_tail;
  p.splits = ch.splits;
  p.kb_per_split = ch.kb_per_split;
  p.units = (int32_t)ch.units;
  p.sk_workers = (int32_t)ch.sk_workers;
  p.ws_slots = (int32_t)ch.ws_slots;
  p.group_m = ch.group_m;
  p.chain_kb = ch.chain_kb;
  p.prefetch_kb = ch.prefetch_kb;
  p.l2_hint = ch.l2_hint;
  p.a_tx_short = (uint32_t)(a_rows(ch.variant, ch.bn, ch.stages) - a_box) * 128u;
  p.vec_store = c_tma ? 1 : 0;
  p.tma_store = c_tma && ch.bn != 320 ? 1 : 0;  // (320 columns: 160 per warp, direct stores)
  p.swap_rows = ch.swap_rows;
  if (ch.swap) {
    p.a_tx_short = 2u * (uint32_t)(kBlockM - ch.swap_rows) * 128u;  // both CTAs' short boxes
    p.vec_store = 0;
    p.tma_store = 0;
  }
  if (fp8) {
    p.idesc = idesc_f8_kmajor(kBlockM * ch.variant, ch.bn, dtype_in == GEMM_E5M2);
    p.idesc_half = idesc_f8_kmajor(kBlockM * ch.variant, ch.bn / 2, dtype_in == GEMM_E5M2);
  } else {
    p.idesc = idesc_f16_kmajor(kBlockM * ch.variant, ch.bn == 320 ? 256 : ch.bn, dtype_in == GEMM_BF16);
    p.idesc_half = idesc_f16_kmajor(kBlockM * ch.variant, ch.bn == 320 ? 64 : ch.bn / 2,
                                    dtype_in == GEMM_BF16);
  }
  if (bs) {
    p.sfa = bs->sfa;
    p.sfb = bs->sfb;
    p.sf_bm = bs->block_m;
    p.sf_lda = (int32_t)ceil_div(M, (int64_t)bs->block_m);
    p.sf_ldb = (int32_t)ceil_div(N, (int64_t)128);
  }
  p.status = h->d_status;
  p.wait_limit_ns = h->wait_limit_ns;
  p.test_stall = h->test_stall;
  if (!ch.kx2 && ((ch.splits > 1 && !ch.half_tail) || ch.sk_workers)) {
    const size_t sliced = (size_t)(ch.tiles - ch.dp_tiles);
    const size_t ws = sliced * ch.ws_slots * kBlockM * ch.variant * ch.bn * sizeof(float);
    st = ensure_workspace(h, ws, sliced * ch.variant * 8);
    if (st != GEMM_OK) return st;
    p.workspace = h->d_ws;
    p.counters = h->d_ctr;
  }
  if ((h->last_cuda = launch_gemm(s)) != cudaSuccess) return GEMM_ERR_CUDA;
  h->last = gemm_config_t{ch.variant,  ch.bn,   ch.sk_workers ? -(int32_t)ch.sk_workers : ch.splits,
                          ch.stages,
                          ch.group_m,  ch.grid, ch.chain_kb, (int32_t)ch.dp_tiles,
                          ch.prefetch_kb ? ch.prefetch_kb : -1, ch.kx2 ? 3 : ch.one_chain ? 2 : 1,
                          ch.l2_hint, ch.swap ? 2 : 1, ch.swap_rows, 1};
  return GEMM_OK;
}

}  // namespace

gemm_status_t gemm_run(gemm_handle_t h, const void* A, const void* B, void* C, int64_t M,
                       int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                       gemm_stream_t stream) {
  return run_impl(h, A, B, C, M, N, K, dtype_in, dtype_out, nullptr, nullptr, stream);
}

gemm_status_t gemm_plan(const gemm_device_model_t* dev, const gemm_config_t* forced,
                        int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                        gemm_dtype_t dtype_out, int32_t fused, int32_t blockwise,
                        gemm_config_t* out) {
  if (!dev || !out || dev->sms < 2 || dev->pairs < 1 || dev->clusters4 < 0)
    return GEMM_ERR_INVALID_ARG;
  if (M < 1 || N < 1 || K < 1) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(dtype_in) || !valid_dtype(dtype_out)) return GEMM_ERR_INVALID_ARG;
  if (dtype_in == GEMM_F32 || is_fp8(dtype_out)) return GEMM_ERR_UNSUPPORTED;
  if (blockwise && !is_fp8(dtype_in)) return GEMM_ERR_UNSUPPORTED;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  if ((K * (int64_t)in_size(dtype_in)) % 16) return GEMM_ERR_UNSUPPORTED;
  // a context that describes the device instead of querying it (no CUDA call below)
  gemm_ctx ctx;
  ctx.model = true;
  ctx.sms = dev->sms;
  ctx.model_pairs = dev->pairs;
  ctx.model_clusters4 = dev->clusters4;
  if (forced) {
    const gemm_status_t st = gemm_set_config(&ctx, forced);
    if (st != GEMM_OK) return st;
  }
  const gemm_config_t& fc = ctx.forced;
  const bool fp8 = is_fp8(dtype_in);
  // the same decisions as gemm_run: the matrix-vector path for a row of A, else choose()
  if (fc.variant == 3 || (!fc.variant && !fc.block_n && !fc.splits && !fc.stages && !fc.epilogue &&
                          !fc.chain_kblocks && fc.swap_ab != 2 && M == 1 && K <= kGemvAutoMaxK &&
                          !fused && !fp8 && !blockwise)) {
    if (M > kGemvMaxRows || fused || fp8 || blockwise) return GEMM_ERR_UNSUPPORTED;
    const int64_t cap = fc.max_ctas ? fc.max_ctas : (int64_t)ctx.sms * 4;
    const int grid = (int)std::min<int64_t>(ceil_div(N, (int64_t)8), cap);
    *out = gemm_config_t{3, 0, 1, 0, 0, grid, 0, (int32_t)N, -1, 1, 1, 1, 0, 1};
    return GEMM_OK;
  }
  if (fc.scheduler == 2) return GEMM_ERR_UNSUPPORTED;
  Choice ch;
  const gemm_status_t st = choose(&ctx, M, N, K, out_kind(dtype_out), fp8 ? 2 * kBlockK : kBlockK,
                                  blockwise != 0, !fp8 && !fused && !blockwise, &ch);
  if (st != GEMM_OK) return st;
  *out = gemm_config_t{ch.variant,  ch.bn,   ch.sk_workers ? -(int32_t)ch.sk_workers : ch.splits,
                       ch.stages,
                       ch.group_m,  ch.grid, ch.chain_kb, (int32_t)ch.dp_tiles,
                       ch.prefetch_kb ? ch.prefetch_kb : -1, ch.kx2 ? 3 : ch.one_chain ? 2 : 1,
                       ch.l2_hint, ch.swap ? 2 : 1, ch.swap_rows, 1};
  return GEMM_OK;
}

gemm_status_t gemm_run_blockwise(gemm_handle_t h, const void* A, const void* B, void* C,
                                 int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                                 gemm_dtype_t dtype_out, const gemm_block_scales_t* scales,
                                 gemm_stream_t stream) {
  if (!scales) return GEMM_ERR_INVALID_ARG;
  return run_impl(h, A, B, C, M, N, K, dtype_in, dtype_out, nullptr, scales, stream);
}

gemm_status_t gemm_run_epilogue(gemm_handle_t h, const void* A, const void* B, void* C,
                                int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                                gemm_dtype_t dtype_out, const gemm_epilogue_t* epilogue,
                                gemm_stream_t stream) {
  return run_impl(h, A, B, C, M, N, K, dtype_in, dtype_out, epilogue, nullptr, stream);
}

gemm_status_t gemm_run_grouped(gemm_handle_t h, const gemm_problem_t* problems, int32_t count,
                               gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                               gemm_stream_t stream_) {
  if (!h || count < 0 || (count > 0 && !problems)) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(dtype_in) || !valid_dtype(dtype_out)) return GEMM_ERR_INVALID_ARG;
  if (dtype_in != GEMM_F16 && dtype_in != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
  if (is_fp8(dtype_out)) return GEMM_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t osz = out_size(dtype_out);
  // Validate everything before queueing anything.
  for (int32_t g = 0; g < count; ++g) {
    const gemm_problem_t& q = problems[g];
    if (q.M < 0 || q.N < 0 || q.K < 0) return GEMM_ERR_INVALID_ARG;
    if (q.M == 0 || q.N == 0) continue;
    if (!q.C || (q.K > 0 && (!q.A || !q.B))) return GEMM_ERR_INVALID_ARG;
    if (q.M > INT32_MAX || q.N > INT32_MAX || q.K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(q.C) % osz) return GEMM_ERR_UNSUPPORTED;
    if (q.K > 0 && (q.K % 8 || reinterpret_cast<uintptr_t>(q.A) % 16 ||
                    reinterpret_cast<uintptr_t>(q.B) % 16))
      return GEMM_ERR_UNSUPPORTED;
  }
  const gemm_config_t& f = h->forced;
  if ((f.splits != 0 && f.splits != 1) || f.epilogue >= 2 || f.swap_ab == 2)
    return GEMM_ERR_UNSUPPORTED;
  // Problems with K = 0 are the empty sum; the rest go into one launch.
  std::vector<int32_t> live;
  int64_t padded[3] = {0, 0, 0};  // MACs with M padded to 128 and to 256 rows
  bool narrow = true;
  for (int32_t g = 0; g < count; ++g) {
    const gemm_problem_t& q = problems[g];
    if (q.M == 0 || q.N == 0) continue;
    if (q.K == 0) {
      if (cudaMemsetAsync(q.C, 0, (size_t)q.M * (size_t)q.N * osz, stream) != cudaSuccess)
        return GEMM_ERR_CUDA;
      continue;
    }
    live.push_back(g);
    for (int v = 1; v <= 2; ++v)
      padded[v] += ceil_div(q.M, (int64_t)kBlockM * v) * kBlockM * v * q.N / 64 * q.K;
    narrow = narrow && q.N <= 128;
  }
  if (live.empty()) return GEMM_OK;
  const int G = (int)live.size();
  // Problems with the longest K first (a stable sort): a tile's time grows with its K, so
  // the long tiles are handed out first and the short ones fill in at the end of the
  // launch, whichever scheduler hands them out (longest processing time first).  The
  // result does not depend on the order.
  std::stable_sort(live.begin(), live.end(),
                   [&](int32_t a, int32_t b) { return problems[a].K > problems[b].K; });
  // A CTA pair when padding every problem's M to 256 rows costs at most 10% more work
  // than padding to 128; 128-column tiles when every N fits one.
  const int cg = f.variant ? f.variant : (padded[2] * 10 <= padded[1] * 11 ? 2 : 1);
  const int bn = f.block_n ? f.block_n : (narrow ? 128 : 256);
  const int stages = f.stages ? f.stages : default_stages(cg, bn);
  if (!kernel_supported(cg, bn, stages)) return GEMM_ERR_INVALID_ARG;
  if (a_rows(cg, bn, stages) < kBlockM || bn == 320) return GEMM_ERR_UNSUPPORTED;  // no grouped kernel

  // The next table of the ring: its host copy is free once its last upload is done.
  const int slot = h->group_next;
  h->group_next = (slot + 1) % gemm_ctx::kGroupRing;
  if (h->group_done[slot]) {
    if (cudaEventSynchronize(h->group_done[slot]) != cudaSuccess) return GEMM_ERR_CUDA;
  } else if (cudaEventCreateWithFlags(&h->group_done[slot], cudaEventDisableTiming) != cudaSuccess) {
    return GEMM_ERR_CUDA;
  }
  if ((size_t)G > h->group_cap[slot]) {
    if (h->h_groups[slot]) cudaFreeHost(h->h_groups[slot]);
    if (h->h_gstart[slot]) cudaFreeHost(h->h_gstart[slot]);
    if (h->d_groups[slot]) cudaFree(h->d_groups[slot]);
    if (h->d_gstart[slot]) cudaFree(h->d_gstart[slot]);
    h->h_groups[slot] = nullptr;
    h->h_gstart[slot] = nullptr;
    h->d_groups[slot] = nullptr;
    h->d_gstart[slot] = nullptr;
    h->group_cap[slot] = 0;
    const size_t cap = std::max<size_t>(G, 16);
    if (cudaMallocHost(&h->h_groups[slot], cap * sizeof(GroupDesc)) != cudaSuccess ||
        cudaMallocHost(&h->h_gstart[slot], (cap + 1) * sizeof(int32_t)) != cudaSuccess ||
        cudaMalloc(&h->d_groups[slot], cap * sizeof(GroupDesc)) != cudaSuccess ||
        cudaMalloc(&h->d_gstart[slot], (cap + 1) * sizeof(int32_t)) != cudaSuccess)
      return GEMM_ERR_OOM;
    h->group_cap[slot] = cap;
  }
  GroupDesc* desc = h->h_groups[slot];
  int32_t* start = h->h_gstart[slot];
  int64_t units = 0;
  int32_t max_num_m = 0;
  for (int i = 0; i < G; ++i) {
    const gemm_problem_t& q = problems[live[i]];
    GroupDesc& d = desc[i];
    std::memset(&d, 0, sizeof(d));
    const int a_box = (cg == 1 && q.M < kBlockM) ? (int)q.M : kBlockM;
    const bool c_tma =
        reinterpret_cast<uintptr_t>(q.C) % 16 == 0 && ((size_t)q.N * osz) % 16 == 0;
    if (!make_map(h, q.A, q.M, q.K, dtype_in, a_box, &d.tmA) ||
        !make_map(h, q.B, q.N, q.K, dtype_in, bn / cg, &d.tmB) ||
        (c_tma && !make_map(h, q.C, q.M, q.N, dtype_out, 32, &d.tmC)))
      return GEMM_ERR_CUDA;
    d.C = q.C;
    d.M = (int32_t)q.M;
    d.N = (int32_t)q.N;
    d.K = (int32_t)q.K;
    d.k_blocks = (int32_t)ceil_div(q.K, (int64_t)kBlockK);
    d.num_m = (int32_t)ceil_div(q.M, (int64_t)kBlockM * cg);
    d.num_n = (int32_t)ceil_div(q.N, (int64_t)bn);
    max_num_m = std::max(max_num_m, d.num_m);
    d.a_tx_short = (uint32_t)(kBlockM - a_box) * 128u;
    d.vec_store = c_tma ? 1 : 0;
    d.tma_store = c_tma ? 1 : 0;
    start[i] = (int32_t)units;
    units += (int64_t)d.num_m * d.num_n;
    if (units > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  }
  start[G] = (int32_t)units;
  if (cudaMemcpyAsync(h->d_groups[slot], desc, G * sizeof(GroupDesc), cudaMemcpyHostToDevice,
                      stream) != cudaSuccess ||
      cudaMemcpyAsync(h->d_gstart[slot], start, (G + 1) * sizeof(int32_t),
                      cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaEventRecord(h->group_done[slot], stream) != cudaSuccess)
    return GEMM_ERR_CUDA;

  int64_t slots = resident_units(h, cg, bn, stages, out_kind(dtype_out));
  if (f.max_ctas) slots = std::min<int64_t>(slots, std::max<int64_t>(f.max_ctas / cg, 1));
  LaunchSpec s;
  std::memset(&s, 0, sizeof(s));
  s.cta_group = cg;
  s.bn = bn;
  s.stages = stages;
  s.out = out_kind(dtype_out);
  // Cluster launch control ("A Blackwell GEMM by Hand in CuTe DSL", section 8): a CTA
  // (pair) per tile in the grid, each running one taking over the tiles of launches not
  // yet started, instead of the resident ones taking the tiles round-robin.
  // Chosen automatically when the tiles' costs differ, i.e. the problems' K do by 2x or
  // more (measured, one GB300, problems longest K first: groups of 16, 24 and 48 problems
  // with K from 256 to 16384, 1.22x / 1.08x / equal against round-robin); with one K for
  // all (MoE layers) every tile costs the same, round-robin is already balanced and was
  // 0.5-3.5% faster.
  int64_t kmin = INT64_MAX, kmax = 0;
  for (int i = 0; i < G; ++i) {
    kmin = std::min<int64_t>(kmin, problems[live[i]].K);
    kmax = std::max<int64_t>(kmax, problems[live[i]].K);
  }
  s.clc = f.scheduler == 2 || (f.scheduler == 0 && !f.max_ctas && kmax >= 2 * kmin);
  if (s.clc && f.max_ctas) return GEMM_ERR_UNSUPPORTED;
  s.grid = (int)((s.clc ? units : std::min<int64_t>(units, slots)) * cg);
  s.grouped = true;
  s.stream = stream;
  // the parameter maps are not read by a grouped kernel; they hold the first problem's
  s.tmA = desc[0].tmA;
  s.tmB = desc[0].tmB;
  s.tmB2 = desc[0].tmB;
  s.tmC = desc[0].tmC;
  GemmParams& p = s.p;
  p.C = desc[0].C;
  p.M = desc[0].M;
  p.N = desc[0].N;
  p.K = desc[0].K;
  p.tiles = (int32_t)units;
  p.units = (int32_t)units;
  p.dp_tiles = (int32_t)units;
  p.splits = 1;
  p.kb_per_split = 0;
  p.group_m = f.group_m ? f.group_m : 16;
  p.chain_kb = f.chain_kblocks ? f.chain_kblocks : kChainKBlocks;
  p.idesc = idesc_f16_kmajor(kBlockM * cg, bn, dtype_in == GEMM_BF16);
  p.idesc_half = p.idesc;
  p.groups = h->d_groups[slot];
  p.group_start = h->d_gstart[slot];
  p.num_groups = G;
  // every problem one row of tiles: its B (an expert's weights) is read once
  p.l2_hint = f.l2_hint ? f.l2_hint : (max_num_m <= 1 ? 2 : 1);
  p.status = h->d_status;
  p.wait_limit_ns = h->wait_limit_ns;
  p.test_stall = h->test_stall;
  if ((h->last_cuda = launch_gemm(s)) != cudaSuccess) return GEMM_ERR_CUDA;
  h->last = gemm_config_t{cg, bn, 1, stages, p.group_m, s.grid, p.chain_kb, (int32_t)units, -1, 1,
                          p.l2_hint, 1, 0, s.clc ? 2 : 1};
  return GEMM_OK;
}

gemm_status_t gemm_device_status(gemm_handle_t h, gemm_stream_t stream_, uint32_t* detail) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  if (cudaStreamSynchronize(stream) != cudaSuccess) return GEMM_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, h->d_status, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess)
    return GEMM_ERR_CUDA;
  if (detail) *detail = word;
  if (word == 0) return GEMM_OK;
  // An aborted split-K run may leave arrival counters behind: clear them too.
  cudaMemset(h->d_status, 0, sizeof(uint32_t));
  if (h->d_ctr) cudaMemset(h->d_ctr, 0, h->ctr_count * sizeof(uint32_t));
  if (cudaDeviceSynchronize() != cudaSuccess) return GEMM_ERR_CUDA;
  return GEMM_ERR_TIMEOUT;
}

gemm_status_t gemm_run_host(gemm_handle_t h, const void* A_host, const void* B_host, void* C_host,
                            int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                            gemm_dtype_t dtype_out, gemm_stream_t stream_) {
  if (!h) return GEMM_ERR_INVALID_ARG;
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  if (!valid_dtype(dtype_in) || !valid_dtype(dtype_out)) return GEMM_ERR_INVALID_ARG;
  if (dtype_in == GEMM_F32 || is_fp8(dtype_out)) return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C_host || (K > 0 && (!A_host || !B_host))) return GEMM_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t isz = in_size(dtype_in);
  const size_t bytes[3] = {(size_t)M * K * isz, (size_t)N * K * isz,
                           (size_t)M * N * out_size(dtype_out)};
  for (int i = 0; i < 3; ++i) {
    if (bytes[i] > h->stage_bytes[i]) {
      if (h->d_stage[i]) cudaFree(h->d_stage[i]);
      h->d_stage[i] = nullptr;
      h->stage_bytes[i] = 0;
      if (cudaMalloc(&h->d_stage[i], bytes[i]) != cudaSuccess) return GEMM_ERR_OOM;
      h->stage_bytes[i] = bytes[i];
    }
  }
  // A pipeline over row chunks of A and C: B goes over first, then every chunk's A rows
  // go over on one copy stream while the GEMM of the chunk before runs on `stream` and
  // the C rows of the chunk before that come back on another copy stream.  One chunk
  // below 2048 rows.
  // about 1024 rows per chunk, two to eight chunks (measured: 4096^3 478 us in four
  // chunks against 489 in eight; 8192^3 1675 us in eight against 1760 in four)
  const int64_t want_chunks =
      std::min<int64_t>(gemm_ctx::kHostChunks, std::max<int64_t>(2, M / 1024));
  const int64_t chunk_rows = M >= 2048 ? ceil_div(ceil_div(M, want_chunks), (int64_t)256) * 256 : M;
  const int nc = (int)ceil_div(M, chunk_rows);
  if (K == 0 || nc == 1) {
    if (K > 0 &&
        (cudaMemcpyAsync(h->d_stage[0], A_host, bytes[0], cudaMemcpyHostToDevice, stream) !=
             cudaSuccess ||
         cudaMemcpyAsync(h->d_stage[1], B_host, bytes[1], cudaMemcpyHostToDevice, stream) !=
             cudaSuccess))
      return GEMM_ERR_CUDA;
    gemm_status_t st = gemm_run(h, h->d_stage[0], h->d_stage[1], h->d_stage[2], M, N, K,
                                dtype_in, dtype_out, stream_);
    if (st != GEMM_OK) return st;
    if (cudaMemcpyAsync(C_host, h->d_stage[2], bytes[2], cudaMemcpyDeviceToHost, stream) !=
        cudaSuccess)
      return GEMM_ERR_CUDA;
    return gemm_device_status(h, stream_, nullptr);
  }
  if (!h->copy_in) {
    if (cudaStreamCreateWithFlags(&h->copy_in, cudaStreamNonBlocking) != cudaSuccess ||
        cudaStreamCreateWithFlags(&h->copy_out, cudaStreamNonBlocking) != cudaSuccess)
      return GEMM_ERR_CUDA;
    for (auto& e : h->host_ev)
      if (cudaEventCreateWithFlags(&e, cudaEventDisableTiming) != cudaSuccess) return GEMM_ERR_CUDA;
  }
  cudaEvent_t* ev = h->host_ev;  // [0] start, [1] done, then per chunk: A in, GEMM, C out
  const size_t osz = out_size(dtype_out);
  const char* Ah = static_cast<const char*>(A_host);
  char* Ch = static_cast<char*>(C_host);
  char* Ad = static_cast<char*>(h->d_stage[0]);
  char* Cd = static_cast<char*>(h->d_stage[2]);
  // the staging buffers are free once the work already queued on `stream` is done
  if (cudaEventRecord(ev[0], stream) != cudaSuccess ||
      cudaStreamWaitEvent(h->copy_in, ev[0], 0) != cudaSuccess ||
      cudaStreamWaitEvent(h->copy_out, ev[0], 0) != cudaSuccess ||
      cudaMemcpyAsync(h->d_stage[1], B_host, bytes[1], cudaMemcpyHostToDevice, h->copy_in) !=
          cudaSuccess)
    return GEMM_ERR_CUDA;
  for (int c = 0; c < nc; ++c) {
    const int64_t r0 = c * chunk_rows, rows = std::min(chunk_rows, M - r0);
    cudaEvent_t e_in = ev[2 + 3 * c], e_gemm = ev[3 + 3 * c], e_out = ev[4 + 3 * c];
    if (cudaMemcpyAsync(Ad + r0 * K * isz, Ah + r0 * K * isz, rows * K * isz,
                        cudaMemcpyHostToDevice, h->copy_in) != cudaSuccess ||
        cudaEventRecord(e_in, h->copy_in) != cudaSuccess ||
        cudaStreamWaitEvent(stream, e_in, 0) != cudaSuccess)
      return GEMM_ERR_CUDA;
    gemm_status_t st = gemm_run(h, Ad + r0 * K * isz, h->d_stage[1], Cd + r0 * N * osz, rows, N,
                                K, dtype_in, dtype_out, stream_);
    if (st != GEMM_OK) {
      cudaStreamSynchronize(h->copy_in);
      cudaStreamSynchronize(h->copy_out);
      return st;
    }
    if (cudaEventRecord(e_gemm, stream) != cudaSuccess ||
        cudaStreamWaitEvent(h->copy_out, e_gemm, 0) != cudaSuccess ||
        cudaMemcpyAsync(Ch + r0 * N * osz, Cd + r0 * N * osz, rows * N * osz,
                        cudaMemcpyDeviceToHost, h->copy_out) != cudaSuccess ||
        cudaEventRecord(e_out, h->copy_out) != cudaSuccess)
      return GEMM_ERR_CUDA;
  }
  // the caller's stream resumes once the last rows of C are back
  if (cudaEventRecord(ev[1], h->copy_out) != cudaSuccess ||
      cudaStreamWaitEvent(stream, ev[1], 0) != cudaSuccess)
    return GEMM_ERR_CUDA;
  return gemm_device_status(h, stream_, nullptr);
}

}  // extern "C"
