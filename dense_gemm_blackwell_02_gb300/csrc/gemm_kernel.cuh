// Persistent, warp-specialised tcgen05 GEMM for sm_103a:  C = A . B^T.
//
// A is M x K and B is N x K, both K-major (K contiguous), fp16 or bf16; fp32
// accumulation in Tensor Memory; C is M x N row-major in fp16, bf16 or fp32.
// ("A Blackwell GEMM by Hand in CuTe DSL", section 1 for the operand convention,
// sections 3 and 8 for the warp roles, the CTA pair and persistence with two TMEM
// accumulator slots; "Optimizing GEMMs using tcgen05 - Part 1", phases 2-5.)
//
// CTA_GROUP = 1: one CTA per 128 x BN tile, tcgen05.mma.cta_group::1 (128 x BN x 16).
// CTA_GROUP = 2: a cluster of two CTAs on neighbouring SMs computes a 256 x BN tile
//   with tcgen05.mma.cta_group::2 (256 x BN x 16).  Each CTA loads its own 128 rows of
//   A and its own BN/2 rows of B; both copies complete on the leader's (rank 0's)
//   full barrier; only the leader issues MMAs, and its commits arrive on the barriers
//   of both CTAs (mask 0b11).  Each CTA's Tensor Memory holds its 128 rows.
//
// Ten warps per CTA, one CTA per SM, looping over work units (tile, K slice):
//   warp 0      TMA producer: one thread fills a STAGES-deep ring of 128B-swizzled
//               A (128 x 64) and B (BN/CTA_GROUP x 64) slices.
//   warp 1      allocates 2*BN TMEM columns (two accumulator slots); in the leader one
//               thread issues the MMAs, four per 64-deep stage, into slot i % 2, commits
//               each stage back to empty[s] and each finished chain to acc_full[slot].
//   warps 2..9  epilogue: warp w reads TMEM lane quarter w % 4 and column half
//               (w - 2) / 4; it loads its 32 x BN/2 block, releases the slot at once
//               (so the next chain's MMAs overlap this epilogue), adds the chain into
//               fp32 registers, and after the unit's last chain converts (RNE) and
//               writes C: through a 128B-swizzled shared staging box and a TMA store,
//               or with direct stores when C's row pitch is not a multiple of 16 bytes.
// A unit's K range is accumulated in chains of at most p.chain_kb k-blocks, each in
// a fresh accumulator; the epilogue sums the chains in order in fp32 registers.
// Split-K units write fp32 partials to a workspace; the last slice to arrive (per
// warp's 32 x BN/2 block, by an atomic counter) sums all slices in slice order, so
// the result does not depend on arrival order ("A Blackwell GEMM by Hand in CuTe
// DSL", section 9).
//
// Every mbarrier wait is bounded by p.wait_limit_ns (globaltimer) and an iteration
// cap; on expiry the waiting thread records the site in the status word and raises a
// shared abort flag that makes every role leave its loop; the CTA then drains its own
// outstanding copies and MMAs before freeing TMEM and returning.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "params.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace gb300 {

struct WaitCtl {
  uint64_t limit_ns;
  uint32_t* status;
  volatile int32_t* abort_flag;
};

__device__ __forceinline__ void record_timeout(const WaitCtl& c, uint32_t site) {
  *c.abort_flag = 1;
  atomicCAS(c.status, 0u, (kDevTimeout << 24) | (site << 16) | (blockIdx.x & 0xFFFFu));
}

// Teardown wait: ignores the abort flag (it is used while aborting) but is bounded.
static __device__ __noinline__ bool wait_parity_drain(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u && (globaltimer_ns() - t0 > c.limit_ns || it > (1u << 26))) {
      record_timeout(c, kSiteDrain);
      return false;
    }
  }
}

// Warp-collective wait: all 32 lanes poll together and leave together (a phase, once
// complete, stays complete, so one lane seeing it is enough), so the warp never
// diverges around the wait.  Lane 0's clock decides the timeout for the warp.
static __device__ __noinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                              uint32_t site) {
  if (__any_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (__any_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
    if ((it & 31u) == 0u) {
      const bool aborting = *c.abort_flag != 0;
      const bool expired = globaltimer_ns() - t0 > c.limit_ns || it > (1u << 26);
      if (__shfl_sync(0xFFFFFFFFu, aborting ? 1u : 0u, 0)) return false;
      if (__shfl_sync(0xFFFFFFFFu, expired ? 1u : 0u, 0)) {
        if (lane_id() == 0) record_timeout(c, site);
        __syncwarp();
        return false;
      }
    }
  }
}

// Inline fast path of the wait: a phase that is already complete costs one test here
// instead of a call (whose register saves cost about 200 cycles per wait, measured with
// clock64 in the MMA warp); the bounded loop above runs only when it is not.  Every wait
// of the kernel's roles is this warp-collective form.  An epilogue warp whose lane 0
// polled alone and broadcast the verdict with a shuffle took longer per accumulator
// hand-over: blockwise FP8 8192^3 589.8 -> 534.1 us, E4M3 4096^3 55.6 -> 51.2 us with
// every lane polling (A/B on one GPU).
__device__ __forceinline__ bool warp_wait_inl(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                              uint32_t site) {
  if (__any_sync(0xFFFFFFFFu, mbar_try_wait(bar, parity))) return true;
  return warp_wait(bar, parity, c, site);
}

// Bounded pause (used by a pair's follower while aborting, so copies it issued can land).
__device__ __forceinline__ void pause_ns(uint64_t ns) {
  const uint64_t t0 = globaltimer_ns();
  while (globaltimer_ns() - t0 < ns) {
  }
}

struct Unit {
  int32_t tile, split, nsplit, m_blk, n_blk, kb0, kb1;
  int32_t half;  // -1: the whole BN columns; 0 / 1: that BN/2-column half of the tile
  int32_t g;     // grouped launches: the problem this unit belongs to
};

// Work unit -> (tile, K slice or column half) -> (m block, n block).
// Units [0, dp_tiles) are whole tiles.  The remaining tiles -- normally the last,
// partial wave -- are spread over more SMs instead of leaving most of them idle ("A
// Blackwell GEMM by Hand in CuTe DSL", section 9, against wave quantisation): either
// as two BN/2-column halves with the whole K (half_tail; no reduction needed), or as
// `splits` K slices reduced in the kernel.  With dp_tiles = 0 every tile is sliced
// along K (split-K for decode shapes).
// Tiles map to (m, n) by grouped rasterisation: group_m M-blocks at a time, walking
// N inside a group, so units running at the same time share A rows and B columns in
// L2 ("Matmul on sm_120", block swizzle; "A Blackwell GEMM by Hand in CuTe DSL",
// section 8).
__device__ __forceinline__ void tile_coords(Unit& w, const GemmParams& p) {
  const int32_t group = p.group_m * p.num_n_tiles;
  const int32_t g = w.tile / group;
  const int32_t first_m = g * p.group_m;
  const int32_t gm = min(p.num_m_tiles - first_m, p.group_m);
  const int32_t r = w.tile - g * group;
  w.m_blk = first_m + r % gm;
  w.n_blk = r / gm;
}

__device__ __forceinline__ Unit decode_unit(int32_t u, const GemmParams& p) {
  Unit w;
  w.half = -1;
  if (u < p.dp_tiles) {
    w.tile = u;
    w.split = 0;
    w.nsplit = 1;
    w.kb0 = 0;
    w.kb1 = p.k_blocks;
  } else if (p.half_tail) {
    const int32_t v = u - p.dp_tiles;
    w.tile = p.dp_tiles + (v >> 1);
    w.half = v & 1;
    w.split = 0;
    w.nsplit = 1;
    w.kb0 = 0;
    w.kb1 = p.k_blocks;
  } else {
    const int32_t v = u - p.dp_tiles;
    w.tile = p.dp_tiles + v / p.splits;
    w.split = v - (w.tile - p.dp_tiles) * p.splits;
    w.nsplit = p.splits;
    w.kb0 = w.split * p.kb_per_split;
    w.kb1 = min(w.kb0 + p.kb_per_split, p.k_blocks);
  }
  tile_coords(w, p);
  return w;
}

// The sequence of units one CTA (pair) processes.  First the whole tiles (and the
// half-tile or K-slice units) numbered first, first + stride, ... < p.units; then, in
// stream-K mode, its own contiguous share of the remaining tiles' (tile, k-block)
// iterations: worker c of W takes iterations [floor(c T / W), floor((c + 1) T / W)),
// T = (tiles - dp_tiles) * k_blocks ("Stream-K", cited in "A Blackwell GEMM by Hand
// in CuTe DSL", section 9 and "CUTLASS Deep Dive", StreamK tile scheduler), cut at
// tile boundaries into segments.  Segment j of a tile covered by n segments is
// reduced like K slice j of n.
struct Walker {
  int32_t u;        // next unit number (unit-numbered phase)
  int32_t sk_done;  // stream-K phase: iterations this worker has taken so far
};

// Stream-K worker holding iteration x (the W-way split above, inverted).  The host
// takes stream-K only when (T + 1) * W fits in 32 bits.
__device__ __forceinline__ uint32_t sk_worker_of(uint32_t x, uint32_t T, uint32_t W) {
  return ((x + 1u) * W - 1u) / T;
}

// Advance worker `first` to its next stream-K segment (false when its range is used
// up).  Kept out of line, with the walker and the unit passed by reference: inlined,
// its divisions raise the register pressure of every role and the epilogue's
// 128-float accumulator spills, which slowed the whole-tile path by ~4% at 4096^3
// (measured against this form on the same GPU).
static __device__ __noinline__ bool sk_next(Walker& k, int32_t first, const GemmParams& p,
                                            Unit& w) {
  const uint32_t W = (uint32_t)p.sk_workers;
  const uint32_t T = (uint32_t)(p.tiles - p.dp_tiles) * (uint32_t)p.k_blocks;
  const uint32_t it = (uint32_t)first * T / W + (uint32_t)k.sk_done;
  const uint32_t end = ((uint32_t)first + 1u) * T / W;
  if (it >= end) return false;
  const uint32_t kb = (uint32_t)p.k_blocks;
  const uint32_t t = it / kb;                       // stream-K tile (relative to dp_tiles)
  w.tile = p.dp_tiles + (int32_t)t;
  w.half = -1;
  w.kb0 = (int32_t)(it - t * kb);
  const uint32_t left = end - it;
  w.kb1 = (kb - (uint32_t)w.kb0) < left ? (int32_t)kb : w.kb0 + (int32_t)left;
  const uint32_t w_lo = sk_worker_of(t * kb, T, W);
  const uint32_t w_hi = sk_worker_of(t * kb + kb - 1u, T, W);
  w.nsplit = (int32_t)(w_hi - w_lo + 1u);
  w.split = first - (int32_t)w_lo;
  tile_coords(w, p);
  k.sk_done += w.kb1 - w.kb0;
  return true;
}

// Grouped launch ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05", Part 6,
// Grouped GEMM: each tile pulls its problem index from the scheduler): unit u is tile
// u - group_start[g] of the problem g whose range holds it (binary search over the
// problems' first units), a whole tile with the problem's whole K, rasterised inside
// the problem as tile_coords does.  Kept out of line like sk_next.
static __device__ __noinline__ void decode_grouped(int32_t u, const GemmParams& p, Unit& w) {
  int32_t lo = 0, hi = p.num_groups - 1;
  while (lo < hi) {
    const int32_t mid = (lo + hi + 1) >> 1;
    if (p.group_start[mid] <= u) lo = mid;
    else hi = mid - 1;
  }
  const GroupDesc& gd = p.groups[lo];
  w.g = lo;
  w.tile = u;
  w.half = -1;
  w.split = 0;
  w.nsplit = 1;
  w.kb0 = 0;
  w.kb1 = gd.k_blocks;
  const int32_t t = u - p.group_start[lo];
  const int32_t group = p.group_m * gd.num_n;
  const int32_t gi = t / group;
  const int32_t first_m = gi * p.group_m;
  const int32_t gm = min(gd.num_m - first_m, p.group_m);
  const int32_t r = t - gi * group;
  w.m_blk = first_m + r % gm;
  w.n_blk = r / gm;
}

// Whether walker_next will return another unit (the walker is not advanced).  Kept out
// of line like sk_next.
static __device__ __noinline__ bool walker_has_next(const Walker& k, int32_t first,
                                                    const GemmParams& p) {
  if (k.u < p.units) return true;
  if (first >= p.sk_workers) return false;
  const uint32_t W = (uint32_t)p.sk_workers;
  const uint32_t T = (uint32_t)(p.tiles - p.dp_tiles) * (uint32_t)p.k_blocks;
  return (uint32_t)first * T / W + (uint32_t)k.sk_done < ((uint32_t)first + 1u) * T / W;
}

// Cluster launch control (CLC): the units of a CTA (pair) are its own, u = blockIdx.x /
// CTA_GROUP, then the one of each launch it cancels.  Answer q (the unit after the CTA's
// q-th) lands in slot q % 4 of a ring in shared memory; the producer warp asks for it when
// it starts its q-th unit, and every warp that walks the units (producer, MMA issuer,
// epilogue warps; in both CTAs of a pair) reads it when it finishes that unit and frees
// the slot on the group leader's clc_empty barrier.
struct ClcLink {
  uint32_t resp0;      // answer slot 0 (16 bytes each)
  uint32_t full0;      // clc_full[0] (8 bytes each): armed by this CTA, completed by the answer
  uint32_t empty0;     // clc_empty[0] of this CTA: the readers of both CTAs arrive on the leader's
  uint32_t leader;     // cluster rank of the group leader
};

// (out of line, like sk_next, so that the epilogue's accumulator keeps its registers)
template <int CTA_GROUP>
static __device__ __noinline__ bool clc_next(const ClcLink& c, uint32_t q, const WaitCtl& ctl,
                                             int32_t& unit) {
  const uint32_t s = q & 3u;
  if (!warp_wait(c.full0 + 8u * s, (q >> 2) & 1u, ctl, kSiteClc)) return false;
  uint32_t x;
  const uint32_t got = clc_query(c.resp0 + 16u * s, x);
  __syncwarp();
  if (lane_id() == 0) {
    if constexpr (CTA_GROUP == 1) mbar_arrive(c.empty0 + 8u * s);
    else mbar_arrive_cluster(mapa_shared(c.empty0 + 8u * s, c.leader));
  }
  unit = (int32_t)(x / (uint32_t)CTA_GROUP);
  return got != 0;
}

// The producer warp asks for answer q (it starts its q-th unit): the leader waits until
// every reader has taken answer q - 4 out of the slot, each CTA arms its own barrier for
// the 16 bytes, and the leader's elected lane sends the request (to the whole cluster for
// a pair).
template <int CTA_GROUP>
__device__ __forceinline__ bool clc_request(const ClcLink& c, uint32_t q, bool leader,
                                            const WaitCtl& ctl) {
  const uint32_t s = q & 3u;
  if (leader && !warp_wait(c.empty0 + 8u * s, ((q >> 2) & 1u) ^ 1u, ctl, kSiteClc)) return false;
  mbar_arrive_expect_tx_elect(c.full0 + 8u * s, 16u);
  if (leader) clc_try_cancel_elect<CTA_GROUP == 2>(c.resp0 + 16u * s, c.full0 + 8u * s);
  return true;
}

// Only two 32-bit counters live across a unit; the stream-K range is recomputed from
// the worker's index on each call.  Under CLC, k.sk_done counts the units walked.
template <bool GROUPED, bool CLC = false, int CTA_GROUP = 1>
__device__ __forceinline__ bool walker_next(Walker& k, int32_t first, int32_t stride,
                                            const GemmParams& p, Unit& w,
                                            const ClcLink* clc = nullptr,
                                            const WaitCtl* ctl = nullptr) {
  if constexpr (CLC) {
    if (k.sk_done > 0 && !clc_next<CTA_GROUP>(*clc, (uint32_t)(k.sk_done - 1), *ctl, k.u))
      return false;
    ++k.sk_done;
    if constexpr (GROUPED) decode_grouped(k.u, p, w);
    else w = decode_unit(k.u, p);
    return true;
  }
  if (k.u < p.units) {
    if constexpr (GROUPED) decode_grouped(k.u, p, w);
    else w = decode_unit(k.u, p);
    k.u += stride;
    return true;
  }
  if constexpr (GROUPED) return false;
  if (first >= p.sk_workers) return false;
  return sk_next(k, first, p, w);
}

__device__ __forceinline__ int32_t chains_of(const Unit& w, int32_t chain_kb) {
  return (w.kb1 - w.kb0 + chain_kb - 1) / chain_kb;
}

// ------------------------------------------------------------- epilogue helpers --
template <int OUT>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (OUT == kOutF16) {
    __half2 h = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  } else {
    __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&h);
  }
}

// Fused epilogue on 32 consecutive values of row m starting at column n0, before they
// are rounded to the output type: v = act(alpha * v + beta * C[m][n] + bias[n])
// ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05", Part 6: Epilogue
// Visitor Trees, D = alpha * acc + beta * C; Classic Fused Epilogue: Bias + ReLU).
// C is read in its own type before this warp writes it; out-of-range columns (and rows)
// read as zero and are not stored.
template <int OUT>
__device__ __forceinline__ void fuse_piece(const GemmParams& p, int32_t m, int32_t n0, float* v) {
  const bool row_ok = m < p.M;
  const bool vec = p.vec_store && n0 + 32 <= p.N;  // C rows and this piece 16-byte aligned
#pragma unroll
  for (int j0 = 0; j0 < 32; j0 += 8) {
    float c[8], b[8];
#pragma unroll
    for (int t = 0; t < 8; ++t) c[t] = 0.0f;
    if (p.beta != 0.0f && row_ok) {
      if constexpr (OUT == kOutF32) {
        const float* src = reinterpret_cast<const float*>(p.C) + (size_t)m * p.N + n0 + j0;
        if (vec) {
          const uint4 x = ld_global_cg_v4(src), y = ld_global_cg_v4(src + 4);
          c[0] = __uint_as_float(x.x); c[1] = __uint_as_float(x.y);
          c[2] = __uint_as_float(x.z); c[3] = __uint_as_float(x.w);
          c[4] = __uint_as_float(y.x); c[5] = __uint_as_float(y.y);
          c[6] = __uint_as_float(y.z); c[7] = __uint_as_float(y.w);
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t)
            if (n0 + j0 + t < p.N) c[t] = src[t];
        }
      } else {
        const uint16_t* src = reinterpret_cast<const uint16_t*>(p.C) + (size_t)m * p.N + n0 + j0;
        uint16_t h[8];
        if (vec) {
          const uint4 x = ld_global_cg_v4(src);
          const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
          for (int t = 0; t < 8; ++t) h[t] = (uint16_t)(w[t >> 1] >> ((t & 1) * 16));
        } else {
#pragma unroll
          for (int t = 0; t < 8; ++t) h[t] = n0 + j0 + t < p.N ? src[t] : (uint16_t)0;
        }
#pragma unroll
        for (int t = 0; t < 8; ++t) {
          if constexpr (OUT == kOutF16) c[t] = __half2float(__ushort_as_half(h[t]));
          else c[t] = __bfloat162float(__ushort_as_bfloat16(h[t]));
        }
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) b[t] = 0.0f;
    if (p.bias) {
      const float* src = p.bias + n0 + j0;
      if (n0 + j0 + 8 <= p.N) {
        const uint4 x = ld_global_cg_v4(src), y = ld_global_cg_v4(src + 4);
        b[0] = __uint_as_float(x.x); b[1] = __uint_as_float(x.y);
        b[2] = __uint_as_float(x.z); b[3] = __uint_as_float(x.w);
        b[4] = __uint_as_float(y.x); b[5] = __uint_as_float(y.y);
        b[6] = __uint_as_float(y.z); b[7] = __uint_as_float(y.w);
      } else {
#pragma unroll
        for (int t = 0; t < 8; ++t)
          if (n0 + j0 + t < p.N) b[t] = src[t];
      }
    }
#pragma unroll
    for (int t = 0; t < 8; ++t) {
      float x = fmaf(p.beta, c[t], p.alpha * v[j0 + t]) + b[t];
      if (p.relu) x = x > 0.0f ? x : 0.0f;  // NaN and -0 become +0, as max(x, 0) reads
      v[j0 + t] = x;
    }
  }
}

// Direct stores of 32 consecutive values of one row (used when C cannot take TMA) into
// the M x N row-major C; vec_store: C's rows are 16-byte aligned.
template <int OUT>
__device__ __forceinline__ void store_row_to(void* C, int32_t M, int32_t N, int32_t vec_store,
                                             int32_t m, int32_t n0, const float* v) {
  struct {
    void* C;
    int32_t M, N, vec_store;
  } p{C, M, N, vec_store};
  if (m >= p.M) return;
  if constexpr (OUT == kOutF32) {
    float* dst = reinterpret_cast<float*>(p.C) + (size_t)m * p.N + n0;
    if (p.vec_store && n0 + 32 <= p.N) {
#pragma unroll
      for (int j = 0; j < 32; j += 4)
        st_global_v4(dst + j, __float_as_uint(v[j]), __float_as_uint(v[j + 1]),
                     __float_as_uint(v[j + 2]), __float_as_uint(v[j + 3]));
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) dst[j] = v[j];
    }
  } else {
    uint32_t packed[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) packed[j] = pack2<OUT>(v[2 * j], v[2 * j + 1]);
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.C) + (size_t)m * p.N + n0;
    if (p.vec_store && n0 + 32 <= p.N) {
#pragma unroll
      for (int j = 0; j < 16; j += 4)
        st_global_v4(dst + 2 * j, packed[j], packed[j + 1], packed[j + 2], packed[j + 3]);
    } else {
#pragma unroll
      for (int j = 0; j < 32; ++j)
        if (n0 + j < p.N) dst[j] = (uint16_t)(packed[j >> 1] >> ((j & 1) * 16));
    }
  }
}

template <int OUT>
__device__ __forceinline__ void store_row_direct(const GemmParams& p, int32_t m, int32_t n0,
                                                 const float* v) {
  store_row_to<OUT>(p.C, p.M, p.N, p.vec_store, m, n0, v);
}

// Direct stores of a warp's 32 rows x 32 columns (rows m_first.., columns n0..; each lane
// holds its own row's 32 values in v), used when C is not written by TMA (its rows are not
// 16-byte aligned, or a tile's columns are not a whole number of staging boxes).  The
// piece goes through the warp's staging box, transposed: each store instruction then
// writes 32 consecutive elements of one row of C, instead of one element of 32 rows.  The
// box's 16-byte chunks are XOR-swizzled by row so that neither side conflicts on banks.
template <int OUT>
__device__ __forceinline__ void store_piece_rows(void* C, int32_t M, int32_t N, int32_t m_first,
                                                 int32_t n0, const float* v, uint32_t staging) {
  const uint32_t lane = lane_id();
#pragma unroll
  for (int c = 0; c < 8; ++c)
    st_shared_v4(staging + lane * 128u + (((uint32_t)c ^ (lane & 7u)) << 4), __float_as_uint(v[4 * c]),
                 __float_as_uint(v[4 * c + 1]), __float_as_uint(v[4 * c + 2]),
                 __float_as_uint(v[4 * c + 3]));
  __syncwarp();
  const int32_t n = n0 + (int32_t)lane;
  const bool col_ok = n < N;
#pragma unroll 4
  for (int r = 0; r < 32; ++r) {
    const int32_t m = m_first + r;
    const float x = __uint_as_float(ld_shared_u32(
        staging + (uint32_t)r * 128u + (((lane >> 2) ^ ((uint32_t)r & 7u)) << 4) + (lane & 3u) * 4u));
    if (col_ok && m < M) {
      if constexpr (OUT == kOutF32) {
        reinterpret_cast<float*>(C)[(size_t)m * N + n] = x;
      } else if constexpr (OUT == kOutF16) {
        reinterpret_cast<uint16_t*>(C)[(size_t)m * N + n] = __half_as_ushort(__float2half_rn(x));
      } else {
        reinterpret_cast<uint16_t*>(C)[(size_t)m * N + n] =
            __bfloat16_as_ushort(__float2bfloat16_rn(x));
      }
    }
  }
  __syncwarp();  // (the box is refilled by the next piece)
}

// The swapped tiling's store: v[j] = C[m0 + j][n] for j < NV, n this thread's column of C
// (in_tile: n is one of the CTA's rows of B).  The 32 lanes of a warp hold 32 consecutive
// columns, so each store instruction writes 32 consecutive elements of one row of C.
template <int OUT, int NV>
__device__ __forceinline__ void store_col_direct(const GemmParams& p, int32_t n, bool in_tile,
                                                 int32_t m0, const float* v) {
  if (!in_tile || n >= p.N) return;
  const int32_t rows = p.M - m0;
  if constexpr (OUT == kOutF32) {
    float* dst = reinterpret_cast<float*>(p.C) + (size_t)m0 * p.N + n;
#pragma unroll
    for (int j = 0; j < NV; ++j)
      if (j < rows) dst[(size_t)j * p.N] = v[j];
  } else {
    uint16_t* dst = reinterpret_cast<uint16_t*>(p.C) + (size_t)m0 * p.N + n;
#pragma unroll
    for (int j = 0; j < NV; j += 2) {
      const uint32_t two = pack2<OUT>(v[j], v[j + 1]);
      if (j < rows) dst[(size_t)j * p.N] = (uint16_t)(two & 0xFFFFu);
      if (j + 1 < rows) dst[(size_t)(j + 1) * p.N] = (uint16_t)(two >> 16);
    }
  }
}

// One 32-column piece of a single-chain unit's output, for the warp's rows: the TMEM
// accumulator at `taddr`, or for a split tile the slices summed in slice order (the
// own slice's partial is the TMEM value itself; two slices add in either order to the
// same bits).  `ws_lane` is this lane's start of the tile's workspace block, `col` the
// piece's first column within the warp's block.  KX: the other K slice of a cluster
// split was received into shared memory at kx_lane (this lane's 16 bytes of the warp's
// block, 512 bytes per 4 columns); 0 for the slice that sent it.
template <bool KX = false>
__device__ __forceinline__ void one_chain_piece(uint32_t taddr, const Unit& w, const float* ws_lane,
                                                size_t slice_stride, int col, float (&v)[32],
                                                uint32_t kx_lane = 0) {
  uint32_t r[32];
  tmem_ld_32x32b_x32(taddr, r);
  tmem_ld_wait(r);
  if constexpr (KX) {
    if (kx_lane != 0) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        const uint4 x = ld_shared_v4(kx_lane + (uint32_t)((col + j) / 4) * 512u);
        v[j] = __uint_as_float(r[j]) + __uint_as_float(x.x);
        v[j + 1] = __uint_as_float(r[j + 1]) + __uint_as_float(x.y);
        v[j + 2] = __uint_as_float(r[j + 2]) + __uint_as_float(x.z);
        v[j + 3] = __uint_as_float(r[j + 3]) + __uint_as_float(x.w);
      }
      return;
    }
  }
  if (w.nsplit <= 1) {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
  } else if (w.nsplit == 2) {
    const float* other = ws_lane + (size_t)(1 - w.split) * slice_stride;
#pragma unroll
    for (int j = 0; j < 32; j += 4) {
      const uint4 x = ld_global_cg_v4(other + (col + j) * 32);
      v[j] = __uint_as_float(r[j]) + __uint_as_float(x.x);
      v[j + 1] = __uint_as_float(r[j + 1]) + __uint_as_float(x.y);
      v[j + 2] = __uint_as_float(r[j + 2]) + __uint_as_float(x.z);
      v[j + 3] = __uint_as_float(r[j + 3]) + __uint_as_float(x.w);
    }
  } else {
#pragma unroll
    for (int j = 0; j < 32; ++j) v[j] = 0.0f;
    for (int32_t sl = 0; sl < w.nsplit; ++sl) {
#pragma unroll
      for (int j = 0; j < 32; j += 4) {
        float t[4];
        if (sl == w.split) {
#pragma unroll
          for (int u = 0; u < 4; ++u) t[u] = __uint_as_float(r[j + u]);
        } else {
          const uint4 x = ld_global_cg_v4(ws_lane + (size_t)sl * slice_stride + (col + j) * 32);
          t[0] = __uint_as_float(x.x);
          t[1] = __uint_as_float(x.y);
          t[2] = __uint_as_float(x.z);
          t[3] = __uint_as_float(x.w);
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) v[j + u] = sl == 0 ? t[u] : v[j + u] + t[u];
      }
    }
  }
}

// ------------------------------------------------------------- shared memory map --
// One-CTA rings deeper than a 128-row A tile allows (10 stages of 128 columns, 5 of 256;
// with the staging in the ring, 12 and 6) hold 16 rows of A per stage, for row tiles of
// M <= 16 rows: A's stage stride is then 2 KiB, and the MMA's 128-row A operand runs on
// over the following stages' bytes.  The rows past 16 are whatever those bytes hold; each
// feeds only its own accumulator row, which is never stored, and the span stays inside
// the ring.  The ring keeps more of B in flight (160 KiB against 96 or 128).
// RING_STAGING (the cluster K split, one unit per CTA): the epilogue's staging boxes lie
// inside the operand ring, after the blocks the K slices exchange, instead of after it:
// the ring is idle once the unit's MMAs have completed, and the 32 KiB go to one more
// stage (a CTA streams at about its bytes in flight over the round trip of a stage).
// NO_STAGING (the swapped tiling, whose epilogue writes C with direct stores): no staging
// boxes at all, and the 32 KiB go to one more stage for the same reason.
template <int CTA_GROUP, int BN, int STAGES, bool RING_STAGING = false, bool NO_STAGING = false>
struct Layout {
  static constexpr int kEpiWarps = 8;
  static constexpr uint32_t kThreads = 32 * (2 + kEpiWarps);
  static constexpr int kRowsB = BN / CTA_GROUP;                // B rows loaded per CTA
  static constexpr bool kSmallA =
      CTA_GROUP == 1 && ((BN == 128 && STAGES > 7) || (BN == 256 && STAGES > 4));
  static constexpr int kARows = kSmallA ? 16 : kBlockM;        // A rows held per stage
  static constexpr uint32_t kABytes = kARows * kBlockK * 2;    // 16 KiB, or 2 KiB
  static constexpr uint32_t kBBytes = kRowsB * kBlockK * 2;
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;   // per CTA
  static constexpr uint32_t kTxBytes = kStageBytes * CTA_GROUP;  // expected on the leader
  static constexpr uint32_t kTxBytesHalf = (kABytes + kBBytes / 2) * CTA_GROUP;  // half-tile unit
  static constexpr uint32_t kStagingBytes = 32 * 128;           // one 32-row x 128 B box
  static constexpr uint32_t kAOff = 0;
  static constexpr uint32_t kBOff = STAGES * kABytes;
  static constexpr uint32_t kRingEnd = kBOff + STAGES * kBBytes;
  // the K slices' exchange blocks: 32 rows x BN/2 fp32 columns per epilogue warp
  static constexpr uint32_t kKxBytes = kEpiWarps * 32u * (BN / 2) * 4u;
  static constexpr uint32_t kCOff = RING_STAGING ? kKxBytes : kRingEnd;
  static constexpr uint32_t kBarOff =
      (RING_STAGING || NO_STAGING) ? kRingEnd : kCOff + kEpiWarps * kStagingBytes;
  // cluster launch control: a ring of 16-byte answers
  static constexpr uint32_t kClcSlots = 4;
  // full[S], empty[S], acc_full[4], acc_empty[4], drain, kx_ready[8], kx_go[8],
  // clc_full[4], clc_empty[4]
  static constexpr uint32_t kNumBars = 2 * STAGES + 9 + 2 * kEpiWarps + 2 * kClcSlots;
  static constexpr uint32_t kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kTmemSlotOff + 4;
  static constexpr uint32_t kClcOff = (kAbortOff + 4 + 15) & ~15u;
  static constexpr uint32_t kEnd = kClcOff + kClcSlots * 16;
  static constexpr uint32_t kDynamicBytes = kEnd + 1024;  // slack for 1024-byte alignment
  static_assert(kABytes % 1024 == 0 && kBBytes % 1024 == 0 && kBOff % 1024 == 0 &&
                    kCOff % 1024 == 0,
                "every operand stage and staging box must start on a 1024-byte boundary");
  static_assert(kDynamicBytes <= 227 * 1024, "shared memory over the per-block limit");
  static_assert(!(RING_STAGING && NO_STAGING), "one staging placement");
  static_assert(!RING_STAGING || kCOff + kEpiWarps * kStagingBytes <= kRingEnd,
                "the staging boxes must fit in the ring after the exchange blocks");
  // the MMA reads 128 rows of A from every stage's A start: inside the ring
  static_assert((STAGES - 1) * kABytes + kBlockM * kBlockK * 2 <= kRingEnd,
                "the A operand's 128-row span must stay inside the operand ring");
};

// ONE_CHAIN: every work unit is a single accumulation chain (at most p.chain_kb
// k-blocks), so the epilogue streams the accumulator out of TMEM in 32-column pieces
// instead of first copying the warp's whole 32 x BN/2 block into registers; the
// registers this frees go to loads in flight in the split-K hand-over.
// FUSED: the fused epilogue (alpha, beta * C, bias, ReLU) is compiled in; kept out of
// the plain kernels, whose general epilogue it would push into more register spills.
// KIND 0: fp16/bf16 operands (tcgen05.mma kind::f16); KIND 1: FP8 operands (kind::f8f6f4);
// KIND 2: FP8 operands with blockwise scales (one chain per K block, general epilogue).
// Either way a K block is one 128-byte row of the swizzle atom: 64 or 128 elements.
// GROUPED: a grouped launch (p.groups): per-problem tensor maps, shapes and C; whole
// tiles only, general epilogue.
// KX2: every tile is two K slices computed by the two CTA groups (CTAs or pairs) of one
// cluster of 2 * CTA_GROUP CTAs; the second slice hands its accumulator to the first
// through distributed shared memory instead of the global workspace.  One unit per CTA
// group, single-chain epilogue.
// STAGED: in the general epilogue, the last K slice of a tile to finish on a CTA's last
// unit brings the other slices' partials into the idle operand ring with asynchronous
// copies instead of reading them into registers, and skips publishing its own when the
// others are all in (the stream-K fix-up).  Built for the plain kernels' split launches;
// the kernel for whole tiles keeps the direct form (its register allocation, and its
// time at 8192^3, measured better with that form than with the staged one or with none).
// SWAP: the operands' roles are exchanged for a few rows of A (decode shapes): B is the
// MMA's row operand, p.swap_rows (<= 128) of its rows per CTA loaded as a short box
// whose rows past the box only feed accumulator lanes that are never stored, and A's
// rows are the MMA's columns, BN of them per tile split over the pair like B's are
// otherwise.  A thread's accumulator row is then a column of C, and the epilogue writes
// it transposed.  CTA pairs, general epilogue, plain fp16/bf16, whole tiles.
// CLC: the units are handed out by cluster launch control instead of round-robin: the grid
// holds a CTA (pair) per unit and each running one takes over the work of launches that
// have not started (ClcLink above).  Grouped launches (whole tiles).
template <int CTA_GROUP, int BN, int STAGES, int OUT, bool ONE_CHAIN, bool FUSED, int KIND = 0,
          bool GROUPED = false, bool KX2 = false, bool STAGED = false, bool SWAP = false,
          bool CLC = false>
__global__ void __launch_bounds__((Layout<CTA_GROUP, BN, STAGES, KX2, SWAP>::kThreads), 1)
    gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                const __grid_constant__ CUtensorMap tmB2, const __grid_constant__ CUtensorMap tmC,
                const GemmParams p) {
  using L = Layout<CTA_GROUP, BN, STAGES, KX2, SWAP>;
  static_assert(BN == 128 || BN == 256 || BN == 320, "BN must be 128, 256 or 320");
  // 320 columns: two MMAs per K step (N = 256 and N = 64) into one 320-column
  // accumulator; built for the pair's cluster K split with single-chain slices only (one
  // unit per CTA group, so one accumulator slot)
  static_assert(BN != 320 || (CTA_GROUP == 2 && KX2 && ONE_CHAIN), "BN 320: pair, cluster K split");
  static_assert(CTA_GROUP == 1 || CTA_GROUP == 2, "CTA_GROUP must be 1 or 2");
  static_assert(KIND != 2 || !ONE_CHAIN, "blockwise scales need the general epilogue");
  static_assert(!GROUPED || (!ONE_CHAIN && !FUSED && KIND == 0),
                "grouped launches use the plain general epilogue");
  static_assert(!KX2 || (!FUSED && KIND == 0 && !GROUPED),
                "the cluster K split uses the plain epilogues");
  static_assert(!SWAP || (CTA_GROUP == 2 && BN != 320 && !ONE_CHAIN && !FUSED && KIND == 0 &&
                          !GROUPED && !KX2 && !STAGED),
                "the swapped tiling is a plain CTA-pair kernel with the general epilogue");
  static_assert(!CLC || (GROUPED && !SWAP), "cluster launch control serves grouped launches");
  // Accumulator slots in Tensor Memory: two, so that a unit's epilogue overlaps the next
  // chain's MMAs; four for blockwise scales with 128-column tiles, whose chains are one K
  // block each (the MMA then runs up to three K blocks ahead of the epilogue that scales
  // them; Tensor Memory holds 512 columns).  One for 320 columns.
  constexpr uint32_t kSlots = (KIND == 2 && BN == 128) ? 4u : 2u;
  constexpr uint32_t kSlotShift = kSlots == 4u ? 2u : 1u;
  constexpr uint32_t kTmemCols = BN == 320 ? 512 : kSlots * BN;
  constexpr int kHalf = BN / 2;                // columns per epilogue warp
  constexpr int kPieces = kHalf / 32;          // tcgen05.ld x32 pieces per warp
  constexpr int kOutBytes = OUT == kOutF32 ? 4 : 2;
  constexpr int kBoxCols = 128 / kOutBytes;    // columns of one 128-byte staging row
  constexpr int kBoxes = kHalf / kBoxCols;     // staging boxes per warp
  constexpr bool kTmaStoreOk = kHalf % kBoxCols == 0;  // (BN 320 writes C with direct stores)
  // rows of the MMA's row operand per CTA and per tile: 128 (A), or with SWAP the
  // p.swap_rows rows of B per CTA
  const int32_t rows_cta = SWAP ? p.swap_rows : kBlockM;
  const int32_t kRowsTile = rows_cta * CTA_GROUP;
  constexpr int kKbElems = KIND == 0 ? kBlockK : 2 * kBlockK;  // K elements per K block

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sA = base + L::kAOff;
  const uint32_t sB = base + L::kBOff;
  const uint32_t sC = base + L::kCOff;
  const uint32_t bar0 = base + L::kBarOff;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto acc_full_bar = [&](uint32_t i) { return bar0 + 8u * (2 * STAGES + i); };
  auto acc_empty_bar = [&](uint32_t i) { return bar0 + 8u * (2 * STAGES + 4 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 8);
  auto kx_ready_bar = [&](uint32_t w) { return bar0 + 8u * (2 * STAGES + 9 + w); };
  auto kx_go_bar = [&](uint32_t w) { return bar0 + 8u * (2 * STAGES + 9 + L::kEpiWarps + w); };
  auto clc_full_bar = [&](uint32_t s) { return bar0 + 8u * (2 * STAGES + 9 + 2 * L::kEpiWarps + s); };
  auto clc_empty_bar = [&](uint32_t s) {
    return bar0 + 8u * (2 * STAGES + 9 + 2 * L::kEpiWarps + L::kClcSlots + s);
  };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOff);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + L::kAbortOff);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const WaitCtl ctl{p.wait_limit_ns, p.status, abort_flag};
  // Cluster rank; with KX2 the cluster holds two CTA groups (K slices 0 and 1), the
  // group of slice s starting at rank s * CTA_GROUP.
  const uint32_t crank = (CTA_GROUP == 2 || KX2) ? cluster_ctarank() : 0u;
  const uint32_t rank = CTA_GROUP == 2 ? (KX2 ? (crank & 1u) : crank) : 0u;  // place in the pair
  const uint32_t group_base = KX2 ? crank - rank : 0u;  // cluster rank of the group's leader
  const uint32_t slice_k = KX2 ? crank / CTA_GROUP : 0u;
  // the same rank of the other K slice's CTA group
  const uint32_t kx_peer = slice_k == 0 ? crank + (uint32_t)CTA_GROUP : crank - (uint32_t)CTA_GROUP;
  const uint16_t pair_mask = (uint16_t)(KX2 ? (0x3u << group_base) : 0x3u);
  // a stage's commit frees it in both CTAs of the pair, whose copies land in it
  const uint16_t stage_mask = pair_mask;
  const bool leader = rank == 0;
  const int32_t first_unit = (int32_t)(blockIdx.x / CTA_GROUP);
  const int32_t unit_stride = (int32_t)(gridDim.x / CTA_GROUP);
  const ClcLink clc{base + L::kClcOff, clc_full_bar(0), clc_empty_bar(0), group_base};

  // ---------------------------------------------------------------- setup --
  if (warp == 0 && lane == 0) {
    for (uint32_t s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);   // the leader's producer arms it; copies complete it
      mbar_init(empty_bar(s), 1);  // one commit per use
    }
    for (uint32_t i = 0; i < kSlots; ++i) {
      mbar_init(acc_full_bar(i), 1);
      mbar_init(acc_empty_bar(i), L::kEpiWarps * CTA_GROUP);  // every epilogue warp of the pair
    }
    if constexpr (KX2) {
      for (uint32_t w = 0; w < L::kEpiWarps; ++w) {
        mbar_init(kx_ready_bar(w), 1);  // the receiving warp arms it; the sender's bytes complete it
        mbar_init(kx_go_bar(w), 1);     // the receiving warp: its ring is free
      }
    }
    if constexpr (CLC) {
      for (uint32_t i = 0; i < L::kClcSlots; ++i) {
        mbar_init(clc_full_bar(i), 1);  // this CTA's producer arms it; the answer completes it
        // every reader: producer, MMA issuer (leader) and epilogue warps of the group
        mbar_init(clc_empty_bar(i), CTA_GROUP == 2 ? 2 * (2 + L::kEpiWarps) - 1 : 2 + L::kEpiWarps);
      }
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    if constexpr (!GROUPED) {  // a grouped launch's maps live in global memory
      tma_prefetch_desc(&tmA);
      tma_prefetch_desc(&tmB);
      if (p.half_tail || BN == 320) tma_prefetch_desc(&tmB2);
      if (p.tma_store) tma_prefetch_desc(&tmC);
    }
  }
  if (warp == 1) {
    tmem_alloc<CTA_GROUP>(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish<CTA_GROUP>();
  }
  tc_fence_before();
  if constexpr (CTA_GROUP == 2 || KX2) cluster_sync();
  else __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  // Launched with programmatic stream serialisation: the setup above overlaps the tail
  // of the preceding kernel; nothing in global memory (A, B, C, the workspace, the
  // status word) is touched before that kernel has completed.  The next kernel may
  // then be scheduled as this one's CTAs exit.
  grid_dependency_wait();
  grid_launch_dependents();

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer --
    // The whole warp runs the loop; one elected lane issues each copy.  B's copy goes
    // out ahead of A's: on the decode shapes B streams from DRAM while A stays in L2
    // (1-3% faster there, neutral on square shapes; measured).
    uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
    uint32_t clc_asked = 0;  // answers this warp has asked for (CLC)
    bool ok = true;
    // When every B element is read by one tile only (one row of tiles), B's lines are
    // marked first to be evicted and A's last: A, re-read by every tile from L2, then
    // stays there however far apart in K the tiles running at once are (stream-K).  The
    // loop is built twice, with and without the hint: the hinted copy, even with the
    // default policy, or a branch between the two forms in the loop, cost 3-4% at
    // 4096^3 (measured).
    auto produce = [&](auto hinted) {
      constexpr bool kHint = decltype(hinted)::value;
      // (with SWAP the row operand, tmA, is B: B's lines go first, A's last either way)
      const uint64_t pol_a = kHint ? (SWAP ? l2_policy_evict_first() : l2_policy_evict_last()) : 0ull;
      const uint64_t pol_b = kHint ? (SWAP ? l2_policy_evict_last() : l2_policy_evict_first()) : 0ull;
      Walker walk{first_unit, 0};
      Unit w;
      while (ok && walker_next<GROUPED, CLC, CTA_GROUP>(walk, first_unit, unit_stride, p, w, &clc, &ctl)) {
        const int32_t a_row = w.m_blk * kRowsTile + (int32_t)rank * rows_cta;
        // a half-tile unit loads half the B rows (through the half-height map tmB2)
        const bool half = w.half >= 0;
        // (BN 320: each CTA's first 128 B rows are columns 128 * rank.. of the tile, its
        // last 32 columns 256 + 32 * rank.., so that the accumulator's columns are in order)
        const int32_t b_row = w.n_blk * BN +
                              (half ? w.half * (BN / 2) + (int32_t)rank * (L::kRowsB / 2)
                                    : (int32_t)rank * (BN == 320 ? 128 : L::kRowsB));
        [[maybe_unused]] const int32_t b_row320 = w.n_blk * BN + 256 + (int32_t)rank * 32;
        const CUtensorMap* mapB = half ? &tmB2 : &tmB;
        const CUtensorMap* mapA = &tmA;
        uint32_t tx = (half ? L::kTxBytesHalf : L::kTxBytes) - p.a_tx_short;
        if constexpr (GROUPED) {
          // the problem's own maps, written by the host before the launch
          const GroupDesc* gd = p.groups + w.g;
          mapA = &gd->tmA;
          mapB = &gd->tmB;
          tx = L::kTxBytes - gd->a_tx_short;
          fence_tensormap_acquire(mapA);
          fence_tensormap_acquire(mapB);
        }
        // Streaming B from DRAM (decode shapes): keep more requests in flight than the
        // shared-memory ring holds by prefetching B into L2 prefetch_kb k-blocks ahead
        // ("A Blackwell GEMM by Hand in CuTe DSL", section 8: TMA prefetch).
        if (p.prefetch_kb > 0)
          for (int32_t kb = w.kb0; kb < min(w.kb0 + p.prefetch_kb, w.kb1); ++kb)
            tma_prefetch_l2_2d_elect(mapB, kb * kKbElems, b_row);
        for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
          if (p.prefetch_kb > 0 && kb + p.prefetch_kb < w.kb1)
            tma_prefetch_l2_2d_elect(mapB, (kb + p.prefetch_kb) * kKbElems, b_row);
          if (!warp_wait_inl(empty_bar(stage), phase ^ 1u, ctl, kSiteEmpty)) {
            ok = false;
            break;
          }
          if constexpr (CTA_GROUP == 1) {
            mbar_arrive_expect_tx_elect(full_bar(stage), tx);
            if constexpr (kHint) {
              tma_load_2d_hint_elect(sB + stage * L::kBBytes, mapB, kb * kKbElems, b_row,
                                     full_bar(stage), pol_b);
              tma_load_2d_hint_elect(sA + stage * L::kABytes, mapA, kb * kKbElems, a_row,
                                     full_bar(stage), pol_a);
            } else {
              tma_load_2d_elect(sB + stage * L::kBBytes, mapB, kb * kKbElems, b_row, full_bar(stage));
              tma_load_2d_elect(sA + stage * L::kABytes, mapA, kb * kKbElems, a_row, full_bar(stage));
            }
          } else {
            // Both CTAs' copies complete on the leader's full barrier; the leader arms it
            // with the bytes of the pair.
            const uint32_t leader_full = mapa_shared(full_bar(stage), group_base);
            if (leader) mbar_arrive_expect_tx_elect(full_bar(stage), tx);
            if constexpr (SWAP) {
              // the row operand (B's rows, streamed from DRAM) first, as B otherwise
              if constexpr (kHint)
                tma_load_2d_pair_hint_elect(sA + stage * L::kABytes, mapA, kb * kKbElems, a_row,
                                            leader_full, pol_a);
              else
                tma_load_2d_pair_elect(sA + stage * L::kABytes, mapA, kb * kKbElems, a_row,
                                       leader_full);
            }
            if constexpr (kHint) {
              tma_load_2d_pair_hint_elect(sB + stage * L::kBBytes, mapB, kb * kKbElems, b_row,
                                          leader_full, pol_b);
              if constexpr (BN == 320)  // rows 256 + 32 * rank.. of the tile (32-row map)
                tma_load_2d_pair_hint_elect(sB + stage * L::kBBytes + 128 * 128, &tmB2,
                                            kb * kKbElems, b_row320, leader_full, pol_b);
              if constexpr (!SWAP)
                tma_load_2d_pair_hint_elect(sA + stage * L::kABytes, mapA, kb * kKbElems, a_row,
                                            leader_full, pol_a);
            } else {
              tma_load_2d_pair_elect(sB + stage * L::kBBytes, mapB, kb * kKbElems, b_row,
                                     leader_full);
              if constexpr (BN == 320)
                tma_load_2d_pair_elect(sB + stage * L::kBBytes + 128 * 128, &tmB2, kb * kKbElems,
                                       b_row320, leader_full);
              if constexpr (!SWAP)
                tma_load_2d_pair_elect(sA + stage * L::kABytes, mapA, kb * kKbElems, a_row,
                                       leader_full);
            }
          }
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if constexpr (CLC) {
          // Ask for the unit after this one only now that this one's loads are all issued:
          // a unit is claimed as late as the ring still hides the answer's latency (its
          // stages are still being multiplied), so that a CTA holds no claimed unit it has
          // not started while others run out of work.  Asking at the unit's start, or as
          // soon as the previous answer was in, balanced worse (measured).
          if (ok) {
            if (!clc_request<CTA_GROUP>(clc, clc_asked, leader, ctl)) {
              ok = false;
              break;
            }
            ++clc_asked;
          }
        }
      }
    };
    if (p.l2_hint == 2) produce(std::true_type{});
    else produce(std::false_type{});
    // No copy may still be landing in shared memory when the CTA exits.
    if (lane == 0) {
      if (leader) {
        for (uint32_t s = 0; s < STAGES; ++s)
          if (armed & (1u << s)) wait_parity_drain(full_bar(s), (armed_phase >> s) & 1u, ctl);
        // nor an answer of cluster launch control (after an abort one may be under way)
        if (CLC && clc_asked > 0)
          wait_parity_drain(clc_full_bar((clc_asked - 1u) & 3u), ((clc_asked - 1u) >> 2) & 1u, ctl);
      } else if (*abort_flag) {
        // The follower's copies complete on the leader's barrier, which it cannot poll;
        // normally every one of them was consumed by an MMA before the teardown.  On an
        // abort, give any copy still in flight time to land.
        pause_ns(200000);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer --
    // In the leader the whole warp runs the loop, one elected lane issues the MMAs
    // and commits; descriptors advance by adding the stage offset (>> 4) to the
    // start-address field and 2 (32 bytes) per 16-deep K step.
    if (leader) {
      uint32_t stage = 0, phase = 0, iter = 0;
      bool ok = true;
      const uint64_t desc_a0 = smem_desc_sw128_kmajor(sA);
      const uint64_t desc_b0 = smem_desc_sw128_kmajor(sB);
      if (p.test_stall) ok = warp_wait(drain_bar, 0, ctl, kSiteTestStall);
      Walker walk{first_unit, 0};
      Unit w;
      while (ok && walker_next<GROUPED, CLC, CTA_GROUP>(walk, first_unit, unit_stride, p, w, &clc, &ctl)) {
        const uint32_t idesc = w.half >= 0 ? p.idesc_half : p.idesc;
        if constexpr (KIND == 2) {
          // Blockwise scales: every K block is a chain of its own, on one operand stage and
          // one accumulator slot, whose stage commit also tells the epilogue.  A flat loop
          // with its bound in a register: re-reading the unit's fields (which the asm
          // statements' memory clobbers force) cost ~140 of the ~830 cycles the loop took
          // per K block (clock64 trace, 8192^3).
          const int32_t kb_end = w.kb1;
          for (int32_t kb = w.kb0; kb < kb_end; ++kb) {
            const uint32_t slot = iter & (kSlots - 1u), acc_phase = (iter >> kSlotShift) & 1u;
            // The slot and the stage tested together, one vote for the two when both are
            // complete (8192^3 514.0 -> 493.9 us against a vote per barrier, A/B on one
            // GPU); the bounded waits otherwise.
            const bool both =
                __any_sync(0xFFFFFFFFu, mbar_try_wait(acc_empty_bar(slot), acc_phase ^ 1u) &&
                                            mbar_try_wait(full_bar(stage), phase));
            if (!both && (!warp_wait_inl(acc_empty_bar(slot), acc_phase ^ 1u, ctl, kSiteAccEmpty) ||
                          !warp_wait_inl(full_bar(stage), phase, ctl, kSiteFull))) {
              ok = false;
              break;
            }
            tc_fence_after();
            umma_stage_elect<CTA_GROUP, KIND>(tmem_base + slot * BN,
                                              desc_a0 + ((stage * L::kABytes) >> 4),
                                              desc_b0 + ((stage * L::kBBytes) >> 4), idesc, 0u,
                                              empty_bar(stage), stage_mask);
            if (++stage == STAGES) {
              stage = 0;
              phase ^= 1u;
            }
            ++iter;
          }
        } else {
          for (int32_t c0 = w.kb0; c0 < w.kb1 && ok; c0 += p.chain_kb) {
            const int32_t c1 = min(c0 + p.chain_kb, w.kb1);
            const uint32_t slot = iter & (kSlots - 1u), acc_phase = (iter >> kSlotShift) & 1u;
            if (!warp_wait_inl(acc_empty_bar(slot), acc_phase ^ 1u, ctl, kSiteAccEmpty)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t d_tmem = tmem_base + slot * BN;
            for (int32_t kb = c0; kb < c1; ++kb) {
              if (!warp_wait_inl(full_bar(stage), phase, ctl, kSiteFull)) {
                ok = false;
                break;
              }
              tc_fence_after();
              const uint64_t da = desc_a0 + ((stage * L::kABytes) >> 4);
              const uint64_t db = desc_b0 + ((stage * L::kBBytes) >> 4);
              // four MMAs of 32 bytes of K, then the commit that frees the stage (in both
              // CTAs) once they are done
              static_assert(kBlockK * 2 == 128, "umma_stage_elect covers 128 bytes of K");
              if constexpr (BN == 320) {
                // columns 0-255 from each CTA's first 128 B rows, 256-319 from the next 32
                umma_stage320_elect(d_tmem, da, db, p.idesc, p.idesc_half, kb > c0 ? 1u : 0u,
                                    empty_bar(stage), stage_mask);
              } else {
                umma_stage_elect<CTA_GROUP, KIND>(d_tmem, da, db, idesc, kb > c0 ? 1u : 0u,
                                                  empty_bar(stage), stage_mask);
              }
              if (++stage == STAGES) {
                stage = 0;
                phase ^= 1u;
              }
            }
            if (!ok) break;
            if constexpr (CTA_GROUP == 1) umma_commit_elect<1>(acc_full_bar(slot));
            else umma_commit_pair_elect(acc_full_bar(slot), pair_mask);
            ++iter;
          }
        }
      }
      // Every issued MMA must finish before TMEM is released.
      umma_commit_elect<CTA_GROUP>(drain_bar);
      if (lane == 0) wait_parity_drain(drain_bar, 0, ctl);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    const uint32_t ew = warp - 2;                // 0..7
    const uint32_t q = warp & 3u;                // TMEM lane quarter this warp may read
    const uint32_t h = ew >> 2;                  // column half
    const uint32_t row = q * 32u + lane;         // accumulator row held by this thread
    const uint32_t staging = sC + ew * L::kStagingBytes;
    uint32_t iter = 0;
    uint32_t e_stage = 0, e_phase = 0;  // (blockwise: the operand stage of chain iter)
    bool ok = true;
    Walker walk{first_unit, 0};
    Unit w;
    if constexpr (ONE_CHAIN) {
      constexpr size_t kBlockFloats = 32 * kHalf;
      constexpr size_t kBlocksPerSlice = (size_t)CTA_GROUP * 8;  // (rank, quarter, half)
      constexpr size_t kSliceStride = kBlocksPerSlice * kBlockFloats;
      const size_t my_block = ((size_t)rank * 4 + q) * 2 + h;
      while (ok && walker_next<GROUPED, CLC, CTA_GROUP>(walk, first_unit, unit_stride, p, w, &clc, &ctl)) {
        // in a half-tile unit the h = 1 warps only take part in the slot hand-over, and
        // so do warps whose 32 rows all lie at or past M (no partial, no store)
        const int32_t m0 = w.m_blk * kRowsTile + (int32_t)rank * rows_cta;
        const bool active = (w.half < 0 || h == 0) && m0 + (int32_t)(q * 32u) < p.M;
        const uint32_t slot = iter & (kSlots - 1u), acc_phase = (iter >> kSlotShift) & 1u;
        if (!warp_wait_inl(acc_full_bar(slot), acc_phase, ctl, kSiteAccFull)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((q * 32u) << 16) + slot * BN + h * kHalf;
        const int32_t n_half = w.n_blk * BN + (w.half >= 0 ? w.half : (int32_t)h) * kHalf;
        bool emit = active;
        const float* ws_lane = nullptr;
        uint32_t kx_lane = 0;
        if constexpr (KX2) {
          // The two K slices of the tile are the two CTA groups of this cluster, and
          // each finishes one column half of it: slice k the warps of half h = k.  A
          // ring is idle once its MMAs completed; the finishing warp takes the other
          // slice's partial there (its 32 rows x BN/2 columns, 16 bytes per lane and 4
          // columns), adds it to its own and emits C; the warp of the other half sends
          // its partial the other way.  A sender's own ring holds the partial until the
          // copy has read it: the teardown's cluster barrier waits for the receiver,
          // which waits for the copy.
          constexpr uint32_t kKxWarpBytes = 32u * kHalf * 4u;
          static_assert(L::kEpiWarps * kKxWarpBytes <= STAGES * L::kStageBytes,
                        "the received partials must fit in the operand ring");
          const uint32_t wbuf = base + L::kAOff + ew * kKxWarpBytes;
          if (active && w.nsplit > 1 && h == slice_k) {
            if (lane == 0) {
              // (its own barrier: a local arm; the go carries no data of this warp's, only
              // that its ring is idle -- its MMAs are complete -- so a relaxed arrive: the
              // cluster-scope release forms cost about a microsecond each, measured)
              mbar_arrive_expect_tx(kx_ready_bar(ew), kKxWarpBytes);
              mbar_arrive_cluster_relaxed(mapa_shared(kx_go_bar(ew), kx_peer));
            }
            if (!warp_wait(kx_ready_bar(ew), 0, ctl, kSiteKx)) {
              ok = false;
              break;
            }
            kx_lane = wbuf + lane * 16u;
          } else if (active && w.nsplit > 1) {
            // The other half: stage the partial in this CTA's own ring (idle too), then,
            // once the other slice's warp is ready for it, one bulk copy into its ring.
#pragma unroll
            for (int pc = 0; pc < kPieces; ++pc) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(taddr + 32u * pc, r);
              tmem_ld_wait(r);
#pragma unroll
              for (int j = 0; j < 32; j += 4)
                st_shared_v4(wbuf + lane * 16u + (uint32_t)((32 * pc + j) / 4) * 512u, r[j],
                             r[j + 1], r[j + 2], r[j + 3]);
            }
            fence_proxy_async_smem();  // the copy engine reads what the threads wrote
            __syncwarp();
            if (!warp_wait(kx_go_bar(ew), 0, ctl, kSiteKx)) {
              ok = false;
              break;
            }
            if (lane == 0)
              bulk_copy_s2cluster(mapa_shared(wbuf, kx_peer), wbuf, kKxWarpBytes,
                                  mapa_shared(kx_ready_bar(ew), kx_peer));
            __syncwarp();
            emit = false;
          }
        } else if (active && w.nsplit > 1) {
          // Split-K: this slice's partial goes to the workspace straight from TMEM
          // (the same block layout as the general epilogue); the last slice to arrive
          // emits C, summing the slices in slice order.
          const size_t sliced = (size_t)(w.tile - p.dp_tiles);
          const float* ws_tile = p.workspace + sliced * p.ws_slots * kSliceStride;
          ws_lane = ws_tile + my_block * kBlockFloats + lane * 4;
          float* mine = p.workspace + sliced * p.ws_slots * kSliceStride +
                        ((size_t)w.split * kBlocksPerSlice + my_block) * kBlockFloats + lane * 4;
#pragma unroll
          for (int pc = 0; pc < kPieces; ++pc) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + 32u * pc, r);
            tmem_ld_wait(r);
#pragma unroll
            for (int j = 0; j < 32; j += 4)
              st_global_cg_v4(mine + (32 * pc + j) * 32, r[j], r[j + 1], r[j + 2], r[j + 3]);
          }
          __syncwarp();
          uint32_t last = 0;
          if (lane == 0) {
            uint32_t* ctr = p.counters + sliced * kBlocksPerSlice + my_block;
            const uint32_t before = atom_add_acq_rel_gpu(ctr, 1u);
            last = (before == (uint32_t)w.nsplit - 1u) ? 1u : 0u;
            if (last) st_relaxed_gpu_u32(ctr, 0u);  // ready for the next launch
          }
          emit = __shfl_sync(0xFFFFFFFFu, last, 0) != 0;
          __syncwarp();
        }
        if (emit) {
          if (kTmaStoreOk && p.tma_store) {
            constexpr int kPiecesPerBox = kBoxCols / 32;
            const uint32_t row_addr = staging + lane * 128u;
#pragma unroll
            for (int bx = 0; bx < kBoxes; ++bx) {
              // the previous store from this staging box must have finished reading it
              if (lane == 0) bulk_wait_group_read<0>();
              __syncwarp();
#pragma unroll
              for (int pp = 0; pp < kPiecesPerBox; ++pp) {
                float v[32];
                const int pc = bx * kPiecesPerBox + pp;
                one_chain_piece<KX2>(taddr + 32u * pc, w, ws_lane, kSliceStride, 32 * pc, v, kx_lane);
                if constexpr (FUSED) fuse_piece<OUT>(p, m0 + (int32_t)row, n_half + 32 * pc, v);
                // 16-byte chunks of the 128-byte row, in the 128-byte swizzled order
                constexpr int kChunks = 8 / kPiecesPerBox;
#pragma unroll
                for (int c = 0; c < kChunks; ++c) {
                  const uint32_t cj = (uint32_t)(pp * kChunks + c);
                  uint32_t w4[4];
                  if constexpr (OUT == kOutF32) {
#pragma unroll
                    for (int t = 0; t < 4; ++t) w4[t] = __float_as_uint(v[c * 4 + t]);
                  } else {
#pragma unroll
                    for (int t = 0; t < 4; ++t) w4[t] = pack2<OUT>(v[c * 8 + 2 * t], v[c * 8 + 2 * t + 1]);
                  }
                  st_shared_v4(row_addr + ((cj ^ (lane & 7u)) << 4), w4[0], w4[1], w4[2], w4[3]);
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
              const int32_t box_n = n_half + bx * kBoxCols, box_m = m0 + (int32_t)(q * 32u);
              if (lane == 0 && box_n < p.N && box_m < p.M) {
                tma_store_2d(&tmC, staging, box_n, box_m);
                bulk_commit_group();
              }
            }
          } else {
#pragma unroll
            for (int pc = 0; pc < kPieces; ++pc) {
              float v[32];
              one_chain_piece<KX2>(taddr + 32u * pc, w, ws_lane, kSliceStride, 32 * pc, v, kx_lane);
              if constexpr (FUSED) fuse_piece<OUT>(p, m0 + (int32_t)row, n_half + 32 * pc, v);
              store_piece_rows<OUT>(p.C, p.M, p.N, m0 + (int32_t)(q * 32u), n_half + 32 * pc, v,
                                    staging);
            }
          }
        }
        // The slot goes back to the MMA warp once this warp's last TMEM read is done.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (CTA_GROUP == 1) mbar_arrive(acc_empty_bar(slot));
          else mbar_arrive_cluster_relaxed(mapa_shared(acc_empty_bar(slot), group_base));
        }
        ++iter;
      }
    } else {
    while (ok && walker_next<GROUPED, CLC, CTA_GROUP>(walk, first_unit, unit_stride, p, w, &clc, &ctl)) {
      // In a half-tile unit the accumulator holds BN/2 columns: the h = 0 warps own
      // them, the h = 1 warps only take part in the slot hand-over.
      const bool active = w.half < 0 || h == 0;
      // (asked before the accumulator is live: a call with it live would spill it)
      bool final_unit = false;
      if constexpr (STAGED) final_unit = w.nsplit > 1 && !walker_has_next(walk, first_unit, p);
      float acc[kHalf];
      const int32_t nchains = chains_of(w, p.chain_kb);
      if constexpr (KIND == 2) {
      // One accumulation chain: wait for it, read it out of Tensor Memory into the fp32
      // registers scaled by sc, hand the slot back.  False when the wait gave up.
      auto consume_chain = [&](int32_t ch, float sc) -> bool {
        const uint32_t slot = iter & (kSlots - 1u);
        // A chain is one K block, i.e. one operand stage (the iter-th of this CTA), and the
        // MMA issuer's commit that frees that stage also tells that its accumulator is
        // complete: wait on the stage's empty barrier (use iter / STAGES of it).  Its next
        // phase cannot complete before this one is seen: the MMAs of stage use
        // iter + STAGES need the slot of chain iter + STAGES - kSlots >= iter released.
        static_assert(STAGES >= (int)kSlots, "a stage must not come round before its slot");
        const uint32_t st_idx = e_stage, st_phase = e_phase;  // (iter % STAGES, its use)
        if (++e_stage == (uint32_t)STAGES) {
          e_stage = 0;
          e_phase ^= 1u;
        }
        // Every lane polls and the warp leaves on one verdict (no broadcast of one lane's),
        // so tcgen05.ld below is executed by the whole, converged warp.
        if (!warp_wait_inl(empty_bar(st_idx), st_phase, ctl, kSiteAccFull)) return false;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((q * 32u) << 16) + slot * BN + h * kHalf;
        // (the sums start at +0: fma(x, sc, +0) is x * sc rounded once, as the first
        // product was before, and needs no select per chain; two per instruction)
        if (active) {
          if constexpr (kPieces == 2) {
            // both pieces in flight behind one wait (64 columns: the registers allow it)
            uint32_t r0[32], r1[32];
            tmem_ld_32x32b_x32(taddr, r0);
            tmem_ld_32x32b_x32(taddr + 32u, r1);
            tmem_ld_wait(r0);
            tie_regs(r1);
#pragma unroll
            for (int j = 0; j < 32; j += 2) {
              fma2_rn(acc[j], acc[j + 1], __uint_as_float(r0[j]), __uint_as_float(r0[j + 1]), sc);
              fma2_rn(acc[32 + j], acc[33 + j], __uint_as_float(r1[j]), __uint_as_float(r1[j + 1]), sc);
            }
          } else {
#pragma unroll
            for (int pc = 0; pc < kPieces; ++pc) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(taddr + 32u * pc, r);
              tmem_ld_wait(r);
              // (one fmaf each here: the packed form raised this 256-column kernel's spills)
#pragma unroll
              for (int j = 0; j < 32; ++j)
                acc[32 * pc + j] = fmaf(__uint_as_float(r[j]), sc, acc[32 * pc + j]);
            }
          }
        }
        // The slot is free for the next chain as soon as the loads are done.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          // the leader's acc_empty, in shared::cluster space (its own, for rank 0)
          if constexpr (CTA_GROUP == 1) mbar_arrive(acc_empty_bar(slot));
          else mbar_arrive_cluster_relaxed(mapa_shared(acc_empty_bar(slot), group_base));
        }
        ++iter;
        return true;
      };
        // Blockwise FP8 scales ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell
        // tcgen05", Part 6, FP8 and Blockwise Scaling): every chain is one 128-element K
        // block kb; its TMEM value is scaled by sfa(row block, kb) * sfb(column block, kb)
        // before it is added.  This thread's row and this warp's columns (one 128-column
        // block: a warp's columns never cross one) fix the two scale columns; the scales
        // are stored K-block-major, so a warp's 32 rows read one line per K block.  The
        // chains go eight at a time with A's scales of the next eight in flight, each in a
        // register of its own: a scale is loaded into the register its chain of eight
        // earlier has just used, and first read eight chains later (loading into one of
        // two registers chosen at run time made every chain wait for its load).
        const int32_t m = min(w.m_blk * kRowsTile + (int32_t)(rank * kBlockM + q * 32u + lane),
                              p.M - 1);
        const int32_t n = min(w.n_blk * BN + (w.half >= 0 ? w.half : (int32_t)h) * kHalf, p.N - 1);
        // (the scale pointers advance by one K block per chain, in registers: indexing
        // from the unit's fields re-read them after every asm statement, ~120 cycles per
        // chain in the epilogue warps, measured).  B's scale is the same for the whole
        // warp, so lane i holds chain c + i's for 32 chains at once and hands it out with
        // a shuffle, the next 32 in flight: a warp then has five scale loads in flight,
        // not eight.
        const size_t lda = (size_t)p.sf_lda, ldb = (size_t)p.sf_ldb;
        const float* pa = p.sfa + m / p.sf_bm + (size_t)w.kb0 * lda;
        const float* pb = p.sfb + (n >> 7) + (size_t)w.kb0 * ldb;
        float sa[8], sbv = 0.0f, sbv_next = 0.0f;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          sa[j] = 0.0f;
          if (active && j < nchains) sa[j] = pa[j * lda];
        }
        // chain 8's, clamped to the last chain so that the load below needs no branch (it
        // reads a valid scale whose value goes unused once fewer than eight chains remain;
        // the branch cost ~2% at 8192^3, measured; eight chains ahead rather than four:
        // 4096^3 79.9 -> 77.8 us)
        pa += (size_t)max(0, min(8, nchains - 1)) * lda;
        if (active && (int32_t)lane < nchains) sbv = pb[lane * ldb];
        if (active && 32 + (int32_t)lane < nchains) sbv_next = pb[(32 + lane) * ldb];
#pragma unroll
        for (int j = 0; j < kHalf; ++j) acc[j] = 0.0f;
        for (int32_t c0 = 0; c0 < nchains && ok; c0 += 8) {
#pragma unroll
          for (int j = 0; j < 8; ++j) {
            const int32_t ch = c0 + j;
            if (ch < nchains && ok) {
              const float sc = sa[j] * __shfl_sync(0xFFFFFFFFu, sbv, ch & 31);
              if (!consume_chain(ch, sc)) ok = false;
              sa[j] = *pa;
              if (ch + 9 < nchains) pa += lda;
              if ((ch & 31) == 31) {
                // chains ch + 1.. are in sbv_next; fetch ch + 33..
                const int32_t nc = ch + 33 + (int32_t)lane;
                sbv = sbv_next;
                sbv_next = active && nc < nchains ? pb[(size_t)nc * ldb] : 0.0f;
              }
            }
          }
        }
      } else {
        for (int32_t ch = 0; ch < nchains; ++ch) {
          const uint32_t slot = iter & (kSlots - 1u), acc_phase = (iter >> kSlotShift) & 1u;
          // Every lane polls and the warp leaves on one verdict, so tcgen05.ld below is
          // always executed by the whole, converged warp.
          if (!warp_wait_inl(acc_full_bar(slot), acc_phase, ctl, kSiteAccFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t taddr = tmem_base + ((q * 32u) << 16) + slot * BN + h * kHalf;
          if (active) {
#pragma unroll
            for (int pc = 0; pc < kPieces; ++pc) {
              uint32_t r[32];
              tmem_ld_32x32b_x32(taddr + 32u * pc, r);
              tmem_ld_wait(r);
              if (ch == 0) {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[32 * pc + j] = __uint_as_float(r[j]);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) acc[32 * pc + j] += __uint_as_float(r[j]);
              }
            }
          }
          // The slot is free for the next chain as soon as the loads are done.
          tc_fence_before();
          __syncwarp();
          if (lane == 0) {
            // the leader's acc_empty, in shared::cluster space (its own, for rank 0)
            if constexpr (CTA_GROUP == 1) mbar_arrive(acc_empty_bar(slot));
            else mbar_arrive_cluster_relaxed(mapa_shared(acc_empty_bar(slot), group_base));
          }
          ++iter;
        }
      }
      if (!ok) break;
      if (!active) continue;

      const int32_t m0 = w.m_blk * kRowsTile + (int32_t)rank * rows_cta;  // first row of this CTA
      // first column written by this warp
      const int32_t n_half = w.n_blk * BN + (w.half >= 0 ? w.half : (int32_t)h) * kHalf;
      bool exchanged = false;
      if constexpr (KX2) {
        if (w.nsplit > 1) {
          // Cluster K split (see the single-chain epilogue): the warp of the column half
          // the other slice finishes stages its summed chains in its own idle ring and
          // copies them into the other slice's ring once that one has finished with it;
          // the receiving warp adds them to its own (p0 + p1 = p1 + p0, the same bits as
          // the workspace path) and stores C.
          constexpr uint32_t kKxWarpBytes = 32u * kHalf * 4u;
          static_assert(L::kEpiWarps * kKxWarpBytes <= STAGES * L::kStageBytes,
                        "the received partials must fit in the operand ring");
          const uint32_t wlane = base + L::kAOff + ew * kKxWarpBytes + lane * 16u;
          if (h == slice_k) {
            if (lane == 0) {
              // (its own barrier: a local arm; the go carries no data of this warp's, only
              // that its ring is idle -- its MMAs are complete -- so a relaxed arrive: the
              // cluster-scope release forms cost about a microsecond each, measured)
              mbar_arrive_expect_tx(kx_ready_bar(ew), kKxWarpBytes);
              mbar_arrive_cluster_relaxed(mapa_shared(kx_go_bar(ew), kx_peer));
            }
            if (!warp_wait(kx_ready_bar(ew), 0, ctl, kSiteKx)) {
              ok = false;
              break;
            }
#pragma unroll
            for (int j = 0; j < kHalf; j += 4) {
              const uint4 x = ld_shared_v4(wlane + (uint32_t)(j / 4) * 512u);
              acc[j] += __uint_as_float(x.x);
              acc[j + 1] += __uint_as_float(x.y);
              acc[j + 2] += __uint_as_float(x.z);
              acc[j + 3] += __uint_as_float(x.w);
            }
            exchanged = true;
          } else {
#pragma unroll
            for (int j = 0; j < kHalf; j += 4)
              st_shared_v4(wlane + (uint32_t)(j / 4) * 512u, __float_as_uint(acc[j]),
                           __float_as_uint(acc[j + 1]), __float_as_uint(acc[j + 2]),
                           __float_as_uint(acc[j + 3]));
            fence_proxy_async_smem();
            __syncwarp();
            if (!warp_wait(kx_go_bar(ew), 0, ctl, kSiteKx)) {
              ok = false;
              break;
            }
            if (lane == 0) {
              const uint32_t wbuf = base + L::kAOff + ew * kKxWarpBytes;
              bulk_copy_s2cluster(mapa_shared(wbuf, kx_peer), wbuf, kKxWarpBytes,
                                  mapa_shared(kx_ready_bar(ew), kx_peer));
            }
            __syncwarp();
            continue;
          }
        }
      }
      if constexpr (STAGED) {
        if (w.nsplit > 1 && !exchanged) {
          // Split-K: this slice's fp32 block (the warp's 32 rows x BN/2 columns) goes to
          // the workspace; the last slice of the block to arrive sums all slices in slice
          // order.  Within a block, each group of 4 columns holds the warp's 32 rows
          // contiguously (float index (col / 4) * 128 + lane * 4 + col % 4), so every
          // warp-wide 16-byte access covers 512 contiguous bytes.
          constexpr size_t kBlockFloats = 32 * kHalf;
          constexpr size_t kBlocksPerSlice = (size_t)CTA_GROUP * 8;  // (rank, quarter, half)
          const size_t sliced = (size_t)(w.tile - p.dp_tiles);      // index among sliced tiles
          const size_t my_block = ((size_t)rank * 4 + q) * 2 + h;
          float* ws_tile = p.workspace + sliced * p.ws_slots * kBlocksPerSlice * kBlockFloats;
          uint32_t* ctr = p.counters + sliced * kBlocksPerSlice + my_block;
          const float* ws_lane = ws_tile + (size_t)my_block * kBlockFloats + lane * 4;
          const size_t slice_stride = kBlocksPerSlice * kBlockFloats;
          // The last unit of this CTA: its operand ring is idle (every MMA has completed
          // and nothing more is loaded), so the other slices' blocks can be staged there.
          // With at most two of them, a slice that finds them all published does not
          // publish its own (the common case for the last segment of a stream-K worker,
          // whose partners ran at the starts of their ranges).
          const bool fast = w.nsplit <= 3 && final_unit;
          uint32_t last = 0;
          if (fast && lane == 0) last = ld_acquire_gpu_u32(ctr) == (uint32_t)w.nsplit - 1u ? 1u : 0u;
          last = __shfl_sync(0xFFFFFFFFu, last, 0);
          if (!last) {
            float* mine = ws_tile + ((size_t)w.split * kBlocksPerSlice + my_block) * kBlockFloats +
                          lane * 4;
  #pragma unroll
            for (int j = 0; j < kHalf; j += 4)
              st_global_cg_v4(mine + j * 32, __float_as_uint(acc[j]), __float_as_uint(acc[j + 1]),
                              __float_as_uint(acc[j + 2]), __float_as_uint(acc[j + 3]));
            // The warp's partial is published by lane 0's release-increment of the block's
            // counter (after the warp barrier); the slice that sees the count reach the
            // number of slices acquires every other slice's partial the same way.
            __syncwarp();
            if (lane == 0) {
              const uint32_t before = atom_add_acq_rel_gpu(ctr, 1u);
              last = (before == (uint32_t)w.nsplit - 1u) ? 1u : 0u;
            }
            last = __shfl_sync(0xFFFFFFFFu, last, 0);
            __syncwarp();
            if (!last) continue;
          }
          if (lane == 0) st_relaxed_gpu_u32(ctr, 0u);  // ready for the next launch
          // Sum the slices in slice order: the result is the same whichever slice arrived
          // last.  With two slices the sum is p0 + p1 = p1 + p0 exactly, so the last one
          // adds the other's partial to its own registers; with three, (p0 + p1) + p2 is
          // formed with its own partial taken from the registers.
          if (fast) {
            // The other blocks come into this warp's share of the idle ring through
            // asynchronous copies (all in flight at once, no registers held), in the
            // block layout above: one block, or the two others' halves of the columns.
            constexpr uint32_t kRegion = 32u * kHalf * 4u;
            static_assert(L::kEpiWarps * kRegion <= STAGES * L::kStageBytes,
                          "the staged partials must fit in the operand ring");
            const uint32_t wreg = base + L::kAOff + ew * kRegion + lane * 16u;
            if (w.nsplit == 2) {
              const float* other = ws_lane + (size_t)(1 - w.split) * slice_stride;
  #pragma unroll
              for (int j = 0; j < kHalf; j += 4) cp_async_cg_16(wreg + (uint32_t)(j / 4) * 512u, other + j * 32);
              cp_async_wait_all();
              __syncwarp();
  #pragma unroll
              for (int j = 0; j < kHalf; j += 4) {
                const uint4 x = ld_shared_v4(wreg + (uint32_t)(j / 4) * 512u);
                acc[j] += __uint_as_float(x.x);
                acc[j + 1] += __uint_as_float(x.y);
                acc[j + 2] += __uint_as_float(x.z);
                acc[j + 3] += __uint_as_float(x.w);
              }
            } else {
              // the two other slices, in slice order
              const int32_t sa = w.split == 0 ? 1 : 0, sb = w.split == 2 ? 1 : 2;
              const float* pa = ws_lane + (size_t)sa * slice_stride;
              const float* pb = ws_lane + (size_t)sb * slice_stride;
              constexpr int kCols = kHalf / 2;
              constexpr uint32_t kSecond = kRegion / 2;
              // one column half at a time (its index a compile-time constant, so that the
              // accumulator stays in registers)
              auto column_half = [&](auto half) {
                constexpr int c0 = decltype(half)::value * kCols;
  #pragma unroll
                for (int j = 0; j < kCols; j += 4) {
                  cp_async_cg_16(wreg + (uint32_t)(j / 4) * 512u, pa + (c0 + j) * 32);
                  cp_async_cg_16(wreg + kSecond + (uint32_t)(j / 4) * 512u, pb + (c0 + j) * 32);
                }
                cp_async_wait_all();
                __syncwarp();
  #pragma unroll
                for (int j = 0; j < kCols; j += 4) {
                  const uint4 xa = ld_shared_v4(wreg + (uint32_t)(j / 4) * 512u);
                  const uint4 xb = ld_shared_v4(wreg + kSecond + (uint32_t)(j / 4) * 512u);
                  // (p0 + p1) + p2 with this slice's own partial in acc
                  if (w.split == 2) {
                    acc[c0 + j] += __uint_as_float(xa.x) + __uint_as_float(xb.x);
                    acc[c0 + j + 1] += __uint_as_float(xa.y) + __uint_as_float(xb.y);
                    acc[c0 + j + 2] += __uint_as_float(xa.z) + __uint_as_float(xb.z);
                    acc[c0 + j + 3] += __uint_as_float(xa.w) + __uint_as_float(xb.w);
                  } else {
                    acc[c0 + j] = (acc[c0 + j] + __uint_as_float(xa.x)) + __uint_as_float(xb.x);
                    acc[c0 + j + 1] = (acc[c0 + j + 1] + __uint_as_float(xa.y)) + __uint_as_float(xb.y);
                    acc[c0 + j + 2] = (acc[c0 + j + 2] + __uint_as_float(xa.z)) + __uint_as_float(xb.z);
                    acc[c0 + j + 3] = (acc[c0 + j + 3] + __uint_as_float(xa.w)) + __uint_as_float(xb.w);
                  }
                }
                __syncwarp();  // the region is refilled for the next half
              };
              column_half(std::integral_constant<int, 0>{});
              column_half(std::integral_constant<int, 1>{});
            }
          } else if (w.nsplit == 2) {
            const float* other = ws_lane + (size_t)(1 - w.split) * slice_stride;
  #pragma unroll
            for (int j = 0; j < kHalf; j += 4) {
              const uint4 x = ld_global_cg_v4(other + j * 32);
              acc[j] += __uint_as_float(x.x);
              acc[j + 1] += __uint_as_float(x.y);
              acc[j + 2] += __uint_as_float(x.z);
              acc[j + 3] += __uint_as_float(x.w);
            }
          } else {
            // every slice's partial (this one's published too) read back in order
            for (int32_t s = 0; s < w.nsplit; ++s) {
              const float* src = ws_lane + (size_t)s * slice_stride;
  #pragma unroll
              for (int j = 0; j < kHalf; j += 4) {
                const uint4 x = ld_global_cg_v4(src + j * 32);
                if (s == 0) {
                  acc[j] = __uint_as_float(x.x);
                  acc[j + 1] = __uint_as_float(x.y);
                  acc[j + 2] = __uint_as_float(x.z);
                  acc[j + 3] = __uint_as_float(x.w);
                } else {
                  acc[j] += __uint_as_float(x.x);
                  acc[j + 1] += __uint_as_float(x.y);
                  acc[j + 2] += __uint_as_float(x.z);
                  acc[j + 3] += __uint_as_float(x.w);
                }
              }
            }
          }
        }

      } else {
        if (w.nsplit > 1 && !exchanged) {
          // Split-K: this slice's fp32 block (the warp's 32 rows x BN/2 columns) goes to
          // the workspace; the last slice of the block to arrive sums all slices in slice
          // order.  Within a block, each group of 4 columns holds the warp's 32 rows
          // contiguously (float index (col / 4) * 128 + lane * 4 + col % 4), so every
          // warp-wide 16-byte access covers 512 contiguous bytes.
          constexpr size_t kBlockFloats = 32 * kHalf;
          constexpr size_t kBlocksPerSlice = (size_t)CTA_GROUP * 8;  // (rank, quarter, half)
          const size_t sliced = (size_t)(w.tile - p.dp_tiles);      // index among sliced tiles
          const size_t my_block = ((size_t)rank * 4 + q) * 2 + h;
          float* ws_tile = p.workspace + sliced * p.ws_slots * kBlocksPerSlice * kBlockFloats;
          float* mine = ws_tile + ((size_t)w.split * kBlocksPerSlice + my_block) * kBlockFloats +
                        lane * 4;
  #pragma unroll
          for (int j = 0; j < kHalf; j += 4)
            st_global_cg_v4(mine + j * 32, __float_as_uint(acc[j]), __float_as_uint(acc[j + 1]),
                            __float_as_uint(acc[j + 2]), __float_as_uint(acc[j + 3]));
          // The warp's partial is published by lane 0's release-increment of the block's
          // counter (after the warp barrier); the slice that sees the count reach the
          // number of slices acquires every other slice's partial the same way.
          __syncwarp();
          uint32_t last = 0;
          if (lane == 0) {
            uint32_t* ctr = p.counters + sliced * kBlocksPerSlice + my_block;
            const uint32_t before = atom_add_acq_rel_gpu(ctr, 1u);
            last = (before == (uint32_t)w.nsplit - 1u) ? 1u : 0u;
            if (last) st_relaxed_gpu_u32(ctr, 0u);  // ready for the next launch
          }
          last = __shfl_sync(0xFFFFFFFFu, last, 0);
          __syncwarp();
          if (!last) continue;
          // Sum the slices in slice order: the result is the same whichever slice arrived
          // last.  With two slices the sum is p0 + p1 = p1 + p0 exactly, so the last one
          // adds the other's partial to its own registers; with more, every partial is
          // read back and added in order.
          const float* ws_lane = ws_tile + (size_t)my_block * kBlockFloats + lane * 4;
          const size_t slice_stride = kBlocksPerSlice * kBlockFloats;
          if (w.nsplit == 2) {
            const float* other = ws_lane + (size_t)(1 - w.split) * slice_stride;
  #pragma unroll
            for (int j = 0; j < kHalf; j += 4) {
              const uint4 x = ld_global_cg_v4(other + j * 32);
              acc[j] += __uint_as_float(x.x);
              acc[j + 1] += __uint_as_float(x.y);
              acc[j + 2] += __uint_as_float(x.z);
              acc[j + 3] += __uint_as_float(x.w);
            }
          } else {
            for (int32_t s = 0; s < w.nsplit; ++s) {
              const float* src = ws_lane + (size_t)s * slice_stride;
  #pragma unroll
              for (int j = 0; j < kHalf; j += 4) {
                const uint4 x = ld_global_cg_v4(src + j * 32);
                if (s == 0) {
                  acc[j] = __uint_as_float(x.x);
                  acc[j + 1] = __uint_as_float(x.y);
                  acc[j + 2] = __uint_as_float(x.z);
                  acc[j + 3] = __uint_as_float(x.w);
                } else {
                  acc[j] += __uint_as_float(x.x);
                  acc[j + 1] += __uint_as_float(x.y);
                  acc[j + 2] += __uint_as_float(x.z);
                  acc[j + 3] += __uint_as_float(x.w);
                }
              }
            }
          }
        }

      }
      if constexpr (FUSED) {
        const int32_t m = m0 + (int32_t)row;
#pragma unroll
        for (int pc = 0; pc < kPieces; ++pc) fuse_piece<OUT>(p, m, n_half + 32 * pc, acc + 32 * pc);
      }
      if constexpr (SWAP) {
        // this thread holds column n = m0 + row of C (row n of B), for the kHalf rows of
        // C (rows of A) from n_half on
        store_col_direct<OUT, kHalf>(p, m0 + (int32_t)row, (int32_t)row < rows_cta, n_half, acc);
        continue;
      }
      // this unit's output: the launch's C, or in a grouped launch its problem's
      const GroupDesc* gd = nullptr;
      if constexpr (GROUPED) gd = p.groups + w.g;
      const bool out_tma = GROUPED ? gd->tma_store != 0 : p.tma_store != 0;
      const int32_t out_m = GROUPED ? gd->M : p.M, out_n = GROUPED ? gd->N : p.N;
      const CUtensorMap* out_map = GROUPED ? &gd->tmC : &tmC;
      if (kTmaStoreOk && out_tma) {
        // Each 128-byte row of a staging box is written in the 128-byte swizzled order
        // (16-byte chunk j of row r at chunk j ^ (r % 8)) that the C tensor map's
        // CU_TENSOR_MAP_SWIZZLE_128B expects ("A Blackwell GEMM by Hand in CuTe DSL",
        // section 6); the TMA store clips rows >= M and columns >= N.
        const uint32_t row_addr = staging + lane * 128u;
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) {
          // the previous store from this staging box must have finished reading it
          if (lane == 0) bulk_wait_group_read<0>();
          __syncwarp();
#pragma unroll
          for (int cj = 0; cj < 8; ++cj) {
            uint32_t w4[4];
            if constexpr (OUT == kOutF32) {
#pragma unroll
              for (int t = 0; t < 4; ++t)
                w4[t] = __float_as_uint(acc[bx * kBoxCols + cj * 4 + t]);
            } else {
#pragma unroll
              for (int t = 0; t < 4; ++t)
                w4[t] = pack2<OUT>(acc[bx * kBoxCols + cj * 8 + 2 * t],
                                   acc[bx * kBoxCols + cj * 8 + 2 * t + 1]);
            }
            st_shared_v4(row_addr + ((cj ^ (lane & 7u)) << 4), w4[0], w4[1], w4[2], w4[3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          const int32_t box_n = n_half + bx * kBoxCols, box_m = m0 + (int32_t)(q * 32u);
          // a box wholly outside C (ragged last tiles) is not stored at all
          if (lane == 0 && box_n < out_n && box_m < out_m) {
            if constexpr (GROUPED) fence_tensormap_acquire(out_map);
            tma_store_2d(out_map, staging, box_n, box_m);
            bulk_commit_group();
          }
        }
      } else {
        // (row stores: the transposed form of the single-chain epilogue raised this
        // epilogue's register spills)
        const int32_t m = m0 + (int32_t)row;
#pragma unroll
        for (int pc = 0; pc < kPieces; ++pc) {
          if constexpr (GROUPED)
            store_row_to<OUT>(gd->C, gd->M, gd->N, gd->vec_store, m, n_half + 32 * pc, acc + 32 * pc);
          else
            store_row_direct<OUT>(p, m, n_half + 32 * pc, acc + 32 * pc);
        }
      }
    }
    }  // general epilogue
    // Every TMA store of this warp must be complete before the CTA exits.
    if ((GROUPED || p.tma_store) && lane == 0) bulk_wait_group<0>();
    __syncwarp();
  }

  // --------------------------------------------------------------- teardown --
  tc_fence_before();
  // no CTA leaves while its pair (or the other K slice) may still signal it
  if constexpr (CTA_GROUP == 2 || KX2) cluster_sync();
  else __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<CTA_GROUP>(tmem_base, kTmemCols);
  }
}

}  // namespace gb300
