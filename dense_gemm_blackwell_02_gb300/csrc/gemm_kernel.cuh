// Persistent, warp-specialised tcgen05 GEMM for sm_103a:  C = A . B^T.
//
// A is M x K and B is N x K, both K-major (K contiguous), fp16 or bf16; fp32
// accumulation in Tensor Memory; C is M x N row-major in fp16, bf16 or fp32.
// ("A Blackwell GEMM by Hand in CuTe DSL", section 1 for the operand convention;
// section 3 for the warp roles; section 8 for persistence with two TMEM slots.)
//
// One CTA of 6 warps per SM, looping over work units (tile, K slice):
//   warp 0      TMA producer: one thread fills a STAGES-deep ring of 128B-swizzled
//               A (128 x 64) and B (BN x 64) slices, arming full[s] with the byte count.
//   warp 1      allocates 2*BN TMEM columns; one thread issues tcgen05.mma
//               (128 x BN x 16, four per 64-deep stage) into accumulator slot i%2,
//               commits each stage back to empty[s] and each finished tile to acc_full.
//   warps 2..5  epilogue: tcgen05.ld of their 32-lane quarter, release acc_empty as soon
//               as the loads are done, convert (RNE) and store C, so tile i's epilogue
//               overlaps tile i+1's mainloop.
// Split-K units write fp32 partials to a workspace; the last of a tile's slices to
// arrive (per 32-row quarter, by an atomic counter) sums all slices in slice order,
// so the result does not depend on arrival order ("A Blackwell GEMM by Hand in CuTe
// DSL", section 9, split-K for decode shapes).
//
// Every mbarrier wait is bounded by p.wait_limit_ns (globaltimer) and an iteration
// cap; on expiry the waiting thread records the site in the status word, raises a
// shared abort flag that makes every role leave its loop, and the CTA drains its own
// outstanding copies and MMAs before freeing TMEM and returning.
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

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

// Wait for the phase of `bar` with parity `parity` to complete.  Returns false when
// the CTA is aborting or the limit ran out (then the abort flag is raised).
__device__ __noinline__ bool wait_parity(uint32_t bar, uint32_t parity, const WaitCtl& c,
                                         uint32_t site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u) {
      if (*c.abort_flag) return false;
      if (globaltimer_ns() - t0 > c.limit_ns || it > (1u << 26)) {
        record_timeout(c, site);
        return false;
      }
    }
  }
}

// Teardown wait: ignores the abort flag (it is used while aborting) but is bounded.
__device__ __noinline__ bool wait_parity_drain(uint32_t bar, uint32_t parity, const WaitCtl& c) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0u && (globaltimer_ns() - t0 > c.limit_ns || it > (1u << 26))) {
      record_timeout(c, kSiteDrain);
      return false;
    }
  }
}

struct Unit {
  int32_t tile, split, m_blk, n_blk, kb0, kb1;
};

// Work unit -> (tile, K slice) -> (m block, n block) with grouped rasterisation:
// tiles are taken group_m M-blocks at a time, walking N inside a group, so units
// running at the same time share A rows and B columns in L2 ("Matmul on sm_120",
// block swizzle; "A Blackwell GEMM by Hand in CuTe DSL", section 8).
__device__ __forceinline__ Unit decode_unit(int32_t u, const GemmParams& p) {
  Unit w;
  w.tile = u / p.splits;
  w.split = u - w.tile * p.splits;
  const int32_t group = p.group_m * p.num_n_tiles;
  const int32_t g = w.tile / group;
  const int32_t first_m = g * p.group_m;
  const int32_t gm = min(p.num_m_tiles - first_m, p.group_m);
  const int32_t r = w.tile - g * group;
  w.m_blk = first_m + r % gm;
  w.n_blk = r / gm;
  w.kb0 = w.split * p.kb_per_split;
  w.kb1 = min(w.kb0 + p.kb_per_split, p.k_blocks);
  return w;
}

// ----------------------------------------------------------------- epilogue stores --
template <int OUT>
__device__ __forceinline__ void store_row_chunk(const GemmParams& p, int32_t m, int32_t n0,
                                                const float (&v)[32]) {
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
    for (int j = 0; j < 16; ++j) {
      if constexpr (OUT == kOutF16) {
        __half2 h = __floats2half2_rn(v[2 * j], v[2 * j + 1]);
        packed[j] = *reinterpret_cast<uint32_t*>(&h);
      } else {
        __nv_bfloat162 h = __floats2bfloat162_rn(v[2 * j], v[2 * j + 1]);
        packed[j] = *reinterpret_cast<uint32_t*>(&h);
      }
    }
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

// --------------------------------------------------------------- shared memory map --
template <int BN, int STAGES>
struct SmemLayout1 {
  static constexpr uint32_t kABytes = kBlockM * kBlockK * 2;  // 16 KiB
  static constexpr uint32_t kBBytes = BN * kBlockK * 2;       // 32 KiB at BN = 256
  static constexpr uint32_t kStageBytes = kABytes + kBBytes;
  static constexpr uint32_t kAOff = 0;
  static constexpr uint32_t kBOff = STAGES * kABytes;
  static constexpr uint32_t kBarOff = kBOff + STAGES * kBBytes;
  // full[S], empty[S], acc_full[2], acc_empty[2], drain
  static constexpr uint32_t kNumBars = 2 * STAGES + 5;
  static constexpr uint32_t kTmemSlotOff = kBarOff + kNumBars * 8;
  static constexpr uint32_t kAbortOff = kTmemSlotOff + 4;
  static constexpr uint32_t kEnd = kAbortOff + 4;
  static constexpr uint32_t kDynamicBytes = kEnd + 1024;  // slack for 1024-byte alignment
  static_assert(kAOff % 1024 == 0 && kBOff % 1024 == 0 && kABytes % 1024 == 0 &&
                    kBBytes % 1024 == 0,
                "every operand stage must start on a 1024-byte boundary (128B swizzle atom)");
  static_assert(kDynamicBytes <= 227 * 1024, "shared memory over the per-block limit");
};

constexpr uint32_t kThreads1 = 192;  // warp 0 producer, warp 1 MMA, warps 2..5 epilogue

template <int BN, int STAGES, int OUT>
__global__ void __launch_bounds__(kThreads1, 1)
    gemm_1cta_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmB, const GemmParams p) {
  using L = SmemLayout1<BN, STAGES>;
  static_assert(BN == 128 || BN == 256, "BN must be 128 or 256");
  constexpr uint32_t kTmemCols = 2 * BN;  // two accumulator slots
  constexpr int kChunks = BN / 32;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (base - raw);

  const uint32_t sA = base + L::kAOff;
  const uint32_t sB = base + L::kBOff;
  const uint32_t bar0 = base + L::kBarOff;
  auto full_bar = [&](uint32_t s) { return bar0 + 8u * s; };
  auto empty_bar = [&](uint32_t s) { return bar0 + 8u * (STAGES + s); };
  auto acc_full_bar = [&](uint32_t i) { return bar0 + 8u * (2 * STAGES + i); };
  auto acc_empty_bar = [&](uint32_t i) { return bar0 + 8u * (2 * STAGES + 2 + i); };
  const uint32_t drain_bar = bar0 + 8u * (2 * STAGES + 4);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kTmemSlotOff);
  volatile int32_t* abort_flag = reinterpret_cast<volatile int32_t*>(smem + L::kAbortOff);

  const uint32_t warp = warp_id();
  const uint32_t lane = lane_id();
  const WaitCtl ctl{p.wait_limit_ns, p.status, abort_flag};

  // ---------------------------------------------------------------- setup --
  if (warp == 0 && lane == 0) {
    for (uint32_t s = 0; s < STAGES; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);
    }
    for (uint32_t i = 0; i < 2; ++i) {
      mbar_init(acc_full_bar(i), 1);
      mbar_init(acc_empty_bar(i), 4);  // one arrival per epilogue warp
    }
    mbar_init(drain_bar, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
    tma_prefetch_desc(&tmA);
    tma_prefetch_desc(&tmB);
  }
  if (warp == 1) {
    tmem_alloc<1>(smem_addr(tmem_slot), kTmemCols);
    tmem_relinquish<1>();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;

  if (warp == 0) {
    // ---------------------------------------------------------- TMA producer --
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, armed = 0, armed_phase = 0;
      bool ok = true;
      for (int32_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const Unit w = decode_unit(u, p);
        for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_parity(empty_bar(stage), phase ^ 1u, ctl, kSiteEmpty)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(full_bar(stage), L::kStageBytes);
          tma_load_2d(sA + stage * L::kABytes, &tmA, kb * kBlockK, w.m_blk * kBlockM,
                      full_bar(stage));
          tma_load_2d(sB + stage * L::kBBytes, &tmB, kb * kBlockK, w.n_blk * BN, full_bar(stage));
          armed |= 1u << stage;
          armed_phase = (armed_phase & ~(1u << stage)) | (phase << stage);
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
      }
      // No copy may still be landing in this CTA's shared memory when it exits.
      for (uint32_t s = 0; s < STAGES; ++s)
        if (armed & (1u << s)) wait_parity_drain(full_bar(s), (armed_phase >> s) & 1u, ctl);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer --
    if (lane == 0) {
      uint32_t stage = 0, phase = 0, iter = 0;
      bool ok = true;
      if (p.test_stall) ok = wait_parity(drain_bar, 0, ctl, kSiteTestStall);
      for (int32_t u = blockIdx.x; u < p.units && ok; u += gridDim.x) {
        const Unit w = decode_unit(u, p);
        const uint32_t slot = iter & 1u, acc_phase = (iter >> 1) & 1u;
        if (!wait_parity(acc_empty_bar(slot), acc_phase ^ 1u, ctl, kSiteAccEmpty)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + slot * BN;
        for (int32_t kb = w.kb0; kb < w.kb1; ++kb) {
          if (!wait_parity(full_bar(stage), phase, ctl, kSiteFull)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t a0 = sA + stage * L::kABytes, b0 = sB + stage * L::kBBytes;
#pragma unroll
          for (uint32_t k = 0; k < kBlockK / 16; ++k)
            umma_f16<1>(d_tmem, smem_desc_sw128_kmajor(a0 + 32u * k),
                        smem_desc_sw128_kmajor(b0 + 32u * k), p.idesc,
                        (kb > w.kb0 || k > 0) ? 1u : 0u);
          umma_commit(empty_bar(stage));  // stage is free once these MMAs are done
          if (++stage == STAGES) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(acc_full_bar(slot));  // accumulator final
        ++iter;
      }
      // Every issued MMA must finish before TMEM is released.
      umma_commit(drain_bar);
      wait_parity_drain(drain_bar, 0, ctl);
    }
    __syncwarp();
  } else {
    // -------------------------------------------------------------- epilogue --
    const uint32_t q = warp & 3u;             // TMEM lane quarter this warp may read
    const uint32_t row = q * 32u + lane;      // accumulator row held by this thread
    uint32_t iter = 0;
    for (int32_t u = blockIdx.x; u < p.units; u += gridDim.x) {
      const Unit w = decode_unit(u, p);
      const uint32_t slot = iter & 1u, acc_phase = (iter >> 1) & 1u;
      // One lane polls; the warp follows its verdict, so tcgen05.ld below is always
      // executed by the whole, converged warp.
      uint32_t ok = 1;
      if (lane == 0) ok = wait_parity(acc_full_bar(slot), acc_phase, ctl, kSiteAccFull) ? 1u : 0u;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) break;
      tc_fence_after();
      const uint32_t taddr = tmem_base + ((q * 32u) << 16) + slot * BN;
      const int32_t m = w.m_blk * kBlockM + (int32_t)row;
      const int32_t n_base = w.n_blk * BN;
      if (p.splits == 1) {
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + 32u * c, r);
          tmem_ld_wait(r);
          if (c == kChunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty_bar(slot));
          }
          float v[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          store_row_chunk<OUT>(p, m, n_base + 32 * c, v);
        }
      } else {
        // Split-K: this slice's fp32 partial rows go to the workspace.
        float* ws_tile = p.workspace + (size_t)w.tile * p.splits * kBlockM * BN;
        float* mine = ws_tile + ((size_t)w.split * kBlockM + row) * BN;
#pragma unroll 1
        for (int c = 0; c < kChunks; ++c) {
          uint32_t r[32];
          tmem_ld_32x32b_x32(taddr + 32u * c, r);
          tmem_ld_wait(r);
          if (c == kChunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty_bar(slot));
          }
#pragma unroll
          for (int j = 0; j < 32; j += 4)
            st_global_cg_v4(mine + 32 * c + j, r[j], r[j + 1], r[j + 2], r[j + 3]);
        }
        __threadfence();
        __syncwarp();
        uint32_t last = 0;
        if (lane == 0) {
          uint32_t* ctr = p.counters + (size_t)w.tile * 4 + q;
          const uint32_t before = atomicAdd(ctr, 1u);
          last = (before == (uint32_t)p.splits - 1u) ? 1u : 0u;
          if (last) atomicExch(ctr, 0u);  // ready for the next launch
          __threadfence();
        }
        last = __shfl_sync(0xFFFFFFFFu, last, 0);
        __syncwarp();
        if (last) {
          // Sum the slices in slice order: the result is the same whichever slice
          // arrived last.
#pragma unroll 1
          for (int c = 0; c < kChunks; ++c) {
            float v[32];
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = 0.0f;
#pragma unroll 1
            for (int32_t s = 0; s < p.splits; ++s) {
              const float* src = ws_tile + ((size_t)s * kBlockM + row) * BN + 32 * c;
#pragma unroll
              for (int j = 0; j < 32; j += 4) {
                const uint4 x = ld_global_cg_v4(src + j);
                if (s == 0) {
                  v[j] = __uint_as_float(x.x);
                  v[j + 1] = __uint_as_float(x.y);
                  v[j + 2] = __uint_as_float(x.z);
                  v[j + 3] = __uint_as_float(x.w);
                } else {
                  v[j] += __uint_as_float(x.x);
                  v[j + 1] += __uint_as_float(x.y);
                  v[j + 2] += __uint_as_float(x.z);
                  v[j + 3] += __uint_as_float(x.w);
                }
              }
            }
            store_row_chunk<OUT>(p, m, n_base + 32 * c, v);
          }
        }
      }
      ++iter;
    }
  }

  // --------------------------------------------------------------- teardown --
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc<1>(tmem_base, kTmemCols);
  }
}

}  // namespace gb300
