// Inline-PTX wrappers for the sm_103a GEMM: mbarriers, TMA (cp.async.bulk.tensor),
// Tensor Memory (tcgen05.alloc/ld/dealloc), the tcgen05 MMA and its commit, fences
// and cluster helpers.  Every wait here is bounded (see warp_wait).
//
// The operations are the four primitives described in "A Blackwell GEMM by Hand in
// CuTe DSL", section 2 (TMA, mbarrier, TMEM, tcgen05.mma), and the wrapper list in
// "Optimizing GEMMs using tcgen05 - Part 1", sections 2.3-2.4.  The PTX spelling
// follows NVIDIA's public PTX ISA (tcgen05 family, cp.async.bulk.tensor, mbarrier).
#pragma once
#include <cstdint>

namespace gb300 {

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint32_t warp_id() { return threadIdx.x >> 5; }
__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ------------------------------------------------------------------ mbarrier --
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbarrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

// Arrive on a barrier given by its shared::cluster address (possibly in the peer CTA).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// The same arrive without release semantics: for a barrier that hands over Tensor Memory
// the arriving warp has finished reading (tcgen05.wait::ld, then the tcgen05 fence before
// the arrive), which orders no memory writes.  The release form waited up to ~1900 cycles
// (measured with clock64 in a CTA pair's epilogue), once per accumulation chain.
__device__ __forceinline__ void mbar_arrive_cluster_relaxed(uint32_t cluster_bar) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_bar)
               : "memory");
}

// Arm a barrier in (possibly) the peer CTA with an expected transaction count.
// Arm this CTA's own barrier for a transfer (one thread).
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// ------------------------------------------------- warp-uniform single issue --
// The producer and MMA warps run their loops with all 32 lanes in lock-step, so the
// compiler keeps loop state and descriptors warp-uniform; each asynchronous
// instruction is then issued by exactly one lane, chosen inside the asm block with
// elect.sync.  (Issuing from a loop that only lane 0 executes measured 227 cycles per
// tcgen05.mma on sm_103a; the warp-uniform form issues a 128 x 256 x 16 MMA every 128
// cycles, the tensor core's rate.)
#define GB300_ELECT "{\n\t.reg .pred e_;\n\t.reg .b32 r_;\n\telect.sync r_|e_, 0xffffffff;\n\t"

__device__ __forceinline__ void mbar_arrive_expect_tx_elect(uint32_t bar, uint32_t bytes) {
  asm volatile(GB300_ELECT "@e_ mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(bar),
               "r"(bytes)
               : "memory");
}

// Programmatic dependent launch: wait until the grids this one depends on (the
// preceding work in the stream) have completed and their memory is visible; and let
// the next grid launch early (its blocks wait in their own grid_dependency_wait).
__device__ __forceinline__ void grid_dependency_wait() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
}
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// --------------------------------------------------------------------- fences --
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ------------------------------------------------------------------- cluster --
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;"
               ::: "memory");
}

__device__ __forceinline__ uint32_t ld_shared_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared.b32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}

// Bulk copy of `bytes` (a multiple of 16) from this CTA's shared memory to another
// CTA's (distributed shared memory); the bytes complete_tx on `remote_bar`, an mbarrier
// of the destination CTA.  Both shared addresses 16-byte aligned; dst and remote_bar in
// the shared::cluster window.
__device__ __forceinline__ void bulk_copy_s2cluster(uint32_t dst, uint32_t src, uint32_t bytes,
                                                    uint32_t remote_bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(dst), "r"(src), "r"(bytes), "r"(remote_bar)
      : "memory");
}

// shared::cta address -> the same offset in CTA `rank` of the cluster (shared::cluster).
__device__ __forceinline__ uint32_t mapa_shared(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}

// ----------------------------------------------------------------------- TMA --
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// A tensor map in global memory written before the launch (a grouped launch's problem
// table): order this thread's later uses of it through the tensor-map proxy after that
// write (PTX ISA, fence.proxy.tensormap::generic, acquire at system scope for a host
// write).
__device__ __forceinline__ void fence_tensormap_acquire(const void* tmap) {
  asm volatile("fence.proxy.tensormap::generic.acquire.sys [%0], 128;"
               ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}

// 2-D tiled load global -> this CTA's shared memory, completing on `bar` (this CTA);
// one elected lane issues it.
__device__ __forceinline__ void tma_load_2d_elect(uint32_t dst, const void* tmap, int32_t c0,
                                                  int32_t c1, uint32_t bar) {
  asm volatile(GB300_ELECT
               "@e_ cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
               " [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(dst),
               "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar)
               : "memory");
}

// 2-D tiled load for a CTA pair: the data lands in this CTA's shared memory, the
// completion is signalled on `cluster_bar`, which may live in the peer CTA.
__device__ __forceinline__ void tma_load_2d_pair_elect(uint32_t dst, const void* tmap, int32_t c0,
                                                       int32_t c1, uint32_t cluster_bar) {
  asm volatile(
      GB300_ELECT
      "@e_ cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%2, %3}], [%4];\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(cluster_bar)
      : "memory");
}

// Bring a tile of a tensor into L2 without a shared-memory destination (elected lane).
__device__ __forceinline__ void tma_prefetch_l2_2d_elect(const void* tmap, int32_t c0, int32_t c1) {
  asm volatile(GB300_ELECT "@e_ cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];\n\t}" ::"l"(
                   reinterpret_cast<uint64_t>(tmap)),
               "r"(c0), "r"(c1)
               : "memory");
}

// L2 cache policies for the hinted loads: the whole access range marked first to be
// evicted (an operand read once), or last (an operand re-read from L2 by many tiles).
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void tma_load_2d_hint_elect(uint32_t dst, const void* tmap, int32_t c0,
                                                       int32_t c1, uint32_t bar, uint64_t policy) {
  asm volatile(
      GB300_ELECT
      "@e_ cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint_elect(uint32_t dst, const void* tmap,
                                                            int32_t c0, int32_t c1,
                                                            uint32_t cluster_bar, uint64_t policy) {
  asm volatile(
      GB300_ELECT
      "@e_ cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;\n\t}" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(cluster_bar), "l"(policy)
      : "memory");
}

// 2-D tiled store shared -> global (bulk-group completion).
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int32_t c0, int32_t c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.global.shared::cta.tile.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
          reinterpret_cast<uint64_t>(tmap)),
      "r"(src), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void bulk_commit_group() {
  asm volatile("cp.async.bulk.commit_group;" ::: "memory");
}

// Wait until at most N bulk groups are still reading their shared-memory source.
template <int N>
__device__ __forceinline__ void bulk_wait_group_read() {
  asm volatile("cp.async.bulk.wait_group.read %0;" ::"n"(N) : "memory");
}

template <int N>
__device__ __forceinline__ void bulk_wait_group() {
  asm volatile("cp.async.bulk.wait_group %0;" ::"n"(N) : "memory");
}

// Two fused multiply-adds in one instruction: (a0, a1) = (x0, x1) * s + (a0, a1), each
// rounded once as fmaf would (fma.rn.f32x2).  Half the issue slots of two fmaf: the
// blockwise epilogue's warps share an SM sub-partition with the MMA warp, and their
// issue rate set the pace (8192^3 497.7 -> 482.3 us, same bits).
__device__ __forceinline__ void fma2_rn(float& a0, float& a1, float x0, float x1, float s) {
  asm("{\n\t.reg .b64 a_, x_, s_;\n\t"
      "mov.b64 a_, {%0, %1};\n\tmov.b64 x_, {%2, %3};\n\tmov.b64 s_, {%4, %4};\n\t"
      "fma.rn.f32x2 a_, x_, s_, a_;\n\tmov.b64 {%0, %1}, a_;\n\t}"
      : "+f"(a0), "+f"(a1)
      : "f"(x0), "f"(x1), "f"(s));
}

// --------------------------------------------------------------- Tensor Memory --
template <int CTA_GROUP>
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  if constexpr (CTA_GROUP == 1)
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}

template <int CTA_GROUP>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (CTA_GROUP == 1)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

template <int CTA_GROUP>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (CTA_GROUP == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

// ------------------------------------------------------------------- tcgen05.mma --
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, fp32 D; issued by one elected lane of a
// warp whose lanes all execute the call.

// One 128-byte-deep stage (64 fp16/bf16 or 128 FP8 values of K): four MMAs of 32 bytes
// of K each (K=16 for kind::f16, K=32 for kind::f8f6f4; descriptor start addresses
// advance by 32 bytes, i.e. +2 in the >>4-encoded field) and the commit that frees the
// stage, issued by one elected lane in a single asm block.  (Four separately elected
// MMAs cost about 120 cycles of issue each on sm_103a; batched, a 128 x 128 x 16 MMA
// issues every 64 cycles, the tensor core's rate.)  `accumulate` applies to the first
// MMA; the other three always accumulate.  For CTA_GROUP == 2 the commit is multicast
// to both CTAs.  KIND 0: kind::f16; KIND 1: kind::f8f6f4.
#define GB300_STAGE_MMA(CG, KINDSTR)                                                     \
  asm volatile(GB300_ELECT                                                               \
               ".reg .pred p_;\n\t.reg .b64 a1_, a2_, a3_, b1_, b2_, b3_;\n\t"           \
               "setp.ne.b32 p_, %4, 0;\n\t"                                              \
               "add.s64 a1_, %1, 2;\n\tadd.s64 a2_, %1, 4;\n\tadd.s64 a3_, %1, 6;\n\t"    \
               "add.s64 b1_, %2, 2;\n\tadd.s64 b2_, %2, 4;\n\tadd.s64 b3_, %2, 6;\n\t"    \
               "@e_ tcgen05.mma.cta_group::" #CG ".kind::" KINDSTR " [%0], %1, %2, %3, p_;\n\t" \
               "@e_ tcgen05.mma.cta_group::" #CG ".kind::" KINDSTR " [%0], a1_, b1_, %3, 1;\n\t" \
               "@e_ tcgen05.mma.cta_group::" #CG ".kind::" KINDSTR " [%0], a2_, b2_, %3, 1;\n\t" \
               "@e_ tcgen05.mma.cta_group::" #CG ".kind::" KINDSTR " [%0], a3_, b3_, %3, 1;\n\t" \
               GB300_STAGE_COMMIT_##CG "\n\t}"                                               \
               ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate),         \
               "r"(empty_bar), "h"(cta_mask)                                               \
               : "memory")
#define GB300_STAGE_COMMIT_1 \
  "@e_ tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%5];"
#define GB300_STAGE_COMMIT_2                                                            \
  "@e_ tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64" \
  " [%5], %6;"

// One 64-deep stage of a 320-column pair tile: per 16-deep K step an N = 256 MMA into
// columns 0-255 (B from the stage start) and an N = 64 MMA into columns 256-319 (B from
// 16 KiB on: the descriptor's address field counts 16-byte units), then the commit.
__device__ __forceinline__ void umma_stage320_elect(uint32_t d_tmem, uint64_t a_desc,
                                                    uint64_t b_desc, uint32_t idesc256,
                                                    uint32_t idesc64, uint32_t accumulate,
                                                    uint32_t empty_bar, uint16_t cta_mask) {
  asm volatile(GB300_ELECT
               ".reg .pred p_;\n\t.reg .b64 a1_, a2_, a3_, b1_, b2_, b3_, c0_, c1_, c2_, c3_;\n\t"
               ".reg .b32 d2_;\n\t"
               "setp.ne.b32 p_, %4, 0;\n\t"
               "add.s64 a1_, %1, 2;\n\tadd.s64 a2_, %1, 4;\n\tadd.s64 a3_, %1, 6;\n\t"
               "add.s64 b1_, %2, 2;\n\tadd.s64 b2_, %2, 4;\n\tadd.s64 b3_, %2, 6;\n\t"
               "add.s64 c0_, %2, 1024;\n\tadd.s64 c1_, %2, 1026;\n\t"
               "add.s64 c2_, %2, 1028;\n\tadd.s64 c3_, %2, 1030;\n\t"
               "add.u32 d2_, %0, 256;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p_;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [d2_], %1, c0_, %7, p_;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [%0], a1_, b1_, %3, 1;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [d2_], a1_, c1_, %7, 1;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [%0], a2_, b2_, %3, 1;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [d2_], a2_, c2_, %7, 1;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [%0], a3_, b3_, %3, 1;\n\t"
               "@e_ tcgen05.mma.cta_group::2.kind::f16 [d2_], a3_, c3_, %7, 1;\n\t"
               GB300_STAGE_COMMIT_2 "\n\t}"
               ::"r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc256), "r"(accumulate),
               "r"(empty_bar), "h"(cta_mask), "r"(idesc64)
               : "memory");
}

// cta_mask: the pair's two CTAs in the cluster (0b11, or 0b1100 for the second pair of
// a four-CTA cluster).
template <int CTA_GROUP, int KIND = 0>
__device__ __forceinline__ void umma_stage_elect(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                                 uint32_t idesc, uint32_t accumulate,
                                                 uint32_t empty_bar, uint16_t cta_mask = 0x3) {
  if constexpr (CTA_GROUP == 1 && KIND == 0) GB300_STAGE_MMA(1, "f16");
  else if constexpr (CTA_GROUP == 2 && KIND == 0) GB300_STAGE_MMA(2, "f16");
  else if constexpr (CTA_GROUP == 1) GB300_STAGE_MMA(1, "f8f6f4");
  else GB300_STAGE_MMA(2, "f8f6f4");
}

// Make `bar` arrive once all MMAs this thread issued before have completed (the
// cta_group must match the one every other tcgen05 instruction of the kernel uses).
template <int CTA_GROUP>
__device__ __forceinline__ void umma_commit_elect(uint32_t bar) {
  if constexpr (CTA_GROUP == 1)
    asm volatile(GB300_ELECT
                 "@e_ tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                     bar)
                 : "memory");
  else
    asm volatile(GB300_ELECT
                 "@e_ tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(
                     bar)
                 : "memory");
}

// Pair form: the arrive lands on the barrier at the same offset in every CTA of cta_mask.
__device__ __forceinline__ void umma_commit_pair_elect(uint32_t bar, uint16_t cta_mask) {
  asm volatile(GB300_ELECT
               "@e_ tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64"
               " [%0], %1;\n\t}" ::"r"(bar),
               "h"(cta_mask)
               : "memory");
}

// 32 lanes x 32 bits, 32 consecutive columns: thread t of the warp receives lane
// (quarter*32 + t), columns [col, col+32).
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32"
      " {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
        "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
        "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}

__device__ __forceinline__ void tmem_ld_wait() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// Wait for outstanding tcgen05.ld and tie the destination registers to the wait, so
// the compiler cannot move a use of them above it.
__device__ __forceinline__ void tmem_ld_wait(uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.wait::ld.sync.aligned;"
      : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
        "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]),
        "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]),
        "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]), "+r"(r[25]),
        "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
      :
      : "memory");
}

// Tie registers loaded by an earlier tcgen05.ld to a wait already executed: an empty
// statement after the wait (both volatile, so kept in order) that the compiler must treat
// as redefining them, so that no use of them moves above the wait.
__device__ __forceinline__ void tie_regs(uint32_t (&r)[32]) {
  asm volatile(""
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]),
                 "+r"(r[7]), "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]),
                 "+r"(r[13]), "+r"(r[14]), "+r"(r[15]), "+r"(r[16]), "+r"(r[17]), "+r"(r[18]),
                 "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]), "+r"(r[24]),
                 "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]),
                 "+r"(r[31])
               :
               : "memory");
}

// ---------------------------------------------------------- global memory helpers --
__device__ __forceinline__ void st_global_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}

__device__ __forceinline__ void st_global_cg_v4(void* p, uint32_t a, uint32_t b, uint32_t c,
                                                uint32_t d) {
  asm volatile("st.global.cg.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// Counter increment that releases this thread's earlier writes (and, through a
// preceding warp barrier, the warp's) at GPU scope and acquires those released by
// earlier increments: the hand-over of split-K partial tiles between CTAs.
__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.add.acq_rel.gpu.global.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Load that acquires, at GPU scope, the writes released by the increments it observes.
__device__ __forceinline__ uint32_t ld_acquire_gpu_u32(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// 16 bytes global -> shared without passing through registers (cached in L2 only), and
// the wait for all of this thread's such copies.
__device__ __forceinline__ void cp_async_cg_16(uint32_t dst, const void* src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_wait_all() {
  asm volatile("cp.async.commit_group;\n\tcp.async.wait_group 0;" ::: "memory");
}

__device__ __forceinline__ void st_relaxed_gpu_u32(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ uint4 ld_global_cg_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.cg.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p)
               : "memory");
  return v;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c),
               "r"(d)
               : "memory");
}

// ---------------------------------------------------------- cluster launch control --
// Dynamic scheduling ("A Blackwell GEMM by Hand in CuTe DSL", section 8: the tutorials'
// cluster-launch-control scheduler): a running CTA asks to cancel the launch of a cluster
// of the same grid that has not started yet, and takes over its work.  The 16-byte answer
// lands in shared memory and completes 16 bytes on the mbarrier.  One elected lane issues
// it; with MULTICAST the answer reaches the same offsets in every CTA of the cluster.
template <bool MULTICAST>
__device__ __forceinline__ void clc_try_cancel_elect(uint32_t resp, uint32_t bar) {
  if constexpr (MULTICAST)
    asm volatile(GB300_ELECT
                 "@e_ clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes"
                 ".multicast::cluster::all.b128 [%0], [%1];\n\t}" ::"r"(resp), "r"(bar)
                 : "memory");
  else
    asm volatile(GB300_ELECT
                 "@e_ clusterlaunchcontrol.try_cancel.async.shared::cta.mbarrier::complete_tx::bytes"
                 ".b128 [%0], [%1];\n\t}" ::"r"(resp), "r"(bar)
                 : "memory");
}

// Decode an answer: 1 and the cancelled cluster's first blockIdx.x if a launch was
// cancelled; 0 if none was left to cancel (the grid's work is all taken).
__device__ __forceinline__ uint32_t clc_query(uint32_t resp, uint32_t& first_ctaid_x) {
  uint32_t ok, x = 0;
  asm volatile(
      "{\n\t.reg .b128 a_;\n\t.reg .pred c_;\n\t"
      "ld.shared.b128 a_, [%2];\n\t"
      "clusterlaunchcontrol.query_cancel.is_canceled.pred.b128 c_, a_;\n\t"
      "selp.u32 %0, 1, 0, c_;\n\t"
      "@c_ clusterlaunchcontrol.query_cancel.get_first_ctaid::x.b32.b128 %1, a_;\n\t}"
      : "=r"(ok), "+r"(x)
      : "r"(resp)
      : "memory");
  first_ctaid_x = x;
  return ok;
}

}  // namespace gb300
