// C = A . B^T for M <= 4 rows of A on the CUDA cores: the product is then a stream
// over B (every element of B used once per row of A, 2M FLOPs per 2 bytes), bound by
// HBM, so it is written as a coalesced stream rather than shaped into tensor-core
// tiles ("A Blackwell GEMM by Hand in CuTe DSL", section 1: decode shapes are bound by
// memory; section 9: decided by how the work fills the machine).
//
// Every warp takes its own rows n = w, w + W, ... of B (w the warp's index in the
// grid, W the grid's warps): its 32 lanes read 16-byte chunks l, l + 32, ... of B_n,
// eight chunks in flight per lane, and the same chunks of the M rows of A (A is small
// and stays in L1/L2), multiply in fp32 and accumulate with fma; the warp then sums its
// lanes with shuffles and lane 0 writes C[m][n].  The order of every addition is fixed,
// so the result does not change from run to run.  Products of two fp16 or bf16 values
// are exact in fp32; only the additions round.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>

#include "launch.h"

namespace gb300 {

namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

template <bool BF16>
__device__ __forceinline__ void widen8(const uint4& x, float (&f)[8]) {
  const uint32_t w[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      const __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      const float2 v = __bfloat1622float2(h);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    } else {
      const __half2 h = *reinterpret_cast<const __half2*>(&w[i]);
      const float2 v = __half22float2(h);
      f[2 * i] = v.x;
      f[2 * i + 1] = v.y;
    }
  }
}

template <int OUT>
__device__ __forceinline__ void store_out(void* C, size_t idx, float v) {
  if constexpr (OUT == kOutF32) reinterpret_cast<float*>(C)[idx] = v;
  else if constexpr (OUT == kOutF16) reinterpret_cast<__half*>(C)[idx] = __float2half_rn(v);
  else reinterpret_cast<__nv_bfloat16*>(C)[idx] = __float2bfloat16_rn(v);
}

// Loads through the read-only path: B streams once, A is re-read by every row.
__device__ __forceinline__ uint4 ldg_stream(const uint4* p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <int MR, bool BF16, int OUT>
__global__ void __launch_bounds__(kGemvThreads) gemv_kernel(const uint4* __restrict__ A,
                                                           const uint4* __restrict__ B,
                                                           void* __restrict__ C, int32_t M,
                                                           int32_t N, int32_t chunks) {
  constexpr int kInFlight = 8;  // 16-byte chunks of B per lane before they are used
  const int lane = threadIdx.x & 31;
  const int32_t warps = (int32_t)gridDim.x * kGemvWarps;
  // Wait for the preceding kernel in the stream (programmatic dependent launch) before
  // any global memory is touched, then let the next one be scheduled.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" :::);
  for (int32_t n = (int32_t)blockIdx.x * kGemvWarps + (threadIdx.x >> 5); n < N; n += warps) {
    const uint4* brow = B + (size_t)n * chunks;
    float acc[MR];
#pragma unroll
    for (int m = 0; m < MR; ++m) acc[m] = 0.0f;
    for (int32_t c0 = lane; c0 < chunks; c0 += kInFlight * 32) {
      uint4 bv[kInFlight];
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int32_t c = c0 + u * 32;
        bv[u] = c < chunks ? ldg_stream(brow + c) : make_uint4(0, 0, 0, 0);
      }
#pragma unroll
      for (int u = 0; u < kInFlight; ++u) {
        const int32_t c = c0 + u * 32;
        if (c >= chunks) break;
        float bf[8];
        widen8<BF16>(bv[u], bf);
#pragma unroll
        for (int m = 0; m < MR; ++m) {
          if (m >= M) break;
          float af[8];
          widen8<BF16>(__ldg(A + (size_t)m * chunks + c), af);
#pragma unroll
          for (int j = 0; j < 8; ++j) acc[m] = fmaf(af[j], bf[j], acc[m]);
        }
      }
    }
#pragma unroll
    for (int m = 0; m < MR; ++m) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) acc[m] += __shfl_xor_sync(0xFFFFFFFFu, acc[m], off);
    }
    if (lane == 0) {
#pragma unroll
      for (int m = 0; m < MR; ++m)
        if (m < M) store_out<OUT>(C, (size_t)m * N + n, acc[m]);
    }
  }
}

template <int MR, bool BF16>
cudaError_t launch_by_out(const GemvSpec& s) {
  void (*k)(const uint4*, const uint4*, void*, int32_t, int32_t, int32_t) =
      s.out == kOutF16 ? gemv_kernel<MR, BF16, kOutF16>
      : s.out == kOutBF16 ? gemv_kernel<MR, BF16, kOutBF16>
                          : gemv_kernel<MR, BF16, kOutF32>;
  // no more CTAs than fit at once: a CTA that waits for a free SM would start its rows late
  static int per_sm = 0;
  if (per_sm == 0 && cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k, kGemvThreads, 0) !=
                         cudaSuccess) {
    cudaGetLastError();
    per_sm = 1;
  }
  int dev = 0, sms = 1;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(std::min(s.grid, std::max(per_sm, 1) * sms), 1, 1);
  cfg.blockDim = dim3(kGemvThreads, 1, 1);
  cfg.stream = s.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, static_cast<const uint4*>(s.A),
                            static_cast<const uint4*>(s.B), s.C, s.M, s.N, s.chunks);
}

}  // namespace

cudaError_t launch_gemv(const GemvSpec& s) {
  if (s.M < 1 || s.M > kGemvMaxRows || s.grid < 1) return cudaErrorInvalidValue;
  if (s.M <= 2) return s.bf16 ? launch_by_out<2, true>(s) : launch_by_out<2, false>(s);
  return s.bf16 ? launch_by_out<4, true>(s) : launch_by_out<4, false>(s);
}

}  // namespace gb300
