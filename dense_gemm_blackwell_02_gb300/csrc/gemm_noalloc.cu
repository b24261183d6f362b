// gemm_run_noalloc: the split-K GEMM for callers that cannot allocate device memory.
//
// Who needs this.  Some code that wants a GEMM is not allowed to call cudaMalloc:
//   * a custom device-memory allocator or memory pool that itself wants to run a
//     GEMM (calling cudaMalloc from inside it would recurse into the allocator or
//     bypass the budget it enforces);
//   * a plug-in whose host framework owns every device allocation and forbids
//     extensions from making their own;
//   * a process that has reserved (almost) all device memory up front for a pool and
//     cannot afford a surprise allocation, or an error path that runs when memory is
//     already exhausted.
// gemm_run cannot serve them: it needs a handle, and gemm_create allocates the
// handle's status word, while gemm_run itself grows a split-K workspace on first use.
//
// What this entry point does instead.  Its scratch -- the status word, the split-K
// arrival counters and the fp32 partial tiles -- is one file-scope static __device__
// array of fixed size (GEMM_NOALLOC_SCRATCH_BYTES in include/gemm.h).  The CUDA driver
// places that array on every GPU that loads this library, where it stays until the
// process exits.  On its first call on a device, with that device current, the entry
// point looks up the array's device address (cudaGetSymbolAddress) and keeps it once the
// lookup has succeeded; a first call that has to do this should therefore come before any
// stream capture.  No call makes
// a device or host allocation: no cudaMalloc, no cudaFree, no allocating library call.
//
// Sharing.  Every call on a device uses the same array, which keeps the previous
// call's contents; each call clears the status word and the counters it will use
// (cudaMemsetAsync on the caller's stream) before its kernel.  Two calls whose work
// overlaps on the GPU (different streams, no ordering between them) race on the
// array and may produce wrong results.
//
// The kernel is the same one-CTA split-K kernel gemm_run launches (BN = 256, 4 stages),
// with its K-slice count chosen by a fixed rule in this file.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstring>
#include <mutex>

#include "gemm.h"
#include "launch.h"
#include "umma.cuh"

using namespace gb300;

namespace {

constexpr size_t kStatusBytes = 256;                               // status word, padded
constexpr size_t kCounterWords = 16384;                            // (tile, quarter, half) counters
constexpr size_t kCounterBytes = kCounterWords * sizeof(uint32_t);
constexpr size_t kWorkspaceBytes = GEMM_NOALLOC_WORKSPACE_BYTES;   // fp32 partial tiles
constexpr size_t kScratchBytes = kStatusBytes + kCounterBytes + kWorkspaceBytes;
static_assert(kScratchBytes == GEMM_NOALLOC_SCRATCH_BYTES, "header and file disagree");
constexpr int kBN = 256;
constexpr int kStages = 4;
constexpr uint64_t kWaitLimitNs = 2000000000ull;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;

struct DeviceSetup {
  bool done = false;                 // set only once the lookup below has succeeded
  unsigned char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
  int sms = 0;
  bool supported = false;
};

DeviceSetup g_setup[kMaxDevices];
std::mutex g_setup_mutex;

// Once per device, with that device current: find the array's device address.  Only a
// successful set-up is remembered: a first call that fails (for instance one made by
// mistake during a stream capture, where the lookup may be refused) leaves the device
// unset, and a later call tries again.
cudaError_t setup_device(int dev, DeviceSetup* s) {
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (s->done) return cudaSuccess;
  int major = 0, minor = 0, sms = 0;
  cudaError_t err = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  if (err == cudaSuccess) err = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (err != cudaSuccess) return err;
  const bool supported = (major == 10 && minor == 3);
  void* p = nullptr;
  if (supported) {
    err = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (err != cudaSuccess) return err;
  }
  s->scratch = static_cast<unsigned char*>(p);
  s->sms = sms;
  s->supported = supported;
  s->done = true;
  return cudaSuccess;
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// rows x cols row-major matrix, 128-byte swizzle, box {128 bytes of columns, box_rows};
// loads zero-fill out-of-range elements, stores skip them.
bool encode_map(const void* ptr, int64_t rows, int64_t cols, gemm_dtype_t dtype, int box_rows,
                CUtensorMap* out) {
  auto fn = encoder();
  if (!fn) return false;
  const cuuint64_t esz = dtype == GEMM_F32 ? 4 : 2;
  const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)cols * esz};
  const cuuint32_t box[2] = {(cuuint32_t)(128 / esz), (cuuint32_t)box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUtensorMapDataType dt = dtype == GEMM_BF16  ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                 : dtype == GEMM_F32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                                     : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  return fn(out, dt, 2, const_cast<void*>(ptr), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M,
                                          int64_t N, int64_t K, gemm_dtype_t dtype_in,
                                          gemm_dtype_t dtype_out, gemm_stream_t stream_) {
  if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
  const bool in_ok = dtype_in == GEMM_F16 || dtype_in == GEMM_BF16;
  const bool out_ok = dtype_out == GEMM_F16 || dtype_out == GEMM_BF16 || dtype_out == GEMM_F32;
  const bool in_known = in_ok || dtype_in == GEMM_F32 || dtype_in == GEMM_E4M3 ||
                        dtype_in == GEMM_E5M2;  // known types this entry point does not take
  if (!out_ok || !in_known) return GEMM_ERR_INVALID_ARG;
  if (!in_ok) return GEMM_ERR_UNSUPPORTED;
  if (M == 0 || N == 0) return GEMM_OK;
  if (!C || (K > 0 && (!A || !B))) return GEMM_ERR_INVALID_ARG;
  if (M > INT32_MAX || N > INT32_MAX || K > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const size_t osz = dtype_out == GEMM_F32 ? 4 : 2;
  if (reinterpret_cast<uintptr_t>(C) % osz) return GEMM_ERR_UNSUPPORTED;
  if (K == 0)
    return cudaMemsetAsync(C, 0, (size_t)M * (size_t)N * osz, stream) == cudaSuccess
               ? GEMM_OK
               : GEMM_ERR_CUDA;
  if (K % 8) return GEMM_ERR_UNSUPPORTED;
  if (reinterpret_cast<uintptr_t>(A) % 16 || reinterpret_cast<uintptr_t>(B) % 16)
    return GEMM_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return GEMM_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
  DeviceSetup& ds = g_setup[dev];
  if (setup_device(dev, &ds) != cudaSuccess) return GEMM_ERR_CUDA;
  if (!ds.supported) return GEMM_ERR_UNSUPPORTED;

  // Fixed K-slice rule: slice K only when there are fewer tiles than half the SMs, and
  // into no more slices than the fixed scratch holds partial tiles for (one slice needs
  // none, so every valid product runs).
  const int64_t k_blocks = cdiv(K, kBlockK);
  const int64_t num_m = cdiv(M, kBlockM), num_n = cdiv(N, kBN);
  const int64_t tiles = num_m * num_n;
  int64_t splits = 1;
  if (tiles * 2 <= ds.sms && k_blocks >= 8) {
    splits = ds.sms / tiles;
    if (splits > k_blocks / 4) splits = k_blocks / 4;
    if (splits > 32) splits = 32;
    const int64_t fit = (int64_t)(kWorkspaceBytes / ((size_t)tiles * kBlockM * kBN * sizeof(float)));
    if (splits > fit) splits = fit;
    if (splits < 1) splits = 1;
  }
  const int64_t per = cdiv(k_blocks, splits);
  splits = cdiv(k_blocks, per);
  const int64_t units = tiles * splits;
  if (units > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
  const size_t ws_need = splits > 1 ? (size_t)tiles * splits * kBlockM * kBN * sizeof(float) : 0;
  const size_t ctr_need = splits > 1 ? (size_t)tiles * 8 : 0;  // (tile, quarter, half)
  // (cannot happen with the rule above; kept as the guard of the fixed-size scratch)
  if (ws_need > kWorkspaceBytes || ctr_need > kCounterWords) return GEMM_ERR_UNSUPPORTED;

  LaunchSpec s;
  std::memset(&s, 0, sizeof(s));
  s.cta_group = 1;
  s.bn = kBN;
  s.stages = kStages;
  s.out = dtype_out == GEMM_F16 ? kOutF16 : dtype_out == GEMM_BF16 ? kOutBF16 : kOutF32;
  s.grid = (int)(units < ds.sms ? units : ds.sms);
  s.stream = stream;
  const bool c_tma = reinterpret_cast<uintptr_t>(C) % 16 == 0 && ((size_t)N * osz) % 16 == 0;
  // one row tile of M < 128 rows: A's box is M rows (see gemm_run)
  const int a_box = M < kBlockM ? (int)M : kBlockM;
  if (!encode_map(A, M, K, dtype_in, a_box, &s.tmA) ||
      !encode_map(B, N, K, dtype_in, kBN, &s.tmB) ||
      (c_tma && !encode_map(C, M, N, dtype_out, 32, &s.tmC)))
    return GEMM_ERR_CUDA;
  s.tmB2 = s.tmB;  // no half-tile units here

  uint32_t* status = reinterpret_cast<uint32_t*>(ds.scratch);
  uint32_t* counters = reinterpret_cast<uint32_t*>(ds.scratch + kStatusBytes);
  float* workspace = reinterpret_cast<float*>(ds.scratch + kStatusBytes + kCounterBytes);
  // The array keeps the last call's contents: the status word and the counters this
  // call uses must start at zero (the partial tiles are written before they are read).
  if (cudaMemsetAsync(ds.scratch, 0, kStatusBytes + ctr_need * sizeof(uint32_t), stream) !=
      cudaSuccess)
    return GEMM_ERR_CUDA;

  GemmParams& p = s.p;
  p.C = C;
  p.M = (int32_t)M;
  p.N = (int32_t)N;
  p.K = (int32_t)K;
  p.num_m_tiles = (int32_t)num_m;
  p.num_n_tiles = (int32_t)num_n;
  p.tiles = (int32_t)tiles;
  p.k_blocks = (int32_t)k_blocks;
  p.dp_tiles = splits > 1 ? 0 : (int32_t)tiles;
  p.half_tail = 0;
  p.splits = (int32_t)splits;
  p.kb_per_split = (int32_t)per;
  p.units = (int32_t)units;
  p.sk_workers = 0;
  p.ws_slots = (int32_t)splits;
  p.group_m = 16;
  p.chain_kb = kChainKBlocks;
  p.prefetch_kb = 0;
  p.l2_hint = 1;
  p.a_tx_short = (uint32_t)(kBlockM - a_box) * 128u;
  p.vec_store = c_tma ? 1 : 0;
  p.tma_store = c_tma ? 1 : 0;
  p.idesc = idesc_f16_kmajor(kBlockM, kBN, dtype_in == GEMM_BF16);
  p.idesc_half = p.idesc;
  p.workspace = workspace;
  p.counters = counters;
  p.status = status;
  p.wait_limit_ns = kWaitLimitNs;
  p.test_stall = 0;
  return launch_gemm(s) == cudaSuccess ? GEMM_OK : GEMM_ERR_CUDA;
}
