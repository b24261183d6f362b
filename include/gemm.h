/*
 * gemm.h -- C ABI of libgemm.so, a GB300 (sm_103a) dense tensor-core GEMM.
 *
 *     C = A . B^T        A: M x K,  B: N x K,  C: M x N
 *
 * The operation is the one defined in "A Blackwell GEMM by Hand in CuTe DSL",
 * section 1 (C_{MxN} = A_{MxK} B_{NxK}^T, both operands K-major), with fp16 or
 * bf16 inputs, fp32 accumulation, and C written as fp16, bf16 or fp32
 * (round-to-nearest-even from the fp32 accumulator).  The kernels are built
 * from TMA, mbarriers, tcgen05.mma into Tensor Memory and warp specialisation
 * (same page, sections 2-3 and 8; "Optimizing GEMMs using tcgen05 - Part 1").
 *
 * Layout.  All matrices are dense and row-major with no padding:
 *   A[i][k] at A + (i*K + k) elements, B[j][k] at B + (j*K + k),
 *   C[i][j] at C + (i*N + j).
 * "K-major" means K is the contiguous dimension of A and B.
 *
 * Ownership.  The caller owns A, B and C (device memory unless stated), and
 * keeps them alive until the work queued on `stream` has finished.  A handle
 * owns its split-K workspace, its device status word, its tensor-map cache and
 * the staging buffers of gemm_run_host.  One handle serves one host thread and
 * one stream at a time: calls that overlap on the GPU through one handle race
 * on its workspace.
 *
 * Errors.  Every call returns a gemm_status_t.  Argument problems are reported
 * synchronously and nothing is launched.  gemm_run is asynchronous: a kernel
 * whose internal wait ran out of time (a hang that was cut short) is reported
 * later by gemm_device_status, which synchronises the stream.
 */
#ifndef GB300_GEMM_H
#define GB300_GEMM_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t (a CUstream); 0 / NULL is the legacy default stream. */
typedef struct CUstream_st* gemm_stream_t;

typedef struct gemm_ctx* gemm_handle_t;

/* Element types.  GEMM_F32 is an output type only; GEMM_E4M3 and GEMM_E5M2 (OCP 8-bit
 * floating point, one byte per element: E4M3 with bias 7, no infinities, largest
 * finite 448; E5M2 IEEE-style with bias 15) are input types only ("CUTLASS Deep
 * Dive: From CuTe Layouts to Blackwell tcgen05", Part 6: FP8 and Blockwise Scaling). */
typedef enum {
  GEMM_F16 = 0,
  GEMM_BF16 = 1,
  GEMM_F32 = 2,
  GEMM_E4M3 = 3,
  GEMM_E5M2 = 4
} gemm_dtype_t;

typedef enum {
  GEMM_OK = 0,
  GEMM_ERR_INVALID_ARG = 1, /* null pointer, negative size, bad handle, bad config */
  GEMM_ERR_UNSUPPORTED = 2, /* dtype combination, K not a multiple of 16 bytes, pointer
                               not 16-byte aligned, no sm_103 device */
  GEMM_ERR_CUDA = 3,        /* a CUDA runtime / driver call failed */
  GEMM_ERR_OOM = 4,         /* device or host allocation failed */
  GEMM_ERR_TIMEOUT = 5      /* a kernel wait exceeded its limit (see gemm_device_status) */
} gemm_status_t;

/*
 * Kernel selection.  Zero in any field means "choose automatically".
 *   variant   1 = one CTA per 128-row tile (cta_group::1)
 *             2 = a CTA pair per 256-row tile (cta_group::2, cluster of 2)
 *             3 = the CUDA-core matrix-vector path for M <= 4 (fp16/bf16 inputs, no
 *                 fused epilogue; other fields ignored except max_ctas); chosen
 *                 automatically for M == 1 with K <= 16384
 *   block_n   128 or 256 columns of C per tile; or 320 (two MMAs per K step, N = 256
 *             and N = 64) for CTA pairs under the cluster K split with single-chain
 *             slices only (epilogue 3; else GEMM_ERR_UNSUPPORTED), chosen automatically
 *             when 256-column tiles cannot be cut into two K slices within the resident
 *             pairs and 320-column tiles can
 *   splits    K slices per tile (1 = no split; >1 = split-K with a deterministic
 *             in-kernel reduction in slice order; -1 = stream-K: every resident unit
 *             takes an equal share of the (tile, K block) iterations).
 *             gemm_last_config reports -W for stream-K over W units.  Stream-K
 *             needs tiles * K blocks * W < 2^32; gemm_run returns
 *             GEMM_ERR_UNSUPPORTED beyond that.
 *   stages    depth of the shared-memory operand ring: 6 (pairs, BN 256), 8 (pairs, BN
 *             128), 4 (one CTA, BN 256), 6 (one CTA, BN 128); or, for one CTA and at most 16
 *             rows of A with fp16/bf16 inputs and no fused epilogue, 5 (BN 256) or 10 (BN
 *             128) stages that hold 16 rows of A each (chosen automatically for M <= 16).
 *             The cluster K split (epilogue 3) keeps its epilogue staging inside the idle
 *             ring and runs one stage deeper: 7 (pairs, BN 256), 9 (pairs, BN 128), 6
 *             (pairs, BN 320), 4 (one CTA, BN 256), 7 (one CTA, BN 128), 6 and 12 with
 *             16-row A stages; a forced depth other than that one refuses it.
 *             gemm_last_config reports the depth used.
 *   group_m   grouped rasterisation: M tiles per group
 *   max_ctas  cap on the persistent grid (0 = one CTA per SM)
 *   chain_kblocks  K blocks (128 bytes of K: 64 fp16/bf16 or 128 FP8 elements)
 *             accumulated in one Tensor-Memory accumulator before the epilogue adds
 *             it into its fp32 registers (0 = K 4096: 64 blocks, or 32 for FP8; the
 *             tensor core's fp32 accumulation error grows with the length of one
 *             accumulation chain)
 *   dp_tiles  reported by gemm_last_config only (must be 0 on input): how many
 *             tiles ran whole.  The rest ran as `splits` K slices each, or, when
 *             `splits` is 1, as two half-width (block_n / 2 column) units each.  A
 *             forced `splits` slices every tile; automatically, only the tiles of a
 *             partial last wave are cut (or all tiles are sliced along K when there
 *             are too few of them for the SMs).
 *   prefetch_kblocks  how many 64-deep K blocks ahead of the shared-memory ring the
 *             producer prefetches B into L2 (0 or -1 = never, the default)
 *   epilogue  1 = general (the accumulator is copied to registers, chains summed
 *             there); 2 = single-chain (streamed out of Tensor Memory in 32-column
 *             pieces), valid only when every work unit spans at most chain_kblocks K
 *             blocks (else gemm_run returns GEMM_ERR_UNSUPPORTED); 0 = 2 when valid
 *             for fp16/bf16 inputs, 1 for FP8 inputs (faster there: an FP8 tile is
 *             half the stages, and the single-chain form holds its accumulator slot
 *             through the stores);
 *             3 = single-chain with a tile's two K slices run by the two CTA groups of
 *             one cluster (2 CTAs, or 4 for pairs) and summed through distributed
 *             shared memory instead of the global workspace (each slice summed in
 *             the single-chain or the general epilogue, whichever its length allows):
 *             valid only for fp16/bf16 inputs without a fused epilogue, when the shape
 *             is cut into exactly 2 K slices, with every tile and every unit resident
 *             at once (else GEMM_ERR_UNSUPPORTED).  Chosen automatically when one of
 *             the two tile widths gives exactly that.
 *             gemm_last_config reports the one used.
 *   l2_hint   L2 cache policy of the operand loads: 1 = none; 2 = B's loads marked
 *             evict-first and A's evict-last (for one row of tiles, where every B
 *             element is read once and A is re-read by every tile); 0 = 2 when the
 *             tiles form one row (M <= 256 for CTA pairs, M <= 128 for one CTA per
 *             tile; with swap_ab, M <= block_n or the tiles form one wave), else 1.
 *             gemm_last_config reports the one used.
 *   swap_ab   2 = the swapped tiling for a few rows of A (decode shapes): B is the
 *             MMA's row operand, swap_rows of its rows per CTA of a pair, and block_n
 *             (128 or 256) rows of A are the MMA's columns, so a tile covers block_n
 *             rows x 2 * swap_rows columns of C, written transposed from Tensor Memory
 *             by direct stores.  Valid for fp16/bf16 inputs without a fused epilogue,
 *             CTA pairs (variant 0 or 2), no K split (splits 0 or 1), the general
 *             epilogue (epilogue 0 or 1); else GEMM_ERR_UNSUPPORTED.  1 = off;
 *             0 = chosen automatically (only when no other field but group_m,
 *             prefetch_kblocks and l2_hint is forced) for 17..128 rows of A with K of
 *             two accumulation chains or more (8192 fp16/bf16 elements) when the plain
 *             one-CTA tiles would leave a quarter of the SMs idle and the swapped tiles,
 *             with at least 96 rows of B per CTA, form one wave (or, with K of at most
 *             two chains, a second wave at least 40% full).
 *             gemm_last_config reports 2 or 1.
 *   swap_rows with swap_ab: rows of B per CTA, 1..128 (0 = the fewest that make one
 *             wave of tiles, rounded up to a multiple of 8, at most 128).
 *             gemm_last_config reports the one used (0 when not swapped).
 *   scheduler how a grouped launch (gemm_run_grouped) hands its tiles to the CTAs:
 *             1 = round-robin over the resident CTAs (pairs), a persistent grid;
 *             2 = cluster launch control ("A Blackwell GEMM by Hand in CuTe DSL",
 *             section 8): a CTA (pair) per tile in the grid, and every running one
 *             takes over the tiles of launches that have not started yet, so CTAs that
 *             finish early take more (not with max_ctas: GEMM_ERR_UNSUPPORTED);
 *             0 = 2 when the problems' K differ by 2x or more (unequal tile costs),
 *             else 1.  Either way the problems' tiles are handed out longest K first.
 *             Other calls refuse 2 with GEMM_ERR_UNSUPPORTED.  gemm_last_config
 *             reports 1 or 2.
 */
typedef struct {
  int32_t variant;
  int32_t block_n;
  int32_t splits;
  int32_t stages;
  int32_t group_m;
  int32_t max_ctas;
  int32_t chain_kblocks;
  int32_t dp_tiles;
  int32_t prefetch_kblocks;
  int32_t epilogue;
  int32_t l2_hint;
  int32_t swap_ab;
  int32_t swap_rows;
  int32_t scheduler;
} gemm_config_t;

/* Create a handle on the current CUDA device.  Fails with GEMM_ERR_UNSUPPORTED
 * if that device is not compute capability 10.3.  *out is NULL on failure. */
gemm_status_t gemm_create(gemm_handle_t* out);

/* Release a handle and everything it owns.  Synchronises the device first.
 * NULL is accepted and ignored. */
gemm_status_t gemm_destroy(gemm_handle_t h);

/*
 * Queue C = A . B^T on `stream`.
 *   A, B, C     device pointers, 16-byte aligned, layouts as above.
 *   M, N, K     sizes >= 0.  M == 0 or N == 0 is a no-op; K == 0 writes C = 0.
 *               A row of K elements must be a multiple of 16 bytes (TMA row
 *               pitch): K % 8 == 0 for fp16/bf16, K % 16 == 0 for FP8.
 *   dtype_in    GEMM_F16, GEMM_BF16, GEMM_E4M3 or GEMM_E5M2 (A and B share it).
 *               FP8 runs tcgen05.mma kind::f8f6f4 with K blocks of 128 elements
 *               ("A Blackwell GEMM by Hand in CuTe DSL", section 6: the 128-byte
 *               swizzle atom holds 128 FP8 values of K); a per-tensor scale pair
 *               (scale_a, scale_b) is applied as gemm_run_epilogue's
 *               alpha = scale_a * scale_b.
 *   dtype_out   GEMM_F16, GEMM_BF16 or GEMM_F32.
 * Neither allocates on the steady path nor synchronises: the split-K workspace
 * grows on the first call that needs more of it (an allocation, outside any
 * stream capture you may be doing, so warm a shape up first).
 */
gemm_status_t gemm_run(gemm_handle_t h, const void* A, const void* B, void* C, int64_t M,
                       int64_t N, int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                       gemm_stream_t stream);

/*
 * Fused epilogue ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05",
 * Part 6: Epilogue Visitor Trees, D = alpha * acc + beta * C; Classic Fused
 * Epilogue: Bias + ReLU).  Applied to the fp32 accumulator before the single
 * rounding to dtype_out:
 *     C[i][j] = act( alpha * sum_k A[i][k] B[j][k] + beta * C_prev[i][j] + bias[j] )
 *   alpha, beta  binary32 scales (alpha = 1, beta = 0: the plain product)
 *   C_prev       the contents of C before the call (read in dtype_out, only when
 *                beta != 0; C is then read and overwritten in place)
 *   bias         N binary32 values, one per column of C, 16-byte aligned; or NULL
 *   activation   GEMM_ACT_NONE (identity) or GEMM_ACT_RELU (max(x, 0); NaN and -0
 *                give +0)
 * The caller owns bias.  Split-K and stream-K tiles apply it once, to the reduced
 * sum.
 */
typedef enum { GEMM_ACT_NONE = 0, GEMM_ACT_RELU = 1 } gemm_activation_t;
typedef struct {
  float alpha;
  float beta;
  const float* bias;
  int32_t activation;
} gemm_epilogue_t;

/* gemm_run with a fused epilogue.  epilogue == NULL (or alpha 1, beta 0, no bias,
 * no activation) is exactly gemm_run.  Errors as gemm_run, and:
 *   GEMM_ERR_INVALID_ARG   an activation other than the two above;
 *   GEMM_ERR_UNSUPPORTED   bias not 16-byte aligned, or K == 0 with a non-trivial
 *                          epilogue. */
gemm_status_t gemm_run_epilogue(gemm_handle_t h, const void* A, const void* B, void* C,
                                int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                                gemm_dtype_t dtype_out, const gemm_epilogue_t* epilogue,
                                gemm_stream_t stream);

/*
 * Blockwise-scaled FP8 product ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell
 * tcgen05", Part 6: FP8 and Blockwise Scaling: one scale per (block_m, block_k) tile
 * of A and one per (block_n, block_k) tile of B, applied during accumulation):
 *     C[i][j] = sum_kb sfa[i / block_m][kb] * sfb[j / 128][kb]
 *                      * sum_{k = 128 kb}^{min(K, 128 kb + 128) - 1} A[i][k] B[j][k]
 *   sfa       the ceil(M / block_m) x ceil(K / 128) binary32 scales of A, stored
 *             K-block-major: scale (r, kb) at sfa[kb * ceil(M / block_m) + r]; device
 *             memory, 4-byte aligned; the caller owns it
 *   sfb       the ceil(N / 128) x ceil(K / 128) scales of B, likewise: scale (c, kb) at
 *             sfb[kb * ceil(N / 128) + c]
 *   block_m   rows of A per scale, >= 1 (1: one scale per row and K block; 128: per
 *             128 x 128 tile)
 *   block_n   rows of B per scale: 128
 * Each 128-element K block is accumulated in its own Tensor-Memory chain, then scaled
 * and added in fp32 registers (fma(P_kb, sfa * sfb, acc)).  Automatically one CTA per
 * 128 x 128 tile (variant 1, block_n 128), whose kernel keeps four accumulator slots.
 */
typedef struct {
  const float* sfa;
  const float* sfb;
  int32_t block_m;
  int32_t block_n;
} gemm_block_scales_t;

/* gemm_run with FP8 operands and block scales.  Errors as gemm_run, and:
 *   GEMM_ERR_INVALID_ARG   scales NULL, block_m < 1;
 *   GEMM_ERR_UNSUPPORTED   dtype_in not FP8, block_n != 128, a scale pointer not
 *                          4-byte aligned, or a forced configuration with
 *                          chain_kblocks > 1 or the single-chain epilogue. */
gemm_status_t gemm_run_blockwise(gemm_handle_t h, const void* A, const void* B, void* C,
                                 int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                                 gemm_dtype_t dtype_out, const gemm_block_scales_t* scales,
                                 gemm_stream_t stream);

/*
 * Grouped GEMM ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05", Part 6,
 * Grouped GEMM: the many differently shaped GEMMs of a Mixture-of-Experts layer in one
 * launch, each tile fetching its problem's pointers and tensor maps).  For every
 * problem g: C_g = A_g . B_g^T, with A_g (M_g x K_g), B_g (N_g x K_g) and C_g
 * (M_g x N_g) laid out, aligned and owned as for gemm_run.
 *   problems   `count` descriptions in HOST memory, read before the call returns
 *   dtype_in   GEMM_F16 or GEMM_BF16 (shared by every problem; FP8 is refused)
 *   dtype_out  GEMM_F16, GEMM_BF16 or GEMM_F32
 * Problems with M_g == 0 or N_g == 0 are skipped; K_g == 0 writes C_g = 0.  One
 * kernel computes the rest: whole tiles of every problem, 128 x block_n (one CTA) or
 * 256 x block_n (a CTA pair; chosen when padding every M_g to 256 rows costs at most
 * 10% more work), handed to the persistent CTAs in problem order.  gemm_set_config's
 * variant, block_n, stages, group_m, max_ctas and chain_kblocks apply; a forced
 * splits other than 1, or the single-chain epilogue, gives GEMM_ERR_UNSUPPORTED.
 * The problem table goes to the device with cudaMemcpyAsync on `stream` from a ring
 * of four pinned buffers owned by the handle; a fifth call waits for the first's copy.
 * Calls on one handle share its buffers: order them on one stream.
 * Errors as gemm_run, checked for every problem before anything is queued.
 */
typedef struct {
  const void* A;
  const void* B;
  void* C;
  int64_t M, N, K;
} gemm_problem_t;

gemm_status_t gemm_run_grouped(gemm_handle_t h, const gemm_problem_t* problems, int32_t count,
                               gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                               gemm_stream_t stream);

/*
 * The same product with HOST buffers: copies A and B to device staging buffers
 * owned by the handle, runs the GEMM and copies C back, then synchronises `stream`
 * and reports kernel timeouts like gemm_device_status.  From M = 2048 rows on, the
 * work is a pipeline of two to eight row chunks of about 1024 rows (a multiple of 256):
 * B goes over first, then chunk c's rows of A
 * go over on a copy stream owned by the handle while the GEMM of chunk c - 1 runs on
 * `stream` and the C rows of chunk c - 2 come back on a second copy stream.
 * Page-locked host memory makes the copies asynchronous DMA; pageable memory
 * works but is slower.
 */
gemm_status_t gemm_run_host(gemm_handle_t h, const void* A_host, const void* B_host, void* C_host,
                            int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                            gemm_dtype_t dtype_out, gemm_stream_t stream);

/* Force a kernel configuration for later runs (NULL restores automatic choice).
 * Invalid combinations are rejected here with GEMM_ERR_INVALID_ARG; a forced
 * choice that cannot serve a given shape makes gemm_run fail the same way. */
gemm_status_t gemm_set_config(gemm_handle_t h, const gemm_config_t* cfg);

/* The configuration the last successful gemm_run on this handle launched. */
gemm_status_t gemm_last_config(gemm_handle_t h, gemm_config_t* out);

/* A GPU described rather than queried, for gemm_plan: its SM count, the CTA pairs that
 * can be resident at once (one CTA per SM), and the clusters of four CTAs (two pairs)
 * that can be resident at once for the pair's cluster K split.  A full GB300:
 * {152, 76, 36}. */
typedef struct {
  int32_t sms;
  int32_t pairs;
  int32_t clusters4;
} gemm_device_model_t;

/* The configuration gemm_run (fused = 0, blockwise = 0), gemm_run_epilogue with a
 * non-trivial epilogue (fused = 1) or gemm_run_blockwise (blockwise = 1) would launch
 * for an M x N x K product on the described device, under `forced` (NULL: automatic
 * choice), without touching a GPU: the same host decisions, with every residency query
 * answered from *dev instead of the driver.  *out is filled as gemm_last_config would
 * be.  Errors: NULL dev or out, dev->sms < 2, dev->pairs < 1, dev->clusters4 < 0,
 * M, N or K < 1, or an invalid dtype -> GEMM_ERR_INVALID_ARG; the combinations gemm_run
 * refuses (K * element size not a multiple of 16, FP8 output, blockwise scales
 * without FP8 inputs, a forced configuration that cannot serve the shape) ->
 * GEMM_ERR_UNSUPPORTED or GEMM_ERR_INVALID_ARG as there.  Pointer alignment, which
 * gemm_run also checks, is not part of the plan. */
gemm_status_t gemm_plan(const gemm_device_model_t* dev, const gemm_config_t* forced,
                        int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype_in,
                        gemm_dtype_t dtype_out, int32_t fused, int32_t blockwise,
                        gemm_config_t* out);

/* Synchronise `stream`, read and clear the handle's device status word.
 * Returns GEMM_ERR_TIMEOUT if a kernel gave up waiting since the last call
 * (the output of that run is undefined), else GEMM_OK.  *detail, if non-NULL,
 * receives the raw word (code << 24 | wait site << 16 | block index). */
gemm_status_t gemm_device_status(gemm_handle_t h, gemm_stream_t stream, uint32_t* detail);

/* Upper bound, in nanoseconds, on any single wait inside the kernels (default
 * 2 s).  Must be > 0. */
gemm_status_t gemm_set_wait_limit(gemm_handle_t h, uint64_t ns);

/* Test hook: when enabled, the MMA-issuing thread of every CTA first waits on
 * a barrier that nothing ever arrives on, so the wait limit runs out and the
 * run ends with GEMM_ERR_TIMEOUT instead of a result.  Off by default. */
gemm_status_t gemm_set_test_stall(gemm_handle_t h, int32_t enable);

/* Number of SMs of the handle's device. */
int32_t gemm_sm_count(gemm_handle_t h);

/* Static description of a status code; never NULL. */
const char* gemm_status_string(gemm_status_t s);

/* The name of the CUDA error (e.g. "cudaErrorLaunchOutOfResources") that made the
 * last kernel launch on this handle fail with GEMM_ERR_CUDA; "" if none did, or for
 * a NULL handle.  Static storage; never NULL. */
const char* gemm_last_cuda_error(gemm_handle_t h);

/*
 * gemm_run_noalloc -- the same product for callers that cannot allocate device
 * memory.  The pages have no counterpart of this call; it exists for users of
 * this library, not for the method.
 *
 * Who needs it: code that must not call cudaMalloc, such as a custom device
 * allocator or memory pool that wants a GEMM (cudaMalloc would recurse into it
 * or escape its budget), a plug-in whose framework owns every device
 * allocation, or a process that has reserved its device memory up front.
 * gemm_run needs a handle (gemm_create allocates) and grows a workspace on
 * demand; this call needs neither and allocates nothing, host or device.
 *
 * Scratch: a fixed static device array of GEMM_NOALLOC_SCRATCH_BYTES bytes in
 * the library, which every GPU that loads the library holds until the process
 * exits.  It carries a status word, split-K arrival counters and up to
 * GEMM_NOALLOC_WORKSPACE_BYTES of fp32 partial tiles.  The first call on a
 * device looks up the array's address on that device (cudaGetSymbolAddress),
 * so make that first call before any stream capture.  Every call shares the
 * array: each call clears the parts it relies on, on `stream`, and calls whose
 * work overlaps on the GPU race on it -- order them on one stream.
 *
 * Arguments, layouts and argument errors are those of gemm_run (no handle), except
 * that FP8 inputs are refused with GEMM_ERR_UNSUPPORTED.
 * The kernel is gemm_run's one-CTA split-K kernel with 256-column tiles; when
 * fewer tiles than half the SMs exist, K is sliced, into no more slices than
 * GEMM_NOALLOC_WORKSPACE_BYTES holds partial tiles for (an unsliced product needs
 * none), so every product gemm_run accepts with these dtypes runs.  The first
 * call on a device that fails its address lookup returns GEMM_ERR_CUDA and is
 * retried by the next call.  The call is
 * asynchronous; a kernel wait that runs out of time leaves C undefined and is
 * not reported (gemm_run with gemm_device_status reports it).
 */
#define GEMM_NOALLOC_WORKSPACE_BYTES (16u << 20)
#define GEMM_NOALLOC_SCRATCH_BYTES (256u + 65536u + GEMM_NOALLOC_WORKSPACE_BYTES)
gemm_status_t gemm_run_noalloc(const void* A, const void* B, void* C, int64_t M, int64_t N,
                               int64_t K, gemm_dtype_t dtype_in, gemm_dtype_t dtype_out,
                               gemm_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* GB300_GEMM_H */
