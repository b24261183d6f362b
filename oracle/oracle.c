/*
 * CPU oracle for the dense GEMM  C = A . B^T  (TEST INFRASTRUCTURE ONLY).
 *
 * Only the test suite, the smoke check and the CPU-baseline leg of the
 * benchmark may load this library.  The CUDA path never calls it and shares
 * no code, header, table or constant with it.
 *
 * What it computes (the plain definition, nothing more):
 *   A is M x K, B is N x K, both row-major with K contiguous ("K-major"),
 *   stored as IEEE binary16 (fp16) or bfloat16 bit patterns.
 *       C[i][j] = round_out( sum_{k=0}^{K-1} double(A[i][k]) * double(B[j][k]) )
 *   - "A Blackwell GEMM by Hand in CuTe DSL", section 1 (C = A B^T, both
 *     operands K-major); "Speed-of-Light GEMM, Part 1", naive matmul listing
 *     (one dot product over k per output element).
 *   - The sum runs over k in increasing order and is accumulated in binary64.
 *     Every product of two fp16 or two bf16 values is exact in binary64
 *     (at most 11+11 significant bits), so only the additions round.
 *   - round_out rounds the binary64 sum directly to the output format with
 *     round-to-nearest, ties-to-even (no intermediate fp32 step), overflowing
 *     to +-inf as IEEE 754 prescribes.  The pages do not state the rounding
 *     mode of the fp32 -> fp16/bf16 output conversion; RNE is the reading
 *     taken here.
 *   - Subnormal inputs are decoded exactly.
 *   - K == 0 gives the empty sum, +0.
 *
 * Fused epilogue (oracle_gemm_epilogue): "CUTLASS Deep Dive: From CuTe Layouts
 * to Blackwell tcgen05", Part 6, Epilogue Visitor Trees (D = alpha * acc +
 * beta * C) and Classic Fused Epilogue: Bias + ReLU (d = max(0, alpha * acc +
 * bias)), taken together:
 *       D[i][j] = act( alpha * S[i][j] + beta * Cprev[i][j] + bias[j] )
 *   with S the sum above, Cprev the previous output (dtype_out bit patterns),
 *   bias one binary32 value per column, act the identity or ReLU (max(x, 0));
 *   alpha, beta and bias are taken exactly, the expression is evaluated in
 *   binary64 and rounded once to dtype_out.
 *
 * FP8 inputs ("CUTLASS Deep Dive: From CuTe Layouts to Blackwell tcgen05",
 * Part 6, FP8 and Blockwise Scaling: E4M3 input): A and B may instead hold
 * 8-bit E4M3 or E5M2 patterns, one byte per element.  The pages name E4M3 but do
 * not define it; the definitions taken are the OCP 8-bit floating point ones:
 *   E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits; no infinities;
 *         exponent 1111 is a normal binade except fraction 111, which is NaN
 *         (largest finite 448); exponent 0000 is subnormal, frac * 2^-9.
 *   E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits, IEEE-style
 *         (exponent 11111: infinity or NaN; largest finite 57344).
 * Products of two such values are exact in binary64, as above.
 *
 * Blockwise scaling (oracle_gemm_blockwise; same page and section: one scale
 * per (block_m, block_k) tile of A and one per (block_n, block_k) tile of B,
 * applied during accumulation):
 *       C[i][j] = round_out( sum_kb  sfa[i / bm][kb] * sfb[j / bn][kb] * P_kb[i][j] )
 *       P_kb[i][j] = sum_{k = kb*bk}^{min(K, (kb+1)*bk) - 1} A[i][k] * B[j][k]
 *   with sfa (ceil(M/bm) x ceil(K/bk)) and sfb (ceil(N/bn) x ceil(K/bk))
 *   row-major binary32 scales.  Each block's partial sum runs over k in
 *   increasing order in binary64; the scale product (exact in binary64) then
 *   multiplies it, and the blocks are summed in increasing kb.
 *
 * The format decoders and the rounding routine below are written from the
 * IEEE 754 / bfloat16 / OCP FP8 format definitions (sign, biased exponent,
 * fraction).
 *
 * Build: gcc -O2 -ffp-contract=off -fPIC -shared -pthread oracle.c -o liboracle.so
 * (-ffp-contract=off keeps "sum += a*b" as a multiply then an add on every
 * host architecture, so x86-64 and aarch64 produce identical results.)
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_F32 = 2, ORACLE_E4M3 = 3, ORACLE_E5M2 = 4 };

/* ---------------------------------------------------------------------- */
/* Format parameters: fraction bits, minimum normal exponent, maximum       */
/* exponent, exponent bias, total width.                                   */
/* ---------------------------------------------------------------------- */
typedef struct {
  int frac_bits;
  int emin;
  int emax;
  int bias;
  int exp_bits;
} fmt_t;

static const fmt_t FMT_F16 = {10, -14, 15, 15, 5};
static const fmt_t FMT_BF16 = {7, -126, 127, 127, 8};
static const fmt_t FMT_F32 = {23, -126, 127, 127, 8};
static const fmt_t FMT_E5M2 = {2, -14, 15, 15, 5};

static const fmt_t* fmt_of(int dtype) {
  switch (dtype) {
    case ORACLE_F16: return &FMT_F16;
    case ORACLE_BF16: return &FMT_BF16;
    case ORACLE_F32: return &FMT_F32;
    default: return NULL;
  }
}

/* Decode a 16- or 32-bit pattern of the given format into its exact value. */
static double decode_bits(uint32_t bits, const fmt_t* f) {
  const int width = 1 + f->exp_bits + f->frac_bits;
  const uint32_t sign = (bits >> (width - 1)) & 1u;
  const uint32_t e = (bits >> f->frac_bits) & ((1u << f->exp_bits) - 1u);
  const uint32_t frac = bits & ((1u << f->frac_bits) - 1u);
  double v;
  if (e == 0) {
    /* zero or subnormal: frac * 2^(emin - frac_bits) */
    v = ldexp((double)frac, f->emin - f->frac_bits);
  } else if (e == (1u << f->exp_bits) - 1u) {
    v = frac ? NAN : INFINITY;
  } else {
    /* normal: (2^frac_bits + frac) * 2^(e - bias - frac_bits) */
    v = ldexp((double)((1u << f->frac_bits) + frac), (int)e - f->bias - f->frac_bits);
  }
  return sign ? -v : v;
}

/* E4M3 (OCP): like an IEEE format of 4 exponent bits (bias 7) and 3 fraction
 * bits, except that the all-ones exponent holds normal numbers and only the
 * all-ones exponent with the all-ones fraction is NaN (there is no infinity). */
static double decode_e4m3(uint32_t bits) {
  const uint32_t sign = (bits >> 7) & 1u;
  const uint32_t e = (bits >> 3) & 15u;
  const uint32_t frac = bits & 7u;
  double v;
  if (e == 15u && frac == 7u) return NAN;
  if (e == 0) v = ldexp((double)frac, 1 - 7 - 3);  /* subnormal: frac * 2^-9 */
  else v = ldexp((double)(8u + frac), (int)e - 7 - 3);
  return sign ? -v : v;
}

/*
 * Round x to the nearest value of format f, ties to even, and return the bit
 * pattern.  Works on the magnitude: find the binade of |x| (clamped to the
 * subnormal binade), express |x| in units of that binade's spacing, round the
 * count to an integer (ties to even), then re-encode.
 */
static uint32_t round_to_bits(double x, const fmt_t* f) {
  const int width = 1 + f->exp_bits + f->frac_bits;
  const uint32_t sign = signbit(x) ? 1u : 0u;
  const uint32_t exp_all_ones = (1u << f->exp_bits) - 1u;
  const uint32_t inf_bits = (sign << (width - 1)) | (exp_all_ones << f->frac_bits);
  if (isnan(x)) return inf_bits | (1u << (f->frac_bits - 1)); /* quiet NaN */
  const double a = fabs(x);
  if (isinf(a)) return inf_bits;
  if (a == 0.0) return sign << (width - 1);

  int e2;
  (void)frexp(a, &e2);          /* a = m * 2^e2, m in [0.5, 1) */
  int e = e2 - 1;               /* exponent of the leading bit */
  if (e < f->emin) e = f->emin; /* subnormal binade shares emin's spacing */
  const int q = e - f->frac_bits;           /* spacing is 2^q */
  const double r = ldexp(a, -q);            /* exact: scaling by a power of two */
  double n = floor(r);
  const double rem = r - n;                 /* exact: r and n share the binade */
  if (rem > 0.5 || (rem == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;

  /* n * 2^q is the rounded magnitude; n may have carried to 2^(frac_bits+1). */
  double nn = n;
  int ee = e;
  if (nn >= ldexp(1.0, f->frac_bits + 1)) { nn /= 2.0; ee += 1; }
  if (ee > f->emax) return inf_bits;        /* rounded past the largest finite */
  uint32_t biased, frac;
  if (nn < ldexp(1.0, f->frac_bits)) {      /* subnormal (only when ee == emin) */
    biased = 0;
    frac = (uint32_t)nn;
  } else {
    biased = (uint32_t)(ee + f->bias);
    frac = (uint32_t)(nn - ldexp(1.0, f->frac_bits));
  }
  return (sign << (width - 1)) | (biased << f->frac_bits) | frac;
}

/* ---------------------------------------------------------------------- */
/* Decode tables (one per 16-bit input format), built once.                 */
/* ---------------------------------------------------------------------- */
static double g_lut[2][65536];
static double g_lut8[2][256];  /* [0]: E4M3, [1]: E5M2 */
static pthread_once_t g_lut_once = PTHREAD_ONCE_INIT;

static void build_luts(void) {
  for (uint32_t b = 0; b < 65536u; ++b) {
    g_lut[ORACLE_F16][b] = decode_bits(b, &FMT_F16);
    g_lut[ORACLE_BF16][b] = decode_bits(b, &FMT_BF16);
  }
  for (uint32_t b = 0; b < 256u; ++b) {
    g_lut8[0][b] = decode_e4m3(b);
    g_lut8[1][b] = decode_bits(b, &FMT_E5M2);
  }
}

static const double* lut_of(int dtype_in) {
  pthread_once(&g_lut_once, build_luts);
  if (dtype_in == ORACLE_E4M3) return g_lut8[0];
  if (dtype_in == ORACLE_E5M2) return g_lut8[1];
  return g_lut[dtype_in];
}

static int in_bytes_of(int dtype_in) {
  return dtype_in == ORACLE_E4M3 || dtype_in == ORACLE_E5M2 ? 1 : 2;
}

/* The sequential binary64 dot product of row i of A and row j of B over
 * k = k0 .. k1-1 (elements of in_bytes bytes, decoded through lut). */
static double dot_row(const void* a_row, const void* b_row, int64_t k0, int64_t k1,
                      int in_bytes, const double* lut) {
  double s = 0.0;
  if (in_bytes == 1) {
    const uint8_t* a8 = (const uint8_t*)a_row;
    const uint8_t* b8 = (const uint8_t*)b_row;
    for (int64_t k = k0; k < k1; ++k) s += lut[a8[k]] * lut[b8[k]];
  } else {
    const uint16_t* a16 = (const uint16_t*)a_row;
    const uint16_t* b16 = (const uint16_t*)b_row;
    for (int64_t k = k0; k < k1; ++k) s += lut[a16[k]] * lut[b16[k]];
  }
  return s;
}

static void store_out(void* C, int64_t idx, double v, int dtype_out) {
  const fmt_t* f = fmt_of(dtype_out);
  const uint32_t bits = round_to_bits(v, f);
  if (dtype_out == ORACLE_F32) ((uint32_t*)C)[idx] = bits;
  else ((uint16_t*)C)[idx] = (uint16_t)bits;
}

/* ---------------------------------------------------------------------- */
/* Threading: a job is a list of (i, j) output coordinates described by a   */
/* row list and a column list; workers take whole rows of that product.     */
/* ---------------------------------------------------------------------- */
typedef struct {
  const void* A;
  const void* B;
  void* C;            /* rounded output, or NULL */
  double* C64;        /* unrounded binary64 output, or NULL */
  int64_t K;
  const int64_t* rows; /* NULL means 0..nrows-1 */
  int64_t nrows;
  const int64_t* cols; /* NULL means 0..ncols-1 */
  int64_t ncols;
  int dtype_out;
  const double* lut;
  int64_t next_row;    /* shared work counter */
  pthread_mutex_t mu;
  /* fused epilogue (all zero: none) */
  int epi;
  double alpha, beta;
  const void* cprev;   /* M x N, dtype_out bit patterns, or NULL */
  int64_t ldc;         /* row length of cprev (N) */
  const float* bias;   /* N values, or NULL */
  int relu;
  int in_bytes;        /* 2: fp16/bf16 operands, 1: fp8 */
  /* blockwise scales (sfa NULL: none) */
  const float* sfa;    /* ceil(M/bm) x nkb */
  const float* sfb;    /* ceil(N/bn) x nkb */
  int64_t bm, bn, bk, nkb;
} job_t;

static void* worker(void* arg) {
  job_t* jb = (job_t*)arg;
  for (;;) {
    pthread_mutex_lock(&jb->mu);
    const int64_t r = jb->next_row++;
    pthread_mutex_unlock(&jb->mu);
    if (r >= jb->nrows) break;
    const int64_t i = jb->rows ? jb->rows[r] : r;
    const char* a_row = (const char*)jb->A + i * jb->K * jb->in_bytes;
    for (int64_t c = 0; c < jb->ncols; ++c) {
      const int64_t j = jb->cols ? jb->cols[c] : c;
      const char* b_row = (const char*)jb->B + j * jb->K * jb->in_bytes;
      double v;
      if (jb->sfa) {
        v = 0.0;
        for (int64_t kb = 0; kb < jb->nkb; ++kb) {
          const int64_t k0 = kb * jb->bk;
          const int64_t k1 = k0 + jb->bk < jb->K ? k0 + jb->bk : jb->K;
          const double scale = (double)jb->sfa[(i / jb->bm) * jb->nkb + kb] *
                               (double)jb->sfb[(j / jb->bn) * jb->nkb + kb];
          v += scale * dot_row(a_row, b_row, k0, k1, jb->in_bytes, jb->lut);
        }
      } else {
        v = dot_row(a_row, b_row, 0, jb->K, jb->in_bytes, jb->lut);
      }
      if (jb->epi) {
        v = jb->alpha * v;
        if (jb->cprev) {
          const fmt_t* f = fmt_of(jb->dtype_out);
          const int64_t idx = i * jb->ldc + j;
          const uint32_t bits = jb->dtype_out == ORACLE_F32
                                    ? ((const uint32_t*)jb->cprev)[idx]
                                    : ((const uint16_t*)jb->cprev)[idx];
          v += jb->beta * decode_bits(bits, f);
        }
        if (jb->bias) v += (double)jb->bias[j];
        if (jb->relu && !(v > 0.0)) v = 0.0;
      }
      const int64_t out = r * jb->ncols + c;
      if (jb->C64) jb->C64[out] = v;
      if (jb->C) store_out(jb->C, out, v, jb->dtype_out);
    }
  }
  return NULL;
}

static int run_job(job_t* jb, int nthreads) {
  if (nthreads <= 0) {
    long n = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = n > 0 ? (int)n : 1;
  }
  if (nthreads > 256) nthreads = 256;
  if (jb->nrows < nthreads) nthreads = jb->nrows > 0 ? (int)jb->nrows : 1;
  jb->next_row = 0;
  pthread_mutex_init(&jb->mu, NULL);
  pthread_t th[256];
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, worker, jb) != 0) break;
    ++started;
  }
  worker(jb);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  pthread_mutex_destroy(&jb->mu);
  return nthreads;
}

static int check_types(int dtype_in, int dtype_out) {
  if (dtype_in != ORACLE_F16 && dtype_in != ORACLE_BF16 && dtype_in != ORACLE_E4M3 &&
      dtype_in != ORACLE_E5M2)
    return -1;
  if (!fmt_of(dtype_out)) return -1;
  return 0;
}

/* ---------------------------------------------------------------------- */
/* Exported entry points.  Each returns the number of threads used, or -1   */
/* on an invalid argument.                                                  */
/* ---------------------------------------------------------------------- */

/* Full C (M x N, row-major), rounded to dtype_out. */
int oracle_gemm(const void* A, const void* B, void* C, int64_t M, int64_t N,
                int64_t K, int dtype_in, int dtype_out, int nthreads) {
  if (check_types(dtype_in, dtype_out) || M < 0 || N < 0 || K < 0) return -1;
  job_t jb = {A, B, C, NULL, K, NULL, M, NULL, N, dtype_out, lut_of(dtype_in), 0};
  jb.in_bytes = in_bytes_of(dtype_in);
  return run_job(&jb, nthreads);
}

/* Selected outputs: out[r][c] = C[rows[r]][cols[c]] (nrows x ncols,
 * row-major).  rows == NULL selects 0..nrows-1, cols == NULL 0..ncols-1.
 * Either C_out (rounded) or C64_out (unrounded binary64 sum) may be NULL. */
int oracle_gemm_select(const void* A, const void* B, void* C_out, double* C64_out,
                       int64_t K, const int64_t* rows, int64_t nrows,
                       const int64_t* cols, int64_t ncols, int dtype_in, int dtype_out,
                       int nthreads) {
  if (check_types(dtype_in, dtype_out) || K < 0 || nrows < 0 || ncols < 0) return -1;
  job_t jb = {A, B, C_out, C64_out, K, rows, nrows, cols, ncols, dtype_out,
              lut_of(dtype_in), 0};
  jb.in_bytes = in_bytes_of(dtype_in);
  return run_job(&jb, nthreads);
}

/* Full D (M x N) with the fused epilogue described at the top: cprev (M x N,
 * dtype_out patterns) may be NULL when beta is 0, bias (N floats) may be NULL,
 * relu is 0 or 1.  D may be the same buffer as cprev only if nthreads == 1. */
int oracle_gemm_epilogue(const void* A, const void* B, const void* cprev,
                         const float* bias, double alpha, double beta, int relu, void* D,
                         int64_t M, int64_t N, int64_t K, int dtype_in, int dtype_out,
                         int nthreads) {
  if (check_types(dtype_in, dtype_out) || M < 0 || N < 0 || K < 0) return -1;
  if (beta != 0.0 && !cprev) return -1;
  job_t jb = {A, B, D, NULL, K, NULL, M, NULL, N, dtype_out, lut_of(dtype_in), 0};
  jb.in_bytes = in_bytes_of(dtype_in);
  jb.epi = 1;
  jb.alpha = alpha;
  jb.beta = beta;
  jb.cprev = beta != 0.0 ? cprev : NULL;
  jb.ldc = N;
  jb.bias = bias;
  jb.relu = relu ? 1 : 0;
  return run_job(&jb, nthreads);
}

/* Selected outputs (as oracle_gemm_select) of the blockwise-scaled product
 * described at the top: sfa holds ceil(M/bm) x ceil(K/bk) and sfb
 * ceil(N/bn) x ceil(K/bk) binary32 scales, row-major; M is the row count of A. */
int oracle_gemm_blockwise(const void* A, const void* B, const float* sfa, const float* sfb,
                          int64_t bm, int64_t bn, int64_t bk, void* C_out, double* C64_out,
                          int64_t M, int64_t K, const int64_t* rows, int64_t nrows,
                          const int64_t* cols, int64_t ncols, int dtype_in, int dtype_out,
                          int nthreads) {
  if (check_types(dtype_in, dtype_out) || M < 0 || K < 0 || nrows < 0 || ncols < 0) return -1;
  if (!sfa || !sfb || bm <= 0 || bn <= 0 || bk <= 0) return -1;
  job_t jb = {A, B, C_out, C64_out, K, rows, nrows, cols, ncols, dtype_out,
              lut_of(dtype_in), 0};
  jb.in_bytes = in_bytes_of(dtype_in);
  jb.sfa = sfa;
  jb.sfb = sfb;
  jb.bm = bm;
  jb.bn = bn;
  jb.bk = bk;
  jb.nkb = (K + bk - 1) / bk;
  (void)M;
  return run_job(&jb, nthreads);
}

/* Exposed for the pins: decode n patterns of dtype to binary64. */
int oracle_decode(const void* bits, double* out, int64_t n, int dtype) {
  if (dtype == ORACLE_E4M3 || dtype == ORACLE_E5M2) {
    for (int64_t t = 0; t < n; ++t) out[t] = lut_of(dtype)[((const uint8_t*)bits)[t]];
    return 0;
  }
  const fmt_t* f = fmt_of(dtype);
  if (!f) return -1;
  for (int64_t t = 0; t < n; ++t) {
    uint32_t b = dtype == ORACLE_F32 ? ((const uint32_t*)bits)[t]
                                     : ((const uint16_t*)bits)[t];
    out[t] = decode_bits(b, f);
  }
  return 0;
}

/* Exposed for the pins: round n binary64 values to dtype (RNE). */
int oracle_round(const double* x, void* out, int64_t n, int dtype) {
  if (!fmt_of(dtype)) return -1;
  for (int64_t t = 0; t < n; ++t) store_out(out, t, x[t], dtype);
  return 0;
}
