/*
 * tl_oracle.c -- CPU oracle for C = epilogue(op(A) . op(B)).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file; only the tests, the smoke check and the benchmark's CPU-baseline leg
 * do.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes (the plain definition, written out):
 *
 *   C[i,j] = round_dtype( epi( sum_{k<K} x(opA[i,k]) * x(opB[k,j]) ) )
 *
 *   - opA[i,k] is A[i*lda+k], or A[k*lda+i] when trans_a; opB[k,j] is
 *     B[k*ldb+j], or B[j*ldb+k] when trans_b.  This is T.gemm's transpose_A /
 *     transpose_B reading: A is [M,K] (or [K,M]) and B is [K,N] (or [N,K])
 *     ("TileLang core primitives" page, section 3.3 "T.gemm").
 *   - x() decodes the exact value of an IEEE binary16 or bfloat16 bit pattern
 *     (decoders below, written from the two formats' definitions).
 *   - the sum runs over k = 0..K-1 in order, in IEEE binary64.  The pages fix the
 *     accumulator at fp32 and the cast "at the end" ("TileLang: from tile dataflow
 *     to controllable AI kernels", section "minimal but complete GEMM skeleton":
 *     fp16 inputs, fp32 accumulation, converted back to the output dtype last);
 *     the oracle accumulates in binary64, which is closer to the exact sum than
 *     any fp32 order, so the GPU/oracle difference is the GPU's own rounding.
 *   - epi is the identity, or ReLU = max(x, 0) applied to the accumulator before
 *     the cast ("TileLang core primitives" page, section 3.8, where the epilogue
 *     takes max(C, 0) on the fp32 accumulator tile; "NVIDIA backend codegen" page,
 *     section 1, the GEMM+ReLU quickstart).  Negative sums give +0.
 *   - round_dtype is round-to-nearest, ties-to-even, from binary64 straight to the
 *     output format (same format as the inputs), with overflow to +-inf and
 *     gradual underflow.
 *
 * Out-of-range elements of a partial tile do not exist here: the oracle sums over
 * exactly K terms, which is what zero padding of partial tiles must reproduce
 * ("TileLang core primitives" page, section 4.2: out-of-bounds source reads give
 * the safe value 0, out-of-bounds destination stores are skipped).
 *
 * Parallelism: OpenMP over output rows only; the summation order of each C[i,j]
 * is the same for every thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1, ORACLE_E4M3 = 2, ORACLE_E5M2 = 3 };

/* ---- format decoders ---------------------------------------------------- */

/* IEEE 754 binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 0x1F;
  const int f = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);                /* subnormal: f * 2^(1-15-10) */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 1024), e - 25);    /* (1024+f) * 2^(e-15-10) */
  }
  return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 7) & 0xFF;
  const int f = h & 0x7F;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -133);               /* f * 2^(1-127-7) */
  } else if (e == 255) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 128), e - 134);    /* (128+f) * 2^(e-127-7) */
  }
  return sign ? -v : v;
}

/* 8-bit E4M3 ("fn" variant: finite only): 1 sign, 4 exponent (bias 7), 3 fraction
 * bits; exponent 15 with fraction 7 is NaN, every other code is finite, so the
 * largest magnitude is 1.75 * 2^8 = 448.  Subnormals: f * 2^(1-7-3). */
double oracle_e4m3_to_f64(uint8_t h) {
  const int sign = (h >> 7) & 1;
  const int e = (h >> 3) & 0xF;
  const int f = h & 0x7;
  double v;
  if (e == 15 && f == 7) {
    v = NAN;
  } else if (e == 0) {
    v = ldexp((double)f, -9);
  } else {
    v = ldexp((double)(f + 8), e - 10);       /* (8+f) * 2^(e-7-3) */
  }
  return sign ? -v : v;
}

/* 8-bit E5M2: 1 sign, 5 exponent (bias 15), 2 fraction bits, IEEE-style: exponent
 * 31 is infinity (fraction 0) or NaN; largest finite 1.75 * 2^15 = 57344. */
double oracle_e5m2_to_f64(uint8_t h) {
  const int sign = (h >> 7) & 1;
  const int e = (h >> 2) & 0x1F;
  const int f = h & 0x3;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -16);                /* f * 2^(1-15-2) */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(f + 4), e - 17);       /* (4+f) * 2^(e-15-2) */
  }
  return sign ? -v : v;
}

/* ---- round to nearest even, binary64 -> 16-bit format -------------------- */

/*
 * Generic RNE encoder for a binary format with `mant` fraction bits and minimum
 * normal exponent `emin` (exponent bias = 1 - emin).  The value is scaled by
 * its quantum q = 2^(max(E, emin) - mant), where E = floor(log2|v|); |v|/q is
 * exact in binary64, and its integer rounding r (ties to even) is the
 * significand.  The encoding (E - emin + 1) << mant + r - 2^mant carries into
 * the exponent when r reaches 2^(mant+1), and equals r for subnormals.
 */
static uint16_t rne_encode(double v, int mant, int emin, uint32_t inf_bits,
                           uint16_t qnan) {
  if (isnan(v)) return qnan;
  const uint16_t sign = signbit(v) ? 0x8000 : 0;
  const double x = fabs(v);
  if (isinf(x)) return (uint16_t)(sign | inf_bits);
  if (x == 0.0) return sign;
  int e2;
  (void)frexp(x, &e2);          /* x = f * 2^e2, f in [0.5, 1) */
  int E = e2 - 1;               /* floor(log2 x) */
  if (E < emin) E = emin;       /* subnormal range shares the quantum of emin */
  if (E > 2000) E = 2000;       /* far past overflow; keeps the shifts small */
  const double q = ldexp(1.0, E - mant);
  const double n = x / q;       /* exact: division by a power of two */
  double r = floor(n);
  const double frac = n - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  const uint32_t hidden = 1u << mant;
  uint32_t bits;
  if (r < (double)hidden) {
    bits = (uint32_t)r;                                   /* subnormal or zero */
  } else {
    bits = ((uint32_t)(E - emin + 1) << mant) + (uint32_t)r - hidden;
  }
  if (bits >= inf_bits) bits = inf_bits;                  /* overflow -> inf */
  return (uint16_t)(sign | bits);
}

uint16_t oracle_f64_to_f16(double v) { return rne_encode(v, 10, -14, 0x7C00, 0x7E00); }
uint16_t oracle_f64_to_bf16(double v) { return rne_encode(v, 7, -126, 0x7F80, 0x7FC0); }

/* ---- the GEMM ----------------------------------------------------------- */

static double decode(uint16_t h, int dtype) {
  return dtype == ORACLE_BF16 ? oracle_bf16_to_f64(h) : oracle_f16_to_f64(h);
}

static uint16_t encode(double v, int dtype) {
  return dtype == ORACLE_BF16 ? oracle_f64_to_bf16(v) : oracle_f64_to_f16(v);
}

static double op_a(const uint16_t* A, int64_t lda, int trans_a, int64_t i, int64_t k,
                   int dtype) {
  return decode(trans_a ? A[k * lda + i] : A[i * lda + k], dtype);
}

static double op_b(const uint16_t* B, int64_t ldb, int trans_b, int64_t k, int64_t j,
                   int dtype) {
  return decode(trans_b ? B[j * ldb + k] : B[k * ldb + j], dtype);
}

/* The binary64 accumulator of one output element, k in order. */
static double dot(const uint16_t* A, const uint16_t* B, int64_t K, int64_t lda,
                  int64_t ldb, int dtype, int trans_a, int trans_b, int64_t i, int64_t j) {
  double s = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    s += op_a(A, lda, trans_a, i, k, dtype) * op_b(B, ldb, trans_b, k, j, dtype);
  }
  return s;
}

static double epilogue(double s, int relu) { return (relu && !(s > 0.0)) ? 0.0 : s; }

static void set_threads(int nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/*
 * Full product: C[i*ldc+j] for i<M, j<N, rounded to dtype.  If `sums` is not NULL
 * it receives the binary64 accumulators after the epilogue (row-major, M x N).
 * Returns 0, or -1 on an invalid argument.
 */
int oracle_gemm(const uint16_t* A, const uint16_t* B, uint16_t* C, double* sums,
                int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                int dtype, int trans_a, int trans_b, int relu, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
  if (M == 0 || N == 0) return 0;
  if (ldc < N) return -1;
  if (K > 0) {
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N)) return -1;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      const double s = epilogue(dot(A, B, K, lda, ldb, dtype, trans_a, trans_b, i, j), relu);
      if (C) C[i * ldc + j] = encode(s, dtype);
      if (sums) sums[i * N + j] = s;
    }
  }
  return 0;
}

/*
 * Selected entries only: out[t] = C[rows[t], cols[t]] (rounded), and, if
 * `sums` is not NULL, sums[t] = its binary64 accumulator after the epilogue.
 */
int oracle_gemm_entries(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
                        int64_t K, int64_t lda, int64_t ldb, int dtype, int trans_a,
                        int trans_b, int relu, const int64_t* rows, const int64_t* cols,
                        int64_t count, uint16_t* out, double* sums, int nthreads) {
  if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return -1;
  for (int64_t t = 0; t < count; ++t) {
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t t = 0; t < count; ++t) {
    const double s =
        epilogue(dot(A, B, K, lda, ldb, dtype, trans_a, trans_b, rows[t], cols[t]), relu);
    if (out) out[t] = encode(s, dtype);
    if (sums) sums[t] = s;
  }
  return 0;
}

/* ---- the FP8 GEMM ------------------------------------------------------------
 *
 *   C[i,j] = round_out( epi( alpha * sum_{k<K} x_a(opA[i,k]) * x_b(opB[k,j]) ) )
 *
 * A and B hold 8-bit codes of E4M3 or E5M2 (each operand its own format), decoded
 * exactly; the sum runs over k in order in binary64 and is multiplied by the
 * per-product scale alpha (binary64) before the epilogue and the cast to the
 * 16-bit output format.  This is the plain definition of a low-precision GEMM with
 * one scale for the whole product: the pages' block-scaled form shares one
 * exponent among 32 consecutive K elements ("NVIDIA backend codegen" page,
 * section 4.6.3; "TileLang: a tile language one level below Triton", block-scaled
 * MMA); with every block scale equal, it reduces to this.
 */
static double decode8(uint8_t h, int type) {
  return type == ORACLE_E5M2 ? oracle_e5m2_to_f64(h) : oracle_e4m3_to_f64(h);
}

static double dot8(const uint8_t* A, const uint8_t* B, int64_t K, int64_t lda, int64_t ldb,
                   int a_type, int b_type, int trans_a, int trans_b, int64_t i, int64_t j) {
  double s = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    const double a = decode8(trans_a ? A[k * lda + i] : A[i * lda + k], a_type);
    const double b = decode8(trans_b ? B[j * ldb + k] : B[k * ldb + j], b_type);
    s += a * b;
  }
  return s;
}

static int fp8_args_ok(int a_type, int b_type, int out_dtype) {
  return (a_type == ORACLE_E4M3 || a_type == ORACLE_E5M2) &&
         (b_type == ORACLE_E4M3 || b_type == ORACLE_E5M2) &&
         (out_dtype == ORACLE_F16 || out_dtype == ORACLE_BF16);
}

int oracle_gemm_fp8(const uint8_t* A, const uint8_t* B, uint16_t* C, double* sums,
                    int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb, int64_t ldc,
                    int a_type, int b_type, int out_dtype, int trans_a, int trans_b,
                    double alpha, int relu, int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (!fp8_args_ok(a_type, b_type, out_dtype)) return -1;
  if (M == 0 || N == 0) return 0;
  if (ldc < N) return -1;
  if (K > 0) {
    if (lda < (trans_a ? M : K) || ldb < (trans_b ? K : N)) return -1;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      const double s = epilogue(
          alpha * dot8(A, B, K, lda, ldb, a_type, b_type, trans_a, trans_b, i, j), relu);
      if (C) C[i * ldc + j] = encode(s, out_dtype);
      if (sums) sums[i * N + j] = s;
    }
  }
  return 0;
}

int oracle_gemm_fp8_entries(const uint8_t* A, const uint8_t* B, int64_t M, int64_t N, int64_t K,
                            int64_t lda, int64_t ldb, int a_type, int b_type, int out_dtype,
                            int trans_a, int trans_b, double alpha, int relu,
                            const int64_t* rows, const int64_t* cols, int64_t count,
                            uint16_t* out, double* sums, int nthreads) {
  if (!fp8_args_ok(a_type, b_type, out_dtype)) return -1;
  for (int64_t t = 0; t < count; ++t) {
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t t = 0; t < count; ++t) {
    const double s = epilogue(alpha * dot8(A, B, K, lda, ldb, a_type, b_type, trans_a, trans_b,
                                           rows[t], cols[t]),
                              relu);
    if (out) out[t] = encode(s, out_dtype);
    if (sums) sums[t] = s;
  }
  return 0;
}

void oracle_decode8_array(const uint8_t* in, double* out, int64_t n, int type) {
  for (int64_t t = 0; t < n; ++t) out[t] = decode8(in[t], type);
}

/* ---- the block-scaled (MX) FP8 GEMM ------------------------------------------
 *
 * The pages' block-scaled form: 8-bit operands in which every 32 consecutive K
 * elements of a row share one power-of-two scale, E8M0 codes SFA (per row of A)
 * and SFB (per column of the product, i.e. per row of the K-major B) ("NVIDIA
 * backend codegen" page, section 4.6.3; "TileLang: a tile language one level
 * below Triton", block-scaled MMA).  Written out:
 *
 *   C[i,j] = round_out( epi( sum_{k<K} x_a(A[i,k]) 2^(SFA[i][k/32] - 127)
 *                                      * x_b(B[j,k]) 2^(SFB[j][k/32] - 127) ) )
 *
 * A is [M,K] and B is [N,K], both K-major (the layout of the MX formats, whose
 * blocks run along K); SFA is [M][sfa_ld] and SFB is [N][sfb_ld] bytes, block b of
 * row r at r*ld + b.  An E8M0 code e is the value 2^(e - 127) for e < 255; e = 255 is
 * NaN.  K must be a multiple of the block size 32.  The sum runs over k in order in
 * binary64 (every scaled product is exact there).
 */
static double e8m0(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

static double dot_mx(const uint8_t* A, const uint8_t* B, const uint8_t* SA, const uint8_t* SB,
                     int64_t K, int64_t lda, int64_t ldb, int64_t sfa_ld, int64_t sfb_ld,
                     int a_type, int b_type, int64_t i, int64_t j) {
  double s = 0.0;
  for (int64_t k = 0; k < K; ++k) {
    const double a = decode8(A[i * lda + k], a_type) * e8m0(SA[i * sfa_ld + k / 32]);
    const double b = decode8(B[j * ldb + k], b_type) * e8m0(SB[j * sfb_ld + k / 32]);
    s += a * b;
  }
  return s;
}

static int mx_args_ok(int64_t M, int64_t N, int64_t K, int64_t lda, int64_t ldb,
                      int64_t sfa_ld, int64_t sfb_ld, int a_type, int b_type, int out_dtype) {
  if (M < 0 || N < 0 || K < 0 || K % 32 != 0) return 0;
  if (!fp8_args_ok(a_type, b_type, out_dtype)) return 0;
  if (K > 0 && (lda < K || ldb < K || sfa_ld < K / 32 || sfb_ld < K / 32)) return 0;
  return 1;
}

int oracle_gemm_mx(const uint8_t* A, const uint8_t* B, const uint8_t* SA, const uint8_t* SB,
                   uint16_t* C, double* sums, int64_t M, int64_t N, int64_t K, int64_t lda,
                   int64_t ldb, int64_t ldc, int64_t sfa_ld, int64_t sfb_ld, int a_type,
                   int b_type, int out_dtype, int relu, int nthreads) {
  if (!mx_args_ok(M, N, K, lda, ldb, sfa_ld, sfb_ld, a_type, b_type, out_dtype)) return -1;
  if (M == 0 || N == 0) return 0;
  if (ldc < N) return -1;
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    for (int64_t j = 0; j < N; ++j) {
      const double s =
          epilogue(dot_mx(A, B, SA, SB, K, lda, ldb, sfa_ld, sfb_ld, a_type, b_type, i, j), relu);
      if (C) C[i * ldc + j] = encode(s, out_dtype);
      if (sums) sums[i * N + j] = s;
    }
  }
  return 0;
}

int oracle_gemm_mx_entries(const uint8_t* A, const uint8_t* B, const uint8_t* SA,
                           const uint8_t* SB, int64_t M, int64_t N, int64_t K, int64_t lda,
                           int64_t ldb, int64_t sfa_ld, int64_t sfb_ld, int a_type, int b_type,
                           int out_dtype, int relu, const int64_t* rows, const int64_t* cols,
                           int64_t count, uint16_t* out, double* sums, int nthreads) {
  if (!mx_args_ok(M, N, K, lda, ldb, sfa_ld, sfb_ld, a_type, b_type, out_dtype)) return -1;
  for (int64_t t = 0; t < count; ++t) {
    if (rows[t] < 0 || rows[t] >= M || cols[t] < 0 || cols[t] >= N) return -1;
  }
  set_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 16)
  for (int64_t t = 0; t < count; ++t) {
    const double s = epilogue(dot_mx(A, B, SA, SB, K, lda, ldb, sfa_ld, sfb_ld, a_type, b_type,
                                     rows[t], cols[t]),
                              relu);
    if (out) out[t] = encode(s, out_dtype);
    if (sums) sums[t] = s;
  }
  return 0;
}

/* ---- attention ---------------------------------------------------------------
 *
 * The pages' second workload on the same primitives is the FlashAttention forward
 * pass ("TileLang: a tile language one level below Triton", section "FlashAttention:
 * online softmax as tile code"): Q, K, V and O are [B, S, H, D] (batch, sequence,
 * heads, head dim), scores are scaled by 1/sqrt(D), and the causal form lets query
 * i see keys j <= i.  The oracle writes out the plain definition, not the online
 * (blockwise, rescaled) form:
 *
 *   s_ij = (1/sqrt(D)) * sum_d Q[b,i,h,d] * K[b,j,h,d]        (j < S, and j <= i if causal)
 *   O[b,i,h,:] = sum_j exp(s_ij - max_j s_ij) V[b,j,h,:] / sum_j exp(s_ij - max_j s_ij)
 *
 * in binary64 with libm's exp, rounded once to the 16-bit output format.  The
 * subtraction of the row maximum changes nothing mathematically (softmax is
 * shift-invariant); it keeps exp in range.
 */
static void attention_row(const uint16_t* Q, const uint16_t* K, const uint16_t* V,
                          int64_t S, int64_t H, int64_t D, int dtype, int causal, int64_t b,
                          int64_t h, int64_t i, double* scores, double* out) {
  const double scale = 1.0 / sqrt((double)D);
  const int64_t row = H * D;                      /* elements between sequence positions */
  const uint16_t* q = Q + (b * S + i) * row + h * D;
  const int64_t n = causal ? i + 1 : S;
  double mx = -INFINITY;
  for (int64_t j = 0; j < n; ++j) {
    const uint16_t* k = K + (b * S + j) * row + h * D;
    double acc = 0.0;
    for (int64_t d = 0; d < D; ++d) acc += decode(q[d], dtype) * decode(k[d], dtype);
    scores[j] = acc * scale;
    if (scores[j] > mx) mx = scores[j];
  }
  double den = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    scores[j] = exp(scores[j] - mx);
    den += scores[j];
  }
  for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
  for (int64_t j = 0; j < n; ++j) {
    const uint16_t* v = V + (b * S + j) * row + h * D;
    for (int64_t d = 0; d < D; ++d) out[d] += scores[j] * decode(v[d], dtype);
  }
  for (int64_t d = 0; d < D; ++d) out[d] /= den;
}

static int attention_args_ok(int64_t B, int64_t S, int64_t H, int64_t D, int dtype) {
  return B >= 0 && S >= 0 && H >= 0 && D > 0 && (dtype == ORACLE_F16 || dtype == ORACLE_BF16);
}

/* All of O; `sums` (if not NULL) receives the binary64 outputs before rounding. */
int oracle_attention(const uint16_t* Q, const uint16_t* K, const uint16_t* V, uint16_t* O,
                     double* sums, int64_t B, int64_t S, int64_t H, int64_t D, int dtype,
                     int causal, int nthreads) {
  if (!attention_args_ok(B, S, H, D, dtype)) return -1;
  set_threads(nthreads);
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double* out = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for collapse(2) schedule(dynamic, 1)
    for (int64_t b = 0; b < B; ++b) {
      for (int64_t h = 0; h < H; ++h) {
        for (int64_t i = 0; i < S; ++i) {
          attention_row(Q, K, V, S, H, D, dtype, causal, b, h, i, scores, out);
          const int64_t base = ((b * S + i) * H + h) * D;
          for (int64_t d = 0; d < D; ++d) {
            if (O) O[base + d] = encode(out[d], dtype);
            if (sums) sums[base + d] = out[d];
          }
        }
      }
    }
    free(scores);
    free(out);
  }
  return 0;
}

/* Selected rows (b[t], i[t], h[t]) only: out[t*D + d], rounded. */
int oracle_attention_rows(const uint16_t* Q, const uint16_t* K, const uint16_t* V, int64_t B,
                          int64_t S, int64_t H, int64_t D, int dtype, int causal,
                          const int64_t* bs, const int64_t* is, const int64_t* hs, int64_t count,
                          uint16_t* out, int nthreads) {
  if (!attention_args_ok(B, S, H, D, dtype)) return -1;
  for (int64_t t = 0; t < count; ++t) {
    if (bs[t] < 0 || bs[t] >= B || is[t] < 0 || is[t] >= S || hs[t] < 0 || hs[t] >= H) return -1;
  }
  set_threads(nthreads);
#pragma omp parallel
  {
    double* scores = (double*)malloc(sizeof(double) * (size_t)(S > 0 ? S : 1));
    double* row = (double*)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 4)
    for (int64_t t = 0; t < count; ++t) {
      attention_row(Q, K, V, S, H, D, dtype, causal, bs[t], hs[t], is[t], scores, row);
      for (int64_t d = 0; d < D; ++d) out[t * D + d] = encode(row[d], dtype);
    }
    free(scores);
    free(row);
  }
  return 0;
}

/* Vector forms of the format conversions, for the pin tests. */
void oracle_decode_array(const uint16_t* in, double* out, int64_t n, int dtype) {
  for (int64_t t = 0; t < n; ++t) out[t] = decode(in[t], dtype);
}

void oracle_encode_array(const double* in, uint16_t* out, int64_t n, int dtype) {
  for (int64_t t = 0; t < n; ++t) out[t] = encode(in[t], dtype);
}
