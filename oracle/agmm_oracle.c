/*
 * CPU oracle for the all-gather matmul.  TEST INFRASTRUCTURE ONLY.
 *
 * Only the test suite, the smoke check and the benchmark's CPU-baseline leg
 * may load this file's library.  The product path (the CUDA library and its
 * Python binding) never calls it and shares no code, header or table with it.
 *
 * What it computes (plain definition, written out with no blocking or fusion):
 *
 *   "Add all gather matmul benchmark" (pytorch/helion PR #400), the statement
 *   of the op:  (a, out) = ag_matmul(a_shared, b)  with  a = all_gather(a_shared)
 *   and  out = a @ b.  With D row shards of m_per_shard rows each, the gathered
 *   matrix is the row concatenation: row r*m_per_shard + i of `a` is row i of
 *   shard r.
 *
 *   "Fused all-gather+GEMM HBM-buffer kernel for iris.ops" (ROCm/iris #346),
 *   section "New kernel": an optional bias is added in the GEMM epilogue; the
 *   fused kernel only changes when tiles are computed, not what is computed.
 *
 *   Precision: 16-bit storage (bf16 or fp16) for a, b and out; products and
 *   sums in fp32, summed over k in increasing order; fp32 bias added after the
 *   sum; one round-to-nearest-even back to the storage type.
 *
 * The 16-bit <-> fp32 conversions are written here from the IEEE-754 binary16
 * and bfloat16 encodings; they use no library conversion routine.
 *
 * Extension (not on the pages): FP8 E4M3 inputs with per-tensor scales,
 * out = bf16(scale_a * scale_b * (a @ b) + bias), b given as [N, K]; the
 * E4M3 decoding is written from the OCP 8-bit floating-point definition.
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -pthread
 * (-ffp-contract=off keeps a*b+c as two roundings on every host, so results
 * do not depend on whether the compiler would emit FMA.)
 */
#define _GNU_SOURCE
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

enum { ORACLE_BF16 = 0, ORACLE_FP16 = 1 };

/* ---------------- bfloat16 (1 sign, 8 exponent, 7 mantissa bits) -------- */

static float bits_to_f32(uint32_t u) {
  float f;
  memcpy(&f, &u, sizeof f);
  return f;
}

static uint32_t f32_to_bits(float f) {
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return u;
}

/* bfloat16 is the upper half of an fp32 encoding: widening is exact. */
float oracle_bf16_to_f32(uint16_t h) { return bits_to_f32((uint32_t)h << 16); }

/* Round-to-nearest-even to bfloat16: keep the upper 16 bits and round on the
 * 16 dropped bits; a tie rounds to the even kept value.  A carry out of the
 * mantissa moves into the exponent, which turns the largest finite values
 * into infinity exactly as RNE overflow requires.  NaN stays a quiet NaN. */
uint16_t oracle_f32_to_bf16(float x) {
  uint32_t u = f32_to_bits(x);
  if ((u & 0x7f800000u) == 0x7f800000u && (u & 0x007fffffu) != 0)
    return (uint16_t)(((u >> 16) & 0x8000u) | 0x7fc0u);
  uint32_t kept = u >> 16;
  uint32_t dropped = u & 0xffffu;
  if (dropped > 0x8000u || (dropped == 0x8000u && (kept & 1u))) kept += 1u;
  return (uint16_t)kept;
}

/* ---------------- IEEE binary16 (1 sign, 5 exponent, 10 mantissa bits) -- */

float oracle_fp16_to_f32(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int m = h & 0x3ff;
  double v;
  if (e == 0x1f) {
    if (m != 0) return bits_to_f32(((uint32_t)sign << 31) | 0x7fc00000u | ((uint32_t)m << 13));
    v = INFINITY;
  } else if (e == 0) {
    v = ldexp((double)m, -24); /* subnormal: m * 2^-24 */
  } else {
    v = ldexp((double)(1024 + m), e - 25); /* (1 + m/1024) * 2^(e-15) */
  }
  return (float)(sign ? -v : v); /* every binary16 value is exact in fp32 */
}

/* Round-to-nearest-even to binary16.  The value is split into a power-of-two
 * quantum (2^-24 in the subnormal range, 2^(e-10) for a normal with exponent
 * e) and an integer count of quanta rounded half-to-even; all of this is
 * exact in double precision because x is an fp32 value. */
uint16_t oracle_f32_to_fp16(float x) {
  uint32_t u = f32_to_bits(x);
  uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
  if (isnan(x)) return (uint16_t)(sign | 0x7e00u | ((u >> 13) & 0x3ffu));
  double ax = fabs((double)x);
  if (ax == 0.0) return sign;
  /* 65504 is the largest finite binary16; halfway to the next power of two,
   * 65520, already rounds (to even) up to 2^16, which is out of range. */
  if (ax >= 65520.0) return (uint16_t)(sign | 0x7c00u);
  int e2;
  frexp(ax, &e2); /* ax = f * 2^e2, f in [0.5, 1): unbiased exponent is e2-1 */
  int e = e2 - 1;
  int quantum_exp = (e < -14) ? -24 : e - 10;
  double q = ldexp(ax, -quantum_exp); /* number of quanta, exact */
  double n = floor(q);
  double frac = q - n;
  if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
  if (e < -14) return (uint16_t)(sign | (uint16_t)n); /* n = 1024 is 2^-14 */
  if (n == 2048.0) { n = 1024.0; e += 1; }
  if (e + 15 >= 31) return (uint16_t)(sign | 0x7c00u);
  return (uint16_t)(sign | (uint16_t)((e + 15) << 10) | (uint16_t)((int)n - 1024));
}

static float to_f32(uint16_t h, int dtype) {
  return dtype == ORACLE_FP16 ? oracle_fp16_to_f32(h) : oracle_bf16_to_f32(h);
}

static uint16_t from_f32(float x, int dtype) {
  return dtype == ORACLE_FP16 ? oracle_f32_to_fp16(x) : oracle_f32_to_bf16(x);
}

/* Widen n 16-bit values (for callers that compare in fp32). */
void oracle_to_f32(const uint16_t* src, int64_t n, int dtype, float* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = to_f32(src[i], dtype);
}

/* Round n fp32 values to the 16-bit type. */
void oracle_from_f32(const float* src, int64_t n, int dtype, uint16_t* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = from_f32(src[i], dtype);
}

/* ---------------- the all-gather: row concatenation of the shards -------- */

/* a_gathered[r*m_per_shard + i][:] = shards[r][i][:], bit for bit. */
void oracle_all_gather(const uint16_t* const* shards, int D, int64_t m_per_shard, int64_t K,
                       uint16_t* a_gathered) {
  size_t shard_elems = (size_t)m_per_shard * (size_t)K;
  for (int r = 0; r < D; ++r)
    memcpy(a_gathered + (size_t)r * shard_elems, shards[r], shard_elems * sizeof(uint16_t));
}

/* ---------------- FP8 E4M3 (an extension the pages do not cover) ----------
 * The OCP 8-bit floating-point format E4M3: 1 sign bit, 4 exponent bits with
 * bias 7, 3 mantissa bits.  Exponent field 0 holds subnormals m * 2^-9;
 * otherwise the value is (1 + m/8) * 2^(e-7) = (8 + m) * 2^(e-10).  There are
 * no infinities; S.1111.111 is NaN, so the largest finite value is 448. */
float oracle_e4m3_to_f32(uint8_t v) {
  const int sign = v >> 7, e = (v >> 3) & 15, m = v & 7;
  if (e == 15 && m == 7) return sign ? -NAN : NAN;
  const float x = e == 0 ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
  return sign ? -x : x;
}

void oracle_e4m3_to_f32_array(const uint8_t* src, int64_t n, float* dst) {
  for (int64_t i = 0; i < n; ++i) dst[i] = oracle_e4m3_to_f32(src[i]);
}

/* Byte-wise all-gather (any element size): row concatenation of D shards of
 * row_bytes * m_per_shard bytes each. */
void oracle_all_gather_bytes(const uint8_t* const* shards, int D, int64_t m_per_shard,
                             int64_t row_bytes, uint8_t* a_gathered) {
  size_t shard_bytes = (size_t)m_per_shard * (size_t)row_bytes;
  for (int r = 0; r < D; ++r) memcpy(a_gathered + (size_t)r * shard_bytes, shards[r], shard_bytes);
}

/* ---------------- the GEMM: naive i-k-j loop, fp32 accumulate ------------ */

typedef struct {
  const uint16_t* a; /* [M, K] gathered, row-major */
  const float* b32;  /* [K, N] row-major, widened once */
  const float* bias; /* [N] or NULL */
  const int64_t* rows;
  int64_t nrows, K, N;
  int dtype;
  float* out_f32;     /* [nrows, N] or NULL */
  uint16_t* out;      /* [nrows, N] or NULL */
  float* abs_ab;      /* [nrows, N] or NULL: sum_k |a_ik| |b_kj| */
  int64_t first, last; /* this worker's slice of `rows` */
} gemm_job;

static void* gemm_worker(void* arg) {
  gemm_job* j = (gemm_job*)arg;
  const int64_t K = j->K, N = j->N;
  float* acc = (float*)malloc((size_t)N * sizeof(float));
  float* absacc = j->abs_ab ? (float*)malloc((size_t)N * sizeof(float)) : NULL;
  for (int64_t t = j->first; t < j->last; ++t) {
    const uint16_t* arow = j->a + (size_t)j->rows[t] * (size_t)K;
    for (int64_t n = 0; n < N; ++n) acc[n] = 0.0f;
    if (absacc)
      for (int64_t n = 0; n < N; ++n) absacc[n] = 0.0f;
    for (int64_t k = 0; k < K; ++k) { /* k increasing for every output */
      const float aik = to_f32(arow[k], j->dtype);
      const float* brow = j->b32 + (size_t)k * (size_t)N;
      for (int64_t n = 0; n < N; ++n) acc[n] = acc[n] + aik * brow[n];
      if (absacc) {
        const float aabs = fabsf(aik);
        for (int64_t n = 0; n < N; ++n) absacc[n] = absacc[n] + aabs * fabsf(brow[n]);
      }
    }
    for (int64_t n = 0; n < N; ++n) {
      float v = acc[n];
      if (j->bias) v = v + j->bias[n];
      if (j->out_f32) j->out_f32[(size_t)t * N + n] = v;
      if (j->out) j->out[(size_t)t * N + n] = from_f32(v, j->dtype);
      if (absacc) j->abs_ab[(size_t)t * N + n] = absacc[n];
    }
  }
  free(acc);
  free(absacc);
  return NULL;
}

/* out rows `rows[0..nrows)` of  a @ b (+ bias), a = [M, K] gathered.
 * Output row t of each result array is for gathered row rows[t].
 * nthreads <= 0 means one thread per online core.  Returns the thread count. */
int oracle_gemm_rows(const uint16_t* a, int64_t M, int64_t K, const uint16_t* b, int64_t N,
                     const float* bias, int dtype, const int64_t* rows, int64_t nrows,
                     float* out_f32, uint16_t* out, float* abs_ab, int nthreads) {
  (void)M;
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
  float* b32 = (float*)malloc((size_t)K * (size_t)N * sizeof(float));
  oracle_to_f32(b, K * N, dtype, b32);
  gemm_job* jobs = (gemm_job*)calloc((size_t)nthreads, sizeof(gemm_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  for (int t = 0; t < nthreads; ++t) {
    gemm_job* j = &jobs[t];
    j->a = a; j->b32 = b32; j->bias = bias; j->rows = rows; j->nrows = nrows;
    j->K = K; j->N = N; j->dtype = dtype;
    j->out_f32 = out_f32; j->out = out; j->abs_ab = abs_ab;
    j->first = nrows * t / nthreads;
    j->last = nrows * (t + 1) / nthreads;
    pthread_create(&tids[t], NULL, gemm_worker, j);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  free(b32);
  return nthreads;
}

/* ---------------- FP8 GEMM: E4M3 a [M, K] and b given as [N, K] ------------
 * out_f32[t, j] = (scale_a * scale_b) * sum_k f32(a[rows[t], k]) * f32(bt[j, k])
 *                 (+ bias[j]),  the sum in fp32 over k in increasing order, the
 * product of the two scales rounded to fp32 once, then bf16 by RNE.
 * abs_ab[t, j] = |scale_a * scale_b| * sum_k |a| |b|  (the tolerance scale). */
typedef struct {
  const uint8_t* a;
  const float* b32; /* [K, N], widened and transposed once */
  const float* bias;
  const int64_t* rows;
  int64_t K, N;
  float scale;
  float* out_f32;
  uint16_t* out;
  float* abs_ab;
  int64_t first, last;
} gemm8_job;

static void* gemm8_worker(void* arg) {
  gemm8_job* j = (gemm8_job*)arg;
  const int64_t K = j->K, N = j->N;
  float* acc = (float*)malloc((size_t)N * sizeof(float));
  float* absacc = j->abs_ab ? (float*)malloc((size_t)N * sizeof(float)) : NULL;
  for (int64_t t = j->first; t < j->last; ++t) {
    const uint8_t* arow = j->a + (size_t)j->rows[t] * (size_t)K;
    for (int64_t n = 0; n < N; ++n) acc[n] = 0.0f;
    if (absacc)
      for (int64_t n = 0; n < N; ++n) absacc[n] = 0.0f;
    for (int64_t k = 0; k < K; ++k) {
      const float aik = oracle_e4m3_to_f32(arow[k]);
      const float* brow = j->b32 + (size_t)k * (size_t)N;
      for (int64_t n = 0; n < N; ++n) acc[n] = acc[n] + aik * brow[n];
      if (absacc) {
        const float aabs = fabsf(aik);
        for (int64_t n = 0; n < N; ++n) absacc[n] = absacc[n] + aabs * fabsf(brow[n]);
      }
    }
    for (int64_t n = 0; n < N; ++n) {
      float v = acc[n] * j->scale;
      if (j->bias) v = v + j->bias[n];
      if (j->out_f32) j->out_f32[(size_t)t * N + n] = v;
      if (j->out) j->out[(size_t)t * N + n] = oracle_f32_to_bf16(v);
      if (absacc) j->abs_ab[(size_t)t * N + n] = absacc[n] * fabsf(j->scale);
    }
  }
  free(acc);
  free(absacc);
  return NULL;
}

int oracle_gemm_rows_fp8(const uint8_t* a, int64_t M, int64_t K, const uint8_t* bt, int64_t N,
                         float scale_a, float scale_b, const float* bias, const int64_t* rows,
                         int64_t nrows, float* out_f32, uint16_t* out, float* abs_ab,
                         int nthreads) {
  (void)M;
  if (nthreads <= 0) {
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    nthreads = c > 0 ? (int)c : 1;
  }
  if (nthreads > nrows) nthreads = nrows > 0 ? (int)nrows : 1;
  float* b32 = (float*)malloc((size_t)K * (size_t)N * sizeof(float));
  for (int64_t n = 0; n < N; ++n)
    for (int64_t k = 0; k < K; ++k)
      b32[(size_t)k * N + n] = oracle_e4m3_to_f32(bt[(size_t)n * K + k]);
  gemm8_job* jobs = (gemm8_job*)calloc((size_t)nthreads, sizeof(gemm8_job));
  pthread_t* tids = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  const float scale = scale_a * scale_b;
  for (int t = 0; t < nthreads; ++t) {
    gemm8_job* j = &jobs[t];
    j->a = a; j->b32 = b32; j->bias = bias; j->rows = rows;
    j->K = K; j->N = N; j->scale = scale;
    j->out_f32 = out_f32; j->out = out; j->abs_ab = abs_ab;
    j->first = nrows * t / nthreads;
    j->last = nrows * (t + 1) / nthreads;
    pthread_create(&tids[t], NULL, gemm8_worker, j);
  }
  for (int t = 0; t < nthreads; ++t) pthread_join(tids[t], NULL);
  free(tids);
  free(jobs);
  free(b32);
  return nthreads;
}
