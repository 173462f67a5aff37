/*
 * Oracle for the tiled dense GEMM -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the CPU-baseline leg of the benchmark use
 * this file.  The CUDA library never links it, includes it or calls it, and it
 * shares no code with the library.
 *
 * What the tiled kernels compute is, up to the order of the floating-point
 * additions, the plain product
 *
 *     C[i][j] = sum_{k<K} A[i][k] * B[k][j]
 *
 * ("CUDA tile", section 2.1, the definition C[i][j] = sum_k A[i][k]*B[k][j];
 * "矩阵乘法中的平铺" (qian.cx), whose traffic model shows that splitting K into
 * l-length stages leaves the total unchanged).  Tiling, staging and K-splitting
 * only regroup that sum, so the oracle is the definition written out: a triple
 * loop in double precision over the exact values stored in A and B.
 *
 *  - Inputs are the raw storage bits the GPU receives (fp32, fp16 or bf16);
 *    the oracle decodes them itself (IEEE binary32 / binary16, and bfloat16 =
 *    the upper half of a binary32).
 *  - Every product of two such values is exact in double (at most 24+24
 *    significant bits), so the only rounding is in the K-term sum; its error
 *    is below K * 2^-53 * S, with S[i][j] = sum_k |A[i][k] * B[k][j]|, which
 *    the oracle returns beside C for the tolerance of the parity tests.
 *  - The loop runs i, k, j: for each output element the terms are added in
 *    increasing k, as in the i, j, k order of the definition.
 *  - Rows are independent; the multi-threaded entry point splits rows only,
 *    so every element's arithmetic, and hence its value, is the same for any
 *    thread count.
 *
 * Storage format codes: 0 = fp32, 1 = fp16, 2 = bf16.
 * Leading dimensions are in elements, row-major.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORACLE_F32 = 0, ORACLE_F16 = 1, ORACLE_BF16 = 2 };

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1F;
  int f = h & 0x3FF;
  double v;
  if (e == 0) {
    v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
  } else if (e == 31) {
    v = f ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

/* bfloat16: the sign, exponent and top 7 fraction bits of a binary32. */
static double decode_bf16(uint16_t h) {
  uint32_t u = (uint32_t)h << 16;
  float x;
  memcpy(&x, &u, sizeof x);
  return (double)x;
}

static double decode_f32(uint32_t u) {
  float x;
  memcpy(&x, &u, sizeof x);
  return (double)x;
}

static double load_elem(const void* base, int fmt, int64_t idx) {
  switch (fmt) {
    case ORACLE_F32: return decode_f32(((const uint32_t*)base)[idx]);
    case ORACLE_F16: return decode_f16(((const uint16_t*)base)[idx]);
    default:         return decode_bf16(((const uint16_t*)base)[idx]);
  }
}

/* Decode a rows x cols block of storage bits into a dense double array. */
void oracle_decode(const void* src, int fmt, int64_t rows, int64_t cols, int64_t ld, double* dst) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c)
      dst[r * cols + c] = load_elem(src, fmt, r * ld + c);
}

/*
 * The definition on rows [row_begin, row_end): C (and S when non-null) are
 * dense double arrays with leading dimension N.  A and B hold storage bits.
 */
void oracle_gemm_rows(int64_t M, int64_t N, int64_t K,
                      const void* A, int64_t lda, const void* B, int64_t ldb, int fmt,
                      double* C, double* S, int64_t row_begin, int64_t row_end) {
  (void)M;
  for (int64_t i = row_begin; i < row_end; ++i) {
    double* c = C + i * N;
    double* s = S ? S + i * N : NULL;
    for (int64_t j = 0; j < N; ++j) {
      c[j] = 0.0;
      if (s) s[j] = 0.0;
    }
    for (int64_t k = 0; k < K; ++k) {
      double a = load_elem(A, fmt, i * lda + k);
      for (int64_t j = 0; j < N; ++j) {
        double p = a * load_elem(B, fmt, k * ldb + j);
        c[j] += p;
        if (s) s[j] += fabs(p);
      }
    }
  }
}

typedef struct {
  int64_t M, N, K, lda, ldb;
  const void* A;
  const void* B;
  int fmt;
  double* C;
  double* S;
  int64_t r0, r1;
} rows_job;

static void* rows_worker(void* p) {
  rows_job* j = (rows_job*)p;
  oracle_gemm_rows(j->M, j->N, j->K, j->A, j->lda, j->B, j->ldb, j->fmt, j->C, j->S, j->r0, j->r1);
  return NULL;
}

/* Full product on `threads` host threads (rows split into contiguous bands). */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const void* A, int64_t lda, const void* B, int64_t ldb, int fmt,
                double* C, double* S, int threads) {
  if (M < 0 || N < 0 || K < 0) return 1;
  if (threads < 1) threads = 1;
  if (threads > M) threads = M > 0 ? (int)M : 1;
  if (threads == 1) {
    oracle_gemm_rows(M, N, K, A, lda, B, ldb, fmt, C, S, 0, M);
    return 0;
  }
  pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * threads);
  rows_job* jobs = (rows_job*)malloc(sizeof(rows_job) * threads);
  if (!tid || !jobs) { free(tid); free(jobs); return 2; }
  for (int t = 0; t < threads; ++t) {
    rows_job j = {M, N, K, lda, ldb, A, B, fmt, C, S, M * t / threads, M * (t + 1) / threads};
    jobs[t] = j;
    pthread_create(&tid[t], NULL, rows_worker, &jobs[t]);
  }
  for (int t = 0; t < threads; ++t) pthread_join(tid[t], NULL);
  free(tid);
  free(jobs);
  return 0;
}

/* Single entries (i, j) of the product, for spot checks at sizes where the full
 * product is too slow.  out_c / out_s receive n values. */
void oracle_gemm_entries(int64_t K, const void* A, int64_t lda, const void* B, int64_t ldb, int fmt,
                         int64_t n, const int64_t* rows, const int64_t* cols,
                         double* out_c, double* out_s) {
  for (int64_t t = 0; t < n; ++t) {
    double c = 0.0, s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      double p = load_elem(A, fmt, rows[t] * lda + k) * load_elem(B, fmt, k * ldb + cols[t]);
      c += p;
      s += fabs(p);
    }
    out_c[t] = c;
    if (out_s) out_s[t] = s;
  }
}

/*
 * Cache-blocked variant of the same product, timed beside the plain oracle as
 * a CPU baseline.  Operands are first decoded into dense double panels; the
 * k loop is split into blocks of KB (the l-length stages of the qian.cx
 * traffic model) and rows/columns into IB x JB output blocks, so a B panel of
 * KB x JB doubles stays in cache while IB rows reuse it.  Results agree with
 * oracle_gemm to within K * 2^-53 * S (same terms, same k order per element:
 * the k blocks are visited in increasing order).
 */
typedef struct {
  int64_t M, N, K;
  const double* Ad;
  const double* Bd;
  double* C;
  int64_t r0, r1;
} blk_job;

enum { IB = 32, JB = 256, KB = 128 };

static void* blocked_worker(void* p) {
  blk_job* j = (blk_job*)p;
  const int64_t N = j->N, K = j->K;
  for (int64_t i = j->r0; i < j->r1; ++i)
    for (int64_t c = 0; c < N; ++c) j->C[i * N + c] = 0.0;
  for (int64_t i0 = j->r0; i0 < j->r1; i0 += IB) {
    int64_t i1 = i0 + IB < j->r1 ? i0 + IB : j->r1;
    for (int64_t j0 = 0; j0 < N; j0 += JB) {
      int64_t j1 = j0 + JB < N ? j0 + JB : N;
      for (int64_t k0 = 0; k0 < K; k0 += KB) {
        int64_t k1 = k0 + KB < K ? k0 + KB : K;
        for (int64_t i = i0; i < i1; ++i) {
          double* crow = j->C + i * N;
          for (int64_t k = k0; k < k1; ++k) {
            double a = j->Ad[i * K + k];
            const double* brow = j->Bd + k * N;
            for (int64_t c = j0; c < j1; ++c) crow[c] += a * brow[c];
          }
        }
      }
    }
  }
  return NULL;
}

int oracle_gemm_blocked(int64_t M, int64_t N, int64_t K,
                        const void* A, int64_t lda, const void* B, int64_t ldb, int fmt,
                        double* C, int threads) {
  if (M < 0 || N < 0 || K < 0) return 1;
  double* Ad = (double*)malloc(sizeof(double) * (size_t)(M * K + 1));
  double* Bd = (double*)malloc(sizeof(double) * (size_t)(K * N + 1));
  if (!Ad || !Bd) { free(Ad); free(Bd); return 2; }
  oracle_decode(A, fmt, M, K, lda, Ad);
  oracle_decode(B, fmt, K, N, ldb, Bd);
  if (threads < 1) threads = 1;
  if (threads > M) threads = M > 0 ? (int)M : 1;
  pthread_t* tid = (pthread_t*)malloc(sizeof(pthread_t) * threads);
  blk_job* jobs = (blk_job*)malloc(sizeof(blk_job) * threads);
  if (!tid || !jobs) { free(Ad); free(Bd); free(tid); free(jobs); return 2; }
  for (int t = 0; t < threads; ++t) {
    blk_job j = {M, N, K, Ad, Bd, C, M * t / threads, M * (t + 1) / threads};
    jobs[t] = j;
    pthread_create(&tid[t], NULL, blocked_worker, &jobs[t]);
  }
  for (int t = 0; t < threads; ++t) pthread_join(tid[t], NULL);
  free(tid);
  free(jobs);
  free(Ad);
  free(Bd);
  return 0;
}
