/*
 * CPU oracle for the dense product  C = A·B (+ bias).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file; only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header or constant with the
 * CUDA library.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *
 *     C[i][j] = ( sum_{k=0}^{K-1} A[i][k] * B[k][j] ) + (bias ? bias[j] : 0)
 *
 * in IEEE binary64 from the exact values of the fp16 / fp32 inputs.
 *   - "Output = Input * Weight + Bias" is the operation the FuseReductionEpilogue
 *     series sets out to fuse (kimm240.github.io/tvm, "[TIR][Schedule] Add
 *     FuseReductionEpilogue primitive ... 1. Problem Analysis").  Starting the
 *     reduction from the bias (part 2 of that series) and adding the bias after
 *     the sum are the same number in exact arithmetic; the oracle adds it last.
 *   - fp16 multiply with a wider accumulator is the tensor-core operation
 *     described on je-d.tistory.com "tvm" (Tensor Core: mixed-precision
 *     multiply and accumulate); the oracle's accumulator is binary64.
 *
 * Sum order: for every output element the k terms are added in ascending k,
 * one multiply and one add each (built with -ffp-contract=off, no fast-math),
 * so the result is reproducible bit for bit on any host.
 *
 * Storage conventions (matching the library's C-ABI):
 *   A is M x K.  a_major = 0: row-major, element (i,k) at i*K + k.
 *                a_major = 1: column-major, element (i,k) at k*M + i.
 *   B is K x N.  b_major = 0: row-major, element (k,j) at k*N + j.
 *                b_major = 1: column-major, element (k,j) at j*K + k.
 *   dtype 0 = IEEE binary16, 1 = IEEE binary32.
 *   bias: NULL or N binary32 values.
 *   C: binary64, row-major, one row of N values per requested row.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_ENOMEM (-3)

/* binary16 -> binary64 by its definition: sign, 5-bit biased exponent
 * (bias 15), 10-bit fraction; exponent 0 = subnormal (no implicit 1,
 * scale 2^-14), exponent 31 = Inf (fraction 0) or NaN. */
double oracle_f16_to_f64(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int expo = (h >> 10) & 0x1f;
  const int frac = h & 0x3ff;
  double v;
  if (expo == 0) {
    v = ldexp((double)frac, -24);           /* frac * 2^-10 * 2^-14 */
  } else if (expo == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), expo - 25); /* (1 + frac/1024) * 2^(e-15) */
  }
  return sign ? -v : v;
}

static double load_elem(const void *base, int dtype, int64_t idx) {
  if (dtype == 0) return oracle_f16_to_f64(((const uint16_t *)base)[idx]);
  return (double)((const float *)base)[idx];
}

static int64_t a_index(int64_t i, int64_t k, int64_t M, int64_t K, int major) {
  return major == 0 ? i * K + k : k * M + i;
}

static int64_t b_index(int64_t k, int64_t j, int64_t K, int64_t N, int major) {
  return major == 0 ? k * N + j : j * K + k;
}

typedef struct {
  int64_t M, N, K;
  const void *A;
  int a_dtype, a_major;
  const double *B64; /* B decoded to binary64, logical K x N, row-major */
  const float *bias;
  const int64_t *rows; /* NULL: all rows 0..M-1 */
  int64_t row_begin, row_end; /* positions in the row list for this worker */
  double *C;
} oracle_job;

/* One worker: for each of its output rows, accumulate over k ascending. */
static void *oracle_worker(void *arg) {
  const oracle_job *jb = (const oracle_job *)arg;
  const int64_t N = jb->N, K = jb->K;
  for (int64_t r = jb->row_begin; r < jb->row_end; ++r) {
    const int64_t i = jb->rows ? jb->rows[r] : r;
    double *acc = jb->C + r * N;
    for (int64_t j = 0; j < N; ++j) acc[j] = 0.0;
    for (int64_t k = 0; k < K; ++k) {
      const double a = load_elem(jb->A, jb->a_dtype,
                                 a_index(i, k, jb->M, K, jb->a_major));
      const double *brow = jb->B64 + k * N;
      for (int64_t j = 0; j < N; ++j) acc[j] += a * brow[j];
    }
    if (jb->bias)
      for (int64_t j = 0; j < N; ++j) acc[j] += (double)jb->bias[j];
  }
  return NULL;
}

/*
 * Computes the requested rows of C.
 *   rows == NULL, nrows == M : the whole product.
 *   otherwise rows[0..nrows) lists row indices in [0, M); output row r of C
 *   holds product row rows[r].
 * threads <= 0 means 1.  Returns 0, or a negative code on bad arguments or
 * allocation failure.
 */
int oracle_gemm_rows(int64_t M, int64_t N, int64_t K, const void *A, int a_dtype,
                     int a_major, const void *B, int b_dtype, int b_major,
                     const float *bias, const int64_t *rows, int64_t nrows,
                     double *C, int threads) {
  if (M < 0 || N < 0 || K < 0 || nrows < 0) return ORACLE_EINVAL;
  if ((a_dtype != 0 && a_dtype != 1) || (b_dtype != 0 && b_dtype != 1))
    return ORACLE_EINVAL;
  if ((a_major != 0 && a_major != 1) || (b_major != 0 && b_major != 1))
    return ORACLE_EINVAL;
  if (rows == NULL && nrows != M) return ORACLE_EINVAL;
  if (nrows == 0 || N == 0) return ORACLE_OK;
  if (!C || (K > 0 && (!A || !B))) return ORACLE_EINVAL;
  if (rows)
    for (int64_t r = 0; r < nrows; ++r)
      if (rows[r] < 0 || rows[r] >= M) return ORACLE_EINVAL;

  /* Read B once into binary64 in its logical K x N order. */
  double *B64 = NULL;
  if (K > 0) {
    B64 = (double *)malloc((size_t)K * (size_t)N * sizeof(double));
    if (!B64) return ORACLE_ENOMEM;
    for (int64_t k = 0; k < K; ++k)
      for (int64_t j = 0; j < N; ++j)
        B64[k * N + j] = load_elem(B, b_dtype, b_index(k, j, K, N, b_major));
  }

  if (threads <= 0) threads = 1;
  if ((int64_t)threads > nrows) threads = (int)nrows;
  oracle_job *jobs = (oracle_job *)calloc((size_t)threads, sizeof(oracle_job));
  pthread_t *tids = (pthread_t *)calloc((size_t)threads, sizeof(pthread_t));
  char *spawned = (char *)calloc((size_t)threads, 1);
  if (!jobs || !tids || !spawned) {
    free(jobs); free(tids); free(spawned); free(B64);
    return ORACLE_ENOMEM;
  }
  /* Contiguous row slices; slice t-1 runs on the calling thread, and a slice
   * whose thread could not be started also runs here. */
  for (int t = 0; t < threads; ++t) {
    oracle_job *jb = &jobs[t];
    jb->M = M; jb->N = N; jb->K = K;
    jb->A = A; jb->a_dtype = a_dtype; jb->a_major = a_major;
    jb->B64 = B64; jb->bias = bias; jb->rows = rows; jb->C = C;
    jb->row_begin = nrows * t / threads;
    jb->row_end = nrows * (t + 1) / threads;
    if (t < threads - 1 && pthread_create(&tids[t], NULL, oracle_worker, jb) == 0)
      spawned[t] = 1;
    else
      oracle_worker(jb);
  }
  for (int t = 0; t < threads; ++t)
    if (spawned[t]) pthread_join(tids[t], NULL);
  free(jobs);
  free(tids);
  free(spawned);
  free(B64);
  return ORACLE_OK;
}
