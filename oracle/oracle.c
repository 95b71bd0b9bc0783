/*
 * oracle.c -- CPU reference for the dense half-precision matrix product
 *             C[M,N] = A[M,K] . B[K,N]
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file.  It may be used by the test suite, by the smoke check and by
 * the CPU-baseline leg of the benchmark, and by nothing else.  It shares no
 * code, header, table or constant with the CUDA path.
 *
 * What it computes (the plain definition, no blocking, no reordering):
 *   "tcgen05 for dummies: a B200 GEMM from scratch" (translated), section
 *   "Recap: how to write a fast matmul kernel": each C[m][n] is the dot product
 *   of row m of A with column n of B, accumulated over k in order.
 *   Layout conventions ("HGEMM: WMMA and MMA PTX study notes", kernel header
 *   comment): TN = A row-major [M,K], B column-major i.e. stored as [N,K],
 *   C row-major [M,N]; NN = A, B, C all row-major (B stored as [K,N]).
 *
 * Precision (the reading this file implements):
 *   - every fp16 / bf16 input is converted EXACTLY to double by decoding its
 *     bits (sign, exponent, fraction) -- both formats embed exactly in double;
 *   - each product a*b is exact in double (at most 2 x 11 significant bits);
 *   - the sum runs in double in k order;
 *   - the double result is rounded ONCE to the output format with IEEE
 *     round-to-nearest, ties-to-even, overflowing to +-Inf.
 *   The same routine serves runs with fp32 and with fp16 accumulation on the
 *   device: the oracle is the exact definition, the tests' tolerance absorbs
 *   the device's accumulation order and precision.
 *
 * Threads: rows (or sampled entries) are split across POSIX threads.  That
 * changes nothing in the arithmetic of any single entry.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#define OR_F16 0
#define OR_BF16 1
#define OR_TN 0
#define OR_NN 1

/* ------------------------------------------------------------------------ */
/* Format parameters: p = significant bits (incl. hidden bit), emin = exponent
 * of the smallest normal, emax = exponent of the largest finite, bias.      */
typedef struct {
  int p, emin, emax, bias, frac_bits, exp_bits;
} fmt_t;

static const fmt_t FMT_F16 = {11, -14, 15, 15, 10, 5};
static const fmt_t FMT_BF16 = {8, -126, 127, 127, 7, 8};

static const fmt_t* fmt_of(int dtype) { return dtype == OR_BF16 ? &FMT_BF16 : &FMT_F16; }

/* Exact bits -> double.  IEEE binary16 (1,5,10) and bfloat16 (1,8,7).       */
double oracle_decode(uint16_t bits, int dtype) {
  const fmt_t* f = fmt_of(dtype);
  int sign = bits >> 15;
  int e = (bits >> f->frac_bits) & ((1 << f->exp_bits) - 1);
  int frac = bits & ((1 << f->frac_bits) - 1);
  int emask = (1 << f->exp_bits) - 1;
  double v;
  if (e == emask) {
    v = frac ? NAN : INFINITY;
  } else if (e == 0) {
    /* subnormal: frac * 2^(emin - frac_bits) */
    v = ldexp((double)frac, f->emin - f->frac_bits);
  } else {
    /* normal: (2^frac_bits + frac) * 2^(e - bias - frac_bits) */
    v = ldexp((double)((1 << f->frac_bits) + frac), e - f->bias - f->frac_bits);
  }
  return sign ? -v : v;
}

/* Round a finite non-negative double n < 2^53 to the nearest integer, ties to
 * the even integer.  floor(n) and n - floor(n) are exact in this range.     */
static double round_half_even(double n) {
  double fl = floor(n);
  double diff = n - fl;
  if (diff > 0.5) return fl + 1.0;
  if (diff < 0.5) return fl;
  return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* double -> bits, IEEE round-to-nearest-even, overflow to Inf.              */
uint16_t oracle_encode(double x, int dtype) {
  const fmt_t* f = fmt_of(dtype);
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  uint16_t exp_all = (uint16_t)(((1 << f->exp_bits) - 1) << f->frac_bits);
  if (isnan(x)) return (uint16_t)(exp_all | (1 << (f->frac_bits - 1))); /* quiet NaN */
  double a = fabs(x);
  if (isinf(a)) return sign | exp_all;
  if (a == 0.0) return sign;

  /* Quantum of the target format at a: 2^(max(floor(log2 a), emin) - (p-1)). */
  int e2;
  frexp(a, &e2); /* a = m * 2^e2, m in [0.5, 1)  =>  floor(log2 a) = e2 - 1 */
  int E = e2 - 1;
  if (E < f->emin) E = f->emin;
  int qexp = E - (f->p - 1);
  double n = ldexp(a, -qexp); /* exact scaling by a power of two */
  double r = round_half_even(n);
  double v = ldexp(r, qexp); /* the rounded value, exponent unbounded above */

  if (v == 0.0) return sign; /* rounded below half the smallest subnormal */
  double maxfinite = ldexp((double)((1 << f->p) - 1), f->emax - (f->p - 1));
  if (v > maxfinite) return sign | exp_all;

  /* Encode the (now exactly representable) value v. */
  frexp(v, &e2);
  E = e2 - 1;
  if (E < f->emin) {
    /* subnormal: fraction = v / 2^(emin - frac_bits) */
    uint32_t frac = (uint32_t)ldexp(v, -(f->emin - f->frac_bits));
    return sign | (uint16_t)frac;
  }
  uint32_t mant = (uint32_t)ldexp(v, -(E - f->frac_bits)); /* in [2^fb, 2^(fb+1)) */
  uint32_t frac = mant - (1u << f->frac_bits);
  uint32_t ef = (uint32_t)(E + f->bias);
  return sign | (uint16_t)((ef << f->frac_bits) | frac);
}

/* Vector forms used by the tests. */
void oracle_decode_array(const uint16_t* in, double* out, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_decode(in[i], dtype);
}
void oracle_encode_array(const double* in, uint16_t* out, int64_t n, int dtype) {
  for (int64_t i = 0; i < n; i++) out[i] = oracle_encode(in[i], dtype);
}

/* ------------------------------------------------------------------------ */
/* One dot product, the definition itself.  The layout selects the storage of
 * B: element B[k][n] lives at B[n*K + k] for TN, at B[k*N + n] for NN.      */
typedef struct {
  const uint16_t* A;
  const uint16_t* B;
  int64_t M, N, K;
  int layout;
  const double* lut; /* 65536-entry exact decode of the input format */
} problem_t;

static void dot(const problem_t* p, int64_t m, int64_t n, double* sum, double* abssum) {
  double s = 0.0, sa = 0.0;
  const uint16_t* arow = p->A + m * p->K;
  for (int64_t k = 0; k < p->K; k++) {
    double a = p->lut[arow[k]];
    double b = (p->layout == OR_TN) ? p->lut[p->B[n * p->K + k]] : p->lut[p->B[k * p->N + n]];
    double prod = a * b; /* exact */
    s += prod;
    sa += fabs(prod);
  }
  *sum = s;
  *abssum = sa;
}

static double* make_lut(int dtype) {
  double* lut = (double*)malloc(sizeof(double) * 65536);
  if (!lut) return NULL;
  for (int i = 0; i < 65536; i++) lut[i] = oracle_decode((uint16_t)i, dtype);
  return lut;
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long c = sysconf(_SC_NPROCESSORS_ONLN);
  return c > 0 ? (int)c : 1;
}

/* ---- full product ---------------------------------------------------------*/
typedef struct {
  const problem_t* p;
  int64_t row0, row1;
  int out_dtype;
  uint16_t* C;      /* nullable: rounded output */
  double* C_exact;  /* nullable: double result before the final rounding */
  double* C_abs;    /* nullable: sum_k |a_mk b_kn| (tolerance scale) */
} rows_job_t;

static void* rows_worker(void* arg) {
  rows_job_t* j = (rows_job_t*)arg;
  const problem_t* p = j->p;
  for (int64_t m = j->row0; m < j->row1; m++) {
    for (int64_t n = 0; n < p->N; n++) {
      double s, sa;
      dot(p, m, n, &s, &sa);
      int64_t idx = m * p->N + n;
      if (j->C) j->C[idx] = oracle_encode(s, j->out_dtype);
      if (j->C_exact) j->C_exact[idx] = s;
      if (j->C_abs) j->C_abs[idx] = sa;
    }
  }
  return NULL;
}

/* Returns 0 on success, -1 on bad arguments or allocation failure. */
int oracle_gemm(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K, int layout,
                int in_dtype, int out_dtype, uint16_t* C, double* C_exact, double* C_abs,
                int nthreads) {
  if (M < 0 || N < 0 || K < 0) return -1;
  if (layout != OR_TN && layout != OR_NN) return -1;
  double* lut = make_lut(in_dtype);
  if (!lut) return -1;
  problem_t p = {A, B, M, N, K, layout, lut};
  int T = resolve_threads(nthreads);
  if (T > M) T = M > 0 ? (int)M : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * T);
  rows_job_t* jobs = (rows_job_t*)malloc(sizeof(rows_job_t) * T);
  if (!th || !jobs) { free(lut); free(th); free(jobs); return -1; }
  for (int t = 0; t < T; t++) {
    jobs[t].p = &p;
    jobs[t].row0 = M * t / T;
    jobs[t].row1 = M * (t + 1) / T;
    jobs[t].out_dtype = out_dtype;
    jobs[t].C = C;
    jobs[t].C_exact = C_exact;
    jobs[t].C_abs = C_abs;
  }
  /* A thread that cannot be started runs its share inline. */
  char* joined = (char*)calloc(T, 1);
  if (!joined) { free(lut); free(th); free(jobs); return -1; }
  for (int t = 1; t < T; t++) {
    if (pthread_create(&th[t], NULL, rows_worker, &jobs[t]) == 0) {
      joined[t] = 1;
    } else {
      rows_worker(&jobs[t]);
    }
  }
  rows_worker(&jobs[0]);
  for (int t = 1; t < T; t++)
    if (joined[t]) pthread_join(th[t], NULL);
  free(joined);
  free(th);
  free(jobs);
  free(lut);
  return 0;
}

/* ---- selected entries -----------------------------------------------------*/
typedef struct {
  const problem_t* p;
  const int64_t* rows;
  const int64_t* cols;
  int64_t i0, i1;
  double* exact;
  double* absdot;
} entries_job_t;

static void* entries_worker(void* arg) {
  entries_job_t* j = (entries_job_t*)arg;
  for (int64_t i = j->i0; i < j->i1; i++) {
    double s, sa;
    dot(j->p, j->rows[i], j->cols[i], &s, &sa);
    j->exact[i] = s;
    if (j->absdot) j->absdot[i] = sa;
  }
  return NULL;
}

/* Computes the double dot products for entries (rows[i], cols[i]), i < count.
 * Indices must lie inside [0,M) x [0,N) and layout must be TN or NN.
 * Returns 0, or -1 on bad arguments (nothing is written then).             */
int oracle_gemm_entries(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                        int layout, int in_dtype, const int64_t* rows, const int64_t* cols,
                        int64_t count, double* exact, double* absdot, int nthreads) {
  if (M < 0 || N < 0 || K < 0 || count < 0) return -1;
  if (layout != OR_TN && layout != OR_NN) return -1;
  for (int64_t i = 0; i < count; i++)
    if (rows[i] < 0 || rows[i] >= M || cols[i] < 0 || cols[i] >= N) return -1;
  double* lut = make_lut(in_dtype);
  if (!lut) return -1;
  problem_t p = {A, B, M, N, K, layout, lut};
  int T = resolve_threads(nthreads);
  if (T > count) T = count > 0 ? (int)count : 1;
  pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * T);
  entries_job_t* jobs = (entries_job_t*)malloc(sizeof(entries_job_t) * T);
  if (!th || !jobs) { free(lut); free(th); free(jobs); return -1; }
  for (int t = 0; t < T; t++) {
    jobs[t].p = &p;
    jobs[t].rows = rows;
    jobs[t].cols = cols;
    jobs[t].i0 = count * t / T;
    jobs[t].i1 = count * (t + 1) / T;
    jobs[t].exact = exact;
    jobs[t].absdot = absdot;
  }
  char* joined = (char*)calloc(T, 1);
  if (!joined) { free(lut); free(th); free(jobs); return -1; }
  for (int t = 1; t < T; t++) {
    if (pthread_create(&th[t], NULL, entries_worker, &jobs[t]) == 0) {
      joined[t] = 1;
    } else {
      entries_worker(&jobs[t]);
    }
  }
  entries_worker(&jobs[0]);
  for (int t = 1; t < T; t++)
    if (joined[t]) pthread_join(th[t], NULL);
  free(joined);
  free(th);
  free(jobs);
  free(lut);
  return 0;
}

/* ---- the tiled form ------------------------------------------------------ */
/* The tiled loop nest of the same section ("tiled_matmul"): output tiles of
 * BM x BN, each with an accumulator tile that is zeroed and then receives the
 * mini-products of BK-wide slices of A and B in k order.  Used only to check
 * that tiling does not change the definition; it keeps the per-entry k order,
 * so in double it agrees with oracle_gemm bit for bit.                      */
int oracle_gemm_tiled(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N, int64_t K,
                      int layout, int in_dtype, int64_t BM, int64_t BN, int64_t BK,
                      double* C_exact) {
  if (M < 0 || N < 0 || K < 0 || BM <= 0 || BN <= 0 || BK <= 0) return -1;
  if (layout != OR_TN && layout != OR_NN) return -1;
  double* lut = make_lut(in_dtype);
  if (!lut) return -1;
  double* acc = (double*)malloc(sizeof(double) * BM * BN);
  if (!acc) { free(lut); return -1; }
  for (int64_t m0 = 0; m0 < M; m0 += BM) {
    for (int64_t n0 = 0; n0 < N; n0 += BN) {
      int64_t bm = (M - m0 < BM) ? M - m0 : BM;
      int64_t bn = (N - n0 < BN) ? N - n0 : BN;
      memset(acc, 0, sizeof(double) * BM * BN);
      for (int64_t k0 = 0; k0 < K; k0 += BK) {
        int64_t bk = (K - k0 < BK) ? K - k0 : BK;
        /* acc += A[m0:m0+bm, k0:k0+bk] @ B[k0:k0+bk, n0:n0+bn] */
        for (int64_t i = 0; i < bm; i++)
          for (int64_t j = 0; j < bn; j++) {
            double s = acc[i * BN + j];
            for (int64_t k = 0; k < bk; k++) {
              double a = lut[A[(m0 + i) * K + (k0 + k)]];
              double b = (layout == OR_TN) ? lut[B[(n0 + j) * K + (k0 + k)]]
                                           : lut[B[(k0 + k) * N + (n0 + j)]];
              s += a * b;
            }
            acc[i * BN + j] = s;
          }
      }
      for (int64_t i = 0; i < bm; i++)
        for (int64_t j = 0; j < bn; j++) C_exact[(m0 + i) * N + (n0 + j)] = acc[i * BN + j];
    }
  }
  free(acc);
  free(lut);
  return 0;
}
