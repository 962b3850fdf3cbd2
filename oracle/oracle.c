/*
 * fp64 CPU oracle for the FC-layer GEMMs -- TEST INFRASTRUCTURE ONLY.
 *
 * Only the tests, the smoke check and the benchmark's CPU-baseline leg load
 * this library.  It shares no code, header or constant with the GPU path.
 *
 * What it computes: the plain matrix product C = A . B that an FC layer's
 * forward and backward passes reduce to (Figure 1 caption of "Democratizing
 * AI: Open-source Scalable LLM Training on GPU-based Supercomputers").  Agarwal's
 * 3D decomposition only reassigns which block of this sum each GPU computes,
 * so the exact result is the definition
 *     C[i][j] = sum_r A[i][r] * B[r][j]
 * evaluated here with a naive loop in i-r-j order and fp64 accumulation.
 * Each bf16 x bf16 product is exact in fp64.  Alongside C it forms
 *     S[i][j] = sum_r |A[i][r]| * |B[r][j]|
 * which scales the per-element error bound |C_gpu - C| <= 1e-2 * S + 1e-5.
 *
 * Storage: operands are bf16 bit patterns.  A logical A[M x R] is stored
 * either as written ("N": element (i,r) at A[i*lda + r]) or transposed ("T":
 * element (i,r) at A[r*lda + i]); likewise B[R x N].  Transposed operands are
 * read through address mapping, never copied.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static inline double bf16_to_f64(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return (double)f;
}

static inline double a_at(const uint16_t* A, int64_t lda, int a_t, int64_t i,
                          int64_t r) {
  return bf16_to_f64(a_t ? A[r * lda + i] : A[i * lda + r]);
}

static inline double b_at(const uint16_t* B, int64_t ldb, int b_t, int64_t r,
                          int64_t j) {
  return bf16_to_f64(b_t ? B[j * ldb + r] : B[r * ldb + j]);
}

/* Full product.  C and S are dense row-major [M x N] (leading dimension N). */
void oracle_gemm_f64(const uint16_t* A, int64_t lda, int a_t,
                     const uint16_t* B, int64_t ldb, int b_t, int64_t M,
                     int64_t N, int64_t R, double* C, double* S) {
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < M; ++i) {
    double* c = C + i * N;
    double* s = S + i * N;
    for (int64_t j = 0; j < N; ++j) {
      c[j] = 0.0;
      s[j] = 0.0;
    }
    for (int64_t r = 0; r < R; ++r) {
      const double a = a_at(A, lda, a_t, i, r);
      const double aa = fabs(a);
      for (int64_t j = 0; j < N; ++j) {
        const double b = b_at(B, ldb, b_t, r, j);
        c[j] += a * b;
        s[j] += aa * fabs(b);
      }
    }
  }
}

/* Selected entries (I[e], J[e]) of the same product, each a dot product over
 * r in ascending order. */
void oracle_gemm_entries_f64(const uint16_t* A, int64_t lda, int a_t,
                             const uint16_t* B, int64_t ldb, int b_t,
                             int64_t R, const int64_t* I, const int64_t* J,
                             int64_t count, double* C, double* S) {
#pragma omp parallel for schedule(dynamic, 64)
  for (int64_t e = 0; e < count; ++e) {
    double c = 0.0, s = 0.0;
    for (int64_t r = 0; r < R; ++r) {
      const double a = a_at(A, lda, a_t, I[e], r);
      const double b = b_at(B, ldb, b_t, r, J[e]);
      c += a * b;
      s += fabs(a) * fabs(b);
    }
    C[e] = c;
    S[e] = s;
  }
}

/* Widen bf16 bits to double (exact). */
void oracle_bf16_to_f64(const uint16_t* in, int64_t n, double* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = bf16_to_f64(in[k]);
}

/*
 * Round a finite double to the nearest bf16 (8 significant bits, 8 exponent
 * bits), ties to even, following the IEEE 754 definition of
 * roundTiesToEven: find the two neighbouring representable values and pick
 * the nearer, the one with an even last significand bit on a tie.  Results
 * beyond the largest finite bf16 become infinity; magnitudes below the
 * smallest normal round on the subnormal grid (spacing 2^-133).
 */
static uint16_t f64_to_bf16_rne(double v) {
  const uint16_t sign = signbit(v) ? 0x8000u : 0u;
  double a = fabs(v);
  if (a == 0.0) return sign;
  int e;
  (void)frexp(a, &e);            /* a = f * 2^e, f in [0.5, 1) */
  int exp_unbiased = e - 1;      /* a = 1.xxx * 2^exp_unbiased */
  if (exp_unbiased < -126) exp_unbiased = -126; /* subnormal grid */
  const double ulp = ldexp(1.0, exp_unbiased - 7);
  const double q = a / ulp;      /* exact: a has <= 53 bits */
  double lo = floor(q);
  const double rem = q - lo;
  double m;                      /* integer multiple of ulp */
  if (rem > 0.5) {
    m = lo + 1.0;
  } else if (rem < 0.5) {
    m = lo;
  } else {
    m = (fmod(lo, 2.0) == 0.0) ? lo : lo + 1.0;
  }
  const double r = m * ulp;
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u); /* +-inf */
  /* Encode r exactly as bf16 bits. */
  if (r < ldexp(1.0, -126)) {
    /* subnormal: r = m' * 2^-133, 0 <= m' < 128 */
    const uint16_t mant = (uint16_t)(r / ldexp(1.0, -133));
    return (uint16_t)(sign | mant);
  }
  int er;
  const double fr = frexp(r, &er); /* r = fr * 2^er, fr in [0.5,1) */
  const uint16_t biased = (uint16_t)(er - 1 + 127);
  const uint16_t mant = (uint16_t)((fr * 2.0 - 1.0) * 128.0);
  return (uint16_t)(sign | (uint16_t)(biased << 7) | mant);
}

void oracle_f64_to_bf16(const double* in, int64_t n, uint16_t* out) {
  for (int64_t k = 0; k < n; ++k) out[k] = f64_to_bf16_rne(in[k]);
}

int oracle_max_threads(void) {
#ifdef _OPENMP
  extern int omp_get_max_threads(void);
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Threads for the calling thread's later parallel loops (n >= 1); returns
 * the count now in effect.  A launcher that sets OMP_NUM_THREADS=1 for each
 * of several processes leaves one process that wants every core. */
int oracle_set_threads(int n) {
#ifdef _OPENMP
  extern void omp_set_num_threads(int);
  if (n >= 1) omp_set_num_threads(n);
#else
  (void)n;
#endif
  return oracle_max_threads();
}
