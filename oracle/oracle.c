/*
 * oracle.c -- plain, slow CPU oracle for the fp16 TN GEMM
 *
 *     D(m,n) = C(m,n) + sum_{k<K} A(m,k) * B(n,k)
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests/, __graft_entry__.smoke() and the
 * CPU-baseline leg of bench.py may load this code.  The product library
 * (dense_fp16_tensor_gb300) never links, imports or calls it, and this file
 * includes nothing from the product.
 *
 * Sources (the five pages on CuTe's SM80 fp16 tensor-core GEMM path):
 *  - "Reading CuTe's make_tiled_mma" (blog.qingsen.net,
 *    cute_make_tiled_mma_walkthrough_zh), section "Fix the matrices and
 *    directions first": A is (M,K), B is (N,K), C is (M,N) and
 *    D(m,n) = C(m,n) + sum A(m,k)*B(n,k); B(n,k) = B_math(k,n).  The same
 *    section defines shape:stride notation: (2,2,1):(1,2,4) maps (wm,wn,wk)
 *    to wm + 2 wn + 4 wk, and a size-1 mode's stride does not matter.
 *  - "CuTe Layout to Tensor Core" (chatdocs.ruinique.com), sections 1-2:
 *    a matrix is a Shape + Stride layout, (M,K):(K,1) when K is contiguous
 *    and (M,K):(1,M) (or a padded leading dimension) when M is; a tensor is
 *    a pointer plus a layout.
 *  - Same page, section "Start from C's four values" of the make_tiled_mma
 *    page and "4.3 reading nested parentheses" of "cute(7) simple_gemm"
 *    (yuyanqi.com): an integer coordinate is decoded with the first mode
 *    varying fastest; nesting only groups modes, the offset is the dot
 *    product of the flattened coordinate and stride.
 *
 * Every function is pinned by tests that do not retype it: values printed on
 * the pages (tests/golden), closed forms (identity / permutation / all-ones
 * operands), invariants (K-major vs MN-major views of the same matrix, padded
 * leading dimensions), a library special case (float64 BLAS matmul) and, for
 * the fp16 codec, numpy's IEEE binary16 conversion over every bit pattern.
 *
 * The scaled, batched form (oracle_gemm_tn_general) follows the
 * "cute(7) simple_gemm" page, section 8.1: its cuBLAS comparison computes
 * D = alpha * A.B^T + beta * C, and local_tile's extra modes there (section
 * 4) carry a batch coordinate; see that function's comment for the
 * conventions taken where the page is silent.
 *
 * Arithmetic: fp16 inputs are decoded exactly to fp64; every fp16 x fp16
 * product is exact in fp64 (22 significant bits), and the k-sum runs in
 * ascending k from the initial C(m,n) with no blocking or reordering, so
 * the result does not depend on the number of threads.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_EXPORT __attribute__((visibility("default")))

/* ------------------------------------------------------------------------ */
/* Layout evaluator (shape:stride)                                           */
/* ------------------------------------------------------------------------ */

/*
 * Evaluate a (possibly nested) shape:stride layout at a hierarchical
 * coordinate.  The layout is given flattened: shape[0..nflat) and
 * stride[0..nflat).  The top-level modes are given by mode_len[0..nmodes):
 * top-level mode t owns the next mode_len[t] flat entries.  coord[t] is one
 * integer per top-level mode; it is decoded colexicographically (first
 * sub-mode fastest) over that mode's flat shapes, and the offset is the sum of
 * sub-coordinate times stride over all flat entries.
 *
 * Passing nmodes = 1 and mode_len[0] = nflat evaluates layout(i) for one
 * integer i over the whole shape.
 *
 * Returns the offset, or -1 when a coordinate is outside its mode's size or
 * the description is inconsistent.
 */
ORACLE_EXPORT int64_t oracle_layout_offset(int nflat, const int64_t* shape,
                                           const int64_t* stride, int nmodes,
                                           const int* mode_len,
                                           const int64_t* coord) {
  int64_t offset = 0;
  int f = 0;
  for (int t = 0; t < nmodes; ++t) {
    int64_t rem = coord[t];
    int64_t mode_size = 1;
    for (int j = 0; j < mode_len[t]; ++j) mode_size *= shape[f + j];
    if (rem < 0 || rem >= mode_size) return -1;
    for (int j = 0; j < mode_len[t]; ++j, ++f) {
      if (f >= nflat || shape[f] <= 0) return -1;
      int64_t c = rem % shape[f];
      rem /= shape[f];
      offset += c * stride[f];
    }
  }
  if (f != nflat) return -1;
  return offset;
}

/* A rank-2 view (rows, cols):(row_stride, col_stride) -- the two-mode case of
 * the evaluator above with one coordinate per mode.  The GEMM loops read
 * every operand element through this. */
typedef struct {
  int64_t rows, cols;
  int64_t s_row, s_col;
} view2_t;

static inline int64_t view2_offset(const view2_t* v, int64_t i, int64_t j) {
  return i * v->s_row + j * v->s_col;
}

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 codec, written from the format's definition             */
/* ------------------------------------------------------------------------ */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN;
 * otherwise value = (1024 + fraction) * 2^(exponent - 25). */
ORACLE_EXPORT double oracle_half_to_double(uint16_t h) {
  int sign = (h >> 15) & 1;
  int e = (h >> 10) & 0x1f;
  int frac = h & 0x3ff;
  double v;
  if (e == 0) {
    v = ldexp((double)frac, -24);
  } else if (e == 31) {
    v = frac ? NAN : INFINITY;
  } else {
    v = ldexp((double)(1024 + frac), e - 25);
  }
  return sign ? -v : v;
}

/* Round a double to the nearest binary16 value, ties to even.
 *
 * With |x| = r * q where q is the binary16 quantum at |x|'s binade
 * (2^-24 below 2^-14, else 2^(e-10) for |x| in [2^e, 2^(e+1))), the result
 * is round_half_even(r) * q.  Magnitudes at or above 65520 (half-way between
 * 65504, the largest finite value, and 2^16) round to infinity.  NaN maps to
 * the canonical quiet NaN with the input's sign. */
ORACLE_EXPORT uint16_t oracle_double_to_half_rne(double x) {
  uint16_t sign = signbit(x) ? 0x8000 : 0;
  if (isnan(x)) return (uint16_t)(sign | 0x7e00);
  double a = fabs(x);
  if (a >= 65520.0) return (uint16_t)(sign | 0x7c00);
  if (a == 0.0) return sign;
  int E;
  (void)frexp(a, &E);      /* a = f * 2^E, f in [0.5, 1) => a in [2^(E-1), 2^E) */
  int e = E - 1;           /* unbiased exponent of a */
  int subnormal = e < -14;
  int qexp = subnormal ? -24 : e - 10;
  double n = ldexp(a, -qexp); /* exact: scaling by a power of two */
  double r = floor(n);
  double frac = n - r;
  if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
  uint32_t ir = (uint32_t)r;
  uint32_t bits;
  if (subnormal) {
    bits = ir; /* 1024 lands on the smallest normal, 0x0400 */
  } else {
    /* ir in [1024, 2048]; 2048 carries into the exponent field */
    bits = ((uint32_t)(e + 15) << 10) + (ir - 1024);
  }
  return (uint16_t)(sign | bits);
}

/* ------------------------------------------------------------------------ */
/* The GEMM                                                                  */
/* ------------------------------------------------------------------------ */

typedef struct {
  int64_t M, N, K;
  const uint16_t *A, *B, *C;
  view2_t vA, vB, vC;
  const double* lut; /* binary16 bits -> double, built by oracle_half_to_double */
  double* out_f64;   /* (M,N) row-major, may be NULL */
  uint16_t* out_f16; /* (M,N) row-major, may be NULL */
  int64_t row_begin, row_end;
  /* sampled mode */
  const int64_t *sm, *sn;
  int64_t s_begin, s_end;
} job_t;

/* One output element, exactly as the definition reads. */
static double dot_one(const job_t* j, int64_t m, int64_t n) {
  double acc = j->C ? j->lut[j->C[view2_offset(&j->vC, m, n)]] : 0.0;
  for (int64_t k = 0; k < j->K; ++k) {
    double a = j->lut[j->A[view2_offset(&j->vA, m, k)]];
    double b = j->lut[j->B[view2_offset(&j->vB, n, k)]];
    acc += a * b; /* exact product; sum in ascending k */
  }
  return acc;
}

static void* rows_worker(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t m = j->row_begin; m < j->row_end; ++m) {
    for (int64_t n = 0; n < j->N; ++n) {
      double d = dot_one(j, m, n);
      if (j->out_f64) j->out_f64[m * j->N + n] = d;
      if (j->out_f16) j->out_f16[m * j->N + n] = oracle_double_to_half_rne(d);
    }
  }
  return NULL;
}

static void* samples_worker(void* arg) {
  job_t* j = (job_t*)arg;
  for (int64_t s = j->s_begin; s < j->s_end; ++s) {
    double d = dot_one(j, j->sm[s], j->sn[s]);
    if (j->out_f64) j->out_f64[s] = d;
    if (j->out_f16) j->out_f16[s] = oracle_double_to_half_rne(d);
  }
  return NULL;
}

static double g_lut[65536];
static int g_lut_ready = 0;
static pthread_mutex_t g_lut_mu = PTHREAD_MUTEX_INITIALIZER;

static const double* half_lut(void) {
  pthread_mutex_lock(&g_lut_mu);
  if (!g_lut_ready) {
    for (uint32_t h = 0; h < 65536; ++h) g_lut[h] = oracle_half_to_double((uint16_t)h);
    g_lut_ready = 1;
  }
  pthread_mutex_unlock(&g_lut_mu);
  return g_lut;
}

/* Operand views from the (ptr, ld, major) description:
 *   major 0 (K / N contiguous): (rows, cols):(ld, 1)
 *   major 1 (M / N contiguous): (rows, cols):(1, ld)                      */
static view2_t make_view(int64_t rows, int64_t cols, int64_t ld, int major) {
  view2_t v = {rows, cols, major ? 1 : ld, major ? ld : 1};
  return v;
}

static int run_threads(job_t* proto, int nthreads, int64_t total, int sampled) {
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (total < nthreads) nthreads = total > 0 ? (int)total : 1;
  pthread_t th[256];
  job_t jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = *proto;
    int64_t b = total * t / nthreads, e = total * (t + 1) / nthreads;
    if (sampled) {
      jobs[t].s_begin = b;
      jobs[t].s_end = e;
    } else {
      jobs[t].row_begin = b;
      jobs[t].row_end = e;
    }
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, sampled ? samples_worker : rows_worker, &jobs[t]) != 0) break;
    started = t;
  }
  /* thread 0's share runs here; shares of threads that failed to start too */
  if (sampled) samples_worker(&jobs[0]); else rows_worker(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) {
    if (sampled) samples_worker(&jobs[t]); else rows_worker(&jobs[t]);
  }
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  return nthreads;
}

/*
 * Full oracle over arbitrary element strides ("CuTe Layout to Tensor Core",
 * sections 1-2: an operand is a pointer plus a shape:stride layout, and no
 * mode has to be stride-1).  A, B, C are raw binary16 bit patterns:
 *   A(m,k) = A[m*sAm + k*sAk],  B(n,k) = B[n*sBn + k*sBk],
 *   C(m,n) = C[m*sCm + n*sCn]   (C may be NULL: treated as zero).
 * out_f64 / out_f16 are (M,N) row-major (either may be NULL).
 * Returns the number of threads used.
 */
ORACLE_EXPORT int oracle_gemm_tn_strided(int64_t M, int64_t N, int64_t K,
                                         const uint16_t* A, int64_t sAm, int64_t sAk,
                                         const uint16_t* B, int64_t sBn, int64_t sBk,
                                         const uint16_t* C, int64_t sCm, int64_t sCn,
                                         double* out_f64, uint16_t* out_f16, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.M = M; j.N = N; j.K = K;
  j.A = A; j.B = B; j.C = C;
  view2_t va = {M, K, sAm, sAk}, vb = {N, K, sBn, sBk}, vc = {M, N, sCm, sCn};
  j.vA = va; j.vB = vb; j.vC = vc;
  j.lut = half_lut();
  j.out_f64 = out_f64;
  j.out_f16 = out_f16;
  return run_threads(&j, nthreads, M, 0);
}

/*
 * Full oracle for (ptr, ld, major) operands -- the strided oracle with
 *   A(m,k): a_major 0 -> A[m*ldA + k], a_major 1 -> A[m + k*ldA]
 *   B(n,k): b_major 0 -> B[n*ldB + k], b_major 1 -> B[n + k*ldB]
 *   C(m,n): C[m*ldC + n].
 */
ORACLE_EXPORT int oracle_gemm_tn(int64_t M, int64_t N, int64_t K,
                                 const uint16_t* A, int64_t ldA, int a_major,
                                 const uint16_t* B, int64_t ldB, int b_major,
                                 const uint16_t* C, int64_t ldC,
                                 double* out_f64, uint16_t* out_f16,
                                 int nthreads) {
  view2_t va = make_view(M, K, ldA, a_major), vb = make_view(N, K, ldB, b_major);
  return oracle_gemm_tn_strided(M, N, K, A, va.s_row, va.s_col, B, vb.s_row, vb.s_col, C, ldC, 1,
                                out_f64, out_f16, nthreads);
}

/* Sampled oracle: out[s] = D(sm[s], sn[s]) for s < count (same definition). */
ORACLE_EXPORT int oracle_gemm_tn_sampled(int64_t M, int64_t N, int64_t K,
                                         const uint16_t* A, int64_t ldA, int a_major,
                                         const uint16_t* B, int64_t ldB, int b_major,
                                         const uint16_t* C, int64_t ldC,
                                         int64_t count, const int64_t* sm,
                                         const int64_t* sn, double* out_f64,
                                         uint16_t* out_f16, int nthreads) {
  job_t j;
  memset(&j, 0, sizeof j);
  j.M = M; j.N = N; j.K = K;
  j.A = A; j.B = B; j.C = C;
  j.vA = make_view(M, K, ldA, a_major);
  j.vB = make_view(N, K, ldB, b_major);
  j.vC = make_view(M, N, ldC, 0);
  j.lut = half_lut();
  j.out_f64 = out_f64;
  j.out_f16 = out_f16;
  j.sm = sm;
  j.sn = sn;
  return run_threads(&j, nthreads, count, 1);
}

/* ------------------------------------------------------------------------ */
/* Scaled and batched form                                                   */
/* ------------------------------------------------------------------------ */

typedef struct {
  int64_t M, N, K, L;
  double alpha, beta;
  const uint16_t *A, *B, *C;
  int64_t sAm, sAk, sAl, sBn, sBk, sBl, sCm, sCn, sCl;
  const double* lut;
  double* out_f64;   /* (L,M,N) row-major, may be NULL */
  uint16_t* out_f16; /* (L,M,N) row-major, may be NULL */
  int64_t begin, end; /* range of (l, m) rows */
} gjob_t;

static void* general_worker(void* arg) {
  const gjob_t* j = (const gjob_t*)arg;
  for (int64_t lm = j->begin; lm < j->end; ++lm) {
    const int64_t l = lm / j->M, m = lm % j->M;
    for (int64_t n = 0; n < j->N; ++n) {
      /* the product term P = alpha * sum and the C term Q = beta * C, each
       * present only when its scalar is nonzero (and K > 0 for P) */
      const int has_p = j->alpha != 0.0 && j->K > 0, has_q = j->beta != 0.0;
      double p = 0.0, q = 0.0;
      if (has_p) {
        /* exact fp16 x fp16 products, ascending k */
        double s = 0.0;
        for (int64_t k = 0; k < j->K; ++k) {
          const double a = j->lut[j->A[l * j->sAl + m * j->sAm + k * j->sAk]];
          const double b = j->lut[j->B[l * j->sBl + n * j->sBn + k * j->sBk]];
          s += a * b;
        }
        p = j->alpha * s;
      }
      if (has_q) q = j->beta * j->lut[j->C[l * j->sCl + m * j->sCm + n * j->sCn]];
      /* an absent term is left out, not added as zero: a lone term keeps its
       * sign of zero; with neither term D is +0 */
      const double d = has_p ? (has_q ? p + q : p) : (has_q ? q : 0.0);
      const int64_t o = (l * j->M + m) * j->N + n;
      if (j->out_f64) j->out_f64[o] = d;
      if (j->out_f16) j->out_f16[o] = oracle_double_to_half_rne(d);
    }
  }
  return NULL;
}

/*
 * D(l,m,n) = alpha * sum_{k<K} A(l,m,k) * B(l,n,k) + beta * C(l,m,n)
 * for l < L (the batch), with
 *   A(l,m,k) = A[l*sAl + m*sAm + k*sAk],  B(l,n,k) = B[l*sBl + n*sBn + k*sBk],
 *   C(l,m,n) = C[l*sCl + m*sCm + n*sCn]   (a batch stride may be 0).
 * The sum is formed in fp64 (exact products, ascending k), scaled by alpha,
 * and beta * C is added; the fp16 result is that fp64 value rounded once.
 * Where the pages are silent the BLAS conventions hold: alpha == 0 or
 * K == 0 leaves out the product term and A, B unread; beta == 0 leaves out
 * the C term and C unread (C may be NULL), so NaN or Inf there does not
 * reach D.  A term left out is not added as a zero: D is the other term
 * alone (its sign of zero kept), or +0 when both are left out.
 * out_f64 / out_f16 are (L,M,N) row-major (either may be NULL).
 * Returns the number of threads used.
 */
ORACLE_EXPORT int oracle_gemm_tn_general(int64_t M, int64_t N, int64_t K, int64_t L,
                                         double alpha,
                                         const uint16_t* A, int64_t sAm, int64_t sAk, int64_t sAl,
                                         const uint16_t* B, int64_t sBn, int64_t sBk, int64_t sBl,
                                         double beta,
                                         const uint16_t* C, int64_t sCm, int64_t sCn, int64_t sCl,
                                         double* out_f64, uint16_t* out_f16, int nthreads) {
  gjob_t proto;
  memset(&proto, 0, sizeof proto);
  proto.M = M; proto.N = N; proto.K = K; proto.L = L;
  proto.alpha = alpha; proto.beta = beta;
  proto.A = A; proto.B = B; proto.C = C;
  proto.sAm = sAm; proto.sAk = sAk; proto.sAl = sAl;
  proto.sBn = sBn; proto.sBk = sBk; proto.sBl = sBl;
  proto.sCm = sCm; proto.sCn = sCn; proto.sCl = sCl;
  proto.lut = half_lut();
  proto.out_f64 = out_f64;
  proto.out_f16 = out_f16;
  const int64_t total = L * M;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > 256) nthreads = 256;
  if (total < nthreads) nthreads = total > 0 ? (int)total : 1;
  pthread_t th[256];
  gjob_t jobs[256];
  for (int t = 0; t < nthreads; ++t) {
    jobs[t] = proto;
    jobs[t].begin = total * t / nthreads;
    jobs[t].end = total * (t + 1) / nthreads;
  }
  int started = 0;
  for (int t = 1; t < nthreads; ++t) {
    if (pthread_create(&th[t], NULL, general_worker, &jobs[t]) != 0) break;
    started = t;
  }
  general_worker(&jobs[0]);
  for (int t = started + 1; t < nthreads; ++t) general_worker(&jobs[t]);
  for (int t = 1; t <= started; ++t) pthread_join(th[t], NULL);
  return nthreads;
}
