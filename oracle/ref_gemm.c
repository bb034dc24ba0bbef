/*
 * ORACLE — test infrastructure only.
 *
 * A plain, slow, obviously-correct CPU reference for the dense tile product
 *     C = alpha * A * B + beta * C0
 * evaluated in IEEE binary64.  Only the test-suite, the smoke check and the
 * CPU-baseline leg of the benchmark may load this file's library; the GPU
 * library never links, includes or calls it, and this file includes nothing
 * from the GPU library.
 *
 * Passages followed (pages on mixed-precision tensor-core matrix products):
 *  - "Tensor Core operands: a matrix instruction still needs a layout contract",
 *    first paragraph: row-major leading dimension = element distance between
 *    successive rows, column-major = distance between successive columns,
 *    padding may make it larger than the visible extent.
 *  - same page, third and fourth paragraphs: FP16 / BF16 / TF32 conversion is a
 *    rounding of the multiplicands; error must be measured both against the
 *    original real-valued problem ("mode R") and against the problem on the
 *    inputs exactly as quantised ("mode Q").
 *  - "qsa_prompt_attn: Volta m8n8k4 kernel - keep the hi and lo halves in
 *    separate accumulator chains", sections "What's going on" and "The fix":
 *    an FP32 operand is split into an FP16 hi half and an FP16 lo half so the
 *    products come out close to FP32 precision.
 *  - "feat(cuda-device): derive the m16n8k16 accumulator fragment layout",
 *    section "The layout is a mixed-radix numeral": the PTX row/col formulas of
 *    the f32 accumulator fragment of mma.sync m16n8k16.
 *
 * Readings of points the pages leave open (each is listed in the design notes):
 *  - FP16 and BF16 conversion is round-to-nearest, ties to even, overflow to
 *    infinity, gradual underflow (the IEEE default).
 *  - TF32 conversion is modelled three ways (truncation of the 13 low fraction
 *    bits, round-half-away, round-half-even); which one the hardware applies
 *    is an open question the GPU tests measure.
 *  - The split is hi = fp16(x*2^s), lo = fp16((x*2^s - hi) * 2^L) with the
 *    value of x represented as (hi + lo*2^-L) * 2^-s.  s is a per-operand
 *    power-of-two scale and L is 11 for the three-chain form and 0 for the
 *    single-chain form (plain lo = fp16(x - hi) when s = L = 0).  Powers of two
 *    are exact, so they only move the operand out of the FP16 subnormal range.
 *  - The three-chain product keeps hi*hi + hi*lo + lo*hi and drops lo*lo;
 *    the four-chain variant (a next step listed for the split) keeps lo*lo.
 *
 *  - "qsa_prompt_attn: ...", section "What's going on": the prompt-attention
 *    pair, scores q.k, then the row softmax, then p.v (the definition of
 *    attention written out in orc_attention_f64 below).
 *
 * Everything here is a direct transcription of a definition: a triple loop in
 * the order (row i, column j, k ascending) or the equivalent (i, k, j) axpy
 * order for full grids; no blocking, no fused reductions, no fast-math.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

/* storage type of an input matrix */
enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2, ORC_F64 = 3 };

/* how an operand is quantised before the products are formed */
enum {
  ORC_Q_NONE = 0,        /* the stored value itself (mode R) */
  ORC_Q_FP16 = 1,        /* fp16 round-to-nearest-even */
  ORC_Q_BF16 = 2,        /* bf16 round-to-nearest-even */
  ORC_Q_TF32_TRUNC = 3,  /* fp32 with the 13 low fraction bits cleared */
  ORC_Q_TF32_RNA = 4,    /* tf32, round half away from zero */
  ORC_Q_TF32_RNE = 5,    /* tf32, round half to even */
  ORC_Q_SPLIT3 = 6,      /* hi/lo split, lo scaled by 2^11 (three chains) */
  ORC_Q_SPLIT1 = 7,      /* hi/lo split, plain lo (single chain) */
  ORC_Q_SPLIT4 = 8       /* hi/lo split, lo scaled by 2^11, lo*lo kept (four chains) */
};

/* ------------------------------------------------------------------------- */
/* IEEE bit-level helpers                                                      */
/* ------------------------------------------------------------------------- */

static uint32_t f32_bits(float f) { uint32_t u; memcpy(&u, &f, 4); return u; }
static float bits_f32(uint32_t u) { float f; memcpy(&f, &u, 4); return f; }

/* Round-half-to-even of a non-negative double that is an exact multiple of
 * 1/2^m for small m (the callers scale by powers of two, so q - floor(q) is
 * exact). */
static double rne_nonneg(double q) {
  double f = floor(q);
  double r = q - f;
  if (r > 0.5) return f + 1.0;
  if (r < 0.5) return f;
  /* exact tie: pick the even neighbour */
  return (fmod(f, 2.0) == 0.0) ? f : f + 1.0;
}

/* Round x to the nearest value of a binary floating-point format with p
 * significand bits (implicit bit included), minimum normal exponent emin and
 * maximum exponent emax; ties to even; gradual underflow; overflow to inf.
 * This is the IEEE 754 rounding rule written out. */
double orc_round_format(double x, int p, int emin, int emax) {
  if (isnan(x) || isinf(x) || x == 0.0) return x;
  double a = fabs(x);
  int E;
  frexp(a, &E);            /* a = f * 2^E with f in [0.5, 1) */
  int e = E - 1;           /* 2^e <= a < 2^(e+1) */
  if (e < emin) e = emin;  /* subnormal range: fixed quantum */
  double quantum = ldexp(1.0, e - p + 1);
  double r = rne_nonneg(a / quantum) * quantum;
  /* the largest finite value is (2 - 2^(1-p)) * 2^emax */
  if (r >= ldexp(1.0, emax + 1)) r = INFINITY;
  return copysign(r, x);
}

double orc_fp16(double x) { return orc_round_format(x, 11, -14, 15); }
double orc_bf16(double x) { return orc_round_format(x, 8, -126, 127); }
double orc_tf32_rne(double x) { return orc_round_format(x, 11, -126, 127); }

/* tf32 by truncation: keep sign, exponent and the 10 high fraction bits of the
 * fp32 pattern, clear the 13 low ones. */
double orc_tf32_trunc(double x) {
  float f = (float)x;
  if (isnan(f) || isinf(f)) return (double)f;
  return (double)bits_f32(f32_bits(f) & 0xFFFFE000u);
}

/* tf32 rounding half away from zero on the magnitude: add half a tf32 ulp to
 * the fp32 pattern, then truncate.  A carry into the exponent is the correct
 * rounding up to the next binade (and to infinity past the largest value). */
double orc_tf32_rna(double x) {
  float f = (float)x;
  if (isnan(f) || isinf(f)) return (double)f;
  uint32_t u = f32_bits(f);
  uint32_t mag = (u & 0x7FFFFFFFu) + 0x00001000u;
  if (mag >= 0x7F800000u) mag = 0x7F800000u;
  else mag &= 0xFFFFE000u;
  return (double)bits_f32((u & 0x80000000u) | mag);
}

/* Decoders of stored 16-bit codes, from the IEEE field layout. */
double orc_fp16_decode(uint16_t h) {
  int s = (h >> 15) & 1, e = (h >> 10) & 0x1F, m = h & 0x3FF;
  double v;
  if (e == 0) v = ldexp((double)m, -24);
  else if (e == 31) v = (m == 0) ? INFINITY : NAN;
  else v = ldexp((double)(1024 + m), e - 25);
  return s ? -v : v;
}

double orc_bf16_decode(uint16_t h) {
  return (double)bits_f32(((uint32_t)h) << 16);
}

/* The hi/lo split of one value (see the header comment for the reading).
 * Returns the represented values, already unscaled:  x ~ hi + lo. */
void orc_split(double x, int s, int L, double* hi, double* lo) {
  double xs = ldexp(x, s);                 /* exact: power of two */
  double h = orc_fp16(xs);
  double r = xs - h;                       /* exact in binary64 */
  double l = orc_fp16(ldexp(r, L));
  *hi = ldexp(h, -s);
  *lo = ldexp(l, -(s + L));
}

static double load_elem(const void* base, int type, int64_t idx) {
  switch (type) {
    case ORC_F32: return (double)((const float*)base)[idx];
    case ORC_F16: return orc_fp16_decode(((const uint16_t*)base)[idx]);
    case ORC_BF16: return orc_bf16_decode(((const uint16_t*)base)[idx]);
    default: return ((const double*)base)[idx];
  }
}

/* quantise one stored value; lo is 0 except in the split modes */
static void quant_elem(double x, int q, int s, double* hi, double* lo) {
  *lo = 0.0;
  switch (q) {
    case ORC_Q_FP16: *hi = orc_fp16(x); break;
    case ORC_Q_BF16: *hi = orc_bf16(x); break;
    case ORC_Q_TF32_TRUNC: *hi = orc_tf32_trunc(x); break;
    case ORC_Q_TF32_RNA: *hi = orc_tf32_rna(x); break;
    case ORC_Q_TF32_RNE: *hi = orc_tf32_rne(x); break;
    case ORC_Q_SPLIT3:
    case ORC_Q_SPLIT4: orc_split(x, s, 11, hi, lo); break;
    case ORC_Q_SPLIT1: orc_split(x, s, 0, hi, lo); break;
    default: *hi = x; break;
  }
}

/* Element (r, c) of a matrix stored with leading dimension ld:
 * row-major -> r*ld + c, column-major -> c*ld + r. */
static int64_t elem_index(int64_t r, int64_t c, int64_t ld, int col_major) {
  return col_major ? c * ld + r : r * ld + c;
}

/* Quantise a rows x cols operand (any storage, any layout) into logical
 * row-major binary64 arrays hi and lo (lo may be NULL when unused). */
void orc_quantize(const void* src, int type, int64_t rows, int64_t cols,
                  int64_t ld, int col_major, int q, int s,
                  double* hi, double* lo) {
  for (int64_t r = 0; r < rows; ++r)
    for (int64_t c = 0; c < cols; ++c) {
      double h, l;
      quant_elem(load_elem(src, type, elem_index(r, c, ld, col_major)), q, s, &h, &l);
      hi[r * cols + c] = h;
      if (lo) lo[r * cols + c] = l;
    }
}

/* ------------------------------------------------------------------------- */
/* The product                                                                  */
/* ------------------------------------------------------------------------- */

typedef struct {
  int64_t m, n, k;
  const double *Ahi, *Alo, *Bhi, *Blo;  /* logical row-major m*k and k*n */
  int split;                             /* 1: hi*hi + hi*lo + lo*hi; 2: also lo*lo */
  const float* C0; int64_t ldc0;
  double alpha, beta;
  double *ref, *den; int64_t ldr;
  int64_t row_begin, row_end;
} full_job;

/* For each output row i: ref[i, :] = alpha * sum_k a(i,k) b(k,:) + beta*C0,
 * den[i, :] = |alpha| * sum_k |a(i,k)| |b(k,:)| + |beta| |C0|.
 * The k sum runs in ascending order for every output element. */
static void* full_worker(void* arg) {
  full_job* J = (full_job*)arg;
  int64_t n = J->n, k = J->k;
  double* acc = (double*)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  double* dac = (double*)calloc((size_t)(n > 0 ? n : 1), sizeof(double));
  for (int64_t i = J->row_begin; i < J->row_end; ++i) {
    memset(acc, 0, sizeof(double) * (size_t)n);
    memset(dac, 0, sizeof(double) * (size_t)n);
    for (int64_t kk = 0; kk < k; ++kk) {
      double ah = J->Ahi[i * k + kk];
      double al = J->split ? J->Alo[i * k + kk] : 0.0;
      double aabs = fabs(ah + al);
      const double* bh = J->Bhi + kk * n;
      if (J->split == 2) {
        const double* bl = J->Blo + kk * n;
        for (int64_t j = 0; j < n; ++j) {
          acc[j] += ah * bh[j] + ah * bl[j] + al * bh[j] + al * bl[j];
          dac[j] += aabs * fabs(bh[j] + bl[j]);
        }
      } else if (J->split) {
        const double* bl = J->Blo + kk * n;
        for (int64_t j = 0; j < n; ++j) {
          acc[j] += ah * bh[j] + ah * bl[j] + al * bh[j];
          dac[j] += aabs * fabs(bh[j] + bl[j]);
        }
      } else {
        for (int64_t j = 0; j < n; ++j) {
          acc[j] += ah * bh[j];
          dac[j] += aabs * fabs(bh[j]);
        }
      }
    }
    for (int64_t j = 0; j < n; ++j) {
      double c0 = (J->beta != 0.0 && J->C0) ? (double)J->C0[i * J->ldc0 + j] : 0.0;
      J->ref[i * J->ldr + j] = J->alpha * acc[j] + J->beta * c0;
      if (J->den) J->den[i * J->ldr + j] = fabs(J->alpha) * dac[j] + fabs(J->beta) * fabs(c0);
    }
  }
  free(acc);
  free(dac);
  return NULL;
}

static int resolve_threads(int nthreads) {
  if (nthreads > 0) return nthreads;
  long p = sysconf(_SC_NPROCESSORS_ONLN);
  return p > 0 ? (int)p : 1;
}

/* Full-grid reference on pre-quantised binary64 operands. */
int orc_gemm_f64(int64_t m, int64_t n, int64_t k,
                 const double* Ahi, const double* Alo,
                 const double* Bhi, const double* Blo, int split,
                 const float* C0, int64_t ldc0, double alpha, double beta,
                 double* ref, double* den, int64_t ldr, int nthreads) {
  if (m < 0 || n < 0 || k < 0) return -1;
  int T = resolve_threads(nthreads);
  if (T > m) T = (int)(m > 0 ? m : 1);
  full_job* jobs = (full_job*)calloc((size_t)T, sizeof(full_job));
  pthread_t* th = (pthread_t*)calloc((size_t)T, sizeof(pthread_t));
  int64_t per = (m + T - 1) / T;
  for (int t = 0; t < T; ++t) {
    full_job J = {m, n, k, Ahi, Alo, Bhi, Blo, split, C0, ldc0, alpha, beta,
                  ref, den, ldr, t * per, (t + 1) * per < m ? (t + 1) * per : m};
    if (J.row_begin > m) J.row_begin = m;
    jobs[t] = J;
    pthread_create(&th[t], NULL, full_worker, &jobs[t]);
  }
  for (int t = 0; t < T; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* Selected output elements, operands quantised on the fly                     */
/* ------------------------------------------------------------------------- */

typedef struct {
  int64_t k;
  const void* A; int a_type; int64_t lda; int a_cm; int a_q; int a_s;
  const void* B; int b_type; int64_t ldb; int b_cm; int b_q; int b_s;
  const float* C0; int64_t ldc0;
  double alpha, beta;
  const int64_t *rows, *cols;
  double *ref, *den;
  int64_t p_begin, p_end;
} pts_job;

static void* pts_worker(void* arg) {
  pts_job* J = (pts_job*)arg;
  int splitA = (J->a_q == ORC_Q_SPLIT3 || J->a_q == ORC_Q_SPLIT1 || J->a_q == ORC_Q_SPLIT4);
  int four = (J->a_q == ORC_Q_SPLIT4);
  for (int64_t p = J->p_begin; p < J->p_end; ++p) {
    int64_t i = J->rows[p], j = J->cols[p];
    double acc = 0.0, dac = 0.0;
    for (int64_t kk = 0; kk < J->k; ++kk) {
      double ah, al, bh, bl;
      quant_elem(load_elem(J->A, J->a_type, elem_index(i, kk, J->lda, J->a_cm)), J->a_q, J->a_s, &ah, &al);
      quant_elem(load_elem(J->B, J->b_type, elem_index(kk, j, J->ldb, J->b_cm)), J->b_q, J->b_s, &bh, &bl);
      if (four) acc += ah * bh + ah * bl + al * bh + al * bl;
      else if (splitA) acc += ah * bh + ah * bl + al * bh;
      else acc += ah * bh;
      dac += fabs(ah + al) * fabs(bh + bl);
    }
    double c0 = (J->beta != 0.0 && J->C0) ? (double)J->C0[i * J->ldc0 + j] : 0.0;
    J->ref[p] = J->alpha * acc + J->beta * c0;
    if (J->den) J->den[p] = fabs(J->alpha) * dac + fabs(J->beta) * fabs(c0);
  }
  return NULL;
}

/* Reference values of the listed output elements (row-major C0 with ldc0).
 * A is m x k and B is k x n in their own storage type and layout; each is
 * quantised element by element as it is read. */
int orc_gemm_points(int64_t k,
                    const void* A, int a_type, int64_t lda, int a_col_major, int a_q, int a_s,
                    const void* B, int b_type, int64_t ldb, int b_col_major, int b_q, int b_s,
                    const float* C0, int64_t ldc0, double alpha, double beta,
                    int64_t npts, const int64_t* rows, const int64_t* cols,
                    double* ref, double* den, int nthreads) {
  if (k < 0 || npts < 0) return -1;
  int T = resolve_threads(nthreads);
  if (T > npts) T = (int)(npts > 0 ? npts : 1);
  pts_job* jobs = (pts_job*)calloc((size_t)T, sizeof(pts_job));
  pthread_t* th = (pthread_t*)calloc((size_t)T, sizeof(pthread_t));
  int64_t per = (npts + T - 1) / T;
  for (int t = 0; t < T; ++t) {
    int64_t b = t * per, e = (t + 1) * per;
    if (b > npts) b = npts;
    if (e > npts) e = npts;
    pts_job J = {k, A, a_type, lda, a_col_major, a_q, a_s,
                 B, b_type, ldb, b_col_major, b_q, b_s,
                 C0, ldc0, alpha, beta, rows, cols, ref, den, b, e};
    jobs[t] = J;
    pthread_create(&th[t], NULL, pts_worker, &jobs[t]);
  }
  for (int t = 0; t < T; ++t) pthread_join(th[t], NULL);
  free(jobs);
  free(th);
  return 0;
}

/* ------------------------------------------------------------------------- */
/* The plain fp32 comparator's own result                                      */
/* ------------------------------------------------------------------------- */

/* "tile_matmul(): use the cuBLASDx register-accumulator API ...", spike
 * results, second bullet: fp32 has no matrix instruction, so the fp32 product
 * is a chain of scalar fused multiply-adds.  Reading (listed in the design
 * notes): each output element is ONE chain in fp32, k ascending from an
 * accumulator of +0, each step one correctly rounded fmaf, then
 * out = alpha*acc rounded to fp32 when beta == 0 (C0 is not read), else
 * fmaf(beta, C0, alpha*acc).  A and B are row-major fp32 (m x k, k x n),
 * C0 row-major with ldc0 (may be NULL when beta == 0), out row-major m x n. */
int orc_gemm_fma_chain_f32(int64_t m, int64_t n, int64_t k, const float* A, const float* B,
                           const float* C0, int64_t ldc0, float alpha, float beta, float* out) {
  if (m < 0 || n < 0 || k < 0) return -1;
  if (beta != 0.0f && !C0) return -1;
  for (int64_t i = 0; i < m; ++i)
    for (int64_t j = 0; j < n; ++j) {
      float acc = 0.0f;
      for (int64_t kk = 0; kk < k; ++kk) acc = fmaf(A[i * k + kk], B[kk * n + j], acc);
      const float t = alpha * acc;
      out[i * n + j] = (beta != 0.0f) ? fmaf(beta, C0[i * ldc0 + j], t) : t;
    }
  return 0;
}

/* ------------------------------------------------------------------------- */
/* The m16n8k16 f32 accumulator fragment, from the PTX row/col formulas        */
/* ------------------------------------------------------------------------- */

/* Lane `lane` (0..31) holds four f32 values j = 0..3 of the 16x8 tile.
 * groupID = lane / 4, threadID_in_group = lane % 4;
 * row = groupID + 8 * (j / 2), col = 2 * threadID_in_group + (j % 2). */
int orc_acc_coords(int lane, int j, int* row, int* col) {
  if (lane < 0 || lane > 31 || j < 0 || j > 3) return -1;
  int group = lane / 4, tig = lane % 4;
  *row = group + 8 * (j / 2);
  *col = 2 * tig + (j % 2);
  return 0;
}

/* The m16n8k16 operand fragments, from the PTX ISA operand layouts
 * (groupID = lane / 4, threadID_in_group = lane % 4):
 *   A (row): register r of a lane holds two consecutive columns;
 *     r = 0: row g,   cols 2t, 2t+1      r = 1: row g+8, cols 2t, 2t+1
 *     r = 2: row g,   cols 2t+8, 2t+9    r = 3: row g+8, cols 2t+8, 2t+9
 *   B (col): r = 0: rows (k) 2t, 2t+1 of column g; r = 1: rows 2t+8, 2t+9.
 * Value i of a lane is half i % 2 of register i / 2. */
int orc_frag_a_coords(int lane, int i, int* row, int* col) {
  if (lane < 0 || lane > 31 || i < 0 || i > 7) return -1;
  int g = lane / 4, t = lane % 4, r = i / 2, h = i % 2;
  *row = g + ((r == 1 || r == 3) ? 8 : 0);
  *col = 2 * t + h + ((r >= 2) ? 8 : 0);
  return 0;
}

int orc_frag_b_coords(int lane, int i, int* k, int* n) {
  if (lane < 0 || lane > 31 || i < 0 || i > 3) return -1;
  int g = lane / 4, t = lane % 4, r = i / 2, h = i % 2;
  *k = 2 * t + h + (r == 1 ? 8 : 0);
  *n = g;
  return 0;
}

/* ------------------------------------------------------------------------- */
/* attention: scores, row softmax, weighted sum of values                      */
/* ------------------------------------------------------------------------- */
/* For every query row i (q is lq x d, k is lk x d, v is lk x dv, all
 * row-major and dense, values in binary64 after whatever quantisation the
 * caller applied):
 *   s_ij   = scale * sum_t q_it k_jt                 (t ascending)
 *   p_ij   = exp(s_ij - max_j s_ij) / sum_j exp(s_ij - max_j s_ij)
 *   o_it   = sum_j p_ij v_jt                          (j ascending)
 *   den_it = sum_j p_ij |v_jt|
 * The maximum is subtracted before exp so that no term overflows; it cancels
 * in the quotient. */
typedef struct {
  int64_t lq, lk, d, dv, r0, r1;
  const double *q, *k, *v;
  double scale;
  double *o, *den;
  int ok;
} att_task;

static void* att_worker(void* arg) {
  att_task* t = (att_task*)arg;
  double* s = (double*)malloc((size_t)(t->lk > 0 ? t->lk : 1) * sizeof(double));
  if (!s) { t->ok = 0; return NULL; }
  for (int64_t i = t->r0; i < t->r1; ++i) {
    const double* qi = t->q + i * t->d;
    double mx = -INFINITY;
    for (int64_t j = 0; j < t->lk; ++j) {
      const double* kj = t->k + j * t->d;
      double acc = 0.0;
      for (int64_t c = 0; c < t->d; ++c) acc += qi[c] * kj[c];
      s[j] = t->scale * acc;
      if (s[j] > mx) mx = s[j];
    }
    double sum = 0.0;
    for (int64_t j = 0; j < t->lk; ++j) {
      s[j] = exp(s[j] - mx);
      sum += s[j];
    }
    double* oi = t->o + i * t->dv;
    double* di = t->den + i * t->dv;
    for (int64_t c = 0; c < t->dv; ++c) { oi[c] = 0.0; di[c] = 0.0; }
    for (int64_t j = 0; j < t->lk; ++j) {
      const double pj = s[j] / sum;
      const double* vj = t->v + j * t->dv;
      for (int64_t c = 0; c < t->dv; ++c) {
        oi[c] += pj * vj[c];
        di[c] += pj * fabs(vj[c]);
      }
    }
  }
  free(s);
  return NULL;
}

int orc_attention_f64(int64_t lq, int64_t lk, int64_t d, int64_t dv, const double* q, const double* k,
                      const double* v, double scale, double* o, double* den, int nthreads) {
  if (lq < 0 || lk < 1 || d < 1 || dv < 1) return -1;
  int nt = resolve_threads(nthreads);
  if (nt > lq) nt = (int)(lq > 0 ? lq : 1);
  att_task* tasks = (att_task*)calloc((size_t)nt, sizeof(att_task));
  pthread_t* th = (pthread_t*)calloc((size_t)nt, sizeof(pthread_t));
  if (!tasks || !th) { free(tasks); free(th); return -2; }
  for (int i = 0; i < nt; ++i) {
    att_task* t = &tasks[i];
    t->lq = lq; t->lk = lk; t->d = d; t->dv = dv; t->q = q; t->k = k; t->v = v; t->scale = scale;
    t->o = o; t->den = den; t->ok = 1;
    t->r0 = lq * i / nt;
    t->r1 = lq * (i + 1) / nt;
    pthread_create(&th[i], NULL, att_worker, t);
  }
  int ok = 1;
  for (int i = 0; i < nt; ++i) {
    pthread_join(th[i], NULL);
    ok &= tasks[i].ok;
  }
  free(tasks);
  free(th);
  return ok ? 0 : -2;
}
