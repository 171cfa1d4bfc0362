/*
 * bi_oracle.c -- plain fp64 CPU oracle for the batch-invariant contractions.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header or table with the CUDA library.
 *
 * What it computes is the plain definition of each operation, written out:
 *
 *  - mm / addmm / bmm: c[m,n] = alpha * sum_k a[m,k]*b[k,n] (+ bias[n]).
 *    "Batch-Invariant VLAs" (section "Thinky's Ops were not enough") and
 *    "Unmasking the True Culprit" (section "Implementation Analysis: the
 *    matmul_persistent function") define mm as the plain matrix product and
 *    addmm as mm plus a bias broadcast over rows; "Batch-Invariant Kernel
 *    Design" (section "Kernel 2: Attention BMM") defines bmm as one
 *    independent matrix product per flattened batch*head element.
 *  - conv2d: the direct definition of a non-transposed 2-D convolution with
 *    stride, padding, dilation and groups ("Batch-Invariant Kernel Design",
 *    section "Kernel 1: Conv2d"), and separately the unfold + matrix product
 *    form that "Batch-Invariant VLAs" (section "Replacing nn.Conv2d") uses.
 *  - softmax over the last dimension: p_j = exp(s_j - max s) / sum_i exp(s_i - max s)
 *    (one row at a time, "ai-infra handbook: deterministic inference",
 *    section on normalisation and softmax reductions).
 *  - row reductions of "Unmasking the True Culprit" (section "Beyond Matrix
 *    Multiplication: Other Critical Operations"): RMSNorm
 *    y_j = x_j * (1 / sqrt(mean_i x_i^2 + eps)) * w_j, log-softmax
 *    y_j = (x_j - max x) - log(sum_i exp(x_i - max x)), and the mean over the
 *    last dimension (aten::mean.dim, "Batch-Invariant VLAs").
 *  - attention: o[i,:] = sum_j softmax_j(scale * q_i . k_j) v[j,:] per query
 *    row i of each head, the whole key range at once ("ai-infra handbook:
 *    deterministic inference", section on fixed splitting, attention: the
 *    key/value range is split by a fixed length or not at all, and the
 *    result must not depend on how the queries are chunked).
 *
 * Inputs are the exact bf16 (or, for the products, fp16) bit patterns
 * handed to the GPU, widened to double.  Every output element is accumulated on one thread, sequentially
 * over ascending reduction index, in double precision.  OpenMP only splits
 * the work over output rows, so results do not depend on the thread count.
 * Rounding to the output type happens once, round-to-nearest-even.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* bf16 / fp32 conversions                                             */
/* ------------------------------------------------------------------ */

/* bf16 bits -> double, exactly (bf16 is the top half of an fp32). */
static double bf16_to_double(uint16_t h) {
  uint32_t u = ((uint32_t)h) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

static double g_bf16_table[65536];
static int g_table_ready = 0;

static void ensure_table(void) {
  if (g_table_ready) return;
  for (uint32_t i = 0; i < 65536u; ++i) g_bf16_table[i] = bf16_to_double((uint16_t)i);
  g_table_ready = 1;
}

/* Exposed so the tests can pin it against an independent conversion. */
double bio_bf16_bits_to_double(uint16_t h) { return bf16_to_double(h); }

/*
 * IEEE 754 binary16 bits -> double, exactly, from the format's definition:
 * 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; exponent 0 is
 * zero / subnormal (fraction * 2^-24), exponent 31 is infinity / NaN.
 */
static double f16_to_double(uint16_t h) {
  const int sign = (h >> 15) & 1;
  const int e = (h >> 10) & 31;
  const int f = h & 1023;
  double v;
  if (e == 0)
    v = ldexp((double)f, -24);
  else if (e == 31)
    v = f ? NAN : INFINITY;
  else
    v = ldexp((double)(1024 + f), e - 25);
  return sign ? -v : v;
}

static double g_f16_table[65536];
static int g_f16_ready = 0;

static void ensure_f16_table(void) {
  if (g_f16_ready) return;
  for (uint32_t i = 0; i < 65536u; ++i) g_f16_table[i] = f16_to_double((uint16_t)i);
  g_f16_ready = 1;
}

double bio_f16_bits_to_double(uint16_t h) { return f16_to_double(h); }

/*
 * double -> bf16 bits with ONE round-to-nearest-even step.
 * bf16: 1 sign bit, 8 exponent bits (same range as fp32), 8 significant bits.
 * Normal numbers: the quantum is 2^(E-8) for |x| in [2^(E-1), 2^E).
 * Subnormals (|x| < 2^-126): fixed quantum 2^-133.
 */
static uint16_t double_to_bf16_bits(double x) {
  if (isnan(x)) return (uint16_t)0x7FC0;
  uint16_t sign = signbit(x) ? 0x8000u : 0u;
  double ax = fabs(x);
  if (isinf(ax)) return (uint16_t)(sign | 0x7F80u);
  if (ax == 0.0) return sign;
  double r;
  if (ax < ldexp(1.0, -126)) {
    r = rint(ldexp(ax, 133));          /* ties-to-even under the default mode */
    r = ldexp(r, -133);
  } else {
    int e;
    double f = frexp(ax, &e);          /* ax = f * 2^e, f in [0.5, 1) */
    double q = rint(ldexp(f, 8));      /* 8 significant bits */
    r = ldexp(q, e - 8);
  }
  if (r >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80u);
  float fr = (float)r;                 /* exact: r has <= 8 significant bits */
  uint32_t u;
  memcpy(&u, &fr, sizeof u);
  return (uint16_t)(sign | (uint16_t)(u >> 16));
}

void bio_round_bf16(const double* x, uint16_t* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = double_to_bf16_bits(x[i]);
}

/* double -> fp32, one RNE rounding (C's conversion under the default mode). */
void bio_round_f32(const double* x, float* out, int64_t n) {
  for (int64_t i = 0; i < n; ++i) out[i] = (float)x[i];
}

/* ------------------------------------------------------------------ */
/* Sequential sums, in the order written (used by the pins).          */
/* ------------------------------------------------------------------ */

double bio_sum_seq_f64(const double* x, int64_t n) {
  double s = 0.0;
  for (int64_t i = 0; i < n; ++i) s = s + x[i];
  return s;
}

float bio_sum_seq_f32(const float* x, int64_t n) {
  float s = 0.0f;
  for (int64_t i = 0; i < n; ++i) s = s + x[i];
  return s;
}

int bio_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* ------------------------------------------------------------------ */
/* Matrix products                                                     */
/* ------------------------------------------------------------------ */

/*
 * One output row: c_row[n] = alpha * sum_k a_row[k] b[k,n] (+ bias[n]).
 * The k loop is outermost so each c_row[n] still receives its terms one at
 * a time in ascending k; abs_row[n] = sum_k |a b| (+ |bias|) is the scale
 * of the error bound.  acc / acc_abs are scratch rows of length N.
 */
static void mm_row(int64_t N, int64_t K, const double* tab,
                   const uint16_t* a_row, int64_t sa_k,
                   const uint16_t* b, int64_t sb_k, int64_t sb_n,
                   const double* bias_tab, const uint16_t* bias, int64_t s_bias, double alpha,
                   double* c_row, double* abs_row, double* acc, double* acc_abs) {
  for (int64_t n = 0; n < N; ++n) { acc[n] = 0.0; acc_abs[n] = 0.0; }
  for (int64_t k = 0; k < K; ++k) {
    double av = tab[a_row[k * sa_k]];
    const uint16_t* brow = b + k * sb_k;
    for (int64_t n = 0; n < N; ++n) {
      double p = av * tab[brow[n * sb_n]];   /* exact in double */
      acc[n] = acc[n] + p;
      acc_abs[n] = acc_abs[n] + fabs(p);
    }
  }
  for (int64_t n = 0; n < N; ++n) {
    double v = alpha * acc[n];
    double va = fabs(alpha) * acc_abs[n];
    if (bias) {
      double bv = bias_tab[bias[n * s_bias]];
      v = v + bv;
      va = va + fabs(bv);
    }
    c_row[n] = v;
    if (abs_row) abs_row[n] = va;
  }
}

/*
 * c [R,N] (row-major, fp64) = alpha * a [M,K] @ b [K,N] (+ bias [N]).
 * Strides are in elements; a transposed operand is a stride swap.
 * in_f16: a and b hold fp16 bits (else bf16); bias_f16: likewise for bias.
 * rows: optional list of n_rows output rows to compute (for sampled checks
 * of very large products); output row i then holds row rows[i].  NULL means
 * all M rows in order.
 */
void bio_mm(int64_t M, int64_t N, int64_t K, int in_f16,
            const uint16_t* a, int64_t sa_m, int64_t sa_k,
            const uint16_t* b, int64_t sb_k, int64_t sb_n,
            int bias_f16, const uint16_t* bias, int64_t s_bias, double alpha,
            const int64_t* rows, int64_t n_rows,
            double* c, double* absum) {
  ensure_table();
  ensure_f16_table();
  const double* tab = in_f16 ? g_f16_table : g_bf16_table;
  const double* bias_tab = bias_f16 ? g_f16_table : g_bf16_table;
  int64_t R = rows ? n_rows : M;
  size_t row_bytes = sizeof(double) * (size_t)(N > 0 ? N : 1);
#pragma omp parallel
  {
    double* acc = (double*)malloc(row_bytes);
    double* acc_abs = (double*)malloc(row_bytes);
#pragma omp for schedule(dynamic, 1)
    for (int64_t i = 0; i < R; ++i) {
      int64_t m = rows ? rows[i] : i;
      mm_row(N, K, tab, a + m * sa_m, sa_k, b, sb_k, sb_n, bias_tab, bias, s_bias, alpha,
             c + i * N, absum ? absum + i * N : NULL, acc, acc_abs);
    }
    free(acc);
    free(acc_abs);
  }
}

/*
 * Batched product: for l in [0, L): c[l] = alpha * a[l] @ b[l].
 * c is [L, M, N] contiguous fp64.  Each batch element is an independent mm.
 */
void bio_bmm(int64_t L, int64_t M, int64_t N, int64_t K, int in_f16,
             const uint16_t* a, int64_t sa_l, int64_t sa_m, int64_t sa_k,
             const uint16_t* b, int64_t sb_l, int64_t sb_k, int64_t sb_n,
             double alpha, double* c, double* absum) {
  ensure_table();
  ensure_f16_table();
  const double* tab = in_f16 ? g_f16_table : g_bf16_table;
  size_t row_bytes = sizeof(double) * (size_t)(N > 0 ? N : 1);
#pragma omp parallel
  {
    double* acc = (double*)malloc(row_bytes);
    double* acc_abs = (double*)malloc(row_bytes);
#pragma omp for collapse(2) schedule(dynamic, 1)
    for (int64_t l = 0; l < L; ++l) {
      for (int64_t m = 0; m < M; ++m) {
        int64_t o = (l * M + m) * N;
        mm_row(N, K, tab, a + l * sa_l + m * sa_m, sa_k, b + l * sb_l, sb_k, sb_n,
               tab, NULL, 0, alpha, c + o, absum ? absum + o : NULL, acc, acc_abs);
      }
    }
    free(acc);
    free(acc_abs);
  }
}

/* ------------------------------------------------------------------ */
/* Convolution                                                         */
/* ------------------------------------------------------------------ */

static int64_t conv_out_size(int64_t in, int64_t k, int64_t s, int64_t p, int64_t d) {
  return (in + 2 * p - d * (k - 1) - 1) / s + 1;
}

int64_t bio_conv_out_size(int64_t in, int64_t k, int64_t s, int64_t p, int64_t d) {
  return conv_out_size(in, k, s, p, d);
}

/*
 * Direct convolution.  x [B,C,H,W], w [Co, C/groups, KH, KW], bias [Co] or
 * NULL, all contiguous bf16 bits.  y [B,Co,Ho,Wo] fp64 contiguous.
 * y[b,co,oh,ow] = bias[co] + sum over (ci in the group of co, kh, kw), in
 * that nesting order, of x[b, ci, oh*sh - ph + kh*dh, ow*sw - pw + kw*dw]
 * * w[co, ci_local, kh, kw]; positions outside the image contribute zero.
 */
void bio_conv2d(int64_t B, int64_t C, int64_t H, int64_t W,
                int64_t Co, int64_t KH, int64_t KW,
                int64_t sh, int64_t sw, int64_t ph, int64_t pw, int64_t dh, int64_t dw,
                int64_t groups,
                const uint16_t* x, const uint16_t* w, const uint16_t* bias,
                double* y, double* absum) {
  ensure_table();
  int64_t Ho = conv_out_size(H, KH, sh, ph, dh);
  int64_t Wo = conv_out_size(W, KW, sw, pw, dw);
  int64_t Cig = C / groups, Cog = Co / groups;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int64_t b = 0; b < B; ++b) {
    for (int64_t co = 0; co < Co; ++co) {
      int64_t g = co / Cog;
      for (int64_t oh = 0; oh < Ho; ++oh) {
        for (int64_t ow = 0; ow < Wo; ++ow) {
          double acc = 0.0, acc_abs = 0.0;
          for (int64_t cl = 0; cl < Cig; ++cl) {
            int64_t ci = g * Cig + cl;
            for (int64_t kh = 0; kh < KH; ++kh) {
              int64_t ih = oh * sh - ph + kh * dh;
              for (int64_t kw = 0; kw < KW; ++kw) {
                int64_t iw = ow * sw - pw + kw * dw;
                double xv = 0.0;
                if (ih >= 0 && ih < H && iw >= 0 && iw < W)
                  xv = g_bf16_table[x[((b * C + ci) * H + ih) * W + iw]];
                double wv = g_bf16_table[w[((co * Cig + cl) * KH + kh) * KW + kw]];
                double p = xv * wv;
                acc = acc + p;
                acc_abs = acc_abs + fabs(p);
              }
            }
          }
          if (bias) {
            double bv = g_bf16_table[bias[co]];
            acc = acc + bv;
            acc_abs = acc_abs + fabs(bv);
          }
          int64_t o = ((b * Co + co) * Ho + oh) * Wo + ow;
          y[o] = acc;
          if (absum) absum[o] = acc_abs;
        }
      }
    }
  }
}

/*
 * Explicit unfold (im2col), the layout torch.nn.functional.unfold produces:
 * cols [B, C*KH*KW, Ho*Wo] bf16 bits, row index k = (ci*KH + kh)*KW + kw,
 * column index l = oh*Wo + ow, zero where the window leaves the image.
 */
void bio_unfold(int64_t B, int64_t C, int64_t H, int64_t W, int64_t KH, int64_t KW,
                int64_t sh, int64_t sw, int64_t ph, int64_t pw, int64_t dh, int64_t dw,
                const uint16_t* x, uint16_t* cols) {
  int64_t Ho = conv_out_size(H, KH, sh, ph, dh);
  int64_t Wo = conv_out_size(W, KW, sw, pw, dw);
  int64_t Kd = C * KH * KW, L = Ho * Wo;
  for (int64_t b = 0; b < B; ++b)
    for (int64_t ci = 0; ci < C; ++ci)
      for (int64_t kh = 0; kh < KH; ++kh)
        for (int64_t kw = 0; kw < KW; ++kw) {
          int64_t k = (ci * KH + kh) * KW + kw;
          for (int64_t oh = 0; oh < Ho; ++oh)
            for (int64_t ow = 0; ow < Wo; ++ow) {
              int64_t ih = oh * sh - ph + kh * dh, iw = ow * sw - pw + kw * dw;
              uint16_t v = 0;
              if (ih >= 0 && ih < H && iw >= 0 && iw < W) v = x[((b * C + ci) * H + ih) * W + iw];
              cols[(b * Kd + k) * L + oh * Wo + ow] = v;
            }
        }
}

/* ------------------------------------------------------------------ */
/* Row softmax                                                         */
/* ------------------------------------------------------------------ */

/*
 * s [R, N] fp32 with row stride ss (elements); p [R, N] fp64 contiguous.
 * Per row: mx = max_j s_j; e_j = exp(s_j - mx); p_j = e_j / sum_j e_j,
 * all in double, the sum taken in ascending j.
 */
void bio_softmax_rows(int64_t R, int64_t N, const float* s, int64_t ss, double* p) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    const float* row = s + r * ss;
    double mx = -INFINITY;
    for (int64_t j = 0; j < N; ++j)
      if ((double)row[j] > mx) mx = (double)row[j];
    double sum = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      double e = exp((double)row[j] - mx);
      p[r * N + j] = e;
      sum = sum + e;
    }
    for (int64_t j = 0; j < N; ++j) p[r * N + j] = p[r * N + j] / sum;
  }
}

/* ------------------------------------------------------------------ */
/* Row reductions over the last dimension (doubles in, doubles out)   */
/* ------------------------------------------------------------------ */

/*
 * RMSNorm of each row of x [R, N] (row stride sx): ms = (sum_j x_j^2) / N in
 * ascending j, r = 1 / sqrt(ms + eps), y_j = (x_j * r) * w_j (w NULL: 1).
 * y [R, N] contiguous.
 */
void bio_rmsnorm_rows(int64_t R, int64_t N, const double* x, int64_t sx, const double* w,
                      double eps, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    const double* xr = x + r * sx;
    double ss = 0.0;
    for (int64_t j = 0; j < N; ++j) ss = ss + xr[j] * xr[j];
    const double rinv = 1.0 / sqrt(ss / (double)N + eps);
    for (int64_t j = 0; j < N; ++j) y[r * N + j] = (xr[j] * rinv) * (w ? w[j] : 1.0);
  }
}

/*
 * Log-softmax of each row of s [R, N]: m = max_j s_j,
 * lse = log(sum_j exp(s_j - m)) in ascending j, y_j = (s_j - m) - lse.
 */
void bio_log_softmax_rows(int64_t R, int64_t N, const double* s, int64_t ss, double* y) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    const double* sr = s + r * ss;
    double m = -INFINITY;
    for (int64_t j = 0; j < N; ++j) m = sr[j] > m ? sr[j] : m;
    double sum = 0.0;
    for (int64_t j = 0; j < N; ++j) sum = sum + exp(sr[j] - m);
    const double lse = log(sum);
    for (int64_t j = 0; j < N; ++j) y[r * N + j] = (sr[j] - m) - lse;
  }
}

/* Mean of each row of x [R, N]: (sum_j x_j in ascending j) / N; absum: sum_j |x_j| / N. */
void bio_mean_rows(int64_t R, int64_t N, const double* x, int64_t sx, double* y, double* absum) {
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    const double* xr = x + r * sx;
    double sum = 0.0, sa = 0.0;
    for (int64_t j = 0; j < N; ++j) {
      sum = sum + xr[j];
      sa = sa + fabs(xr[j]);
    }
    y[r] = sum / (double)N;
    if (absum) absum[r] = sa / (double)N;
  }
}

/* ------------------------------------------------------------------ */
/* Attention (doubles in, doubles out)                                */
/* ------------------------------------------------------------------ */

/*
 * q [L, Tq, D], k and v [L, Tk, D], all contiguous.  Per head l and query
 * row i:
 *   s_j   = scale * sum_d q[i,d] * k[j,d]       (ascending d)
 *   m     = max_j s_j
 *   e_j   = exp(s_j - m),  den = sum_j e_j      (ascending j)
 *   o[i,d]     = (sum_j e_j * v[j,d]) / den     (ascending j)
 *   absum[i,d] = (sum_j e_j * |v[j,d]|) / den   (the size of the terms)
 *   smax[i]    = scale * max_j sum_d |q[i,d] * k[j,d]|
 * absum and smax feed the tests' error bounds; either may be NULL.
 */
void bio_attention(int64_t L, int64_t Tq, int64_t Tk, int64_t D, const double* q, const double* k,
                   const double* v, double scale, double* o, double* absum, double* smax) {
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t row = 0; row < L * Tq; ++row) {
    const int64_t l = row / Tq;
    const double* qi = q + row * D;
    const double* kl = k + l * Tk * D;
    const double* vl = v + l * Tk * D;
    double* e = (double*)malloc((size_t)Tk * sizeof(double));
    double m = -INFINITY, sm = 0.0;
    for (int64_t j = 0; j < Tk; ++j) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t d = 0; d < D; ++d) {
        acc = acc + qi[d] * kl[j * D + d];
        aacc = aacc + fabs(qi[d] * kl[j * D + d]);
      }
      e[j] = scale * acc;
      if (e[j] > m) m = e[j];
      if (fabs(scale) * aacc > sm) sm = fabs(scale) * aacc;
    }
    double den = 0.0;
    for (int64_t j = 0; j < Tk; ++j) {
      e[j] = exp(e[j] - m);
      den = den + e[j];
    }
    for (int64_t d = 0; d < D; ++d) {
      double num = 0.0, anum = 0.0;
      for (int64_t j = 0; j < Tk; ++j) {
        num = num + e[j] * vl[j * D + d];
        anum = anum + e[j] * fabs(vl[j * D + d]);
      }
      o[row * D + d] = num / den;
      if (absum) absum[row * D + d] = anum / den;
    }
    if (smax) smax[row] = sm;
    free(e);
  }
}
