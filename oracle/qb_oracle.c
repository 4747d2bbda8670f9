/*
 * qb_oracle.c -- plain CPU oracle for bias-based quantile balancing.
 *
 * TEST INFRASTRUCTURE ONLY (see qb_oracle.h).  Slow on purpose: per-token
 * full sorts, per-expert full sorts, direct counting.  Compiled with
 * -O2 -ffp-contract=off, never with -ffast-math.
 *
 * Parity pins (what each function is checked against, outside itself) are
 * listed in tests/test_oracle_*.py; every function here is pinned.
 */
#include "qb_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Pinned logistic function.                                                 */
/*                                                                           */
/* The pages name only "the raw sigmoid router score" ([QB-PR] "Quantile     */
/* estimator").  Histogram counts are integers decided by fp32 margins, so    */
/* the score must be one fixed, reproducible binary32 function.  This is it: */
/*                                                                           */
/*   x  = clamp(x, -104, 104)       (beyond, exp(-x) over/underflows anyway) */
/*   t  = fma(x, -L2E, M)           M = 1.5*2^23: n = t - M = rint(-x*log2 e)*/
/*   n  = t - M                     (exact)                                   */
/*   w  = fma(n, LN2_HI, x)         Cody & Waite (1980) two-part reduction:   */
/*   w  = fma(n, LN2_LO, w)         w = x + n*ln2, so exp(-x) = 2^n*exp(-w)   */
/*   p  = sum_{i=0..7} (-w)^i / i!  degree-7 Taylor polynomial of exp(-w),    */
/*                                  Horner form in w, one fma per degree,     */
/*                                  coefficients RN((-1)^i / i!)              */
/*   e  = RN(p * 2^n)               (one rounding; +inf when it overflows)    */
/*   s  = RN(1 / RN(1 + e))         (correctly rounded reciprocal)            */
/*                                                                           */
/* so s = 1/(1+exp(-x)); for x < -88.72 e overflows and s = 0 (the exact     */
/* value there is below 3e-39).                                              */
/* ------------------------------------------------------------------------ */

static const float kL2E = 0x1.715476p+0f;     /* RN(log2(e)) */
static const float kMagic = 0x1.8p+23f;       /* 12582912 */
static const float kLn2Hi = 0x1.62e4p-1f;     /* 0.693145751953125 */
static const float kLn2Lo = 0x1.7f7d1cp-20f;  /* RN(ln 2 - kLn2Hi) */

static const float kExpCoef[8] = {
    0x1.0p+0f,        /* +1/0! */
    -0x1.0p+0f,       /* -1/1! */
    0x1.0p-1f,        /* +1/2! */
    -0x1.555556p-3f,  /* -1/3! */
    0x1.555556p-5f,   /* +1/4! */
    -0x1.111112p-7f,  /* -1/5! */
    0x1.6c16c2p-10f,  /* +1/6! */
    -0x1.a01a02p-13f, /* -1/7! */
};

void orc_exp_coeffs(float* c8) {
  for (int i = 0; i < 8; ++i) c8[i] = kExpCoef[i];
}

float orc_exp_neg(float x) {
  float xc = x;
  if (xc > 104.0f) xc = 104.0f;
  if (xc < -104.0f) xc = -104.0f;
  float t = fmaf(xc, -kL2E, kMagic);
  float n = t - kMagic;
  float w = fmaf(n, kLn2Hi, xc);
  w = fmaf(n, kLn2Lo, w);
  float p = kExpCoef[7];
  for (int i = 6; i >= 0; --i) p = fmaf(p, w, kExpCoef[i]);
  /* RN(p * 2^n): the product is exact in binary64 (|n| <= 151), and the cast
   * to binary32 rounds it once (to +inf on overflow). */
  return (float)ldexp((double)p, (int)n);
}

float orc_sigmoid(float x) {
  float e = orc_exp_neg(x);
  float d = 1.0f + e;
  return 1.0f / d;
}

void orc_sigmoid_array(const float* x, float* s, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) s[i] = orc_sigmoid(x[i]);
}

/* ------------------------------------------------------------------------ */
/* BF16 rounding and the order-preserving key ([EQB] EQB paragraph).        */
/* ------------------------------------------------------------------------ */

static float f32_from_bits(uint32_t u) {
  float f;
  memcpy(&f, &u, 4);
  return f;
}

static uint32_t bits_from_f32(float f) {
  uint32_t u;
  memcpy(&u, &f, 4);
  return u;
}

/* Definition of round-to-nearest-even onto the bf16 grid: take the two bf16
 * magnitudes that bracket |r| (truncation toward zero, and the next one up),
 * compare the exact distances in binary64, and break an exact tie toward the
 * candidate with an even last mantissa bit.  Above the largest finite bf16
 * the upper candidate stands for 2^128 and becomes infinity, as IEEE-754
 * rounding with an unbounded exponent prescribes. */
uint16_t orc_bf16_rne(float r) {
  uint32_t u = bits_from_f32(r);
  uint32_t sign = u & 0x80000000u;
  uint32_t mag = u & 0x7FFFFFFFu;
  if (mag > 0x7F800000u) return (uint16_t)((sign >> 16) | 0x7FC0u); /* NaN */
  if (mag == 0x7F800000u) return (uint16_t)((sign >> 16) | 0x7F80u); /* inf */
  uint32_t lo = mag & 0xFFFF0000u;
  uint32_t hi = lo + 0x10000u;
  double vr = (double)f32_from_bits(mag);
  double vlo = (double)f32_from_bits(lo);
  double vhi = (hi == 0x7F800000u) ? ldexp(1.0, 128) : (double)f32_from_bits(hi);
  double dlo = vr - vlo;
  double dhi = vhi - vr;
  uint32_t pick;
  if (dlo < dhi)
    pick = lo;
  else if (dhi < dlo)
    pick = hi;
  else
    pick = ((lo >> 16) & 1u) ? hi : lo;
  return (uint16_t)((sign | pick) >> 16);
}

uint16_t orc_key(float r) {
  uint16_t h = orc_bf16_rne(r);
  if (h == 0x8000u) h = 0; /* -0 folds to +0 */
  return (h & 0x8000u) ? (uint16_t)(h ^ 0xFFFFu) : (uint16_t)(h ^ 0x8000u);
}

float orc_key_decode(uint16_t key) {
  uint16_t h = (key & 0x8000u) ? (uint16_t)(key ^ 0x8000u) : (uint16_t)(key ^ 0xFFFFu);
  return f32_from_bits((uint32_t)h << 16);
}

void orc_keys_array(const float* r, uint16_t* keys, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) keys[i] = orc_key(r[i]);
}

void orc_bf16_array(const float* r, uint16_t* bits, int64_t n) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) bits[i] = orc_bf16_rne(r[i]);
}

/* ------------------------------------------------------------------------ */
/* Routing: alpha, margins, top-k ([QB-PR] "Quantile estimator").            */
/* ------------------------------------------------------------------------ */

typedef struct {
  float v;
  int32_t j;
} vj_t;

/* v descending, then expert index ascending. */
static int cmp_vj(const void* pa, const void* pb) {
  const vj_t* a = (const vj_t*)pa;
  const vj_t* b = (const vj_t*)pb;
  if (a->v > b->v) return -1;
  if (a->v < b->v) return 1;
  return (a->j < b->j) ? -1 : (a->j > b->j);
}

static void route_token(const float* s, const float* bias, int E, int k, vj_t* buf,
                        float* alpha, float* margins, int32_t* topk) {
  for (int j = 0; j < E; ++j) {
    buf[j].v = s[j] + bias[j];
    buf[j].j = j;
  }
  qsort(buf, (size_t)E, sizeof(vj_t), cmp_vj);
  float a = buf[k].v; /* the (k+1)-th largest, counted with multiplicity */
  if (alpha) *alpha = a;
  if (margins)
    for (int j = 0; j < E; ++j) margins[j] = a - s[j];
  if (topk)
    for (int t = 0; t < k; ++t) topk[t] = buf[t].j;
}

static void route_impl(const float* logits, const uint16_t* logits_bf16, const float* bias,
                       int64_t N, int E, int k, float* alpha, float* scores, float* margins,
                       int32_t* topk) {
#pragma omp parallel
  {
    vj_t* buf = (vj_t*)malloc(sizeof(vj_t) * (size_t)E);
    float* s = (float*)malloc(sizeof(float) * (size_t)E);
#pragma omp for schedule(static)
    for (int64_t i = 0; i < N; ++i) {
      for (int j = 0; j < E; ++j) {
        float x = logits ? logits[i * E + j]
                         : f32_from_bits((uint32_t)logits_bf16[i * E + j] << 16);
        s[j] = orc_sigmoid(x);
      }
      if (scores) memcpy(scores + i * E, s, sizeof(float) * (size_t)E);
      route_token(s, bias, E, k, buf, alpha ? alpha + i : NULL,
                  margins ? margins + i * E : NULL, topk ? topk + i * k : NULL);
    }
    free(buf);
    free(s);
  }
}

void orc_route(const float* logits, const float* bias, int64_t N, int E, int k, float* alpha,
               float* scores, float* margins, int32_t* topk) {
  route_impl(logits, NULL, bias, N, E, k, alpha, scores, margins, topk);
}

void orc_route_bf16(const uint16_t* logits_bf16, const float* bias, int64_t N, int E, int k,
                    float* alpha, float* scores, float* margins, int32_t* topk) {
  route_impl(NULL, logits_bf16, bias, N, E, k, alpha, scores, margins, topk);
}

/* ------------------------------------------------------------------------ */
/* EQB: rank, histograms, selection, exact order statistic.                  */
/* ------------------------------------------------------------------------ */

int64_t orc_rank(int64_t n_pool, int E, int k) {
  return ((int64_t)k * n_pool + (int64_t)E - 1) / (int64_t)E;
}

void orc_hist_hi(const uint16_t* keys, int64_t N, int E, int32_t* hist_hi) {
#pragma omp parallel for schedule(static)
  for (int j = 0; j < E; ++j)
    for (int64_t i = 0; i < N; ++i) hist_hi[(int64_t)j * 256 + (keys[i * E + j] >> 8)] += 1;
}

void orc_hist_lo(const uint16_t* keys, int64_t N, int E, const int32_t* sel, int32_t* hist_lo) {
#pragma omp parallel for schedule(static)
  for (int j = 0; j < E; ++j)
    for (int64_t i = 0; i < N; ++i) {
      uint16_t key = keys[i * E + j];
      if ((int32_t)(key >> 8) == sel[j]) hist_lo[(int64_t)j * 256 + (key & 0xFF)] += 1;
    }
}

/* First bin b with sum_{b'<=b} h[b'] >= R; *before = sum_{b'<b} h[b'].
 * Returns -1 when the row holds fewer than R samples. */
static int first_bin_reaching(const int32_t* h, int nb, int64_t R, int64_t* before) {
  int64_t cum = 0;
  for (int b = 0; b < nb; ++b) {
    if (cum + h[b] >= R) {
      *before = cum;
      return b;
    }
    cum += h[b];
  }
  *before = cum;
  return -1;
}

void orc_select_hi(const int32_t* hist_hi, int E, int64_t R, int32_t* sel, int32_t* r_lo) {
  for (int j = 0; j < E; ++j) {
    int64_t before = 0;
    int b = first_bin_reaching(hist_hi + (int64_t)j * 256, 256, R, &before);
    sel[j] = b;
    r_lo[j] = (b < 0) ? 0 : (int32_t)(R - before);
  }
}

void orc_select_lo(const int32_t* hist_lo, int E, const int32_t* r_lo, int32_t* lo) {
  for (int j = 0; j < E; ++j) {
    int64_t before = 0;
    lo[j] = first_bin_reaching(hist_lo + (int64_t)j * 256, 256, r_lo[j], &before);
  }
}

static int cmp_u16(const void* pa, const void* pb) {
  uint16_t a = *(const uint16_t*)pa, b = *(const uint16_t*)pb;
  return (a > b) - (a < b);
}

void orc_kth_key_sort(const uint16_t* keys, int64_t n_pool, int E, int64_t R, uint16_t* qkey) {
#pragma omp parallel
  {
    uint16_t* col = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n_pool > 0 ? n_pool : 1));
#pragma omp for schedule(dynamic, 1)
    for (int j = 0; j < E; ++j) {
      for (int64_t i = 0; i < n_pool; ++i) col[i] = keys[i * E + j];
      qsort(col, (size_t)n_pool, sizeof(uint16_t), cmp_u16);
      qkey[j] = col[R - 1];
    }
    free(col);
  }
}

void orc_center(const double* q, int E, float* b_out) {
  double sum = 0.0;
  for (int j = 0; j < E; ++j) sum += q[j];
  double mu = sum / (double)E;
  for (int j = 0; j < E; ++j) b_out[j] = (float)(q[j] - mu);
}

/* ------------------------------------------------------------------------ */
/* K3 uniform histogram ([QB-PR] "Quantile estimator", "Implementation").    */
/* ------------------------------------------------------------------------ */

void orc_k3_hist(const float* margins, int64_t N, int E, float lo, float hi, int nbins,
                 int32_t* hist) {
  float w = hi - lo;
  float scale = (float)nbins / w;
#pragma omp parallel for schedule(static)
  for (int j = 0; j < E; ++j)
    for (int64_t i = 0; i < N; ++i) {
      float t = (margins[i * E + j] - lo) * scale;
      int idx;
      if (!(t >= 0.0f))
        idx = 0; /* below the range (or NaN): first bin */
      else if (t >= (float)nbins)
        idx = nbins - 1; /* at or above the top edge: last bin */
      else
        idx = (int)floorf(t);
      if (idx > nbins - 1) idx = nbins - 1;
      hist[(int64_t)j * nbins + idx] += 1;
    }
}

void orc_k3_finalize(const int32_t* hist, int E, int nbins, int64_t R, float lo, float hi,
                     float* b_out, float* bounds_out, double* q_out) {
  double dlo = (double)lo;
  double width = ((double)hi - dlo) / (double)nbins;
  double* q = (double*)malloc(sizeof(double) * (size_t)E);
  for (int j = 0; j < E; ++j) {
    int64_t before = 0;
    int b = first_bin_reaching(hist + (int64_t)j * nbins, nbins, R, &before);
    if (b < 0) {
      q[j] = (double)hi; /* fewer than R samples: not reachable for valid input */
      continue;
    }
    double edge = dlo + (double)b * width; /* lower edge of bin b */
    double frac = (double)(R - before) / (double)hist[(int64_t)j * nbins + b];
    q[j] = edge + width * frac;
  }
  orc_center(q, E, b_out);
  float mn = b_out[0], mx = b_out[0];
  for (int j = 1; j < E; ++j) {
    if (b_out[j] < mn) mn = b_out[j];
    if (b_out[j] > mx) mx = b_out[j];
  }
  if (bounds_out) {
    bounds_out[0] = mn - 1.0f;
    bounds_out[1] = mx + 1.0f;
  }
  if (q_out) memcpy(q_out, q, sizeof(double) * (size_t)E);
  free(q);
}

/* ------------------------------------------------------------------------ */
/* Load-error injection ([EQB] LEI paragraph).                               */
/* ------------------------------------------------------------------------ */

void orc_lei(float* grad, const int32_t* topk, int64_t N, int E, int k, float eta,
             int64_t* load_out, double* rho_out) {
  int64_t* load = (int64_t*)calloc((size_t)E, sizeof(int64_t));
  double* rho = (double*)malloc(sizeof(double) * (size_t)E);
  float* c = (float*)malloc(sizeof(float) * (size_t)E);
  for (int64_t i = 0; i < N * (int64_t)k; ++i) load[topk[i]] += 1;
  double T = (double)(N * (int64_t)k) / (double)E;
  double tsum = 0.0;
  for (int e = 0; e < E; ++e) {
    double rho_raw = ((double)load[e] - T) / T;
    rho[e] = tanh(rho_raw);
    tsum += rho[e];
  }
  double tmean = tsum / (double)E;
  for (int e = 0; e < E; ++e) {
    rho[e] = rho[e] - tmean;
    c[e] = (float)((double)eta * rho[e]);
  }
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < N; ++i)
    for (int e = 0; e < E; ++e) grad[i * E + e] = grad[i * E + e] + c[e];
  if (load_out) memcpy(load_out, load, sizeof(int64_t) * (size_t)E);
  if (rho_out) memcpy(rho_out, rho, sizeof(double) * (size_t)E);
  free(load);
  free(rho);
  free(c);
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
