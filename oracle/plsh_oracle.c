/*
 * Positional LSH oracle: a plain, slow, fp64 CPU statement of what the
 * approximate-ALiBi hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file; only the test suite, the smoke check and the CPU-baseline
 * leg of the benchmark do.  It shares no code, header, constant table or
 * helper with the CUDA library: every routine below is written independently
 * from the method's definition.
 *
 * Source of the method ("Positional LSH: Binary Block Matrix Approximation
 * for Attention with Linear Biases", Wolfson & Wagner, technical summary):
 *   - Methodology, item 1 (theoretical framework): L*_ij = exp(-|i-j|/sigma)
 *     is a Laplacian kernel on token positions; a random-binning hash of the
 *     integer positions splits 0..n-1 into contiguous bins and M(h) is 1 where
 *     i and j share a bin; L* = E_h[M(h)].
 *   - Methodology, item 2 (Theorem 2.1): the bias is approximated by the
 *     empirical mean of s i.i.d. masks; the widths follow the Gamma law that
 *     underlies random binning.
 *   - Methodology, item 3 (Theorem 2.2): ALiBi attention reduces to a set of
 *     short block attentions with no positional bias; numerator and row sums
 *     are both taken against the averaged mask.
 *
 * Readings adopted where the pages are silent (each one is listed in the
 * design notes):
 *   - random numbers: Philox4x32-10 (Salmon et al., SC'11), key = seed,
 *     counter = (t, h, 0, 0), uniforms (x + 0.5) * 2^-32;
 *   - width w = sigma * (E1 + E2) with E = -ln U  ->  Gamma(shape 2, scale
 *     sigma); offset u = w * U3  ->  U(0, w);
 *   - bin starts: 0, then ceil(u + k*w) for k = 0, 1, ... below n, with
 *     u + k*w one fused multiply-add (rounded once), de-duplicated; all
 *     singletons when w < 1;
 *   - ln is this file's own atanh-series logarithm built from correctly
 *     rounded +, -, *, / and fused multiply-add (Horner steps) only, so that
 *     another implementation of the same recipe reproduces the widths bit
 *     for bit.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off (no fast-math).  fp contraction
 * must stay off: the sampler's arithmetic is defined operation by operation.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* Philox4x32-10, as published by Salmon, Moraes, Dror and Shaw,            */
/* "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11).                   */
/* ------------------------------------------------------------------------ */
#define PHILOX_MUL_A 0xD2511F53u
#define PHILOX_MUL_B 0xCD9E8D57u
#define PHILOX_WEYL_A 0x9E3779B9u
#define PHILOX_WEYL_B 0xBB67AE85u

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2],
                          uint32_t out[4]) {
  uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
  uint32_t k0 = key_in[0], k1 = key_in[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {            /* key schedule: Weyl sequence */
      k0 += PHILOX_WEYL_A;
      k1 += PHILOX_WEYL_B;
    }
    uint64_t prod_a = (uint64_t)PHILOX_MUL_A * (uint64_t)c0;
    uint64_t prod_b = (uint64_t)PHILOX_MUL_B * (uint64_t)c2;
    uint32_t n0 = (uint32_t)(prod_b >> 32) ^ c1 ^ k0;
    uint32_t n1 = (uint32_t)prod_b;
    uint32_t n2 = (uint32_t)(prod_a >> 32) ^ c3 ^ k1;
    uint32_t n3 = (uint32_t)prod_a;
    c0 = n0; c1 = n1; c2 = n2; c3 = n3;
  }
  out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

/* ------------------------------------------------------------------------ */
/* Natural logarithm from the series ln m = 2 atanh(z), z = (m-1)/(m+1),    */
/* after reducing m into [sqrt(1/2), sqrt(2)).  Only IEEE-754 correctly     */
/* rounded operations are used, each one explicitly.                        */
/* ------------------------------------------------------------------------ */
static const double ORACLE_LN2_HI = 0x1.62e42fef00000p-1; /* 20 low bits zero */
static const double ORACLE_LN2_LO = 0x1.473de6af278edp-34;
static const double ORACLE_SQRT2 = 0x1.6a09e667f3bcdp+0;
#define ORACLE_LN_TERMS 11

double oracle_ln64(double x) {
  /* defined for positive normal x, which is all the sampler feeds it */
  uint64_t bits;
  memcpy(&bits, &x, sizeof bits);
  int64_t e = (int64_t)((bits >> 52) & 0x7ffu) - 1023;
  uint64_t mbits = (bits & 0x000fffffffffffffull) | 0x3ff0000000000000ull;
  double m;
  memcpy(&m, &mbits, sizeof m);
  if (m > ORACLE_SQRT2) {         /* halve m (exact), bump the exponent */
    m = m * 0.5;
    e = e + 1;
  }
  double num = m - 1.0;           /* exact for m in [0.70, 1.42] */
  double den = m + 1.0;
  double z = num / den;
  double z2 = z * z;
  /* Horner over 1/(2k+1), k = ORACLE_LN_TERMS .. 0 */
  double poly = 1.0 / (double)(2 * ORACLE_LN_TERMS + 1);
  for (int k = ORACLE_LN_TERMS - 1; k >= 0; --k) {
    double ck = 1.0 / (double)(2 * k + 1);
    poly = fma(poly, z2, ck);     /* one rounding per step */
  }
  double two_z = z + z;
  double ln_m = two_z * poly;
  double ed = (double)e;
  double hi = ed * ORACLE_LN2_HI;            /* exact */
  double tail = fma(ed, ORACLE_LN2_LO, ln_m);
  return hi + tail;
}

/* One hash draw (w, u) for head h, sample t. */
void oracle_draw(double sigma, int32_t h, int32_t t, uint64_t seed,
                 double* w_out, double* u_out) {
  uint32_t ctr[4] = {(uint32_t)t, (uint32_t)h, 0u, 0u};
  uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
  uint32_t x[4];
  oracle_philox4x32_10(ctr, key, x);
  const double two_m32 = 0x1p-32;
  double u0 = ((double)x[0] + 0.5) * two_m32;
  double u1 = ((double)x[1] + 0.5) * two_m32;
  double u2 = ((double)x[2] + 0.5) * two_m32;
  double e0 = -oracle_ln64(u0);
  double e1 = -oracle_ln64(u1);
  double esum = e0 + e1;
  double w = sigma * esum;
  double u = w * u2;
  *w_out = w;
  *u_out = u;
}

/* Bin starts of one hash on positions 0..n-1, followed by the terminal n.
 * Returns the number of entries written (bins + 1); writes at most cap
 * entries and returns -1 if cap is too small. */
int64_t oracle_bins_one(int64_t n, double w, double u, int32_t* starts,
                        int64_t cap) {
  int64_t cnt = 0;
  if (w < 1.0) {                  /* every position is its own bin */
    if (cap < n + 1) return -1;
    for (int64_t i = 0; i < n; ++i) starts[cnt++] = (int32_t)i;
    starts[cnt++] = (int32_t)n;
    return cnt;
  }
  if (cap < 2) return -1;
  starts[cnt++] = 0;
  double last = 0.0;
  const double nd = (double)n;
  for (int64_t k = 0;; ++k) {
    double p = fma((double)k, w, u);   /* u + k w, rounded once */
    double c = ceil(p);
    if (c >= nd) break;
    if (c > last) {
      if (cnt + 1 >= cap) return -1;
      starts[cnt++] = (int32_t)c;
      last = c;
    }
  }
  starts[cnt++] = (int32_t)n;
  return cnt;
}

/* Draws and bins of every (h, t); layout per (h, t) in order h-major:
 * offsets[h*s + t] .. offsets[h*s + t + 1] index into starts.
 * Pass starts = NULL to only count (offsets still filled).  Returns the
 * total number of entries, or -1 on a capacity error. */
int64_t oracle_sample_bins(int64_t n, const double* sigma, int32_t H, int32_t s,
                           uint64_t seed, int64_t* offsets, int32_t* starts,
                           int64_t cap, double* w_out, double* u_out) {
  int64_t total = 0;
  int32_t* scratch = NULL;
  if (starts == NULL) {
    scratch = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n + 2));
    if (!scratch) return -1;
  }
  for (int32_t h = 0; h < H; ++h) {
    for (int32_t t = 0; t < s; ++t) {
      double w, u;
      oracle_draw(sigma[h], h, t, seed, &w, &u);
      if (w_out) w_out[h * s + t] = w;
      if (u_out) u_out[h * s + t] = u;
      offsets[h * s + t] = total;
      int64_t got;
      if (starts) {
        got = oracle_bins_one(n, w, u, starts + total, cap - total);
      } else {
        got = oracle_bins_one(n, w, u, scratch, n + 2);
      }
      if (got < 0) { free(scratch); return -1; }
      total += got;
    }
  }
  offsets[(int64_t)H * s] = total;
  free(scratch);
  return total;
}

/* ------------------------------------------------------------------------ */
/* Attention.  Q [B,Hq,n,d], K and V [B,Hkv,n,d], float32 values converted  */
/* exactly to double.  Query head h reads KV head h / (Hq/Hkv).             */
/* ------------------------------------------------------------------------ */

/* bin [lo, hi) of position i in one hash's start list (terminal included) */
static void oracle_bin_of(const int32_t* st, int64_t cnt, int64_t i,
                          int64_t* lo, int64_t* hi) {
  int64_t a = 0, b = cnt - 1;     /* st[a] <= i < st[b] */
  while (b - a > 1) {
    int64_t mid = a + (b - a) / 2;
    if ((int64_t)st[mid] <= i) a = mid; else b = mid;
  }
  *lo = st[a];
  *hi = st[b];
}

static double oracle_dot(const float* x, const float* y, int64_t d) {
  double acc = 0.0;
  for (int64_t c = 0; c < d; ++c) acc += (double)x[c] * (double)y[c];
  return acc;
}

typedef struct {
  int64_t B, Hq, Hkv, n, d;
} oracle_shape;

static const float* row_ptr(const float* base, int64_t b, int64_t h,
                            int64_t H, int64_t n, int64_t d, int64_t i) {
  return base + (((b * H + h) * n + i) * d);
}

/*
 * Approximate ALiBi attention, evaluated directly per sample and per bin:
 *   J_t(i) = bin of i under hash t (clipped to j <= i when causal)
 *   N_i = sum_t sum_{j in J_t(i)} exp(S_ij - m_i) v_j
 *   D_i = sum_t sum_{j in J_t(i)} exp(S_ij - m_i)
 *   out_i = N_i / D_i,   S_ij = q_i . k_j / sqrt(d)
 * The shift m_i is the largest S_ij that takes part (or 0 when zero_shift).
 * Rows are given as (b, h, i) triples.  When num_out/den_out are non-NULL
 * the unnormalised parts are written too.
 */
static void oracle_plsh_rows_impl(const float* Q, const float* K, const float* V,
                                  oracle_shape sh, const int64_t* offsets,
                                  const int32_t* starts, int32_t s,
                                  int32_t causal, const int32_t* rb,
                                  const int32_t* rh, const int32_t* ri,
                                  int64_t R, int32_t zero_shift, double* out,
                                  double* num_out, double* den_out) {
  const int64_t group = sh.Hq / sh.Hkv;
  const double inv_sqrt_d = 1.0 / sqrt((double)sh.d);
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < R; ++r) {
    const int64_t b = rb[r], h = rh[r], i = ri[r];
    const int64_t kvh = h / group;
    const float* q = row_ptr(Q, b, h, sh.Hq, sh.n, sh.d, i);
    double m = -INFINITY;
    if (!zero_shift) {
      for (int32_t t = 0; t < s; ++t) {
        const int64_t o0 = offsets[h * s + t], o1 = offsets[h * s + t + 1];
        int64_t lo, hi;
        oracle_bin_of(starts + o0, o1 - o0, i, &lo, &hi);
        if (causal && hi > i + 1) hi = i + 1;
        for (int64_t j = lo; j < hi; ++j) {
          const float* k = row_ptr(K, b, kvh, sh.Hkv, sh.n, sh.d, j);
          double sij = oracle_dot(q, k, sh.d) * inv_sqrt_d;
          if (sij > m) m = sij;
        }
      }
    } else {
      m = 0.0;
    }
    double* acc = (double*)calloc((size_t)sh.d, sizeof(double));
    double den = 0.0;
    for (int32_t t = 0; t < s; ++t) {
      const int64_t o0 = offsets[h * s + t], o1 = offsets[h * s + t + 1];
      int64_t lo, hi;
      oracle_bin_of(starts + o0, o1 - o0, i, &lo, &hi);
      if (causal && hi > i + 1) hi = i + 1;
      for (int64_t j = lo; j < hi; ++j) {
        const float* k = row_ptr(K, b, kvh, sh.Hkv, sh.n, sh.d, j);
        const float* v = row_ptr(V, b, kvh, sh.Hkv, sh.n, sh.d, j);
        double e = exp(oracle_dot(q, k, sh.d) * inv_sqrt_d - m);
        den += e;
        for (int64_t c = 0; c < sh.d; ++c) acc[c] += e * (double)v[c];
      }
    }
    for (int64_t c = 0; c < sh.d; ++c) {
      if (out) out[r * sh.d + c] = acc[c] / den;
      if (num_out) num_out[r * sh.d + c] = acc[c];
    }
    if (den_out) den_out[r] = den;
    free(acc);
  }
}

void oracle_plsh_attn_rows(const float* Q, const float* K, const float* V,
                           int64_t B, int64_t Hq, int64_t Hkv, int64_t n,
                           int64_t d, const int64_t* offsets,
                           const int32_t* starts, int32_t s, int32_t causal,
                           const int32_t* rb, const int32_t* rh,
                           const int32_t* ri, int64_t R, double* out) {
  oracle_shape sh = {B, Hq, Hkv, n, d};
  oracle_plsh_rows_impl(Q, K, V, sh, offsets, starts, s, causal, rb, rh, ri, R,
                        0, out, NULL, NULL);
}

/* Unnormalised numerator and denominator with no shift (m_i = 0). */
void oracle_plsh_parts_rows(const float* Q, const float* K, const float* V,
                            int64_t B, int64_t Hq, int64_t Hkv, int64_t n,
                            int64_t d, const int64_t* offsets,
                            const int32_t* starts, int32_t s, int32_t causal,
                            const int32_t* rb, const int32_t* rh,
                            const int32_t* ri, int64_t R, double* num,
                            double* den) {
  oracle_shape sh = {B, Hq, Hkv, n, d};
  oracle_plsh_rows_impl(Q, K, V, sh, offsets, starts, s, causal, rb, rh, ri, R,
                        1, NULL, num, den);
}

/*
 * Exact ALiBi attention T*_i = sum_j exp(S_ij - |i-j|/sigma_h - m_i) v_j
 *                              / sum_j exp(S_ij - |i-j|/sigma_h - m_i)
 * over all j (j <= i when causal).
 */
void oracle_alibi_exact_rows(const float* Q, const float* K, const float* V,
                             int64_t B, int64_t Hq, int64_t Hkv, int64_t n,
                             int64_t d, const double* sigma, int32_t causal,
                             const int32_t* rb, const int32_t* rh,
                             const int32_t* ri, int64_t R, double* out) {
  const int64_t group = Hq / Hkv;
  const double inv_sqrt_d = 1.0 / sqrt((double)d);
#pragma omp parallel for schedule(dynamic, 4)
  for (int64_t r = 0; r < R; ++r) {
    const int64_t b = rb[r], h = rh[r], i = ri[r];
    const int64_t kvh = h / group;
    const float* q = row_ptr(Q, b, h, Hq, n, d, i);
    const int64_t jend = causal ? i + 1 : n;
    double m = -INFINITY;
    for (int64_t j = 0; j < jend; ++j) {
      const float* k = row_ptr(K, b, kvh, Hkv, n, d, j);
      double dist = (double)(i > j ? i - j : j - i);
      double x = oracle_dot(q, k, d) * inv_sqrt_d - dist / sigma[h];
      if (x > m) m = x;
    }
    double* acc = (double*)calloc((size_t)d, sizeof(double));
    double den = 0.0;
    for (int64_t j = 0; j < jend; ++j) {
      const float* k = row_ptr(K, b, kvh, Hkv, n, d, j);
      const float* v = row_ptr(V, b, kvh, Hkv, n, d, j);
      double dist = (double)(i > j ? i - j : j - i);
      double e = exp(oracle_dot(q, k, d) * inv_sqrt_d - dist / sigma[h] - m);
      den += e;
      for (int64_t c = 0; c < d; ++c) acc[c] += e * (double)v[c];
    }
    for (int64_t c = 0; c < d; ++c) out[r * d + c] = acc[c] / den;
    free(acc);
  }
}

void oracle_set_threads(int32_t nthreads) {
#ifdef _OPENMP
  if (nthreads > 0) omp_set_num_threads(nthreads);
#else
  (void)nthreads;
#endif
}

int32_t oracle_max_threads(void) {
#ifdef _OPENMP
  return (int32_t)omp_get_max_threads();
#else
  return 1;
#endif
}
