// Device hash sampler: random-binning draws and their bin boundaries.
//
// "Positional LSH: Binary Block Matrix Approximation for Attention with
// Linear Biases", technical summary, Methodology 1 (random binning of the
// integer positions into contiguous bins) and Methodology 2 (Gamma-law
// widths).  Recipe per (head h, sample t):
//   Philox4x32-10(key = seed, counter = (t, h, 0, 0)) -> x0, x1, x2
//   U_k = (x_k + 0.5) 2^-32
//   w = sigma_h (-ln U0 - ln U1)   ~ Gamma(shape 2, scale sigma_h)
//   u = w U2                        ~ U(0, w)
//   bin starts: 0 and ceil(u + k w), k = 0, 1, ... below n (all positions
//   when w < 1).
// All fp64 arithmetic is done one correctly rounded operation at a time
// (__dadd_rn etc.), with the library's own logarithm, so the boundaries are
// reproducible bit for bit by any implementation of the same recipe.
//
// Output layout: for every hash, one BinRecord per 32 positions (bitmap of
// bin starts plus the neighbouring starts), which the attention kernels read
// to find each row's bin in O(1).
#include <cuda_runtime.h>
#include <stdint.h>

#include "plsh_internal.h"

namespace plsh {
namespace {

// Philox4x32-10 (Salmon et al., SC'11): multipliers and Weyl increments of the
// published generator.
__device__ __forceinline__ void philox4x32_10(uint32_t c[4], uint32_t k0,
                                              uint32_t k1) {
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r) {
      k0 += 0x9E3779B9u;
      k1 += 0xBB67AE85u;
    }
    const uint32_t lo_a = 0xD2511F53u * c[0];
    const uint32_t hi_a = __umulhi(0xD2511F53u, c[0]);
    const uint32_t lo_b = 0xCD9E8D57u * c[2];
    const uint32_t hi_b = __umulhi(0xCD9E8D57u, c[2]);
    const uint32_t n0 = hi_b ^ c[1] ^ k0;
    const uint32_t n2 = hi_a ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo_b;
    c[2] = n2;
    c[3] = lo_a;
  }
}

// Natural log of a positive normal double: x = 2^e m, m reduced to
// [sqrt(1/2), sqrt(2)), ln m = 2 atanh(z) = 2 z sum_k z^2k / (2k+1) with
// z = (m-1)/(m+1), 12 terms by Horner, then e ln2 added in two parts
// (ln2 split so that e * hi is exact).
__device__ double ln_rn(double x) {
  const double kLn2Hi = 0x1.62e42fef00000p-1;
  const double kLn2Lo = 0x1.473de6af278edp-34;
  const double kSqrt2 = 0x1.6a09e667f3bcdp+0;
  const long long bits = __double_as_longlong(x);
  long long e = ((bits >> 52) & 0x7ff) - 1023;
  double m = __longlong_as_double((bits & 0x000fffffffffffffll) |
                                  0x3ff0000000000000ll);
  if (m > kSqrt2) {
    m = __dmul_rn(m, 0.5);
    e += 1;
  }
  const double z = __ddiv_rn(__dadd_rn(m, -1.0), __dadd_rn(m, 1.0));
  const double z2 = __dmul_rn(z, z);
  double poly = __ddiv_rn(1.0, 23.0);
#pragma unroll
  for (int k = 10; k >= 0; --k) {
    poly = __dadd_rn(__dmul_rn(poly, z2), __ddiv_rn(1.0, (double)(2 * k + 1)));
  }
  const double ln_m = __dmul_rn(__dadd_rn(z, z), poly);
  const double ed = (double)e;
  return __dadd_rn(__dmul_rn(ed, kLn2Hi),
                   __dadd_rn(__dmul_rn(ed, kLn2Lo), ln_m));
}

__global__ void draw_kernel(const double* __restrict__ sigma, int H, int s,
                            uint64_t seed, double* __restrict__ w_out,
                            double* __restrict__ u_out) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= H * s) return;
  const int h = idx / s, t = idx % s;
  uint32_t c[4] = {(uint32_t)t, (uint32_t)h, 0u, 0u};
  philox4x32_10(c, (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32));
  const double two_m32 = 0x1p-32;
  const double u0 = __dmul_rn(__dadd_rn((double)c[0], 0.5), two_m32);
  const double u1 = __dmul_rn(__dadd_rn((double)c[1], 0.5), two_m32);
  const double u2 = __dmul_rn(__dadd_rn((double)c[2], 0.5), two_m32);
  const double e0 = -ln_rn(u0);
  const double e1 = -ln_rn(u1);
  const double w = __dmul_rn(sigma[h], __dadd_rn(e0, e1));
  w_out[idx] = w;
  u_out[idx] = __dmul_rn(w, u2);
}

// ceil(u + k w) with the multiply and the add rounded separately.
__device__ __forceinline__ double start_of(long long k, double w, double u) {
  return ceil(__dadd_rn(u, __dmul_rn((double)k, w)));
}

// Bitmap word `word` of hash `hs`: bit r set when position 32*word + r opens
// a bin.  One thread per (hash, word).
__global__ void bits_from_draws_kernel(int64_t n, int64_t W, int HS,
                                       const double* __restrict__ w_in,
                                       const double* __restrict__ u_in,
                                       BinRecord* __restrict__ rec) {
  const int64_t gid = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (gid >= (int64_t)HS * W) return;
  const int hs = (int)(gid / W);
  const int64_t word = gid % W;
  const double w = w_in[hs], u = u_in[hs];
  const int64_t p0 = word * 32;
  const int64_t p1 = (p0 + 32 < n) ? p0 + 32 : n;   // positions [p0, p1)
  uint32_t bits = 0;
  if (w < 1.0) {
    const int64_t cnt = p1 - p0;
    bits = cnt >= 32 ? 0xffffffffu : ((1u << cnt) - 1u);
  } else {
    if (p0 == 0) bits |= 1u;
    // first k whose start can reach p0: k ~ (p0 - 1 - u) / w, stepped back two
    // to absorb rounding, then walk forward over the exact starts.
    double est = floor(((double)(p0 - 1) - u) / w) - 2.0;
    long long k = est > 0.0 ? (long long)est : 0ll;
    const double lim = (double)p1;
    for (;; ++k) {
      const double c = start_of(k, w, u);
      if (c >= lim) break;
      if (c >= (double)p0) bits |= 1u << ((int64_t)c - p0);
    }
  }
  rec[gid].bits = bits;
}

// One thread per listed start (terminal entries excluded): set its bit.
__global__ void bits_from_starts_kernel(int64_t W, int HS, int64_t n,
                                        const int64_t* __restrict__ offsets,
                                        const int32_t* __restrict__ starts,
                                        int64_t total,
                                        BinRecord* __restrict__ rec) {
  const int64_t e = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (e >= total) return;
  // hash owning entry e: binary search over offsets
  int lo = 0, hi = HS;   // offsets[lo] <= e < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= e) lo = mid; else hi = mid;
  }
  const int32_t p = starts[e];
  if (p >= n) return;    // terminal
  atomicOr(&rec[(int64_t)lo * W + (p >> 5)].bits, 1u << (p & 31));
}

// prev[word] = last start at or before 32*word; next[word] = first start at or
// after 32*(word+1), else n.  One block per hash; sequential segments with a
// running carry, block-wide scans inside a segment.
constexpr int kScanThreads = 256;

__global__ void __launch_bounds__(kScanThreads)
prev_next_kernel(int64_t n, int64_t W, BinRecord* __restrict__ rec) {
  const int hs = blockIdx.x;
  BinRecord* r = rec + (int64_t)hs * W;
  __shared__ int32_t warp_buf[kScanThreads / 32];
  __shared__ int32_t carry_s;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  // forward pass: running maximum of the highest start so far
  int32_t carry = -1;
  for (int64_t base = 0; base < W; base += kScanThreads) {
    const int64_t wd = base + threadIdx.x;
    uint32_t bits = wd < W ? r[wd].bits : 0u;
    int32_t hi_pos = bits ? (int32_t)(wd * 32 + 31 - __clz(bits)) : -1;
    // inclusive max-scan of hi_pos across the block
    int32_t v = hi_pos;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v = max(v, t);
    }
    if (lane == 31) warp_buf[wid] = v;
    __syncthreads();
    int32_t before = carry;
    for (int q = 0; q < wid; ++q) before = max(before, warp_buf[q]);
    int32_t excl = __shfl_up_sync(0xffffffffu, v, 1);
    if (lane == 0) excl = -1;
    excl = max(excl, before);
    if (wd < W) {
      // last start <= 32*wd: position 32*wd itself, else the scan before it
      r[wd].prev = (bits & 1u) ? (int32_t)(wd * 32) : excl;
    }
    if (threadIdx.x == kScanThreads - 1) carry_s = max(before, v);
    __syncthreads();
    carry = carry_s;
    __syncthreads();
  }
  // backward pass: running minimum of the lowest start after the word
  int32_t carry_b = (int32_t)n;
  const int64_t nseg = (W + kScanThreads - 1) / kScanThreads;
  for (int64_t sg = nseg - 1; sg >= 0; --sg) {
    const int64_t wd = sg * kScanThreads + (kScanThreads - 1 - threadIdx.x);
    uint32_t bits = (wd >= 0 && wd < W) ? r[wd].bits : 0u;
    int32_t lo_pos = bits ? (int32_t)(wd * 32 + __ffs(bits) - 1) : (int32_t)n;
    int32_t v = lo_pos;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int32_t t = __shfl_up_sync(0xffffffffu, v, o);
      if (lane >= o) v = min(v, t);
    }
    if (lane == 31) warp_buf[wid] = v;
    __syncthreads();
    int32_t before = carry_b;
    for (int q = 0; q < wid; ++q) before = min(before, warp_buf[q]);
    int32_t excl = __shfl_up_sync(0xffffffffu, v, 1);
    if (lane == 0) excl = (int32_t)n;
    excl = min(excl, before);
    if (wd >= 0 && wd < W) r[wd].next = excl;
    if (threadIdx.x == kScanThreads - 1) carry_s = min(before, v);
    __syncthreads();
    carry_b = carry_s;
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_sample(plsh_bins* b, uint64_t seed, cudaStream_t st) {
  const int HS = b->H * b->s;
  draw_kernel<<<(HS + 127) / 128, 128, 0, st>>>(b->d_sigma, b->H, b->s, seed,
                                                 b->d_w, b->d_u);
  const int64_t total = (int64_t)HS * b->W;
  bits_from_draws_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
      b->n, b->W, HS, b->d_w, b->d_u, b->d_rec);
  prev_next_kernel<<<HS, kScanThreads, 0, st>>>(b->n, b->W, b->d_rec);
  return cudaGetLastError();
}

cudaError_t launch_bins_from_starts(plsh_bins* b, const int32_t* d_starts,
                                    const int64_t* d_offsets, int64_t total,
                                    cudaStream_t st) {
  const int HS = b->H * b->s;
  cudaError_t e = cudaMemsetAsync(b->d_rec, 0,
                                  sizeof(BinRecord) * (size_t)HS * b->W, st);
  if (e != cudaSuccess) return e;
  if (total > 0) {
    bits_from_starts_kernel<<<(unsigned)((total + 255) / 256), 256, 0, st>>>(
        b->W, HS, b->n, d_offsets, d_starts, total, b->d_rec);
  }
  prev_next_kernel<<<HS, kScanThreads, 0, st>>>(b->n, b->W, b->d_rec);
  return cudaGetLastError();
}

}  // namespace plsh
