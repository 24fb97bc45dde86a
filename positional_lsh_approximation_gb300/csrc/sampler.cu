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
//   bin starts: 0 and ceil(u + k w), k = 0, 1, ... below n, u + k w one
//   fused multiply-add (all positions when w < 1).
// All fp64 arithmetic is done one correctly rounded operation at a time
// (__dadd_rn, __fma_rn etc.), with a logarithm of its own built from such
// operations, so the boundaries are reproducible bit for bit by any
// implementation of the same recipe.  Steps that are exact in any case (an
// integer to double, a double's ceiling, scaling by a power of two, the
// comparison of two doubles of one binade) are done on the bits with integer
// instructions: this part issues fp64 instructions, conversions included, at
// a small fraction of its integer rate and with a long latency.
//
// Output layout: for every hash, one BinRecord per 32 positions (bitmap of
// bin starts plus the neighbouring starts), which the attention kernels read
// to find each row's bin in O(1).
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include <algorithm>

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

// Bits of a double as an unsigned integer and back.
__device__ __forceinline__ uint64_t dbits(double x) {
  return (uint64_t)__double_as_longlong(x);
}
__device__ __forceinline__ double dfrom(uint64_t b) { return __longlong_as_double((long long)b); }

// (double)k for 0 <= k < 2^53, exactly: the leading one sets the exponent.
__device__ __forceinline__ double ll_to_double(uint64_t k) {
  if (k == 0) return 0.0;
  const int e = 63 - __clzll((long long)k);    // 2^e <= k < 2^(e+1)
  return dfrom(((uint64_t)(1023 + e) << 52) | ((k << (52 - e)) & 0x000fffffffffffffull));
}

// ceil(r) for 0 <= r < 2^62, exactly: the integer part of the significand,
// plus one when a fraction bit is set.
__device__ __forceinline__ long long ceil_to_ll(double r) {
  const uint64_t b = dbits(r);
  const int ex = (int)(b >> 52) - 1023;        // r = 1.f 2^ex
  if (ex < 0) return b == 0 ? 0 : 1;
  const uint64_t m = (b & 0x000fffffffffffffull) | (1ull << 52);
  if (ex >= 52) return (long long)(m << (ex - 52));
  const int fr = 52 - ex;
  return (long long)((m >> fr) + ((m & ((1ull << fr) - 1ull)) != 0ull));
}

// A positive normal double within float's normal range as a float,
// truncated (error below 2^-23 relative).
__device__ __forceinline__ float to_float_rz(double x) {
  const uint64_t b = dbits(x);
  const uint32_t e = (uint32_t)((b >> 52) & 0x7ff) - 1023u + 127u;
  return __uint_as_float((e << 23) | (uint32_t)((b >> 29) & 0x7fffffu));
}

// Natural log of a positive normal double: x = 2^e m, m reduced to
// [sqrt(1/2), sqrt(2)), ln m = 2 atanh(z) = 2 z sum_k z^2k / (2k+1) with
// z = (m-1)/(m+1), 12 terms by Horner with fused multiply-adds, then e ln2
// added in two parts
// (ln2 split so that e * hi is exact).
__device__ double ln_rn(double x) {
  const double kLn2Hi = 0x1.62e42fef00000p-1;
  const double kLn2Lo = 0x1.473de6af278edp-34;
  const double kSqrt2 = 0x1.6a09e667f3bcdp+0;
  const long long bits = __double_as_longlong(x);
  long long e = ((bits >> 52) & 0x7ff) - 1023;
  double m = __longlong_as_double((bits & 0x000fffffffffffffll) |
                                  0x3ff0000000000000ll);
  // m and sqrt(2) share a binade, so they compare as integers; halving m
  // lowers its exponent by one
  if (dbits(m) > dbits(kSqrt2)) {
    m = dfrom(dbits(m) - (1ull << 52));
    e += 1;
  }
  // 1/(2k+1), each the correctly rounded quotient (folded by the compiler)
  constexpr double kInvOdd[12] = {1.0 / 1,  1.0 / 3,  1.0 / 5,  1.0 / 7,
                                  1.0 / 9,  1.0 / 11, 1.0 / 13, 1.0 / 15,
                                  1.0 / 17, 1.0 / 19, 1.0 / 21, 1.0 / 23};
  const double z = __ddiv_rn(__dadd_rn(m, -1.0), __dadd_rn(m, 1.0));
  const double z2 = __dmul_rn(z, z);
  double poly = kInvOdd[11];
#pragma unroll
  for (int k = 10; k >= 0; --k) poly = __fma_rn(poly, z2, kInvOdd[k]);
  const double ln_m = __dmul_rn(__dadd_rn(z, z), poly);
  const double ed = (double)e;
  return __dadd_rn(__dmul_rn(ed, kLn2Hi),          // exact product
                   __fma_rn(ed, kLn2Lo, ln_m));
}

// ceil(u + k w), the multiply-add rounded once (0 <= k < 2^53, 0 < u + k w
// < 2^62).
__device__ __forceinline__ long long start_of(long long k, double w, double u) {
  return ceil_to_ll(__fma_rn(ll_to_double((uint64_t)k), w, u));
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

// The sampler, one CTA per (hash, segment of kSegWords words): the draw (two
// threads, one logarithm each; every CTA of a hash computes the same bits),
// the segment's bin starts set in a shared-memory bitmap (one thread per k,
// start ceil(u + k w)), the last start before the segment and the first after
// it taken from the same k walk, and the records from two block scans.
constexpr int kSampThreads = 256;
constexpr int kSegWords = 128;

// Block-wide exclusive scan of `v` with operator max (fwd) or min (!fwd):
// thread t receives the combination of threads before it (after it for !fwd)
// and `ident` when there are none.  All threads must call it.
__device__ __forceinline__ int32_t block_excl_scan(int32_t v, bool fwd, int32_t ident,
                                                   int32_t* warp_buf) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  constexpr int nw = kSampThreads / 32;
  int32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int32_t t = fwd ? __shfl_up_sync(0xffffffffu, incl, o)
                          : __shfl_down_sync(0xffffffffu, incl, o);
    const bool take = fwd ? lane >= o : lane + o < 32;
    if (take) incl = fwd ? max(incl, t) : min(incl, t);
  }
  int32_t excl = fwd ? __shfl_up_sync(0xffffffffu, incl, 1)
                     : __shfl_down_sync(0xffffffffu, incl, 1);
  if (fwd ? lane == 0 : lane == 31) excl = ident;
  if (fwd ? lane == 31 : lane == 0) warp_buf[wid] = incl;
  __syncthreads();
  int32_t before = ident;
#pragma unroll
  for (int q = 0; q < nw; ++q) {
    if (fwd ? q < wid : q > wid)
      before = fwd ? max(before, warp_buf[q]) : min(before, warp_buf[q]);
  }
  __syncthreads();
  return fwd ? max(excl, before) : min(excl, before);
}

__global__ void __launch_bounds__(kSampThreads)
sample_kernel(int64_t n, int64_t W, int nseg, int spc, int s,
              const double* __restrict__ sigma, uint64_t seed,
              double* __restrict__ w_out, double* __restrict__ u_out,
              BinRecord* __restrict__ rec) {
  const int cps = (nseg + spc - 1) / spc;      // CTAs per hash
  const int hs = blockIdx.x / cps;
  const int sg0 = (blockIdx.x % cps) * spc;
  __shared__ double lnv[2], wu[2];
  __shared__ uint32_t bits_s[kSegWords];
  __shared__ int32_t warp_buf[kSampThreads / 32];
  __shared__ int32_t next_s, prev_s;
  __shared__ long long k0_s, k1_s;
  // the attention kernel that follows may start its set-up now; it waits
  // for this grid's completion before it reads the records
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if (threadIdx.x < 2) {
    const int h = hs / s, t = hs % s;
    uint32_t c[4] = {(uint32_t)t, (uint32_t)h, 0u, 0u};
    philox4x32_10(c, (uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32));
    // U = (x + 0.5) 2^-32 = (2x + 1) 2^-33, exact: the odd integer 2x + 1 as
    // a double, its exponent lowered by 33
    auto unit = [](uint32_t x) {
      return dfrom(dbits(ll_to_double(2ull * x + 1ull)) - (33ull << 52));
    };
    lnv[threadIdx.x] = ln_rn(unit(c[threadIdx.x]));
    if (threadIdx.x == 0) wu[1] = unit(c[2]);
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    const double w = __dmul_rn(sigma[hs / s], __dadd_rn(-lnv[0], -lnv[1]));
    const double u = __dmul_rn(w, wu[1]);
    wu[0] = w;
    wu[1] = u;
    if (sg0 == 0) {
      w_out[hs] = w;
      u_out[hs] = u;
    }
  }
  __syncthreads();
  const double w = wu[0], u = wu[1];
  const bool wide = dbits(w) >= dbits(1.0);    // w >= 1 (w > 0)
  for (int sg = sg0; sg < min(nseg, sg0 + spc); ++sg) {
    const int64_t seg = (int64_t)sg * kSegWords;
    const int nw = (int)min((int64_t)kSegWords, W - seg);
    const int64_t P0 = seg * 32;
    const int64_t P1 = min(P0 + (int64_t)nw * 32, n);
    if (threadIdx.x < kSegWords) bits_s[threadIdx.x] = 0u;
    if (threadIdx.x == 0) {
      next_s = (int32_t)n;
      prev_s = P0 > 0 ? 0 : -1;    // position 0 always opens a bin
      // k range of the walk, from just below the first start that can reach
      // the segment to just past the first start at or beyond P1; estimated
      // in fp32 (no fp64 division; a fast reciprocal, positions as int32 and
      // k as uint32, so that no conversion takes the fp64 pipe) with a slack
      // that covers its rounding (relative error below 2^-20)
      if (wide) {
        const float wf = to_float_rz(w), uf = to_float_rz(u);
        const float rw = __fdividef(1.0f, wf);
        const float ka = ((float)(int32_t)(P0 - 1) - uf) * rw;
        const float kb = ((float)(int32_t)P1 - uf) * rw;
        const float slack = 2.0f + fmaxf(fabsf(ka), fabsf(kb)) * 0x1p-18f;
        const float lo = floorf(ka - slack), hi = fminf(ceilf(kb + slack), 4294967040.0f);
        k0_s = lo > 0.0f ? (long long)(uint32_t)lo : 0ll;
        k1_s = hi > 0.0f ? (long long)(uint32_t)hi : 0ll;
      }
    }
    __syncthreads();
    if (!wide) {     // w < 1: every position opens a bin
      if (threadIdx.x < nw) {
        const int64_t lo = P0 + (int64_t)threadIdx.x * 32;
        const int64_t cnt = min((int64_t)32, P1 - lo);
        bits_s[threadIdx.x] = cnt >= 32 ? 0xffffffffu : ((1u << cnt) - 1u);
      }
      if (threadIdx.x == 0) {
        if (P0 > 0) prev_s = (int32_t)(P0 - 1);
        if (P1 < n) next_s = (int32_t)P1;
      }
    } else {
      if (P0 == 0 && threadIdx.x == 0) atomicOr(&bits_s[0], 1u);
      // every k of the range (no data-dependent exit, so the loads of
      // independent k overlap): starts below P0 give the last start before
      // the segment, the smallest at or past P1 the next one
      const long long k0 = k0_s, k1 = k1_s;
      int32_t before = -1, after = INT_MAX;
#pragma unroll 4
      for (long long k = k0 + threadIdx.x; k <= k1; k += kSampThreads) {
        const long long c = start_of(k, w, u);
        if (c >= P1) {
          if (c < n) after = min(after, (int32_t)c);
        } else if (c >= P0) {
          const int64_t off = c - P0;
          atomicOr(&bits_s[off >> 5], 1u << (off & 31));
        } else {
          before = max(before, (int32_t)c);
        }
      }
      if (after != INT_MAX) atomicMin(&next_s, after);
      if (before >= 0) atomicMax(&prev_s, before);
    }
    __syncthreads();
    const uint32_t bits = threadIdx.x < nw ? bits_s[threadIdx.x] : 0u;
    const int64_t wd = seg + threadIdx.x;
    const int32_t hi_pos = bits ? (int32_t)(wd * 32 + 31 - __clz(bits)) : -1;
    const int32_t lo_pos = bits ? (int32_t)(wd * 32 + __ffs(bits) - 1) : (int32_t)n;
    const int32_t prev = max(block_excl_scan(hi_pos, true, -1, warp_buf), prev_s);
    const int32_t next = min(block_excl_scan(lo_pos, false, (int32_t)n, warp_buf), next_s);
    if (threadIdx.x < nw) {
      BinRecord o;
      o.bits = bits;
      o.prev = (bits & 1u) ? (int32_t)(wd * 32) : prev;
      o.next = next;
      o.pad = 0;
      rec[(int64_t)hs * W + wd] = o;
    }
    __syncthreads();
  }
}

}  // namespace

cudaError_t launch_sample(plsh_bins* b, uint64_t seed, cudaStream_t st) {
  const int HS = b->H * b->s;
  // about 1024 CTAs whatever the shape: each takes spc consecutive segments
  // of one hash and computes that hash's draw once
  const int64_t nseg = (b->W + kSegWords - 1) / kSegWords;
  const int64_t target = 1024;
  const int64_t spc = std::max<int64_t>(1, (HS * nseg + target - 1) / target);
  const int64_t cps = (nseg + spc - 1) / spc;
  sample_kernel<<<(unsigned)(HS * cps), kSampThreads, 0, st>>>(
      b->n, b->W, (int)nseg, (int)spc, b->s, b->d_sigma, seed, b->d_w, b->d_u, b->d_rec);
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

// Fixed blocks (the deterministic baseline the summary's fine-tuning
// experiment compares against): hash (h, t) cuts 0..n-1 into blocks of width
// w starting at offset o (integers held in d_w, d_u), starts
// {0} u {o + k w : k >= 0} inside [1, n).  One thread per record word, in
// closed form: the word's starts from the first one at or after it, the last
// start at or before its first position, the first start after it.
__global__ void fixed_bins_kernel(int n, int64_t W, int64_t HS, const double* __restrict__ d_w,
                                  const double* __restrict__ d_u, BinRecord* __restrict__ rec) {
  const int64_t idx = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (idx >= HS * W) return;
  const int64_t hs = idx / W;
  const int wd = (int)(idx - hs * W);
  // 64-bit positions: a width may be as large as 2^31 - 1
  const int64_t w = (int64_t)d_w[hs], o = (int64_t)d_u[hs];
  const int64_t a = (int64_t)wd * 32;
  uint32_t bits = wd == 0 ? 1u : 0u;
  for (int64_t p = a <= o ? o : o + (a - o + w - 1) / w * w; p < a + 32 && p < n; p += w)
    bits |= 1u << (int)(p - a);
  const int64_t prev = a < o ? 0 : o + (a - o) / w * w;
  const int64_t z = a + 32;
  int64_t next = z >= n ? n : (z <= o ? o : o + (z - o + w - 1) / w * w);
  if (next > n) next = n;
  BinRecord r;
  r.bits = bits;
  r.prev = (int32_t)prev;
  r.next = (int32_t)next;
  r.pad = 0;
  rec[idx] = r;
}

cudaError_t launch_bins_fixed(plsh_bins* b, cudaStream_t st) {
  const int64_t HS = (int64_t)b->H * b->s;
  const int64_t words = HS * b->W;
  fixed_bins_kernel<<<(unsigned)((words + 255) / 256), 256, 0, st>>>((int)b->n, b->W, HS, b->d_w,
                                                                      b->d_u, b->d_rec);
  return cudaGetLastError();
}

}  // namespace plsh
