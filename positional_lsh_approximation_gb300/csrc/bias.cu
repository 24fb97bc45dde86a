// The bias of the averaged mask at scale: ||L* - M~|| in max norm and in
// spectral norm for one head, without forming either n x n matrix.
//
// "Positional LSH: Binary Block Matrix Approximation for Attention with Linear
// Biases", technical summary: L*_ij = e^{-|i-j|/sigma} (Problem statement),
// M~ = (1/s) sum_t M(h_t) with M(h_t)_ij = 1 when i and j share a bin of hash t
// (Methodology 1-2); the convergence experiment (Results) measures both norms
// of L* - M~ against s.
//
// Max norm, exactly: outside row i's key envelope [min_t lo_t(i),
// max_t hi_t(i)) M~ is zero, so the largest |L*_ij| there sits next to the
// envelope; inside it M~_ij = c_ij / s is counted per key.  One thread per row.
//
// Spectral norm: L* - M~ is symmetric, so the norm is its largest eigenvalue
// magnitude, estimated by Lanczos iteration.  Both products are O(n):
//   (L* x)_i = f_i + g_i - x_i,  f_i = x_i + r f_{i-1},  g_i = x_i + r g_{i+1},
//   r = e^{-1/sigma} (two linear recurrences, scanned in three passes), and
//   (M~ x)_i = (1/s) sum_t (P[hi_t(i)] - P[lo_t(i)]),  P the prefix sums of x
//   (the same scan with r = 1).
// The extreme eigenvalues of the Lanczos tridiagonal matrix come from Sturm
// sequence bisection on the host.  All vectors are fp64.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <algorithm>
#include <vector>

#include "bins_dev.cuh"
#include "plsh_internal.h"

namespace plsh {
namespace {

constexpr int kScanThreads = 256;
constexpr int kScanPer = 16;                        // elements per thread
constexpr int kScanChunk = kScanThreads * kScanPer;  // elements per block
constexpr int kRedThreads = 256;

// ---------------------------------------------------------------- max norm
// Row i: left of i the multiplicity is c(j) = #{t : lo_t <= j}, right of it
// #{t : hi_t > j}; two sweeps outward from i with the bounds sorted once, the
// kernel value carried as a running product of r = e^{-1/sigma}.
__global__ void rowmax_kernel(int n, int s, int64_t W, const BinRecord* __restrict__ rec,
                              double sigma, unsigned long long* __restrict__ out) {
  const double r = exp(-1.0 / sigma);
  double best = 0.0;
  int lo[kMaxS], hi[kMaxS];
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    for (int t = 0; t < s; ++t) {
      const BinRecord rc = load_record(rec, (int64_t)t * W + (i >> 5));
      int a = bin_lo(rc, i), b = bin_hi(rc, i);
      // insertion: lo descending, hi ascending
      int k = t;
      while (k > 0 && lo[k - 1] < a) { lo[k] = lo[k - 1]; --k; }
      lo[k] = a;
      k = t;
      while (k > 0 && hi[k - 1] > b) { hi[k] = hi[k - 1]; --k; }
      hi[k] = b;
    }
    const double inv_s = 1.0 / s;
    // left: j = i - 1 down to the lowest start; c drops below each start
    int c = s, k = 0;
    double p = 1.0;
    for (int j = i - 1; j >= lo[s - 1]; --j) {
      p *= r;
      while (k < s && lo[k] > j) { --c; ++k; }
      best = fmax(best, fabs(p - c * inv_s));
    }
    if (lo[s - 1] > 0) best = fmax(best, p * r);      // first key outside: M~ = 0
    // right: j = i (c = s, L* = 1) up to the last end; c drops at each end
    c = s;
    k = 0;
    p = 1.0;
    for (int j = i + 1; j < hi[s - 1]; ++j) {
      p *= r;
      while (k < s && hi[k] <= j) { --c; ++k; }
      best = fmax(best, fabs(p - c * inv_s));
    }
    if (hi[s - 1] < n) best = fmax(best, p * r);
  }
  // the bit patterns of non-negative doubles order like their values
  for (int o = 16; o > 0; o >>= 1) best = fmax(best, __shfl_xor_sync(0xffffffffu, best, o));
  if ((threadIdx.x & 31) == 0) atomicMax(out, (unsigned long long)__double_as_longlong(best));
}

// ------------------------------------------------- linear recurrence scan
// y_k = r y_{k-1} + x_k over k = 0..n-1 of the sequence read forwards
// (x[k]) or backwards (x[n-1-k]), written in the same order.
__device__ __forceinline__ int64_t seq_index(int64_t k, int n, bool rev) { return rev ? n - 1 - k : k; }

// pass 1: each block scans its chunk with no carry in and writes the chunk's
// last value
__global__ void __launch_bounds__(kScanThreads)
scan_local_kernel(const double* __restrict__ x, double* __restrict__ y, int n, double r, int rev,
                  double* __restrict__ chunk_end) {
  __shared__ double sa[kScanThreads], sb[kScanThreads];
  const int64_t base = (int64_t)blockIdx.x * kScanChunk + (int64_t)threadIdx.x * kScanPer;
  double loc[kScanPer];
  double acc = 0.0;
#pragma unroll
  for (int k = 0; k < kScanPer; ++k) {
    const int64_t q = base + k;
    acc = r * acc + (q < n ? x[seq_index(q, n, rev)] : 0.0);
    loc[k] = acc;
  }
  // scan of (multiplier, value) pairs across the threads:
  // (a1, b1) then (a2, b2) = (a1 a2, a2 b1 + b2)
  double a = pow(r, (double)kScanPer), b = acc;
  sa[threadIdx.x] = a;
  sb[threadIdx.x] = b;
  __syncthreads();
  for (int off = 1; off < kScanThreads; off <<= 1) {
    double pa = 1.0, pb = 0.0;
    if ((int)threadIdx.x >= off) {
      pa = sa[threadIdx.x - off];
      pb = sb[threadIdx.x - off];
    }
    __syncthreads();
    if ((int)threadIdx.x >= off) {
      b = a * pb + b;
      a = pa * a;
      sa[threadIdx.x] = a;
      sb[threadIdx.x] = b;
    }
    __syncthreads();
  }
  // value carried into this thread's run: the inclusive result of the thread before
  const double carry = threadIdx.x == 0 ? 0.0 : sb[threadIdx.x - 1];
  double rk = r;
#pragma unroll
  for (int k = 0; k < kScanPer; ++k) {
    const int64_t q = base + k;
    if (q < n) y[seq_index(q, n, rev)] = loc[k] + rk * carry;
    rk *= r;
  }
  if (threadIdx.x == kScanThreads - 1) chunk_end[blockIdx.x] = sb[threadIdx.x];
}

// pass 2: the value carried into every chunk (one thread; chunks are few)
__global__ void scan_carry_kernel(double* __restrict__ chunk_end, int chunks, double r) {
  if (blockIdx.x != 0 || threadIdx.x != 0) return;
  const double rc = pow(r, (double)kScanChunk);
  double carry = 0.0;
  for (int c = 0; c < chunks; ++c) {
    const double e = chunk_end[c];
    chunk_end[c] = carry;                 // carried into chunk c
    carry = rc * carry + e;               // the global value at its end
  }
}

// pass 3: add each chunk's carry, decayed by r^(k + 1)
__global__ void scan_apply_kernel(double* __restrict__ y, int n, double r, int rev,
                                  const double* __restrict__ carry_in) {
  const int64_t q = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (q >= n) return;
  const int64_t c = q / kScanChunk, k = q - c * kScanChunk;
  const double carry = carry_in[c];
  if (carry != 0.0) y[seq_index(q, n, rev)] += pow(r, (double)(k + 1)) * carry;
}

// ------------------------------------------------------ (L* - M~) x
// y_i = f_i + g_i - x_i - (1/s) sum_t (S[hi_t(i) - 1] - S[lo_t(i) - 1]),
// S the inclusive prefix sums of x (S[-1] = 0)
__global__ void combine_kernel(int n, int s, int64_t W, const BinRecord* __restrict__ rec,
                               const double* __restrict__ x, const double* __restrict__ f,
                               const double* __restrict__ g, const double* __restrict__ S,
                               double* __restrict__ y) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  double m = 0.0;
  for (int t = 0; t < s; ++t) {
    const BinRecord rc = load_record(rec, (int64_t)t * W + (i >> 5));
    const int lo = bin_lo(rc, i), hi = bin_hi(rc, i);
    m += S[hi - 1] - (lo > 0 ? S[lo - 1] : 0.0);
  }
  y[i] = f[i] + g[i] - x[i] - m / s;
}

// ------------------------------------------------------- small vector ops
// block partials of a . b, summed on the host in a fixed order
__global__ void __launch_bounds__(kRedThreads)
dot_kernel(const double* __restrict__ a, const double* __restrict__ b, int n,
           double* __restrict__ part) {
  __shared__ double red[kRedThreads / 32];
  double v = 0.0;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
    v = fma(a[i], b[i], v);
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < kRedThreads / 32; ++w) t += red[w];
    part[blockIdx.x] = t;
  }
}

// w = w - alpha v - beta v_prev
__global__ void lanczos_update_kernel(double* __restrict__ w, const double* __restrict__ v,
                                      const double* __restrict__ vp, int n, double alpha,
                                      double beta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) w[i] = w[i] - alpha * v[i] - beta * vp[i];
}

// v_prev = v; v = w / beta
__global__ void lanczos_shift_kernel(double* __restrict__ vp, double* __restrict__ v,
                                     const double* __restrict__ w, int n, double inv_beta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) {
    vp[i] = v[i];
    v[i] = w[i] * inv_beta;
  }
}

// number of eigenvalues below x of the symmetric tridiagonal matrix with
// diagonal a and off-diagonal b (Sturm sequence of the LDL^T pivots)
int sturm_below(const std::vector<double>& a, const std::vector<double>& b, double x) {
  int cnt = 0;
  double d = 1.0;
  for (size_t i = 0; i < a.size(); ++i) {
    d = a[i] - x - (i > 0 ? b[i - 1] * b[i - 1] / d : 0.0);
    if (d == 0.0) d = -1e-300;
    if (d < 0.0) ++cnt;
  }
  return cnt;
}

// the k-th smallest eigenvalue (0-based) by bisection inside the Gershgorin bound
double tridiag_eig(const std::vector<double>& a, const std::vector<double>& b, int k) {
  double g = 0.0;
  for (size_t i = 0; i < a.size(); ++i) {
    double r = fabs(a[i]);
    if (i > 0) r += fabs(b[i - 1]);
    if (i + 1 < a.size()) r += fabs(b[i]);
    g = std::max(g, r);
  }
  double lo = -g - 1.0, hi = g + 1.0;
  for (int it = 0; it < 200 && hi - lo > 1e-15 * std::max(1.0, fabs(lo) + fabs(hi)); ++it) {
    const double mid = 0.5 * (lo + hi);
    if (sturm_below(a, b, mid) > k) hi = mid;
    else lo = mid;
  }
  return 0.5 * (lo + hi);
}

// a seeded start vector (splitmix64 -> uniform in (-1, 1))
void start_vector(std::vector<double>& v, uint64_t seed) {
  uint64_t z = seed;
  for (double& e : v) {
    z += 0x9e3779b97f4a7c15ull;
    uint64_t q = z;
    q = (q ^ (q >> 30)) * 0xbf58476d1ce4e5b9ull;
    q = (q ^ (q >> 27)) * 0x94d049bb133111ebull;
    q ^= q >> 31;
    e = ((double)(q >> 11) + 0.5) * (1.0 / 9007199254740992.0) * 2.0 - 1.0;
  }
}

struct Scan {
  int n, chunks;
  double* ends;
  cudaError_t run(const double* x, double* y, double r, bool rev, cudaStream_t st) const {
    scan_local_kernel<<<chunks, kScanThreads, 0, st>>>(x, y, n, r, rev ? 1 : 0, ends);
    scan_carry_kernel<<<1, 1, 0, st>>>(ends, chunks, r);
    scan_apply_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, n, r, rev ? 1 : 0, ends);
    return cudaGetLastError();
  }
};

}  // namespace

// Both norms of L* - M~ for head h of `b` (records of hash t of head h at
// rec + (h s + t) W).  max_abs / spectral may be null to skip one.  Blocks on
// `st`; returns the first CUDA error.
cudaError_t bias_error(const plsh_bins* bn, double sigma, int h, int iters, uint64_t seed,
                       double* max_abs, double* spectral, cudaStream_t st) {
  const int n = (int)bn->n, s = bn->s;
  const BinRecord* rec = bn->d_rec + (int64_t)h * s * bn->W;
  cudaError_t e = cudaSuccess;
  if (max_abs) {
    unsigned long long* d_best = nullptr;
    if ((e = cudaMalloc(&d_best, sizeof(unsigned long long))) != cudaSuccess) return e;
    e = cudaMemsetAsync(d_best, 0, sizeof(unsigned long long), st);
    if (e == cudaSuccess) {
      const int blocks = std::min((n + 255) / 256, 4096);
      rowmax_kernel<<<blocks, 256, 0, st>>>(n, s, bn->W, rec, sigma, d_best);
      e = cudaGetLastError();
    }
    unsigned long long bits = 0;
    if (e == cudaSuccess) e = cudaMemcpyAsync(&bits, d_best, sizeof(bits), cudaMemcpyDeviceToHost, st);
    if (e == cudaSuccess) e = cudaStreamSynchronize(st);
    cudaFree(d_best);
    if (e != cudaSuccess) return e;
    double v;
    memcpy(&v, &bits, sizeof(v));
    *max_abs = v;
  }
  if (!spectral) return cudaSuccess;

  // Lanczos on A = L* - M~: vectors v, v_prev, w and the scan outputs f, g, S
  const int red_blocks = std::min((n + kRedThreads - 1) / kRedThreads, 1024);
  const int chunks = (n + kScanChunk - 1) / kScanChunk;
  double* buf = nullptr;
  const size_t vec = (size_t)n;
  if ((e = cudaMalloc(&buf, sizeof(double) * (6 * vec + chunks + red_blocks))) != cudaSuccess)
    return e;
  double *v = buf, *vp = buf + vec, *w = buf + 2 * vec, *f = buf + 3 * vec, *g = buf + 4 * vec,
         *S = buf + 5 * vec, *ends = buf + 6 * vec, *part = ends + chunks;
  const Scan scan{n, chunks, ends};
  const double r = exp(-1.0 / sigma);
  std::vector<double> hv(vec), hp(red_blocks), al, be;
  auto dot = [&](const double* a, const double* b2, double* out) -> cudaError_t {
    dot_kernel<<<red_blocks, kRedThreads, 0, st>>>(a, b2, n, part);
    cudaError_t e2 = cudaMemcpyAsync(hp.data(), part, sizeof(double) * red_blocks,
                                     cudaMemcpyDeviceToHost, st);
    if (e2 == cudaSuccess) e2 = cudaStreamSynchronize(st);
    double t = 0.0;
    for (double x : hp) t += x;
    *out = t;
    return e2;
  };
  start_vector(hv, seed);
  double nrm = 0.0;
  for (double x : hv) nrm += x * x;
  nrm = sqrt(nrm);
  for (double& x : hv) x /= nrm;
  e = cudaMemcpyAsync(v, hv.data(), sizeof(double) * vec, cudaMemcpyHostToDevice, st);
  if (e == cudaSuccess) e = cudaMemsetAsync(vp, 0, sizeof(double) * vec, st);
  double beta = 0.0;
  const unsigned eb = (unsigned)((n + 255) / 256);
  for (int k = 0; k < iters && e == cudaSuccess; ++k) {
    // w = (L* - M~) v
    if ((e = scan.run(v, f, r, false, st)) != cudaSuccess) break;
    if ((e = scan.run(v, g, r, true, st)) != cudaSuccess) break;
    if ((e = scan.run(v, S, 1.0, false, st)) != cudaSuccess) break;
    combine_kernel<<<eb, 256, 0, st>>>(n, s, bn->W, rec, v, f, g, S, w);
    double alpha = 0.0, bnew = 0.0;
    if ((e = dot(v, w, &alpha)) != cudaSuccess) break;
    lanczos_update_kernel<<<eb, 256, 0, st>>>(w, v, vp, n, alpha, beta);
    if ((e = dot(w, w, &bnew)) != cudaSuccess) break;
    bnew = sqrt(bnew);
    al.push_back(alpha);
    if (k + 1 == iters || bnew < 1e-14) break;
    be.push_back(bnew);
    lanczos_shift_kernel<<<eb, 256, 0, st>>>(vp, v, w, n, 1.0 / bnew);
    if ((e = cudaGetLastError()) != cudaSuccess) break;
    beta = bnew;
  }
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  cudaFree(buf);
  if (e != cudaSuccess) return e;
  be.resize(al.size() > 0 ? al.size() - 1 : 0);
  const double lmin = tridiag_eig(al, be, 0), lmax = tridiag_eig(al, be, (int)al.size() - 1);
  *spectral = std::max(fabs(lmin), fabs(lmax));
  return cudaSuccess;
}

}  // namespace plsh
