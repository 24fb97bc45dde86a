// Backward pass of Positional LSH attention on the CUDA cores (a first,
// correctness-first form; the forward runs on the tensor cores).
//
// "Positional LSH: Binary Block Matrix Approximation for Attention with Linear
// Biases", technical summary, Methodology 3: row i of the approximation is
//   O_i = sum_j P_ij v_j,  P_ij = w_ij / l_i,  w_ij = c_ij e^{S_ij - m_i},
//   S_ij = q_i . k_j / sqrt(d),  l_i = sum_j w_ij,
// with c_ij the number of hashes that put i and j in one bin (j <= i when
// causal).  The multiplicities do not depend on Q, K, V, so with dO given:
//   dP_ij = dO_i . v_j,  Delta_i = sum_j P_ij dP_ij,
//   dS_ij = P_ij (dP_ij - Delta_i),
//   dQ_i = sum_j dS_ij k_j / sqrt(d),  dK_j = sum_i dS_ij q_i / sqrt(d),
//   dV_j = sum_i P_ij dO_i,
// a KV head collecting the sums of every query head that reads it.
//
// i and j share a bin of hash t exactly when the bin of j contains i, so the
// rows that see key j form an envelope too, [min_t lo_t(j), max_t hi_t(j))
// (from j up when causal).  Two kernels, no atomics:
//   row kernel   a warp per (b, h, i): m_i, l_i and Delta_i over the row's
//                keys (stored), then dQ_i;
//   key kernel   a warp per (b, kv head, j): for each query head of the
//                group, P_ij and dS_ij over the key's rows, then dK_j, dV_j.
// Scores take a key (or row) per lane with the whole row dot product;
// accumulations take a 16-byte slice of a row per lane.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bins_dev.cuh"
#include "plsh_internal.h"

namespace plsh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr float kLog2e = 1.4426950408889634f;

template <typename T> struct Row;
template <> struct Row<__nv_bfloat16> {
  using Raw = uint4;   // eight elements
  __device__ static Raw raw(const __nv_bfloat16* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ static float elem(const Raw& r, int e) {
    const uint32_t w = e < 2 ? r.x : (e < 4 ? r.y : (e < 6 ? r.z : r.w));
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <> struct Row<float> {
  struct Raw {
    float4 a, b;
  };
  __device__ static Raw raw(const float* p) {
    return Raw{*reinterpret_cast<const float4*>(p), *reinterpret_cast<const float4*>(p + 4)};
  }
  __device__ static float elem(const Raw& r, int e) {
    const float4& h = e < 4 ? r.a : r.b;
    const int k = e & 3;
    return k == 0 ? h.x : (k == 1 ? h.y : (k == 2 ? h.z : h.w));
  }
  __device__ static float one(const float* p) { return *p; }
  __device__ static void store(float* p, float v) { *p = v; }
};

// a . row over D elements, a in shared memory (fp32), row in global memory
template <typename T, int D>
__device__ __forceinline__ float dot_row(const float* __restrict__ a, const T* __restrict__ row) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll 4
  for (int e0 = 0; e0 < D; e0 += 8) {
    const typename Row<T>::Raw r = Row<T>::raw(row + e0);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
      s0 = fmaf(a[e0 + e], Row<T>::elem(r, e), s0);
      s1 = fmaf(a[e0 + e + 1], Row<T>::elem(r, e + 1), s1);
    }
  }
  return s0 + s1;
}

__device__ __forceinline__ float warp_max(float v) {
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

struct BwdParams {
  const void* Q;      // [B, Hq, n, D]
  const void* K;      // [B, Hkv, n, D]
  const void* V;
  const void* dO;     // [B, Hq, n, D]
  void* dQ;           // [B, Hq, n, D]
  void* dK;           // [B, Hkv, n, D]
  void* dV;
  float* stats;       // [B * Hq * n][3]: m (log2 units), l, Delta
  const BinRecord* rec;  // [Hq * s][W]
  int B, Hq, Hkv, n, s, causal;
  int64_t W;
};

// bin bounds of position x under every hash of head h into lo[], hi[]; the
// union [min lo, max hi) of the bins containing x
__device__ __forceinline__ void bounds(const BwdParams& p, int h, int x, int* lo, int* hi,
                                       int lane, int& umin, int& umax) {
  int a = x, b = x + 1;
  for (int t = lane; t < p.s; t += 32) {
    const BinRecord rc = load_record(p.rec, ((int64_t)h * p.s + t) * p.W + (x >> 5));
    lo[t] = bin_lo(rc, x);
    hi[t] = bin_hi(rc, x);
    a = min(a, lo[t]);
    b = max(b, hi[t]);
  }
  for (int o = 16; o > 0; o >>= 1) {
    a = min(a, __shfl_xor_sync(0xffffffffu, a, o));
    b = max(b, __shfl_xor_sync(0xffffffffu, b, o));
  }
  umin = a;
  umax = b;
  __syncwarp();
}

__device__ __forceinline__ int count_in(const int* lo, const int* hi, int s, int y) {
  int c = 0;
  for (int t = 0; t < s; ++t) c += (lo[t] <= y && y < hi[t]) ? 1 : 0;
  return c;
}

// ------------------------------------------------------------- row kernel
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
bwd_row_kernel(BwdParams p) {
  constexpr int S8 = D / 8, R = 32 / S8;
  __shared__ float qs_all[kWarps][D], dos_all[kWarps][D];
  __shared__ int lo_all[kWarps][kMaxS], hi_all[kWarps][kMaxS];
  __shared__ float ds_all[kWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  if (row >= (int64_t)p.B * p.Hq * p.n) return;
  float* qs = qs_all[warp];
  float* dos = dos_all[warp];
  int* lo = lo_all[warp];
  int* hi = hi_all[warp];
  float* ds = ds_all[warp];
  const int i = (int)(row % p.n);
  const int64_t bh = row / p.n;
  const int h = (int)(bh % p.Hq), b = (int)(bh / p.Hq);
  const int kvh = h / (p.Hq / p.Hkv);
  const float scale = kLog2e * rsqrtf((float)D);     // scores in log2 units
  const T* qrow = static_cast<const T*>(p.Q) + row * D;
  const T* dorow = static_cast<const T*>(p.dO) + row * D;
  for (int e = lane; e < D; e += 32) {
    qs[e] = Row<T>::one(qrow + e) * scale;
    dos[e] = Row<T>::one(dorow + e);
  }
  int umin, umax;
  bounds(p, h, i, lo, hi, lane, umin, umax);
  const int j0 = umin, j1 = p.causal ? i + 1 : umax;   // keys [j0, j1)
  const T* Kh = static_cast<const T*>(p.K) + ((int64_t)b * p.Hkv + kvh) * p.n * D;
  const T* Vh = static_cast<const T*>(p.V) + ((int64_t)b * p.Hkv + kvh) * p.n * D;

  // max, then the row sum and sum_j w_ij dP_ij
  float mx = -INFINITY;
  for (int j = j0 + lane; j < j1; j += 32)
    if (count_in(lo, hi, p.s, j) > 0) mx = fmaxf(mx, dot_row<T, D>(qs, Kh + (int64_t)j * D));
  const float m = warp_max(mx);
  float l = 0.f, wdp = 0.f;
  for (int j = j0 + lane; j < j1; j += 32) {
    const int c = count_in(lo, hi, p.s, j);
    if (c == 0) continue;
    const float w = c * exp2f(dot_row<T, D>(qs, Kh + (int64_t)j * D) - m);
    l += w;
    wdp = fmaf(w, dot_row<T, D>(dos, Vh + (int64_t)j * D), wdp);
  }
  l = warp_sum(l);
  const float delta = warp_sum(wdp) / l;
  if (lane == 0) {
    p.stats[row * 3 + 0] = m;
    p.stats[row * 3 + 1] = l;
    p.stats[row * 3 + 2] = delta;
  }

  // dQ_i = sum_j dS_ij k_j / sqrt(d): 32 keys' dS at a time, then slices
  const int sl = lane % S8, rg = lane / S8;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int base = j0; base < j1; base += 32) {
    const int j = base + lane;
    float dsv = 0.f;
    if (j < j1) {
      const int c = count_in(lo, hi, p.s, j);
      if (c > 0) {
        const float pij = c * exp2f(dot_row<T, D>(qs, Kh + (int64_t)j * D) - m) / l;
        dsv = pij * (dot_row<T, D>(dos, Vh + (int64_t)j * D) - delta);
      }
    }
    ds[lane] = dsv;
    __syncwarp();
    const int cnt = min(32, j1 - base);
    for (int r = rg; r < cnt; r += R) {
      const typename Row<T>::Raw kr = Row<T>::raw(Kh + (int64_t)(base + r) * D + sl * 8);
      const float w = ds[r];
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, Row<T>::elem(kr, e), acc[e]);
    }
    __syncwarp();
  }
  for (int o = S8; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  if (rg == 0) {
    const float inv = rsqrtf((float)D);
    T* out = static_cast<T*>(p.dQ) + row * D + sl * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) Row<T>::store(out + e, acc[e] * inv);
  }
}

// ------------------------------------------------------------- key kernel
template <typename T, int D>
__global__ void __launch_bounds__(kThreads)
bwd_key_kernel(BwdParams p) {
  constexpr int S8 = D / 8, R = 32 / S8;
  __shared__ float ks_all[kWarps][D], vs_all[kWarps][D];
  __shared__ int lo_all[kWarps][kMaxS], hi_all[kWarps][kMaxS];
  __shared__ float pp_all[kWarps][32], ds_all[kWarps][32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t key = (int64_t)blockIdx.x * kWarps + warp;
  if (key >= (int64_t)p.B * p.Hkv * p.n) return;
  float* ks = ks_all[warp];
  float* vs = vs_all[warp];
  int* lo = lo_all[warp];
  int* hi = hi_all[warp];
  float* pp = pp_all[warp];
  float* ds = ds_all[warp];
  const int j = (int)(key % p.n);
  const int64_t bk = key / p.n;
  const int kvh = (int)(bk % p.Hkv), b = (int)(bk / p.Hkv);
  const int group = p.Hq / p.Hkv;
  const float scale = kLog2e * rsqrtf((float)D);
  const T* krow = static_cast<const T*>(p.K) + key * D;
  const T* vrow = static_cast<const T*>(p.V) + key * D;
  for (int e = lane; e < D; e += 32) {
    ks[e] = Row<T>::one(krow + e) * scale;
    vs[e] = Row<T>::one(vrow + e);
  }
  __syncwarp();
  const int sl = lane % S8, rg = lane / S8;
  float dk[8], dv[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) dk[e] = dv[e] = 0.f;
  for (int hh = 0; hh < group; ++hh) {
    const int h = kvh * group + hh;
    int umin, umax;
    bounds(p, h, j, lo, hi, lane, umin, umax);
    const int i0 = p.causal ? j : umin, i1 = umax;      // rows [i0, i1)
    const int64_t rbase = ((int64_t)b * p.Hq + h) * p.n;
    const T* Qh = static_cast<const T*>(p.Q) + rbase * D;
    const T* dOh = static_cast<const T*>(p.dO) + rbase * D;
    for (int base = i0; base < i1; base += 32) {
      const int i = base + lane;
      float pv = 0.f, dsv = 0.f;
      if (i < i1) {
        const int c = count_in(lo, hi, p.s, i);
        if (c > 0) {
          const float* st = p.stats + (rbase + i) * 3;
          const float pij = c * exp2f(dot_row<T, D>(ks, Qh + (int64_t)i * D) - st[0]) / st[1];
          pv = pij;
          dsv = pij * (dot_row<T, D>(vs, dOh + (int64_t)i * D) - st[2]);
        }
      }
      pp[lane] = pv;
      ds[lane] = dsv;
      __syncwarp();
      const int cnt = min(32, i1 - base);
      for (int r = rg; r < cnt; r += R) {
        const typename Row<T>::Raw dr = Row<T>::raw(dOh + (int64_t)(base + r) * D + sl * 8);
        const typename Row<T>::Raw qr = Row<T>::raw(Qh + (int64_t)(base + r) * D + sl * 8);
        const float a = pp[r], g = ds[r];
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          dv[e] = fmaf(a, Row<T>::elem(dr, e), dv[e]);
          dk[e] = fmaf(g, Row<T>::elem(qr, e), dk[e]);
        }
      }
      __syncwarp();
    }
  }
  for (int o = S8; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      dk[e] += __shfl_xor_sync(0xffffffffu, dk[e], o);
      dv[e] += __shfl_xor_sync(0xffffffffu, dv[e], o);
    }
  if (rg == 0) {
    const float inv = rsqrtf((float)D);
    T* ok = static_cast<T*>(p.dK) + key * D + sl * 8;
    T* ov = static_cast<T*>(p.dV) + key * D + sl * 8;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      Row<T>::store(ok + e, dk[e] * inv);
      Row<T>::store(ov + e, dv[e]);
    }
  }
}

template <typename T, int D>
cudaError_t launch_typed(const BwdParams& p, cudaStream_t st) {
  const int64_t rows = (int64_t)p.B * p.Hq * p.n, keys = (int64_t)p.B * p.Hkv * p.n;
  bwd_row_kernel<T, D><<<(unsigned)((rows + kWarps - 1) / kWarps), kThreads, 0, st>>>(p);
  bwd_key_kernel<T, D><<<(unsigned)((keys + kWarps - 1) / kWarps), kThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

// Gradients of sum(O * dO) with respect to Q, K, V (see the file comment);
// stats: scratch of 3 B Hq n floats.
cudaError_t launch_attn_bwd(const void* Q, const void* K, const void* V, const void* dO, void* dQ,
                            void* dK, void* dV, float* stats, const plsh_bins* bn, int B, int Hq,
                            int Hkv, int n, int d, int causal, int dtype, cudaStream_t st) {
  BwdParams p;
  p.Q = Q;
  p.K = K;
  p.V = V;
  p.dO = dO;
  p.dQ = dQ;
  p.dK = dK;
  p.dV = dV;
  p.stats = stats;
  p.rec = bn->d_rec;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.n = n;
  p.s = bn->s;
  p.causal = causal;
  p.W = bn->W;
  if (dtype == PLSH_BF16)
    return d == 64 ? launch_typed<__nv_bfloat16, 64>(p, st) : launch_typed<__nv_bfloat16, 128>(p, st);
  return d == 64 ? launch_typed<float, 64>(p, st) : launch_typed<float, 128>(p, st);
}

}  // namespace plsh
