// CUDA-core attention for fp32 inputs and for d = 64 (one warp per query
// row).  Same result as the tensor-core path:
//   Positional LSH ("Positional LSH: Binary Block Matrix Approximation for
//   Attention with Linear Biases", technical summary, Methodology 3):
//     O_i = sum_j c_ij e^{S_ij} v_j / sum_j c_ij e^{S_ij},
//     c_ij = #{t : j in the bin of i under hash t} (j <= i when causal)
//   exact ALiBi (Problem statement, Methodology 1):
//     O_i = sum_j e^{S_ij - |i-j|/sigma_h} v_j / sum_j e^{S_ij - |i-j|/sigma_h}
// Lane l of the warp owns key j0 + l of each 32-key chunk for the scores and
// output columns l, l+32, ... for the accumulator; online softmax in fp32
// (log2 domain).
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bins_dev.cuh"
#include "plsh_internal.h"

namespace plsh {
namespace {

constexpr int kWarps = 8;

template <typename T>
__device__ __forceinline__ float to_f(T v);
template <>
__device__ __forceinline__ float to_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ float to_f<__nv_bfloat16>(__nv_bfloat16 v) {
  return __bfloat162float(v);
}

template <typename T>
__device__ __forceinline__ T from_f(float v);
template <>
__device__ __forceinline__ float from_f<float>(float v) { return v; }
template <>
__device__ __forceinline__ __nv_bfloat16 from_f<__nv_bfloat16>(float v) {
  return __float2bfloat16_rn(v);
}

struct SimtParams {
  AttnArgs a;
  float slope_log2[512];   // exact mode: log2(e) / sigma_h
};

template <typename T, int D>
__global__ void __launch_bounds__(kWarps * 32)
attn_simt_kernel(const __grid_constant__ SimtParams p) {
  const AttnArgs& a = p.a;
  constexpr int PER_LANE = D / 32;
  __shared__ float q_s[kWarps][D];
  __shared__ int lo_s[kWarps][kMaxS];
  __shared__ int hi_s[kWarps][kMaxS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t row = (int64_t)blockIdx.x * kWarps + warp;
  const int64_t total = (int64_t)a.B * a.Hq * a.n;
  if (row >= total) return;
  const int i = (int)(row % a.n);
  const int64_t bh = row / a.n;
  const int h = (int)(bh % a.Hq);
  const int b = (int)(bh / a.Hq);
  const int kvh = h / (a.Hq / a.Hkv);
  const T* Q = static_cast<const T*>(a.Q);
  const T* K = static_cast<const T*>(a.K) + ((int64_t)b * a.Hkv + kvh) * a.n * D;
  const T* V = static_cast<const T*>(a.V) + ((int64_t)b * a.Hkv + kvh) * a.n * D;
  const float scale_log2 = 1.4426950408889634f / sqrtf((float)D);
  for (int c = lane; c < D; c += 32) q_s[warp][c] = to_f(Q[row * D + c]);

  int jlo, jhi;
  if (a.exact) {
    jlo = 0;
    jhi = a.causal ? i + 1 : a.n;
  } else {
    int mylo = a.n, myhi = 0;
    for (int t = lane; t < a.s; t += 32) {
      const BinRecord r = load_record(a.rec, ((int64_t)h * a.s + t) * a.W + (i >> 5));
      const int lo = bin_lo(r, i);
      int hi = bin_hi(r, i);
      if (a.causal && hi > i + 1) hi = i + 1;
      lo_s[warp][t] = lo;
      hi_s[warp][t] = hi;
      mylo = min(mylo, lo);
      myhi = max(myhi, hi);
    }
    jlo = __reduce_min_sync(0xffffffffu, mylo);
    jhi = __reduce_max_sync(0xffffffffu, myhi);
  }
  __syncwarp();
  const float slope = a.exact ? p.slope_log2[h] : 0.f;

  float m = -INFINITY, l = 0.f;
  float acc[PER_LANE];
#pragma unroll
  for (int k = 0; k < PER_LANE; ++k) acc[k] = 0.f;

  for (int j0 = jlo; j0 < jhi; j0 += 32) {
    const int j = j0 + lane;
    float x = -INFINITY;
    if (j < jhi) {
      const T* kr = K + (int64_t)j * D;
      float dot = 0.f;
#pragma unroll 16
      for (int c = 0; c < D; ++c) dot = fmaf(q_s[warp][c], to_f(kr[c]), dot);
      if (a.exact) {
        const float dist = (float)(i > j ? i - j : j - i);
        x = fmaf(dot, scale_log2, -dist * slope);
      } else {
        int cnt = 0;
        for (int t = 0; t < a.s; ++t)
          cnt += (lo_s[warp][t] <= j) & (j < hi_s[warp][t]);
        if (cnt > 0) x = fmaf(dot, scale_log2, log2f((float)cnt));
      }
    }
    float mc = x;
#pragma unroll
    for (int o = 16; o; o >>= 1) mc = fmaxf(mc, __shfl_xor_sync(0xffffffffu, mc, o));
    const float m_new = fmaxf(m, mc);
    if (m_new == -INFINITY) continue;
    const float alpha = exp2f(m - m_new);
    const float pj = (x == -INFINITY) ? 0.f : exp2f(x - m_new);
    float ps = pj;
#pragma unroll
    for (int o = 16; o; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    l = l * alpha + ps;
#pragma unroll
    for (int k = 0; k < PER_LANE; ++k) acc[k] *= alpha;
    const int nk = min(32, jhi - j0);
    for (int jj = 0; jj < nk; ++jj) {
      const float w = __shfl_sync(0xffffffffu, pj, jj);
      if (w == 0.f) continue;
      const T* vr = V + (int64_t)(j0 + jj) * D;
#pragma unroll
      for (int k = 0; k < PER_LANE; ++k) acc[k] = fmaf(w, to_f(vr[lane + 32 * k]), acc[k]);
    }
    m = m_new;
  }
  T* O = static_cast<T*>(a.O);
  const float inv = 1.f / l;
#pragma unroll
  for (int k = 0; k < PER_LANE; ++k) O[row * D + lane + 32 * k] = from_f<T>(acc[k] * inv);
}

}  // namespace

cudaError_t launch_attn_simt(const AttnArgs& a, const float* slopes_host,
                             int dtype, cudaStream_t st) {
  SimtParams p;
  p.a = a;
  for (int h = 0; h < 512; ++h) p.slope_log2[h] = (slopes_host && h < a.Hq) ? slopes_host[h] : 0.f;
  const int64_t rows = (int64_t)a.B * a.Hq * a.n;
  const unsigned grid = (unsigned)((rows + kWarps - 1) / kWarps);
  if (dtype == PLSH_F32) {
    if (a.d == 64) attn_simt_kernel<float, 64><<<grid, kWarps * 32, 0, st>>>(p);
    else attn_simt_kernel<float, 128><<<grid, kWarps * 32, 0, st>>>(p);
  } else {
    if (a.d == 64) attn_simt_kernel<__nv_bfloat16, 64><<<grid, kWarps * 32, 0, st>>>(p);
    else attn_simt_kernel<__nv_bfloat16, 128><<<grid, kWarps * 32, 0, st>>>(p);
  }
  return cudaGetLastError();
}

}  // namespace plsh
