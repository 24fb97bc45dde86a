// One decode step of Positional LSH attention: the query of one new position
// against the cached keys and values.
//
// "Positional LSH: Binary Block Matrix Approximation for Attention with Linear
// Biases", technical summary, Methodology 3: row i of the approximation is
//   O_i = sum_t sum_{j in J_t(i)} e^{S_ij} v_j / sum_t sum_{j in J_t(i)} e^{S_ij},
// with J_t(i) the bin of i under hash t clipped to j <= i.  For a decode step
// i = pos is the newest position and every key sits at or before it, so
// J_t(pos) = [lo_t(pos), pos] and the row is
//   O = sum_j c_j e^{S_j} v_j / sum_j c_j e^{S_j},  c_j = #{t : lo_t(pos) <= j},
// over j in [min_t lo_t(pos), pos]: a short attention over the row's key
// envelope with integer weights, bound by the bytes of K and V it reads.
//
// Work is split over the envelope (flash-decoding style): each (batch
// element, head) gets S splits (S chosen on the host so that the GPU holds
// enough warps), a warp per split.  The warp finds the row's envelope from
// its s bin records, takes its share of it in blocks of 64 keys with an
// online softmax (scores a key per lane, P V with a row slice of 16 bytes per
// lane, no block-wide barrier anywhere) and writes its max m, row sum l and
// unnormalised P V; a second kernel merges the S splits of each (batch
// element, head) and writes O = P V / l.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "bins_dev.cuh"
#include "plsh_internal.h"

namespace plsh {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

template <typename T> struct Vec;
template <> struct Vec<__nv_bfloat16> {
  // raw 16 bytes of a row, converted element by element where they are used
  using Raw = uint4;
  __device__ static Raw raw(const __nv_bfloat16* p) { return *reinterpret_cast<const uint4*>(p); }
  __device__ static float elem(const Raw& r, int e) {
    const uint32_t w = e < 2 ? r.x : (e < 4 ? r.y : (e < 6 ? r.z : r.w));
    return __uint_as_float((e & 1) ? (w & 0xffff0000u) : (w << 16));
  }
  __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <> struct Vec<float> {
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

// q . k over one row of D elements, eight per load, half a bf16 row (a
// quarter of an fp32 row) in flight at a time
template <typename T, int D>
__device__ __forceinline__ float row_dot(const float* __restrict__ qs, const T* __restrict__ k) {
  constexpr int L = sizeof(T) == 2 ? D / 16 : D / 32;  // loads in flight (64 bytes each lane)
  float a0 = 0.f, a1 = 0.f;
#pragma unroll
  for (int e0 = 0; e0 < D; e0 += 8 * L) {
    typename Vec<T>::Raw r[L];
#pragma unroll
    for (int u = 0; u < L; ++u) r[u] = Vec<T>::raw(k + e0 + 8 * u);
#pragma unroll
    for (int u = 0; u < L; ++u) {
#pragma unroll
      for (int e = 0; e < 8; e += 2) {
        a0 = fmaf(qs[e0 + 8 * u + e], Vec<T>::elem(r[u], e), a0);
        a1 = fmaf(qs[e0 + 8 * u + e + 1], Vec<T>::elem(r[u], e + 1), a1);
      }
    }
  }
  return a0 + a1;
}

struct DecodeParams {
  const void* q;        // [B, Hq, 1, D]
  const void* K;        // [B, Hkv, n, D]
  const void* V;
  const BinRecord* rec;  // [Hq * s][W]
  int B, Hq, Hkv, n, s;
  int64_t W;
  int pos;
  int splits;           // S
  float* part_m;        // [B * Hq * S]
  float* part_l;
  float* part_o;        // [B * Hq * S][D]
};

constexpr int kBlockKeys = 64;            // keys a warp scores at a time

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
__device__ __forceinline__ int warp_min_int(int v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

template <typename T, int D>
__global__ void __launch_bounds__(kThreads, 3)
decode_partial_kernel(DecodeParams p) {
  constexpr int S8 = D / 8;               // lanes per row in P V (16 bytes of bf16 each)
  constexpr int R = 32 / S8;              // rows per warp-wide load
  __shared__ float qs_all[kWarps][D];
  __shared__ float ps_all[kWarps][kBlockKeys];
  __shared__ int los_all[kWarps][kMaxS];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * kWarps + warp;
  if (item >= p.B * p.Hq * p.splits) return;   // whole warps only
  float* qs = qs_all[warp];
  float* ps = ps_all[warp];
  int* los = los_all[warp];
  const int bh = item / p.splits, split = item % p.splits;
  const int b = bh / p.Hq, h = bh % p.Hq;
  const int kvh = h / (p.Hq / p.Hkv);

  // the row's bin start under every hash of head h (s <= 64), its minimum,
  // and the query in log2 units
  int lo_a = p.pos, lo_b = p.pos;
  const int64_t rbase = (int64_t)h * p.s * p.W + (p.pos >> 5);
  if (lane < p.s) lo_a = bin_lo(load_record(p.rec, rbase + (int64_t)lane * p.W), p.pos);
  if (lane + 32 < p.s) lo_b = bin_lo(load_record(p.rec, rbase + (int64_t)(lane + 32) * p.W), p.pos);
  los[lane] = lo_a;
  los[lane + 32] = lo_b;
  const float scale = 1.4426950408889634f * rsqrtf((float)D);   // log2(e) / sqrt(d)
  const T* q = static_cast<const T*>(p.q) + (int64_t)bh * D;
  for (int e = lane; e < D; e += 32) qs[e] = Vec<T>::one(q + e) * scale;
  const int lo_min = warp_min_int(min(lo_a, lo_b));
  __syncwarp();

  // this split's share of the envelope [lo_min, pos]
  const int env = p.pos - lo_min + 1;
  const int len = (env + p.splits - 1) / p.splits;
  const int j_begin = lo_min + split * len;
  const int j_end = min(p.pos + 1, j_begin + len);

  const T* Kh = static_cast<const T*>(p.K) + ((int64_t)b * p.Hkv + kvh) * p.n * D;
  const int sl = lane % S8, rg = lane / S8;
  const T* Vh = static_cast<const T*>(p.V) + ((int64_t)b * p.Hkv + kvh) * p.n * D + sl * 8;
  float m = -INFINITY, l = 0.f;
  float acc[8];
#pragma unroll
  for (int e = 0; e < 8; ++e) acc[e] = 0.f;
  for (int j0 = j_begin; j0 < j_end; j0 += kBlockKeys) {
    const int cnt = min(kBlockKeys, j_end - j0);
    // scores of keys j0 + lane and j0 + lane + 32, the multiplicity folded
    // into the exponent: c_j 2^x = 2^(x + log2 c_j), c_j >= 1 in the envelope
    float x[2];
#pragma unroll 1
    for (int u = 0; u < 2; ++u) {
      const int jj = lane + 32 * u;
      x[u] = -INFINITY;
      if (jj < cnt) {
        const int j = j0 + jj;
        int c = 0;
        for (int t = 0; t < p.s; ++t) c += los[t] <= j ? 1 : 0;
        x[u] = row_dot<T, D>(qs, Kh + (int64_t)j * D) + __log2f((float)c);
      }
    }
    const float m_new = fmaxf(m, warp_max(fmaxf(x[0], x[1])));
    const float f = exp2f(m - m_new);        // 0 on the first block (m = -inf)
    const float p0 = exp2f(x[0] - m_new), p1 = exp2f(x[1] - m_new);
    l = l * f + warp_sum(p0 + p1);
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] *= f;
    ps[lane] = p0;
    ps[lane + 32] = p1;
    __syncwarp();
    // P V over the block's rows, R rows per warp-wide load, U loads in flight
    constexpr int U = sizeof(T) == 2 ? 8 : 4;
    for (int r0 = rg; r0 < cnt; r0 += U * R) {
      typename Vec<T>::Raw v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rr = r0 + u * R;
        if (rr < cnt) v[u] = Vec<T>::raw(Vh + (int64_t)(j0 + rr) * D);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int rr = r0 + u * R;
        if (rr < cnt) {
          const float w = ps[rr];
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[e] = fmaf(w, Vec<T>::elem(v[u], e), acc[e]);
        }
      }
    }
    m = m_new;
    __syncwarp();   // ps is rewritten by the next block
  }
  // lanes holding the same slice of different rows add up
#pragma unroll
  for (int o = S8; o < 32; o <<= 1)
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  if (rg == 0) {
#pragma unroll
    for (int e = 0; e < 8; ++e) p.part_o[(int64_t)item * D + sl * 8 + e] = acc[e];
  }
  if (lane == 0) {
    p.part_m[item] = m;    // -inf and 0 for a split past the envelope
    p.part_l[item] = l;
  }
}

// O = sum_k 2^(m_k - m) P V_k / sum_k 2^(m_k - m) l_k over the non-empty splits
template <typename T, int D>
__global__ void __launch_bounds__(D)
decode_merge_kernel(DecodeParams p, void* out) {
  const int bh = blockIdx.x, e = threadIdx.x;
  const int64_t first = (int64_t)bh * p.splits;
  float m = -INFINITY;
  for (int k = 0; k < p.splits; ++k) m = fmaxf(m, p.part_m[first + k]);
  float l = 0.f, o = 0.f;
  for (int k = 0; k < p.splits; ++k) {
    if (p.part_l[first + k] == 0.f) continue;
    const float f = exp2f(p.part_m[first + k] - m);
    l = fmaf(f, p.part_l[first + k], l);
    o = fmaf(f, p.part_o[(first + k) * D + e], o);
  }
  Vec<T>::store(static_cast<T*>(out) + (int64_t)bh * D + e, o / l);
}

template <typename T, int D>
cudaError_t launch_typed(const DecodeParams& p, void* out, cudaStream_t st) {
  const int64_t warps = (int64_t)p.B * p.Hq * p.splits;
  decode_partial_kernel<T, D><<<(unsigned)((warps + kWarps - 1) / kWarps), kThreads, 0, st>>>(p);
  decode_merge_kernel<T, D><<<(unsigned)(p.B * p.Hq), D, 0, st>>>(p, out);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st) {
  DecodeParams p;
  p.q = a.q;
  p.K = a.K;
  p.V = a.V;
  p.rec = a.rec;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.n = a.n;
  p.s = a.s;
  p.W = a.W;
  p.pos = a.pos;
  p.splits = decode_splits(a.B, a.Hq, a.num_sms);
  p.part_m = a.work;
  p.part_l = a.work + (size_t)a.B * a.Hq * p.splits;
  p.part_o = a.work + 2 * (size_t)a.B * a.Hq * p.splits;
  if (a.dtype == PLSH_BF16)
    return a.d == 64 ? launch_typed<__nv_bfloat16, 64>(p, a.o, st)
                     : launch_typed<__nv_bfloat16, 128>(p, a.o, st);
  return a.d == 64 ? launch_typed<float, 64>(p, a.o, st) : launch_typed<float, 128>(p, a.o, st);
}

}  // namespace plsh
