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
// A CTA serves the query heads of one KV group (up to eight, a warp each) of
// one batch element, over a share of the union of their envelopes (the work
// is split over the envelope, flash-decoding style, into about twelve CTAs
// per SM in all; on large grids each group takes as many shares as its own
// expected envelope wants; the groups with the widest scales come first in
// the grid).  The group's key and value rows of a block (16 KB of each, 8 KB
// on large bf16 grids) arrive in shared memory by bulk asynchronous copies, double
// buffered, completing on an mbarrier with a bounded wait: in bf16 the key
// rows as one or two tensor-map tiles (128-byte rows of the tile, 128-byte
// swizzle: chunk c of row r lands at chunk c ^ (r & 7)), in fp32 a copy per
// key row into rows padded by 16 bytes, and one copy for the value rows.
// Every head of the group then reads them from shared memory: scores with a
// key per lane (the swizzle, or the padding, puts the same 16-byte chunk of
// consecutive rows in different banks, and every lane reads the same chunk
// of the query), an online softmax per head, P V with a slice of every row
// per lane.  Each (batch element, head, share) writes its max m, row
// sum l and unnormalised P V; a second kernel merges the shares into
// O = P V / l.
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include "bins_dev.cuh"
#include "plsh_internal.h"
#include "tc_ptx.cuh"

namespace plsh {
namespace {

using namespace ptx;

// bytes of K (and of V) per block: 16 KB, or 8 KB for bf16 grids of many
// CTAs (more CTAs resident per SM, each block sooner done)
constexpr int kStageBytes = 16384;
constexpr int kSmallStageBytes = 8192;
constexpr unsigned FULL = 0xffffffffu;
constexpr int kMaxGroupOrder = 32;   // more KV groups: index order, uniform shares

// 1-D bulk copy global -> shared memory, completion counted in bytes on an
// mbarrier of this CTA (both addresses 16-byte aligned, size a multiple of 16)
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

template <typename T> struct Elem;
template <> struct Elem<__nv_bfloat16> {
  __device__ static float one(const __nv_bfloat16* p) { return __bfloat162float(*p); }
  __device__ static void store(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }
};
template <> struct Elem<float> {
  __device__ static float one(const float* p) { return *p; }
  __device__ static void store(float* p, float v) { *p = v; }
};

// the 2 (f32) or 4 (bf16) consecutive values of a 32-bit word pair / quad
__device__ __forceinline__ float lo16(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float hi16(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

struct DecodeParams {
  const void* q;        // [B, Hq, 1, D]
  const void* K;        // [B, Hkv, n, D]
  const void* V;
  const BinRecord* rec;  // [Hq * s][W]
  int B, Hq, Hkv, n, s;
  int64_t W;
  int pos;
  int heads;            // query heads per CTA (<= 8)
  int hchunks;          // CTAs per KV group and share
  int splits;           // shares of the envelope
  // (kept small: the parameters are copied at every launch)
  uint8_t g_order[kMaxGroupOrder];    // KV groups, widest expected envelope first
  uint8_t g_shares[kMaxGroupOrder];   // shares of each group in that order (<= splits)
  uint8_t shares_of[kMaxGroupOrder];  // shares of group g (index order)
  int g_first[kMaxGroupOrder + 1];    // first CTA of each group in order; [Hkv]: the grid
  int ordered;          // 0: groups in index order, `splits` shares each
  float* part_m;        // [B * Hq * splits]
  float* part_l;
  float* part_o;        // [B * Hq * splits][D]
  int* err;
  uint64_t wait_ns;
};

template <typename T, int D, int kStage = kStageBytes>
struct Cfg {
  static constexpr int kRowBytes = D * (int)sizeof(T);
  static constexpr int kKeys = kStage / kRowBytes;             // keys per block
  static constexpr int kChunks = kRowBytes / 16;               // 16-byte chunks of a row
  static constexpr int kE = 16 / (int)sizeof(T);               // values per chunk
  static constexpr int kPV = D / 32;                           // values of a row per lane
  // bf16 keys by tensor-map tiles of 64 values x kKeys rows, swizzled; fp32
  // keys row by row into padded rows
  static constexpr bool kTiled = sizeof(T) == 2;
  static constexpr int kBoxes = kTiled ? kRowBytes / 128 : 0;  // tiles per block
  static_assert(!kTiled || (kBoxes >= 1 && kKeys <= 256), "a tile is 128 bytes x kKeys rows");
  static constexpr int kKStride = kTiled ? kRowBytes : kRowBytes + 16;
  static constexpr uint32_t kKStage = (uint32_t)(kKeys * kKStride);
  // K, V x two stages, and room to align the swizzled K stages to 1024 bytes
  static constexpr uint32_t kSmem = 2u * kKStage + 2u * kStage + (kTiled ? 1024u : 0u);
  // byte offset of chunk k of key row r in a K stage
  __device__ static uint32_t koff(int r, int k) {
    if constexpr (kTiled)
      return (uint32_t)((k >> 3) * (kKeys * 128) + r * 128 + (((k & 7) ^ (r & 7)) << 4));
    else
      return (uint32_t)(r * kKStride + k * 16);
  }
};

template <typename T, int D, int STAGE>
__global__ void __launch_bounds__(256)
decode_group_kernel(const __grid_constant__ CUtensorMap tmK, DecodeParams p) {
  using C = Cfg<T, D, STAGE>;
  extern __shared__ __align__(128) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  if constexpr (C::kTiled)
    smem += (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;   // swizzle atoms: 1 KB
  __shared__ float qs_all[8][D];
  __shared__ float ps_all[8][C::kKeys];
  __shared__ int los_all[8][kMaxS];
  __shared__ int lo_warp[8];
  __shared__ __align__(8) uint64_t full[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // a programmatic dependent of the kernel before it: nothing in global
  // memory is read before that kernel has completed
  grid_dep_wait();
  const int G = p.Hq / p.Hkv;
  // KV groups with the widest expected envelopes first (the CTAs with the
  // most blocks start in the first wave), every batch element of a group
  // together, each group cut into as many shares as its own envelope wants
  int cta = blockIdx.x, S = p.splits, gr = 0;
  if (p.ordered) {
    while (gr + 1 < p.Hkv && cta >= p.g_first[gr + 1]) ++gr;
    cta -= p.g_first[gr];
    S = p.g_shares[gr];
  }
  const int split = cta % S;
  cta /= S;
  const int hc = cta % p.hchunks;
  cta /= p.hchunks;
  const int b = cta % p.B;
  if (!p.ordered) gr = cta / p.B;
  const int g = p.ordered ? p.g_order[gr] : gr;
  const int hg = hc * p.heads + warp;                // head within the group
  const bool valid = hg < G;
  const int h = g * G + (valid ? hg : 0);
  float* qs = qs_all[warp];
  float* ps = ps_all[warp];
  int* los = los_all[warp];
  const volatile int* no_abort = nullptr;

  // this head's bin start under every hash (s <= 64), the query in log2 units
  int lo_a = p.pos, lo_b = p.pos;
  const int64_t rbase = (int64_t)h * p.s * p.W + (p.pos >> 5);
  if (lane < p.s) lo_a = bin_lo(load_record(p.rec, rbase + (int64_t)lane * p.W), p.pos);
  if (lane + 32 < p.s) lo_b = bin_lo(load_record(p.rec, rbase + (int64_t)(lane + 32) * p.W), p.pos);
  los[lane] = lo_a;
  los[lane + 32] = lo_b;
  const float scale = 1.4426950408889634f * rsqrtf((float)D);   // log2(e) / sqrt(d)
  const T* q = static_cast<const T*>(p.q) + ((int64_t)b * p.Hq + h) * D;
  for (int e = lane; e < D; e += 32) qs[e] = Elem<T>::one(q + e) * scale;
  int lo_min = min(lo_a, lo_b);
  for (int o = 16; o > 0; o >>= 1) lo_min = min(lo_min, __shfl_xor_sync(FULL, lo_min, o));
  if (lane == 0) lo_warp[warp] = valid ? lo_min : p.pos;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&full[0]), 1);
    mbar_init(smem_u32(&full[1]), 1);
    fence_barrier_init();
  }
  __syncthreads();

  // this CTA's share of the union of its heads' envelopes
  int lo_cta = p.pos;
  for (int w = 0; w < p.heads; ++w) lo_cta = min(lo_cta, lo_warp[w]);
  const int env = p.pos - lo_cta + 1;
  const int len = (env + S - 1) / S;
  const int j_begin = lo_cta + split * len;
  const int j_end = min(p.pos + 1, j_begin + len);
  const int nblk = j_begin < j_end ? (j_end - j_begin + C::kKeys - 1) / C::kKeys : 0;
  const uint8_t* Kg = static_cast<const uint8_t*>(p.K) +
                      ((int64_t)b * p.Hkv + g) * p.n * C::kRowBytes;
  const uint8_t* Vg = static_cast<const uint8_t*>(p.V) +
                      ((int64_t)b * p.Hkv + g) * p.n * C::kRowBytes;
  const uint32_t sK = smem_u32(smem), sV = sK + 2 * C::kKStage;
  // block blk into stage blk & 1, issued by warp 0: lane 0 posts the bytes,
  // then every lane copies its share of the key rows
  auto issue = [&](int blk) {
    const int j0 = j_begin + blk * C::kKeys;
    const int cnt = min(C::kKeys, j_end - j0);
    const uint32_t bytes = (uint32_t)(cnt * C::kRowBytes);
    const uint32_t st = (uint32_t)(blk & 1);
    const uint32_t fb = smem_u32(&full[st]);
    if constexpr (C::kTiled) {
      // whole tiles (rows past the block are loaded too; past n, zeros)
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, bytes + (uint32_t)(C::kBoxes * C::kKeys * 128));
        bulk_load(sV + st * STAGE, Vg + (int64_t)j0 * C::kRowBytes, bytes, fb);
#pragma unroll
        for (int x = 0; x < C::kBoxes; ++x)
          tma_load_3d(sK + st * C::kKStage + (uint32_t)(x * C::kKeys * 128), &tmK, fb, 64 * x,
                      j0, b * p.Hkv + g);
      }
    } else {
      if (lane == 0) {
        mbar_arrive_expect_tx(fb, 2 * bytes);
        bulk_load(sV + st * STAGE, Vg + (int64_t)j0 * C::kRowBytes, bytes, fb);
      }
      __syncwarp();
      for (int r = lane; r < cnt; r += 32)
        bulk_load(sK + st * C::kKStage + (uint32_t)r * C::kKStride,
                  Kg + (int64_t)(j0 + r) * C::kRowBytes, C::kRowBytes, fb);
    }
  };
  int issued = 0;
  if (warp == 0) {
    for (; issued < 2 && issued < nblk; ++issued) issue(issued);
  }

  float m = -INFINITY, l = 0.f;
  float acc[C::kPV];
#pragma unroll
  for (int e = 0; e < C::kPV; ++e) acc[e] = 0.f;
  bool ok = true;
  int blk = 0;
  for (; blk < nblk; ++blk) {
    const uint32_t st = (uint32_t)(blk & 1);
    const bool got = mbar_wait(smem_u32(&full[st]), (uint32_t)(blk >> 1) & 1u, no_abort, p.wait_ns);
    ok = __syncthreads_and(got) != 0;
    if (!ok) break;
    const int j0 = j_begin + blk * C::kKeys;
    const int cnt = min(C::kKeys, j_end - j0);
    const uint32_t kst = sK + st * C::kKStage;
    const uint8_t* vst = smem + 2 * C::kKStage + st * STAGE;
    if (valid) {
      // scores of keys j0 + lane + 32 u, the multiplicity folded into the
      // exponent: c_j 2^x = 2^(x + log2 c_j); c_j = 0 outside this head's
      // envelope
      float x[C::kKeys / 32];
#pragma unroll
      for (int u = 0; u < C::kKeys / 32; ++u) {
        const int jj = lane + 32 * u;
        x[u] = -INFINITY;
        if (jj < cnt) {
          const int j = j0 + jj;
          int c = 0;
          for (int t = 0; t < p.s; ++t) c += los[t] <= j ? 1 : 0;
          if (c > 0) {
            float a0 = 0.f, a1 = 0.f;
#pragma unroll 4
            for (int k = 0; k < C::kChunks; ++k) {
              const uint4 kv = ld_shared_v4(kst + C::koff(jj, k));
              const float* qq = qs + k * C::kE;
              if constexpr (sizeof(T) == 2) {
                a0 = fmaf(qq[0], lo16(kv.x), a0);
                a1 = fmaf(qq[1], hi16(kv.x), a1);
                a0 = fmaf(qq[2], lo16(kv.y), a0);
                a1 = fmaf(qq[3], hi16(kv.y), a1);
                a0 = fmaf(qq[4], lo16(kv.z), a0);
                a1 = fmaf(qq[5], hi16(kv.z), a1);
                a0 = fmaf(qq[6], lo16(kv.w), a0);
                a1 = fmaf(qq[7], hi16(kv.w), a1);
              } else {
                a0 = fmaf(qq[0], __uint_as_float(kv.x), a0);
                a1 = fmaf(qq[1], __uint_as_float(kv.y), a1);
                a0 = fmaf(qq[2], __uint_as_float(kv.z), a0);
                a1 = fmaf(qq[3], __uint_as_float(kv.w), a1);
              }
            }
            x[u] = a0 + a1 + __log2f((float)c);
          }
        }
      }
      float mx = x[0];
#pragma unroll
      for (int u = 1; u < C::kKeys / 32; ++u) mx = fmaxf(mx, x[u]);
      for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, o));
      const float m_new = fmaxf(m, mx);
      if (m_new > -INFINITY) {
        const float f = exp2f(m - m_new);        // 0 while m = -inf
        float sum = 0.f;
#pragma unroll
        for (int u = 0; u < C::kKeys / 32; ++u) {
          const float pu = exp2f(x[u] - m_new);
          ps[lane + 32 * u] = pu;
          sum += pu;
        }
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(FULL, sum, o);
        l = l * f + sum;
#pragma unroll
        for (int e = 0; e < C::kPV; ++e) acc[e] *= f;
        m = m_new;
        __syncwarp();
        // P V: lane takes values lane * kPV .. of every row of the block
        const uint8_t* vcol = vst + lane * C::kPV * (int)sizeof(T);
#pragma unroll 4
        for (int jj = 0; jj < cnt; ++jj) {
          const float w = ps[jj];
          const uint8_t* vr = vcol + jj * C::kRowBytes;
          if constexpr (sizeof(T) == 2 && C::kPV == 4) {
            const uint2 v2 = *reinterpret_cast<const uint2*>(vr);
            acc[0] = fmaf(w, lo16(v2.x), acc[0]);
            acc[1] = fmaf(w, hi16(v2.x), acc[1]);
            acc[2] = fmaf(w, lo16(v2.y), acc[2]);
            acc[3] = fmaf(w, hi16(v2.y), acc[3]);
          } else if constexpr (sizeof(T) == 2) {
            const uint32_t v1 = *reinterpret_cast<const uint32_t*>(vr);
            acc[0] = fmaf(w, lo16(v1), acc[0]);
            acc[1] = fmaf(w, hi16(v1), acc[1]);
          } else {
            const float* vf = reinterpret_cast<const float*>(vr);
#pragma unroll
            for (int e = 0; e < C::kPV; ++e) acc[e] = fmaf(w, vf[e], acc[e]);
          }
        }
        __syncwarp();   // ps is rewritten by the next block
      }
    }
    // every warp is done with this stage: refill it with the block after next
    __syncthreads();
    if (warp == 0 && issued < nblk) {
      issue(issued);
      ++issued;
    }
  }
  if (!ok) {
    // let the copies issued and not yet waited for land before the CTA's
    // memory goes away
    if (warp == 0) {
      for (int k = blk; k < issued; ++k)
        mbar_wait(smem_u32(&full[k & 1]), (uint32_t)(k >> 1) & 1u, no_abort, p.wait_ns);
      if (lane == 0) atomicOr(p.err, 1);
    }
    return;
  }
  if (valid) {
    const int64_t item = ((int64_t)b * p.Hq + h) * p.splits + split;
#pragma unroll
    for (int e = 0; e < C::kPV; ++e) p.part_o[item * D + lane * C::kPV + e] = acc[e];
    if (lane == 0) {
      p.part_m[item] = m;    // -inf and 0 for a share with no key of this head
      p.part_l[item] = l;
    }
  }
}

// O = sum_k 2^(m_k - m) P V_k / sum_k 2^(m_k - m) l_k over the non-empty shares
template <typename T, int D>
__global__ void __launch_bounds__(D)
decode_merge_kernel(DecodeParams p, void* out) {
  // launched as a programmatic dependent of the group kernel: its launch
  // overlaps that kernel's tail, and it reads the partials once it is done
  grid_dep_wait();
  const int bh = blockIdx.x, e = threadIdx.x;
  const int64_t first = (int64_t)bh * p.splits;
  const int S = p.ordered ? p.shares_of[(bh % p.Hq) / (p.Hq / p.Hkv)] : p.splits;
  float m = -INFINITY;
  for (int k = 0; k < S; ++k)
    if (p.part_l[first + k] > 0.f) m = fmaxf(m, p.part_m[first + k]);
  float l = 0.f, o = 0.f;
  for (int k = 0; k < S; ++k) {
    if (!(p.part_l[first + k] > 0.f)) continue;
    const float f = exp2f(p.part_m[first + k] - m);
    l = fmaf(f, p.part_l[first + k], l);
    o = fmaf(f, p.part_o[(first + k) * D + e], o);
  }
  Elem<T>::store(static_cast<T*>(out) + (int64_t)bh * D + e, o / l);
}

template <typename T, int D, int STAGE>
cudaError_t launch_staged(const DecodeParams& p, void* out, cudaStream_t st) {
  using C = Cfg<T, D, STAGE>;
  auto kern = decode_group_kernel<T, D, STAGE>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)C::kSmem);
  if (e != cudaSuccess) return e;
  // K as [B * Hkv planes, n rows, D] in tiles of 64 values x kKeys rows (bf16)
  CUtensorMap mk;
  memset(&mk, 0, sizeof mk);
  if (C::kTiled && !make_rows_map_bf16(&mk, p.K, (int64_t)p.B * p.Hkv, p.n, C::kKeys, D))
    return cudaErrorInvalidValue;
  const int64_t ctas =
      p.ordered ? p.g_first[p.Hkv] : (int64_t)p.B * p.Hkv * p.hchunks * p.splits;
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas);
    cfg.blockDim = dim3(32 * p.heads);
    cfg.dynamicSmemBytes = C::kSmem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, mk, p);
    if (e != cudaSuccess) return e;
  }
  {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * p.Hq));
    cfg.blockDim = dim3(D);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e2 = cudaLaunchKernelEx(&cfg, decode_merge_kernel<T, D>, p, out);
    if (e2 != cudaSuccess) return e2;
  }
  return cudaGetLastError();
}

// bf16 grids of at least four CTAs per SM take 8 KB stages (measured on the
// Mistral shape: 64 sequences 37.5 -> 33.7 us; at 8 sequences, 448 CTAs,
// the 16 KB stages stay ahead)
template <typename T, int D>
cudaError_t launch_typed(const DecodeParams& p, void* out, int num_sms, cudaStream_t st) {
  if constexpr (sizeof(T) == 2) {
    const int64_t ctas =
        p.ordered ? p.g_first[p.Hkv] : (int64_t)p.B * p.Hkv * p.hchunks * p.splits;
    if (ctas >= 4LL * num_sms) return launch_staged<T, D, kSmallStageBytes>(p, out, st);
  }
  return launch_staged<T, D, kStageBytes>(p, out, st);
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
  p.heads = decode_heads(a.Hq / a.Hkv);
  p.hchunks = (a.Hq / a.Hkv + p.heads - 1) / p.heads;
  p.splits = decode_splits(a.B, a.Hq, a.Hkv, a.num_sms, a.useful_splits);
  // the envelope of a group reaches about its widest scale back: groups by
  // their largest sigma, descending (stable)
  p.ordered = 0;
  if (a.sigma != nullptr && a.Hkv <= kMaxGroupOrder) {
    const int G = a.Hq / a.Hkv;
    double key[kMaxGroupOrder];
    for (int g = 0; g < a.Hkv; ++g) {
      key[g] = 0.0;
      for (int h = g * G; h < (g + 1) * G; ++h) key[g] = a.sigma[h] > key[g] ? a.sigma[h] : key[g];
      p.g_order[g] = (uint8_t)g;
    }
    for (int i = 1; i < a.Hkv; ++i)        // insertion sort, stable
      for (int j = i; j > 0 && key[p.g_order[j]] > key[p.g_order[j - 1]]; --j) {
        const uint8_t t = p.g_order[j];
        p.g_order[j] = p.g_order[j - 1];
        p.g_order[j - 1] = t;
      }
    // a grid of eight or more CTAs per SM: each group cut into shares of
    // about 64 keys of its own expected envelope (about 1.2 sigma + 32 keys;
    // at most `splits`, the call's share count, which sized the partials),
    // so that narrow groups do not spread a few keys over many CTAs; smaller
    // grids keep `splits` shares for every group (more CTAs run in parallel
    // there).  Measured on the Mistral shape: 32 and 64 sequences 20.1 ->
    // 17.5 and 24.8 -> 23.0 us back to back; at 1, 8 and 16 sequences the
    // per-group shares were slower.
    const bool per_group =
        (int64_t)a.B * a.Hkv * p.hchunks * p.splits >= 8LL * a.num_sms;
    int64_t first = 0;
    for (int gr = 0; gr < a.Hkv; ++gr) {
      const int g = p.g_order[gr];
      const double keys = 1.2 * key[g] + 32.0;
      const double lim = a.pos + 1.0 < keys ? a.pos + 1.0 : keys;
      const int want = per_group ? (int)(lim / 64.0 + 1.0) : p.splits;
      const int sh = want < 1 ? 1 : (want > p.splits ? p.splits : want);
      p.g_shares[gr] = (uint8_t)sh;
      p.shares_of[g] = (uint8_t)sh;
      p.g_first[gr] = (int)first;
      first += (int64_t)a.B * p.hchunks * sh;
    }
    p.g_first[a.Hkv] = (int)first;
    p.ordered = 1;
  }
  p.part_m = a.work;
  p.part_l = a.work + (size_t)a.B * a.Hq * p.splits;
  p.part_o = a.work + 2 * (size_t)a.B * a.Hq * p.splits;
  p.err = a.err;
  p.wait_ns = a.wait_ns;
  if (a.dtype == PLSH_BF16)
    return a.d == 64 ? launch_typed<__nv_bfloat16, 64>(p, a.o, a.num_sms, st)
                     : launch_typed<__nv_bfloat16, 128>(p, a.o, a.num_sms, st);
  return a.d == 64 ? launch_typed<float, 64>(p, a.o, a.num_sms, st)
                   : launch_typed<float, 128>(p, a.o, a.num_sms, st);
}

}  // namespace plsh
