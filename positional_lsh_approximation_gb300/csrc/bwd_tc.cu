// Backward pass of Positional LSH attention on the sm_103a tensor cores.
//
// "Positional LSH: Binary Block Matrix Approximation for Attention with Linear
// Biases", technical summary, Methodology 3: row i of the approximation is
//   O_i = sum_j P_ij v_j,  P_ij = c_ij 2^{x_ij - m_i} / l_i,
//   x_ij = q_i . k_j log2(e) / sqrt(d),
// c_ij the number of hashes that put i and j in one bin (j <= i when causal),
// m_i a per-row shift and l_i the row sum.  The multiplicities do not depend
// on Q, K, V, so with dO given
//   dV_j = sum_i P_ij dO_i,  dP_ij = dO_i . v_j,  Delta_i = dO_i . O_i,
//   dS_ij = P_ij (dP_ij - Delta_i),
//   dK_j = sum_i dS_ij q_i / sqrt(d),  dQ_i = sum_j dS_ij k_j / sqrt(d),
// a KV head collecting the sums of every query head that reads it.  (m, l,
// Delta) come from the forward kernel run in its row statistics mode.
//
// Transposed orientation: a work item is (batch element, KV head, 128-key
// tile); it walks every query head of the group and every 128-row query tile
// whose rows share a bin with its keys (the key j's bins end at hi_t(j), which
// grows with j, so those rows are [j, max_t hi_t(last key)) when causal).
// Per (head, query tile) step, five tcgen05 products with the keys on the
// TMEM lanes:
//   S^T  = K Q^T          (A = K, B = Q; both K-major, TMEM cols 0-127)
//   dP^T = V dO^T         (A = V, B = dO; TMEM cols 128-255)
//   dV  += P^T dO         (A = P^T from TMEM, B = dO MN-major; cols 256-383)
//   dK  += dS^T Q         (A = dS^T from TMEM, B = Q MN-major; cols 384-511)
//   dQ_p = dS K           (A = dS from shared memory, MN-major; B = K MN-major;
//                          into cols 0-127 once dV has read P^T there)
// and one thread per key turns a row of S^T, dP^T into P^T, dS^T (bf16): the
// multiplicity of key j and query i is the number of its bins whose end lies
// above i (and whose start lies at or below i without the causal mask).  The
// same threads add each step's dQ_p rows to an fp32 accumulator in global
// memory (vector atomics; several key tiles reach a query row) and, at the end
// of an item, write dK and dV of their key.
//
// Warps: 0-3 compute (thread = TMEM lane), 4 producer (item queue, query-tile
// ranges from the bin records, TMA of K, V per item and of Q, dO plus the
// rows' statistics per step), 5 one thread issuing tcgen05.mma.  Every
// mbarrier wait is bounded; on expiry the CTA raises the error flag, lets its
// copies and MMAs drain, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include "bins_dev.cuh"
#include "plsh_internal.h"
#include "tc_ptx.cuh"

namespace plsh {
namespace {

using namespace ptx;

constexpr int BM = 128;                          // keys per tile (M of S^T)
constexpr int BQ = 128;                          // queries per step
constexpr int HD = 128;
constexpr int kThreads = 192;
constexpr int kProdWarp = 4;
constexpr int kMmaWarp = 5;
constexpr int kMaxG = 64;                        // query heads per KV head
constexpr int kMaxSlotsB = 16;                   // bin ends kept per key thread
constexpr uint32_t kTile = BM * HD * 2;          // 32 KB bf16 tile
constexpr uint32_t kHalf = kTile / 2;
constexpr uint32_t OFF_K = 0, OFF_V = kTile, OFF_Q = 2 * kTile, OFF_DO = 3 * kTile,
                   OFF_DS = 4 * kTile, OFF_END = 5 * kTile;
constexpr uint32_t kTmemCols = 512;
constexpr unsigned FULL = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

enum {
  B_KVFULL = 0, B_KVEMPTY, B_QFULL, B_QEMPTY, B_SFULL, B_PDS, B_DQFULL, B_DQEMPTY,
  B_ACCFULL, B_ACCEMPTY, B_IFULL, B_IFULL1, B_IEMPTY, B_IEMPTY1, B_DRAIN, NUM_BARS
};

struct ItemB {
  int valid, b, kvh, kt, steps;
  int lo[kMaxG], hi[kMaxG];                      // query tiles [lo, hi) per head of the group
};

struct CtlB {
  uint64_t bars[NUM_BARS];
  ItemB ring[2];
  float stats[2][BQ][3];                         // m, 1/l, Delta of the step's rows
  uint32_t tmem_base;
  int abort;
};

struct BwdTcParams {
  const BinRecord* rec;
  int s;
  int64_t W;
  int B, Hq, Hkv, n, causal;
  const float* stats;                            // [B * Hq * n][3]
  float* dq_acc;                                 // [B * Hq * n][128] fp32, zeroed
  __nv_bfloat16* dK;                             // [B, Hkv, n, 128]
  __nv_bfloat16* dV;
  int num_items;                                 // B * Hkv * key tiles
  int* queue;                                    // {next item, finished CTAs}
  int* err;
  uint64_t wait_ns;
};

__device__ __forceinline__ void read_itemb(const CtlB* ctl, int slot, ItemB& it) {
  const volatile int* v = reinterpret_cast<const volatile int*>(&ctl->ring[slot]);
  it.valid = v[0];
  it.b = v[1];
  it.kvh = v[2];
  it.kt = v[3];
  it.steps = v[4];
}

// (head within the group, query tile) of step k of an item
__device__ __forceinline__ void step_of(const CtlB* ctl, int slot, int G, int k, int& hg, int& qt) {
  const volatile int* lo = ctl->ring[slot].lo;
  const volatile int* hi = ctl->ring[slot].hi;
  for (hg = 0; hg < G; ++hg) {
    const int len = hi[hg] - lo[hg];
    if (k < len) {
      qt = lo[hg] + k;
      return;
    }
    k -= len;
  }
  hg = G - 1;
  qt = 0;
}

__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ BwdTcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_u32);
  CtlB* ctl = reinterpret_cast<CtlB*>(smem + OFF_END);
  auto bar = [&](int k) { return smem_u32(&ctl->bars[k]); };
  volatile int* abort = &ctl->abort;
  const uint64_t lim = p.wait_ns;
  const int G = p.Hq / p.Hkv;
  const int n = p.n, s = p.s;
  const int KT = (n + BM - 1) / BM;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_KVFULL), 1);
    mbar_init(bar(B_KVEMPTY), 1);
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PDS), BM);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQEMPTY), BM);
    mbar_init(bar(B_ACCFULL), 1);
    mbar_init(bar(B_ACCEMPTY), BM);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_IFULL + k), 1);
      mbar_init(bar(B_IEMPTY + k), 1 + BM);      // the MMA thread and every compute thread
    }
    mbar_init(bar(B_DRAIN), 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProdWarp && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
    prefetch_tensormap(&tmDO);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_wait();
  const uint32_t tmem = ctl->tmem_base;

  if (warp == kProdWarp) {
    // ------------------------------------------------ producer / scheduler
    bool ok = true;
    int gstep = 0;                               // steps loaded so far (all items)
    int kv_loads = 0;                            // items whose K and V were loaded
    for (int seq = 0; ok; ++seq) {
      const int slot = seq & 1;
      const uint32_t use = (uint32_t)(seq >> 1);
      int idx = 0;
      if (lane == 0) {
        ok = mbar_wait(bar(B_IEMPTY + slot), (use & 1u) ^ 1u, abort, lim);
        if (ok) idx = atomicAdd(p.queue, 1);
      }
      ok = __shfl_sync(FULL, (int)ok, 0) != 0;
      idx = __shfl_sync(FULL, idx, 0);
      if (!ok) break;
      volatile int* it = reinterpret_cast<volatile int*>(&ctl->ring[slot]);
      if (idx >= p.num_items) {
        if (lane == 0) {
          it[0] = 0;
          mbar_arrive(bar(B_IFULL + slot));
        }
        break;
      }
      // key tiles in ascending order (the first ones reach the most rows)
      const int kt = idx % KT, bk = idx / KT;
      const int kvh = bk % p.Hkv, b = bk / p.Hkv;
      const int j_first = kt * BM, j_last = min(kt * BM + BM - 1, n - 1);
      // query tiles whose rows share a bin with a key of this tile, per head
      int steps = 0;
      for (int hg = 0; hg < G; ++hg) {
        const int h = kvh * G + hg;
        int hmax = j_last + 1, lmin = j_first;
        for (int t = lane; t < s; t += 32) {
          const BinRecord rl = load_record(p.rec, ((int64_t)h * s + t) * p.W + (j_last >> 5));
          hmax = max(hmax, bin_hi(rl, j_last));
          if (!p.causal) {
            const BinRecord rf = load_record(p.rec, ((int64_t)h * s + t) * p.W + (j_first >> 5));
            lmin = min(lmin, bin_lo(rf, j_first));
          }
        }
        hmax = __reduce_max_sync(FULL, hmax);
        lmin = __reduce_min_sync(FULL, lmin);
        const int qlo = p.causal ? kt : lmin / BQ;
        const int qhi = (hmax + BQ - 1) / BQ;
        if (lane == 0) {
          it[5 + hg] = qlo;                      // ring[slot].lo[hg]
          it[5 + kMaxG + hg] = qhi;              // ring[slot].hi[hg]
        }
        steps += qhi - qlo;
      }
      if (lane == 0) {
        it[0] = 1;
        it[1] = b;
        it[2] = kvh;
        it[3] = kt;
        it[4] = steps;
        mbar_arrive(bar(B_IFULL + slot));
      }
      __syncwarp();
      // K and V of the item, once the item before has issued its last dQ
      if (lane == 0) {
        ok = mbar_wait(bar(B_KVEMPTY), ((uint32_t)seq & 1u) ^ 1u, abort, lim);
        if (ok) {
          mbar_arrive_expect_tx(bar(B_KVFULL), 2 * kTile);
          const int plane = b * p.Hkv + kvh;
          tma_load_3d(sbase + OFF_K, &tmK, bar(B_KVFULL), 0, kt * BM, plane);
          tma_load_3d(sbase + OFF_K + kHalf, &tmK, bar(B_KVFULL), 64, kt * BM, plane);
          tma_load_3d(sbase + OFF_V, &tmV, bar(B_KVFULL), 0, kt * BM, plane);
          tma_load_3d(sbase + OFF_V + kHalf, &tmV, bar(B_KVFULL), 64, kt * BM, plane);
          ++kv_loads;
        }
      }
      ok = __shfl_sync(FULL, (int)ok, 0) != 0;
      // per step: the rows' statistics, then Q and dO
      for (int k = 0; ok && k < steps; ++k, ++gstep) {
        int hg, qt;
        step_of(ctl, slot, G, k, hg, qt);
        const int h = kvh * G + hg;
        if (lane == 0) ok = mbar_wait(bar(B_QEMPTY), ((uint32_t)gstep & 1u) ^ 1u, abort, lim);
        ok = __shfl_sync(FULL, (int)ok, 0) != 0;
        if (!ok) break;
        const int buf = gstep & 1;
        const int64_t rowbase = ((int64_t)b * p.Hq + h) * n;
        for (int r = lane; r < BQ; r += 32) {
          const int i = qt * BQ + r;
          float m = 0.f, il = 0.f, dl = 0.f;
          if (i < n) {
            const float* st = p.stats + (rowbase + i) * 3;
            m = st[0];
            il = st[1] > 0.f ? 1.f / st[1] : 0.f;
            dl = st[2];
          }
          ctl->stats[buf][r][0] = m;
          ctl->stats[buf][r][1] = il;
          ctl->stats[buf][r][2] = dl;
        }
        __syncwarp();
        if (lane == 0) {
          const int plane = b * p.Hq + h;
          mbar_arrive_expect_tx(bar(B_QFULL), 2 * kTile);
          tma_load_3d(sbase + OFF_Q, &tmQ, bar(B_QFULL), 0, qt * BQ, plane);
          tma_load_3d(sbase + OFF_Q + kHalf, &tmQ, bar(B_QFULL), 64, qt * BQ, plane);
          tma_load_3d(sbase + OFF_DO, &tmDO, bar(B_QFULL), 0, qt * BQ, plane);
          tma_load_3d(sbase + OFF_DO + kHalf, &tmDO, bar(B_QFULL), 64, qt * BQ, plane);
        }
        __syncwarp();
      }
    }
    if (!ok && lane == 0) {
      *abort = 1;
      atomicOr(p.err, 1);
    }
    // every copy this warp started lands before the CTA can exit
    if (lane == 0 && gstep > 0) mbar_wait(bar(B_QFULL), (uint32_t)(gstep - 1) & 1u, nullptr, lim);
    if (lane == 0 && kv_loads > 0)
      mbar_wait(bar(B_KVFULL), (uint32_t)(kv_loads - 1) & 1u, nullptr, lim);
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(BM, BQ, 0, 0);   // S^T, dP^T
      constexpr uint32_t id_tm = idesc_bf16_f32(BM, HD, 0, 1);   // dV, dK (A from TMEM)
      constexpr uint32_t id_mm = idesc_bf16_f32(BQ, HD, 1, 1);   // dQ_p (both MN-major)
      const uint64_t dK0 = desc_sw128(sbase + OFF_K, 16, 1024);
      const uint64_t dV0 = desc_sw128(sbase + OFF_V, 16, 1024);
      const uint64_t dQ0 = desc_sw128(sbase + OFF_Q, 16, 1024);
      const uint64_t dO0 = desc_sw128(sbase + OFF_DO, 16, 1024);
      const uint64_t dOm = desc_sw128(sbase + OFF_DO, kHalf, 1024);   // dO, MN-major
      const uint64_t dQm = desc_sw128(sbase + OFF_Q, kHalf, 1024);    // Q, MN-major
      const uint64_t dKm = desc_sw128(sbase + OFF_K, kHalf, 1024);    // K, MN-major
      const uint64_t dSm = desc_sw128(sbase + OFF_DS, kHalf, 1024);   // dS, MN-major
      bool ok = true;
      int gstep = 0;
      for (int seq = 0; ok; ++seq) {
        const int slot = seq & 1;
        ok = mbar_wait(bar(B_IFULL + slot), (uint32_t)(seq >> 1) & 1u, abort, lim);
        if (!ok) break;
        ItemB it;
        read_itemb(ctl, slot, it);
        if (!it.valid) break;
        ok = mbar_wait(bar(B_KVFULL), (uint32_t)seq & 1u, abort, lim);
        // the compute threads have read the item before's dV, dK
        if (ok && seq > 0) ok = mbar_wait(bar(B_ACCEMPTY), (uint32_t)(seq - 1) & 1u, abort, lim);
        for (int k = 0; ok && k < it.steps; ++k, ++gstep) {
          ok = mbar_wait(bar(B_QFULL), (uint32_t)gstep & 1u, abort, lim);
          if (ok && gstep > 0)
            ok = mbar_wait(bar(B_DQEMPTY), (uint32_t)(gstep - 1) & 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
          // S^T = K Q^T and dP^T = V dO^T over the head dimension
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tmem, desc_add(dK0, off), desc_add(dQ0, off), id_kk, kk > 0 ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tmem + 128, desc_add(dV0, off), desc_add(dO0, off), id_kk,
                        kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL));
          ok = mbar_wait(bar(B_PDS), (uint32_t)gstep & 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
          // dV += P^T dO and dK += dS^T Q over the step's queries; P^T and
          // dS^T of queries 16kk.. fill the first 16 columns of their chunk
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint32_t ac = (kk >> 1) * 32 + (kk & 1) * 8;
            mma_f16kind_ts(tmem + 256, tmem + ac, desc_add(dOm, kk * (2048 >> 4)), id_tm,
                           (k == 0 && kk == 0) ? 0u : 1u);
          }
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint32_t ac = 128 + (kk >> 1) * 32 + (kk & 1) * 8;
            mma_f16kind_ts(tmem + 384, tmem + ac, desc_add(dQm, kk * (2048 >> 4)), id_tm,
                           (k == 0 && kk == 0) ? 0u : 1u);
          }
          mma_commit(bar(B_QEMPTY));
          // dQ_p = dS K over the tile's keys, into columns 0-127 (the
          // products above have read P^T from there: tcgen05 MMAs of one
          // thread run in issue order)
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_bf16_ss(tmem, desc_add(dSm, kk * (2048 >> 4)), desc_add(dKm, kk * (2048 >> 4)),
                        id_mm, kk > 0 ? 1u : 0u);
          mma_commit(bar(B_DQFULL));
        }
        if (!ok) break;
        // dV, dK complete; K and V free
        mma_commit(bar(B_ACCFULL));
        mma_commit(bar(B_KVEMPTY));
        mbar_arrive(bar(B_IEMPTY + slot));
      }
      if (!ok) {
        *abort = 1;
        atomicOr(p.err, 1);
      }
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr, lim);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------- compute
    const int r = threadIdx.x;                   // TMEM lane: key row, or query row of dQ_p
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base, t_dp = t_s + 128, t_dv = t_s + 256, t_dk = t_s + 384;
    const float scale_log2 = kLog2e * 0.08838834764831845f;      // log2(e) / sqrt(128)
    const uint32_t ds_row = sbase + OFF_DS + (uint32_t)r * 128u;  // this key's row of dS^T
    bool ok = true;
    int gstep = 0;
    for (int seq = 0; ok; ++seq) {
      const int slot = seq & 1;
      ok = __all_sync(FULL, mbar_wait(bar(B_IFULL + slot), (uint32_t)(seq >> 1) & 1u, abort, lim));
      if (!ok) break;
      ItemB it;
      read_itemb(ctl, slot, it);
      if (!it.valid) break;
      const int j = it.kt * BM + r;              // this thread's key
      const bool key_ok = j < n;
      const int jj = min(j, n - 1);
      int cur_h = -1;
      int his[kMaxSlotsB], los[kMaxSlotsB];
      for (int k = 0; ok && k < it.steps; ++k, ++gstep) {
        int hg, qt;
        step_of(ctl, slot, G, k, hg, qt);
        const int h = it.kvh * G + hg;
        if (h != cur_h) {
          // this key's bins under the head's hashes: [lo_t, hi_t)
#pragma unroll
          for (int t = 0; t < kMaxSlotsB; ++t) {
            his[t] = INT_MIN;
            los[t] = INT_MAX;
            if (t < s) {
              const BinRecord rc = load_record(p.rec, ((int64_t)h * s + t) * p.W + (jj >> 5));
              his[t] = bin_hi(rc, jj);
              los[t] = bin_lo(rc, jj);
            }
          }
          cur_h = h;
        }
        const int buf = gstep & 1;
        ok = __all_sync(FULL, mbar_wait(bar(B_QFULL), (uint32_t)gstep & 1u, abort, lim) &&
                                  mbar_wait(bar(B_SFULL), (uint32_t)gstep & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();
        const int i0 = qt * BQ;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t sv[32], dv[32];
          tmem_ld32(t_s + q * 32, sv);
          tmem_ld32(t_dp + q * 32, dv);
          tmem_wait_ld();
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            float pe[2], de[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int e = 2 * e2 + u;
              const int i = i0 + q * 32 + e;
              int c = 0;
#pragma unroll
              for (int t = 0; t < kMaxSlotsB; ++t)
                c += (his[t] > i && los[t] <= i) ? 1 : 0;
              const bool live = key_ok && i < n && c > 0 && (!p.causal || i >= j);
              const float* st = ctl->stats[buf][q * 32 + e];
              const float pv = live ? (float)c * ex2(fmaf(__uint_as_float(sv[e]), scale_log2,
                                                          -st[0])) * st[1]
                                    : 0.f;
              pe[u] = pv;
              de[u] = pv * (__uint_as_float(dv[e]) - st[2]);
            }
            pk[e2] = pack_bf16(pe[0], pe[1]);
            dk[e2] = pack_bf16(de[0], de[1]);
          }
          tmem_st16(t_s + q * 32, pk);
          tmem_st16(t_dp + q * 32, dk);
          // dS^T into shared memory as the MN-major A operand of dQ_p: two
          // 64-query halves of 128 key rows x 128 bytes, 128-byte swizzle
          const uint32_t half = (uint32_t)(q >> 1);
#pragma unroll
          for (int v = 0; v < 4; ++v) {
            const uint32_t c16 = (uint32_t)((q & 1) * 4 + v);
            st_shared_v4(ds_row + half * kHalf + ((c16 ^ (uint32_t)(r & 7)) << 4), dk[4 * v],
                         dk[4 * v + 1], dk[4 * v + 2], dk[4 * v + 3]);
          }
        }
        tmem_wait_st();
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(bar(B_PDS));
        // this step's dQ rows (TMEM lane = query row) into the accumulator
        ok = __all_sync(FULL, mbar_wait(bar(B_DQFULL), (uint32_t)gstep & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();
        {
          const int i = i0 + r;
          float4* dst = reinterpret_cast<float4*>(p.dq_acc + (((int64_t)it.b * p.Hq + h) * n + i) * HD);
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(t_s + q * 32, o);
            tmem_wait_ld();
            if (i < n) {
#pragma unroll
              for (int v = 0; v < 8; ++v)
                atomicAdd(dst + q * 8 + v,
                          make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                      __uint_as_float(o[4 * v + 2]), __uint_as_float(o[4 * v + 3])));
            }
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_DQEMPTY));
      }
      if (!ok) break;
      // dK, dV of this thread's key
      ok = __all_sync(FULL, mbar_wait(bar(B_ACCFULL), (uint32_t)seq & 1u, abort, lim));
      if (!ok) break;
      tc_fence_after();
      if (it.steps > 0) {
        const int64_t krow = ((int64_t)it.b * p.Hkv + it.kvh) * n + j;
#pragma unroll 1
        for (int q = 0; q < 4; ++q) {
          uint32_t a[32], g[32];
          tmem_ld32(t_dv + q * 32, a);
          tmem_ld32(t_dk + q * 32, g);
          tmem_wait_ld();
          if (key_ok) {
            uint4* ov = reinterpret_cast<uint4*>(p.dV + krow * HD + q * 32);
            uint4* ok4 = reinterpret_cast<uint4*>(p.dK + krow * HD + q * 32);
            const float inv = 0.08838834764831845f;                 // 1 / sqrt(128)
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              ov[v] = make_uint4(pack_bf16(__uint_as_float(a[8 * v]), __uint_as_float(a[8 * v + 1])),
                                 pack_bf16(__uint_as_float(a[8 * v + 2]), __uint_as_float(a[8 * v + 3])),
                                 pack_bf16(__uint_as_float(a[8 * v + 4]), __uint_as_float(a[8 * v + 5])),
                                 pack_bf16(__uint_as_float(a[8 * v + 6]), __uint_as_float(a[8 * v + 7])));
              ok4[v] = make_uint4(
                  pack_bf16(__uint_as_float(g[8 * v]) * inv, __uint_as_float(g[8 * v + 1]) * inv),
                  pack_bf16(__uint_as_float(g[8 * v + 2]) * inv, __uint_as_float(g[8 * v + 3]) * inv),
                  pack_bf16(__uint_as_float(g[8 * v + 4]) * inv, __uint_as_float(g[8 * v + 5]) * inv),
                  pack_bf16(__uint_as_float(g[8 * v + 6]) * inv, __uint_as_float(g[8 * v + 7]) * inv));
            }
          }
        }
      } else if (key_ok) {
        // no query row shares a bin with this key: zero gradients
        const int64_t krow = ((int64_t)it.b * p.Hkv + it.kvh) * n + j;
        uint4* ov = reinterpret_cast<uint4*>(p.dV + krow * HD);
        uint4* ok4 = reinterpret_cast<uint4*>(p.dK + krow * HD);
        for (int v = 0; v < HD / 8; ++v) ov[v] = ok4[v] = make_uint4(0u, 0u, 0u, 0u);
      }
      tc_fence_before();
      mbar_arrive(bar(B_ACCEMPTY));
      mbar_arrive(bar(B_IEMPTY + slot));
    }
    if (!ok && lane == 0) {
      *abort = 1;
      atomicOr(p.err, 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(p.queue + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(p.queue, 0);
      atomicExch(p.queue + 1, 0);
      __threadfence();
    }
  }
}

// dQ = dq_acc / sqrt(128) in bf16
__global__ void dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ out,
                                  int64_t count4) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count4) return;
  const float4 v = acc[i];
  const float inv = 0.08838834764831845f;
  out[i] = make_uint2(pack_bf16(v.x * inv, v.y * inv), pack_bf16(v.z * inv, v.w * inv));
}

}  // namespace

size_t bwd_tc_smem_bytes() { return 1024 + OFF_END + sizeof(CtlB); }

cudaError_t launch_attn_bwd_tc(const void* Q, const void* K, const void* V, const void* dO,
                               void* dQ, void* dK, void* dV, const float* stats, float* dq_acc,
                               const plsh_bins* bn, int B, int Hq, int Hkv, int n, int causal,
                               int* queue, int* err, uint64_t wait_ns, int num_sms,
                               cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo;
  if (!make_tile_map_bf16(&mq, Q, (int64_t)B * Hq, n) ||
      !make_tile_map_bf16(&mk, K, (int64_t)B * Hkv, n) ||
      !make_tile_map_bf16(&mv, V, (int64_t)B * Hkv, n) ||
      !make_tile_map_bf16(&mdo, dO, (int64_t)B * Hq, n))
    return cudaErrorInvalidValue;
  BwdTcParams p;
  p.rec = bn->d_rec;
  p.s = bn->s;
  p.W = bn->W;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.n = n;
  p.causal = causal;
  p.stats = stats;
  p.dq_acc = dq_acc;
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.num_items = B * Hkv * ((n + BM - 1) / BM);
  p.queue = queue;
  p.err = err;
  p.wait_ns = wait_ns;
  const size_t smem = bwd_tc_smem_bytes();
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)B * Hq * n * HD, st);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(bwd_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.num_items < num_sms ? p.num_items : num_sms;
  bwd_tc_kernel<<<grid, kThreads, smem, st>>>(mq, mk, mv, mdo, p);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int64_t count4 = (int64_t)B * Hq * n * HD / 4;
  dq_convert_kernel<<<(unsigned)((count4 + 255) / 256), 256, 0, st>>>(
      reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(dQ), count4);
  return cudaGetLastError();
}

}  // namespace plsh
