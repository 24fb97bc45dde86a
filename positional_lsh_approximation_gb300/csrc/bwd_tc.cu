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
//                          into cols 128-255 once dK has read dS^T there)
// Q is double buffered, so the next step's S^T runs while this step's dQ_p
// is being drained; the next dP^T waits for that drain.
//
// Two threads per key (warps w and w + 4 share a TMEM lane quarter, each
// taking half of the step's query columns) turn a row of S^T, dP^T into P^T,
// dS^T (bf16).  A key's multiplicities over a chunk of 32 query rows are a
// running count: the hashes whose bin around the key is open at the chunk's
// first row, minus the bins that end at each row inside the chunk (plus
// those that start there when not causal), held as binary planes; rows past
// every bin end or before every start are masked.  Chunks that every bin of
// every key of the warp spans take c = s, folded into the exponent.  The bins
// sit in a compile-time number of register slots (SREG >= s).  The same
// threads stage each step's dQ_p rows in shared memory, where TMA reductions
// add them to an fp32 accumulator in global memory (several key tiles reach
// a query row), and, at the end of an item, write their half of dK and dV of
// their key.
//
// Warps: 0-7 compute (thread = TMEM lane, two warps per lane quarter), 8
// producer (item queue, query-tile ranges from the bin records, TMA of K, V
// per item and of Q, dO per step, the rows' statistics and the head's bin
// records per step into shared memory, L2 prefetch of the next step's
// tiles), 9 one thread issuing tcgen05.mma.  Items are taken in the order of
// their KV group's expected work, largest first.
// Every mbarrier wait is bounded; on expiry the CTA raises the error flag,
// lets its copies and MMAs drain, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <math.h>
#include <stdint.h>

#include <algorithm>
#include <numeric>
#include <vector>

#include "bins_dev.cuh"
#include "plsh_internal.h"
#include "tc_ptx.cuh"

namespace plsh {
namespace {

using namespace ptx;

constexpr int BM = 128;                          // keys per tile (M of S^T)
constexpr int BQ = 128;                          // queries per step
constexpr int HD = 128;
constexpr int kCompute = 256;                    // two warps per TMEM lane quarter
constexpr int kThreads = kCompute + 64;
constexpr int kProdWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kMaxG = 64;                        // query heads per KV head
constexpr int kMaxSlotsB = 16;                   // bins kept per key thread
constexpr int kMaxOrder = 64;                    // KV heads with a work order
constexpr uint32_t kTile = BM * HD * 2;          // 32 KB bf16 tile
constexpr uint32_t kHalf = kTile / 2;
constexpr uint32_t OFF_K = 0, OFF_V = kTile, OFF_Q = 2 * kTile,   // two Q buffers
                   OFF_DO = 4 * kTile, OFF_DS = 5 * kTile, OFF_END = 6 * kTile;
constexpr uint32_t kTmemCols = 512;
constexpr unsigned FULL = 0xffffffffu;
constexpr float kLog2e = 1.4426950408889634f;

enum {
  B_KVFULL = 0, B_KVEMPTY, B_QFULL, B_QFULL1, B_QEMPTY, B_QEMPTY1, B_DOFULL, B_DOEMPTY,
  B_SFULL, B_PDS, B_DQFULL, B_DQEMPTY, B_ACCFULL, B_ACCEMPTY, B_IFULL, B_IFULL1, B_IEMPTY,
  B_IEMPTY1, B_DRAIN, NUM_BARS
};

struct ItemB {
  int valid, b, kvh, kt, steps;
  int lo[kMaxG], hi[kMaxG];                      // query tiles [lo, hi) per head of the group
};

struct CtlB {
  uint64_t bars[NUM_BARS];
  ItemB ring[2];
  // per step buffer: -(m + log2 l) of the step's rows, then their Delta
  alignas(16) float stats[2][2][BQ];
  // per step buffer: the bin records of the step's head over the item's four
  // 32-key words, per hash
  uint4 recs[2][kMaxSlotsB][BM / 32];
  uint32_t tmem_base;
  int abort;
};

struct BwdTcParams {
  const BinRecord* rec;
  int s;
  int64_t W;
  int B, Hq, Hkv, n;
  const float* stats;                            // [B * Hq * n][2]: -lse, Delta
  float* dq_acc;                                 // [B * Hq * n][128] fp32, zeroed
  __nv_bfloat16* dK;                             // [B, Hkv, n, 128]
  __nv_bfloat16* dV;
  int num_items;                                 // B * Hkv * key tiles
  int ordered;                                   // kv_order holds the KV heads' order
  int kv_order[kMaxOrder];
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

// TMA reduction of a shared-memory box into global memory (add), tracked by
// the issuing thread's bulk async-group.
__device__ __forceinline__ void tma_reduce_add_3d(const CUtensorMap* map, uint32_t src, int x,
                                                  int y, int z) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], "
      "[%1];" ::"l"(map), "r"(src), "r"(x), "r"(y), "r"(z)
      : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// the group's reads of shared memory are done (the writes may still be in flight)
__device__ __forceinline__ void bulk_wait_read() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// A box of a tensor into L2 ahead of its load.
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int x, int y, int z) {
  asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(map),
               "r"(x), "r"(y), "r"(z)
               : "memory");
}

// Rows [a, b] of a 32-row chunk as a bit mask (relative to the chunk).
__device__ __forceinline__ uint32_t row_mask(int a, int b) {
  if (a > 31 || b < 0 || a > b) return 0u;
  const uint32_t up = b >= 31 ? 0xffffffffu : ((2u << b) - 1u);
  const uint32_t dn = a <= 0 ? 0xffffffffu : ~((1u << a) - 1u);
  return up & dn;
}

// Adds one step at the positions of `m` to a five-plane binary counter (the
// step count at each row, up to 31).
__device__ __forceinline__ void plane_add5(uint32_t (&pl)[5], uint32_t m) {
#pragma unroll
  for (int b = 0; b < 5; ++b) {
    const uint32_t c = pl[b] & m;
    pl[b] ^= m;
    m = c;
  }
}

// Multiplies the chunk's weights by the running count c(e): base plus the
// steps at rows 1..e, up steps (bin starts, non-causal only) adding and dn
// steps (bin ends) subtracting, the step counts held as P binary planes;
// four independent runs of eight rows.
template <bool UP, int P>
__device__ __forceinline__ void count_planes(float (&pv)[32], int base, const uint32_t (&up)[5],
                                             const uint32_t (&dn)[5]) {
  float c[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t le = (2u << (8 * g)) - 1u;    // rows 0 .. 8g
    int cb = base;
#pragma unroll
    for (int b = 0; b < P; ++b) {
      cb -= __popc(dn[b] & le) << b;
      if (UP) cb += __popc(up[b] & le) << b;
    }
    c[g] = (float)cb;
  }
#pragma unroll
  for (int k = 0; k < 8; ++k) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int e = 8 * g + k;
      if (k > 0) {
#pragma unroll
        for (int b = 0; b < P; ++b) {
          if (dn[b] & (1u << e)) c[g] -= (float)(1 << b);
          if (UP && (up[b] & (1u << e))) c[g] += (float)(1 << b);
        }
      }
      pv[e] *= c[g];
    }
  }
}

// SREG: register slots per key thread for its bins (s <= SREG; the slots past
// s hold bins that count nowhere), a compile-time count so that the per-chunk
// loop over them is unrolled without branches.
template <bool CAUSAL, int SREG>
__global__ void __launch_bounds__(kThreads, 1)
bwd_tc_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
              const __grid_constant__ CUtensorMap tmAcc, const __grid_constant__ BwdTcParams p) {
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
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_QFULL + k), 1);
      mbar_init(bar(B_QEMPTY + k), 8);           // the compute warps, once dQ staged there is read
    }
    mbar_init(bar(B_DOFULL), 1);
    mbar_init(bar(B_DOEMPTY), 1);
    mbar_init(bar(B_SFULL), 1);
    mbar_init(bar(B_PDS), kCompute);
    mbar_init(bar(B_DQFULL), 1);
    mbar_init(bar(B_DQEMPTY), kCompute);
    mbar_init(bar(B_ACCFULL), 1);
    mbar_init(bar(B_ACCEMPTY), kCompute);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_IFULL + k), 1);
      mbar_init(bar(B_IEMPTY + k), 1 + kCompute);   // the MMA thread and every compute thread
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
    prefetch_tensormap(&tmAcc);
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
    int nq0 = 0, nq1 = 0;                        // Q loads per buffer
    int ndo = 0;                                 // dO loads
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
      ItemB* ring = &ctl->ring[slot];
      volatile int* it = reinterpret_cast<volatile int*>(ring);
      if (idx >= p.num_items) {
        if (lane == 0) {
          it[0] = 0;
          mbar_arrive(bar(B_IFULL + slot));
        }
        break;
      }
      // KV groups in the host's order, then batch elements, then key tiles
      // in ascending order (the first ones reach the most rows)
      const int per = p.B * KT;
      const int gs = idx / per, rem = idx - (idx / per) * per;
      const int b = rem / KT, kt = rem - (rem / KT) * KT;
      const int kvh = p.ordered ? p.kv_order[gs] : gs;
      const int j_first = kt * BM, j_last = min(kt * BM + BM - 1, n - 1);
      // query tiles whose rows share a bin with a key of this tile, per
      // head: the (head, hash) records spread over the lanes and combined in
      // shared memory
      for (int hg = lane; hg < G; hg += 32) {
        ring->hi[hg] = j_last + 1;
        ring->lo[hg] = j_first;
      }
      __syncwarp();
      const int GS = G * s;
      for (int base = 0; base < GS; base += 128) {
        BinRecord rl[4], rf[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ht = base + u * 32 + lane;
          if (ht < GS) {
            const int hg = ht / s, t = ht - (ht / s) * s;
            const int64_t rb = ((int64_t)(kvh * G + hg) * s + t) * p.W;
            rl[u] = load_record(p.rec, rb + (j_last >> 5));
            if (!CAUSAL) rf[u] = load_record(p.rec, rb + (j_first >> 5));
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int ht = base + u * 32 + lane;
          if (ht < GS) {
            const int hg = ht / s;
            atomicMax(&ring->hi[hg], bin_hi(rl[u], j_last));
            if (!CAUSAL) atomicMin(&ring->lo[hg], bin_lo(rf[u], j_first));
          }
        }
      }
      __syncwarp();
      int steps = 0;
      for (int hg = lane; hg < G; hg += 32) {
        const int qlo = CAUSAL ? kt : ring->lo[hg] / BQ;
        const int qhi = (ring->hi[hg] + BQ - 1) / BQ;
        ring->lo[hg] = qlo;
        ring->hi[hg] = qhi;
        steps += qhi - qlo;
      }
      steps = __reduce_add_sync(FULL, steps);
      __threadfence_block();
      __syncwarp();
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
      // the rows' statistics of the next step, read ahead into registers
      float sm[4], sd[4];
      uint4 rr[2];
      auto load_stats = [&](int k) {
        int hg, qt;
        step_of(ctl, slot, G, k, hg, qt);
        const int64_t rowbase = ((int64_t)b * p.Hq + kvh * G + hg) * n;
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int tw = u * 32 + lane;          // (hash, word of the key tile)
          rr[u] = make_uint4(0u, 0u, 0u, 0u);
          if (tw < s * 4) {
            const int64_t word = min((int64_t)kt * 4 + (tw & 3), p.W - 1);
            rr[u] = __ldg(reinterpret_cast<const uint4*>(p.rec) +
                          ((int64_t)(kvh * G + hg) * s + (tw >> 2)) * p.W + word);
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int i = qt * BQ + u * 32 + lane;
          sm[u] = -INFINITY;
          sd[u] = 0.f;
          if (i < n) {
            const float2 st = __ldg(reinterpret_cast<const float2*>(p.stats) + rowbase + i);
            sm[u] = st.x;
            sd[u] = st.y;
          }
        }
      };
      if (ok && steps > 0) load_stats(0);
      for (int k = 0; ok && k < steps; ++k, ++gstep) {
        int hg, qt;
        step_of(ctl, slot, G, k, hg, qt);
        const int plane = b * p.Hq + kvh * G + hg;
        const int qb = gstep & 1;
        // Q into its buffer once the step two back has finished dK
        if (lane == 0) {
          ok = mbar_wait(bar(B_QEMPTY + qb), ((uint32_t)(gstep >> 1) & 1u) ^ 1u, abort, lim);
          if (ok) {
            const uint32_t dst = sbase + OFF_Q + (uint32_t)qb * kTile;
            mbar_arrive_expect_tx(bar(B_QFULL + qb), kTile);
            tma_load_3d(dst, &tmQ, bar(B_QFULL + qb), 0, qt * BQ, plane);
            tma_load_3d(dst + kHalf, &tmQ, bar(B_QFULL + qb), 64, qt * BQ, plane);
            if (qb) ++nq1;
            else ++nq0;
          }
        }
        ok = __shfl_sync(FULL, (int)ok, 0) != 0;
        if (!ok) break;
        // dO and the rows' statistics once the step before has finished dV
        if (lane == 0) ok = mbar_wait(bar(B_DOEMPTY), ((uint32_t)gstep & 1u) ^ 1u, abort, lim);
        ok = __shfl_sync(FULL, (int)ok, 0) != 0;
        if (!ok) break;
        float* sv = ctl->stats[gstep & 1][0];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int r = u * 32 + lane;
          sv[r] = sm[u];
          sv[BQ + r] = sd[u];
        }
        uint4* rv = &ctl->recs[gstep & 1][0][0];
#pragma unroll
        for (int u = 0; u < 2; ++u)
          if (u * 32 + lane < s * 4) rv[u * 32 + lane] = rr[u];
        __syncwarp();
        if (lane == 0) {
          mbar_arrive_expect_tx(bar(B_DOFULL), kTile);
          tma_load_3d(sbase + OFF_DO, &tmDO, bar(B_DOFULL), 0, qt * BQ, plane);
          tma_load_3d(sbase + OFF_DO + kHalf, &tmDO, bar(B_DOFULL), 64, qt * BQ, plane);
          ++ndo;
        }
        __syncwarp();
        if (k + 1 < steps) {
          load_stats(k + 1);
          // the next step's Q and dO into L2 while this step runs
          int hg2, qt2;
          step_of(ctl, slot, G, k + 1, hg2, qt2);
          const int plane2 = b * p.Hq + kvh * G + hg2;
          if (lane < 4)
            tma_prefetch_3d(lane < 2 ? &tmQ : &tmDO, (lane & 1) * 64, qt2 * BQ, plane2);
        }
      }
    }
    if (!ok && lane == 0) {
      *abort = 1;
      atomicOr(p.err, 1);
    }
    // every copy this warp started lands before the CTA can exit
    if (lane == 0) {
      if (nq0 > 0) mbar_wait(bar(B_QFULL), (uint32_t)(nq0 - 1) & 1u, nullptr, lim);
      if (nq1 > 0) mbar_wait(bar(B_QFULL1), (uint32_t)(nq1 - 1) & 1u, nullptr, lim);
      if (ndo > 0) mbar_wait(bar(B_DOFULL), (uint32_t)(ndo - 1) & 1u, nullptr, lim);
      if (kv_loads > 0) mbar_wait(bar(B_KVFULL), (uint32_t)(kv_loads - 1) & 1u, nullptr, lim);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ----------------------------------------------------------- MMA issue
    if (lane == 0) {
      constexpr uint32_t id_kk = idesc_bf16_f32(BM, BQ, 0, 0);   // S^T, dP^T
      constexpr uint32_t id_tm = idesc_bf16_f32(BM, HD, 0, 1);   // dV, dK (A from TMEM)
      constexpr uint32_t id_mm = idesc_bf16_f32(BQ, HD, 1, 1);   // dQ_p (both MN-major)
      const uint64_t dK0 = desc_sw128(sbase + OFF_K, 16, 1024);
      const uint64_t dV0 = desc_sw128(sbase + OFF_V, 16, 1024);
      const uint64_t dO0 = desc_sw128(sbase + OFF_DO, 16, 1024);
      const uint64_t dOm = desc_sw128(sbase + OFF_DO, kHalf, 1024);   // dO, MN-major
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
        for (int k = 0; ok && k < it.steps; ++k, ++gstep) {
          const int qb = gstep & 1;
          const uint32_t q_addr = sbase + OFF_Q + (uint32_t)qb * kTile;
          const uint64_t dQ0 = desc_sw128(q_addr, 16, 1024);
          const uint64_t dQm = desc_sw128(q_addr, kHalf, 1024);       // Q, MN-major
          ok = mbar_wait(bar(B_QFULL + qb), (uint32_t)(gstep >> 1) & 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
          // S^T = K Q^T over the head dimension (the products before have
          // read P^T from these columns: tcgen05 MMAs of one thread run in
          // issue order)
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tmem, desc_add(dK0, off), desc_add(dQ0, off), id_kk, kk > 0 ? 1u : 0u);
          }
          // dP^T = V dO^T, once dO has landed and the step before's dQ_p
          // has been read out of columns 128-255
          ok = mbar_wait(bar(B_DOFULL), (uint32_t)gstep & 1u, abort, lim);
          if (ok && gstep > 0)
            ok = mbar_wait(bar(B_DQEMPTY), (uint32_t)(gstep - 1) & 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t off = ((kk >> 2) * kHalf + (kk & 3) * 32) >> 4;
            mma_bf16_ss(tmem + 128, desc_add(dV0, off), desc_add(dO0, off), id_kk,
                        kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL));
          // the compute threads have read the item before's dV, dK
          if (k == 0 && seq > 0)
            ok = mbar_wait(bar(B_ACCEMPTY), (uint32_t)(seq - 1) & 1u, abort, lim);
          if (ok) ok = mbar_wait(bar(B_PDS), (uint32_t)gstep & 1u, abort, lim);
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
          mma_commit(bar(B_DOEMPTY));
#pragma unroll
          for (int kk = 0; kk < BQ / 16; ++kk) {
            const uint32_t ac = 128 + (kk >> 1) * 32 + (kk & 1) * 8;
            mma_f16kind_ts(tmem + 384, tmem + ac, desc_add(dQm, kk * (2048 >> 4)), id_tm,
                           (k == 0 && kk == 0) ? 0u : 1u);
          }
          // dQ_p = dS K over the tile's keys, into columns 128-255
#pragma unroll
          for (int kk = 0; kk < BM / 16; ++kk)
            mma_bf16_ss(tmem + 128, desc_add(dSm, kk * (2048 >> 4)),
                        desc_add(dKm, kk * (2048 >> 4)), id_mm, kk > 0 ? 1u : 0u);
          mma_commit(bar(B_DQFULL));
        }
        if (!ok) break;
        // an item without steps still hands its (zero) gradients over in turn
        if (it.steps == 0 && seq > 0)
          ok = mbar_wait(bar(B_ACCEMPTY), (uint32_t)(seq - 1) & 1u, abort, lim);
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
    // warps w and w + 4 share TMEM lanes 32 (w % 4) ...; ch = w / 4 picks the
    // half of the query columns (of d for dQ_p, dV and dK) a warp handles
    const int r = threadIdx.x & (BM - 1);        // TMEM lane: key row, or query row of dQ_p
    const int ch = warp >> 2;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t t_s = tmem + lane_base, t_dp = t_s + 128, t_dv = t_s + 256, t_dk = t_s + 384;
    const float scale_log2 = kLog2e * 0.08838834764831845f;      // log2(e) / sqrt(128)
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    const uint32_t ds_row = sbase + OFF_DS + (uint32_t)r * 128u;  // this key's row of dS^T
    const int wq = warp & 3;
    // the warp's rows of its dS^T half, 4 KB (1024-byte aligned): the only
    // part of the dS buffer it writes
    const uint32_t wpiece = sbase + OFF_DS + (uint32_t)ch * kHalf + (uint32_t)wq * 4096u;
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
      // this key's bins under the head's hashes, [lo_t, hi_t), and the rows
      // [ilo, ihi] that share at least one of them
      int his[SREG], los[SREG];
      int ilo = 0, ihi = -1, himin = 0, lomax = 0;
      for (int k = 0; ok && k < it.steps; ++k, ++gstep) {
        int hg, qt;
        step_of(ctl, slot, G, k, hg, qt);
        const int h = it.kvh * G + hg;
        const float* sv = ctl->stats[gstep & 1][0];
        // the step's row statistics and bin records have landed
        ok = __all_sync(FULL, mbar_wait(bar(B_DOFULL), (uint32_t)gstep & 1u, abort, lim));
        if (!ok) break;
        if (h != cur_h) {
          const uint4* rv = &ctl->recs[gstep & 1][0][(jj >> 5) - it.kt * (BM / 32)];
          int hmax = 0, lmin = INT_MAX;
          himin = INT_MAX;
          lomax = 0;
#pragma unroll
          for (int t = 0; t < SREG; ++t) {
            his[t] = CAUSAL ? -1 : (1 << 30);    // unused slots: no count, no step
            los[t] = 1 << 30;
            if (t < s) {
              const uint4 v = rv[t * (BM / 32)];
              BinRecord rc;
              rc.bits = v.x;
              rc.prev = (int32_t)v.y;
              rc.next = (int32_t)v.z;
              rc.pad = 0;
              his[t] = bin_hi(rc, jj);
              los[t] = bin_lo(rc, jj);
              hmax = max(hmax, his[t]);
              himin = min(himin, his[t]);
              lmin = min(lmin, los[t]);
              lomax = max(lomax, los[t]);
            }
          }
          ilo = CAUSAL ? j : lmin;
          ihi = key_ok ? min(hmax, n) - 1 : -1;
          cur_h = h;
        }
        ok = __all_sync(FULL, mbar_wait(bar(B_SFULL), (uint32_t)gstep & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();
        // the copy engine has read the step before's staged dQ rows: the
        // warp's dS^T rows may be written again and that step's Q buffer is
        // free for the producer
        if (lane == 0) {
          bulk_wait_read();
          if (gstep > 0) mbar_arrive(bar(B_QEMPTY + ((gstep - 1) & 1)));
        }
        __syncwarp();
        const int i0 = qt * BQ;
#pragma unroll 1
        for (int q = 2 * ch; q < 2 * ch + 2; ++q) {
          const int ic = i0 + q * 32;
          const uint32_t vm = row_mask(ilo - ic, ihi - ic);
          const uint32_t half = (uint32_t)(q >> 1);
          if (!__any_sync(FULL, vm != 0u)) {
            // no row of the chunk shares a bin with a key of this warp
            const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u,
                                    0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            tmem_st16(t_s + q * 32, z);
            tmem_st16(t_dp + q * 32, z);
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint32_t c16 = (uint32_t)((q & 1) * 4 + v);
              st_shared_v4(ds_row + half * kHalf + ((c16 ^ (uint32_t)(r & 7)) << 4), 0u, 0u, 0u,
                           0u);
            }
            continue;
          }
          uint32_t sv32[32], dv32[32];
          tmem_ld32(t_s + q * 32, sv32);
          tmem_ld32(t_dp + q * 32, dv32);
          // multiplicities over the chunk's rows: the hashes whose bin
          // around the key is open at its first row (base), and the number
          // of bins that end (dn) or, not causal, start (up) at each row
          // inside it, as binary planes; a step at a masked row only touches
          // masked rows after it (vm is one run of rows), so it is dropped
          int base = s;
          int planes = 0;                          // warp-wide planes in use (0: flat)
          uint32_t up[5] = {0u, 0u, 0u, 0u, 0u}, dn[5] = {0u, 0u, 0u, 0u, 0u};
          const bool deep = himin > ic + 31 && (CAUSAL || lomax <= ic);
          if (!__all_sync(FULL, deep || vm == 0u)) {
            int nh = 0, nl = 0;
#pragma unroll
            for (int t = 0; t < SREG; ++t) {
              const int dh = his[t] - ic;
              nh += dh > 0 ? 1 : 0;
              plane_add5(dn, shl_clamp(2u, dh - 1) & vm);
              if (!CAUSAL) {
                const int dl = los[t] - ic;
                nl += dl > 0 ? 0 : 1;
                plane_add5(up, shl_clamp(2u, dl - 1) & vm);
              }
            }
            // not causal, a slot counts lo <= ic < hi as [hi > ic] + [lo <= ic] - 1
            // (an unused one: 1 + 0 - 1)
            base = CAUSAL ? nh : nh + nl - SREG;
            planes = __any_sync(FULL, (dn[4] | up[4]) != 0u)   ? 5
                     : __any_sync(FULL, (dn[3] | up[3]) != 0u) ? 4
                     : __any_sync(FULL, (dn[2] | up[2]) != 0u) ? 3
                     : __any_sync(FULL, (dn[1] | up[1]) != 0u) ? 2
                     : __any_sync(FULL, (dn[0] | up[0]) != 0u) ? 1
                                                               : 0;
          }
          const float lgb = planes == 0 ? lg2((float)max(base, 1)) : 0.f;
          const uint64_t lgb2 = f2_pack(lgb, lgb);
          tmem_wait_ld();
          float pv[32];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 nm = *reinterpret_cast<const float2*>(sv + q * 32 + e);
            const uint64_t a2 =
                f2_fma(f2_pack(__uint_as_float(sv32[e]), __uint_as_float(sv32[e + 1])), scale2,
                       f2_add(f2_pack(nm.x, nm.y), lgb2));
            f2_unpack(a2, pv[e], pv[e + 1]);
          }
          if (__any_sync(FULL, vm != 0xffffffffu)) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (!(vm & (1u << e))) pv[e] = -INFINITY;
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) pv[e] = ex2(pv[e]);
          switch (planes) {
            case 1: count_planes<!CAUSAL, 1>(pv, base, up, dn); break;
            case 2: count_planes<!CAUSAL, 2>(pv, base, up, dn); break;
            case 3: count_planes<!CAUSAL, 3>(pv, base, up, dn); break;
            case 4: count_planes<!CAUSAL, 4>(pv, base, up, dn); break;
            case 5: count_planes<!CAUSAL, 5>(pv, base, up, dn); break;
            default: break;
          }
          uint32_t pk[16], dk[16];
#pragma unroll
          for (int e = 0; e < 32; e += 2) {
            const float2 dl = *reinterpret_cast<const float2*>(sv + BQ + q * 32 + e);
            const uint64_t g2 =
                f2_sub(f2_pack(__uint_as_float(dv32[e]), __uint_as_float(dv32[e + 1])),
                       f2_pack(dl.x, dl.y));
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(pv[e], pv[e + 1]), g2), d0, d1);
            pk[e >> 1] = pack_bf16(pv[e], pv[e + 1]);
            dk[e >> 1] = pack_bf16(d0, d1);
          }
          tmem_st16(t_s + q * 32, pk);
          tmem_st16(t_dp + q * 32, dk);
          // dS^T into shared memory as the MN-major A operand of dQ_p: two
          // 64-query halves of 128 key rows x 128 bytes, 128-byte swizzle
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
        // this step's dQ rows (TMEM lane = query row) into the accumulator:
        // each warp stages its 32 rows and 64 of the d columns as two
        // 128-byte swizzled fp32 boxes of 32 columns, one in its own piece
        // of the dS buffer and one in its piece of the step's Q buffer (both
        // free once dQ_p has run), which TMA adds to the accumulator; the
        // warp waits for the copy engine's reads only before it next writes
        // there (the start of the next step, which also hands the Q buffer
        // back)
        ok = __all_sync(FULL, mbar_wait(bar(B_DQFULL), (uint32_t)gstep & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();
        {
          const int row0 = i0 + wq * 32;
          const int plane = it.b * p.Hq + h;
          const uint32_t qpiece = sbase + OFF_Q + (uint32_t)(gstep & 1) * kTile +
                                  (uint32_t)ch * kHalf + (uint32_t)wq * 4096u;
          uint32_t o[64];
          tmem_ld32(t_dp + ch * 64, *reinterpret_cast<uint32_t(*)[32]>(&o[0]));
          tmem_ld32(t_dp + ch * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&o[32]));
          tmem_wait_ld();
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t row = (u == 0 ? wpiece : qpiece) + (uint32_t)lane * 128u;
#pragma unroll
            for (int c = 0; c < 8; ++c)
              st_shared_v4(row + (((uint32_t)c ^ (uint32_t)(lane & 7)) << 4), o[32 * u + 4 * c],
                           o[32 * u + 4 * c + 1], o[32 * u + 4 * c + 2], o[32 * u + 4 * c + 3]);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0 && row0 < n) {
            tma_reduce_add_3d(&tmAcc, wpiece, ch * 64, row0, plane);
            tma_reduce_add_3d(&tmAcc, qpiece, ch * 64 + 32, row0, plane);
            bulk_commit();
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
        for (int q = 2 * ch; q < 2 * ch + 2; ++q) {
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
        uint4* ov = reinterpret_cast<uint4*>(p.dV + krow * HD + ch * 64);
        uint4* ok4 = reinterpret_cast<uint4*>(p.dK + krow * HD + ch * 64);
        for (int v = 0; v < 8; ++v) ov[v] = ok4[v] = make_uint4(0u, 0u, 0u, 0u);
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

  // the accumulator's reductions are complete before the CTA exits
  if (warp < kCompute / 32 && lane == 0) bulk_wait_all();
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

// The rows' statistics from a saved O and its base-2 log-sum-exp: (-lse,
// Delta = dO . O) per row, and the row of the dQ accumulator cleared.  A warp
// per row, four values of the head dimension per lane.
__global__ void __launch_bounds__(256)
bwd_delta_kernel(const uint2* __restrict__ O, const uint2* __restrict__ dO,
                 const float* __restrict__ lse, float2* __restrict__ stats,
                 float4* __restrict__ acc, int64_t rows) {
  grid_dep_wait();   // launched as a programmatic dependent: O, dO, lse ready
  const int64_t row = (int64_t)blockIdx.x * 8 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  const uint2 o = O[row * 32 + lane], g = dO[row * 32 + lane];
  float d = __uint_as_float(o.x << 16) * __uint_as_float(g.x << 16);
  d = fmaf(__uint_as_float(o.x & 0xffff0000u), __uint_as_float(g.x & 0xffff0000u), d);
  d = fmaf(__uint_as_float(o.y << 16), __uint_as_float(g.y << 16), d);
  d = fmaf(__uint_as_float(o.y & 0xffff0000u), __uint_as_float(g.y & 0xffff0000u), d);
  for (int k = 16; k > 0; k >>= 1) d += __shfl_xor_sync(FULL, d, k);
  acc[row * 32 + lane] = make_float4(0.f, 0.f, 0.f, 0.f);
  if (lane == 0) stats[row] = make_float2(-lse[row], d);
}

// dQ = dq_acc / sqrt(128) in bf16
__global__ void dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ out,
                                  int64_t count4) {
  grid_dep_wait();   // launched as a programmatic dependent of the backward kernel
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= count4) return;
  const float4 v = acc[i];
  const float inv = 0.08838834764831845f;
  out[i] = make_uint2(pack_bf16(v.x * inv, v.y * inv), pack_bf16(v.z * inv, v.w * inv));
}

typedef CUresult (*EncodeTiledFnB)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// The dQ accumulator [planes, n, 128] fp32 as a 3-D tensor with 32 x 32 x 1
// boxes (128-byte rows) and 128-byte swizzle; rows past n are not written.
bool make_acc_map(CUtensorMap* map, float* base, int64_t planes, int64_t n) {
  static EncodeTiledFnB fn = nullptr;
  if (!fn) {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return false;
    fn = reinterpret_cast<EncodeTiledFnB>(ptr);
  }
  const cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)n, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)HD * 4, (cuuint64_t)n * HD * 4};
  const cuuint32_t box[3] = {32, 32, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Launches `kern` as a programmatic dependent of the kernel before it on `st`
// (each of these kernels waits for that kernel before it touches global
// memory), so that its launch overlaps that kernel's tail.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), unsigned grid, unsigned block, size_t smem,
                             cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(block);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace

size_t bwd_tc_smem_bytes() { return 1024 + OFF_END + sizeof(CtlB); }

cudaError_t launch_bwd_delta(const void* O, const void* dO, const float* lse, float* stats,
                             float* dq_acc, int64_t rows, cudaStream_t st) {
  if (rows <= 0) return cudaSuccess;
  return launch_dependent(bwd_delta_kernel, (unsigned)((rows + 7) / 8), 256, 0, st,
                          static_cast<const uint2*>(O), static_cast<const uint2*>(dO), lse,
                          reinterpret_cast<float2*>(stats), reinterpret_cast<float4*>(dq_acc),
                          rows);
}

cudaError_t launch_attn_bwd_tc(const void* Q, const void* K, const void* V, const void* dO,
                               void* dQ, void* dK, void* dV, const float* stats, float* dq_acc,
                               bool clear_acc, const plsh_bins* bn, int B, int Hq, int Hkv, int n,
                               int causal, int* queue, int* err, uint64_t wait_ns, int num_sms,
                               cudaStream_t st) {
  CUtensorMap mq, mk, mv, mdo, macc;
  if (!make_tile_map_bf16(&mq, Q, (int64_t)B * Hq, n) ||
      !make_tile_map_bf16(&mk, K, (int64_t)B * Hkv, n) ||
      !make_tile_map_bf16(&mv, V, (int64_t)B * Hkv, n) ||
      !make_tile_map_bf16(&mdo, dO, (int64_t)B * Hq, n) ||
      !make_acc_map(&macc, dq_acc, (int64_t)B * Hq, n))
    return cudaErrorInvalidValue;
  BwdTcParams p;
  p.rec = bn->d_rec;
  p.s = bn->s;
  p.W = bn->W;
  p.B = B;
  p.Hq = Hq;
  p.Hkv = Hkv;
  p.n = n;
  p.stats = stats;
  p.dq_acc = dq_acc;
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.num_items = B * Hkv * ((n + BM - 1) / BM);
  // KV groups by expected work, largest first: the rows a key reaches grow
  // with its heads' bin widths, which scale with sigma
  p.ordered = 0;
  const int G = Hq / Hkv;
  if (Hkv <= kMaxOrder && (int)bn->sigma_host.size() == Hq) {
    std::vector<double> cost(Hkv, 0.0);
    for (int g = 0; g < Hkv; ++g)
      for (int h = g * G; h < (g + 1) * G; ++h) cost[g] += 1.0 + bn->sigma_host[h] / BQ;
    std::vector<int> order(Hkv);
    std::iota(order.begin(), order.end(), 0);
    std::stable_sort(order.begin(), order.end(), [&](int a, int b) { return cost[a] > cost[b]; });
    for (int g = 0; g < Hkv; ++g) p.kv_order[g] = order[g];
    p.ordered = 1;
  }
  p.queue = queue;
  p.err = err;
  p.wait_ns = wait_ns;
  const size_t smem = bwd_tc_smem_bytes();
  cudaError_t e = cudaSuccess;
  if (clear_acc) e = cudaMemsetAsync(dq_acc, 0, sizeof(float) * (size_t)B * Hq * n * HD, st);
  if (e != cudaSuccess) return e;
  using Kern = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap,
                        BwdTcParams);
  const int sreg = p.s <= 4 ? 4 : p.s <= 8 ? 8 : p.s <= 10 ? 10 : p.s <= 12 ? 12 : 16;
  Kern kern = nullptr;
  switch (sreg) {
    case 4: kern = causal ? bwd_tc_kernel<true, 4> : bwd_tc_kernel<false, 4>; break;
    case 8: kern = causal ? bwd_tc_kernel<true, 8> : bwd_tc_kernel<false, 8>; break;
    case 10: kern = causal ? bwd_tc_kernel<true, 10> : bwd_tc_kernel<false, 10>; break;
    case 12: kern = causal ? bwd_tc_kernel<true, 12> : bwd_tc_kernel<false, 12>; break;
    default: kern = causal ? bwd_tc_kernel<true, 16> : bwd_tc_kernel<false, 16>; break;
  }
  e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  const int grid = p.num_items < num_sms ? p.num_items : num_sms;
  e = launch_dependent(kern, (unsigned)grid, kThreads, smem, st, mq, mk, mv, mdo, macc, p);
  if (e != cudaSuccess) return e;
  const int64_t count4 = (int64_t)B * Hq * n * HD / 4;
  return launch_dependent(dq_convert_kernel, (unsigned)((count4 + 255) / 256), 256, 0, st,
                          reinterpret_cast<const float4*>(dq_acc), static_cast<uint2*>(dQ),
                          count4);
}

}  // namespace plsh
