// Fused block attention on the sm_103a tensor cores (tcgen05 + TMEM + TMA).
//
// Positional LSH ("Positional LSH: Binary Block Matrix Approximation for
// Attention with Linear Biases", technical summary, Methodology 3 /
// Theorem 2.2): ALiBi attention becomes short block attentions without
// positional bias, numerator and row sums both averaged over s masks:
//   O_i = sum_t sum_{j in J_t(i)} e^{S_ij} v_j / sum_t sum_{j in J_t(i)} e^{S_ij}.
// Every hash shares the scores S = QK^T/sqrt(d); only the mask differs.  So
// each (query tile, key tile) score block is computed once, over the union of
// the rows' bins, and weighted by the multiplicity
//   c_ij = #{t : i and j share a bin of hash t}      (j <= i when causal),
// which gives the same sums as the per-sample loop.  Every bin of row i
// contains i, so the keys with c_ij > 0 form one interval [lo_min(i), i]
// (or [lo_min, hi_max) without the causal mask), and inside it c_i(j) is a
// step function of j that rises at the bin starts lo_t(i) (and falls at the
// bin ends hi_t(i) when not causal).  The row's thread keeps those starts
// sorted in shared memory and walks them while it sweeps the key tiles: a
// 32-key chunk with no step takes log2(c) into the exponent's FMA offset, a
// chunk with steps adds one ramp per distinct step position.
//
// Exact ALiBi (the dense comparator) runs on the same pipeline with weight
// e^{S_ij - |i-j|/sigma_h} over every key tile.
//
// Pipeline (one persistent CTA per SM, 6 warps):
//   warp 4      producer: pops work items (b, h, 128-row query tile) from a
//               global queue ordered by expected cost, stages the item's bin
//               records in shared memory, finds its key envelope, TMA-loads Q
//               (two item stages) and K/V tiles (two stages each) from the
//               diagonal tile down;
//   warp 5      one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//               score buffers, then O += P V into the TMEM accumulator
//               (tcgen05 MMAs of one thread execute in issue order, so the
//               next S into a buffer lands after the P V that reads it);
//   warps 0-3   one thread per query row: tcgen05.ld of the score row, running
//               max over the valid keys, lazy rescale of O in TMEM (only when
//               the max grows by more than 2^8), P = 2^(x - m) split into two
//               bf16 terms P = P_hi + P_lo written back over the consumed
//               score columns, row sums in fp32, and the final O / l epilogue.
//   O += P_hi V + P_lo V runs as two tensor-core products with A read from
//   TMEM: a single bf16 P carries a 2^-9 relative error per weight, which
//   shows in rows whose few keys cancel; the pair carries about 2^-17.
// Every wait on an mbarrier is bounded; on expiry the CTA raises the library
// error flag, drains its in-flight copies and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_runtime.h>
#include <limits.h>
#include <stdint.h>

#include <mutex>

#include "bins_dev.cuh"
#include "plsh_internal.h"
#include "tc_ptx.cuh"

namespace plsh {
namespace {

using namespace ptx;

constexpr int BM = 128;      // query rows per tile (MMA M)
constexpr int BN = 128;      // keys per tile (MMA N of QK^T, K of PV)
constexpr int HD = 128;      // head dim (MMA K of QK^T, N of PV)
constexpr int kThreads = 192;
constexpr uint32_t kTileBytes = BM * HD * 2;     // 32 KB bf16 tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 64-column TMA box
constexpr uint32_t OFF_Q = 0;                        // two item stages
constexpr uint32_t OFF_K = OFF_Q + 2 * kTileBytes;   // two tile stages
constexpr uint32_t OFF_V = OFF_K + 2 * kTileBytes;   // two tile stages
constexpr uint32_t OFF_BP = OFF_V + 2 * kTileBytes;
constexpr uint32_t kTmemCols = 512;   // S0 | S1 | O | unused; P over S
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)
constexpr unsigned FULL = 0xffffffffu;
constexpr int kWordsPerTile = BM / 32;

enum {
  B_QFULL = 0, B_QFULL1, B_QEMPTY, B_QEMPTY1, B_KFULL, B_KFULL1, B_KEMPTY,
  B_KEMPTY1, B_VFULL, B_VFULL1, B_VEMPTY, B_VEMPTY1, B_SFULL, B_SFULL1,
  B_PFULL, B_PVDONE, B_IFULL, B_IFULL1, B_IEMPTY, B_IEMPTY1, B_DRAIN, NUM_BARS
};

struct Item {
  int valid, b, h, qt, kt_lo, kt_hi;
};

struct Ctl {
  uint64_t bars[NUM_BARS];
  Item ring[2];
  uint32_t tmem_base;
  int abort;
};

struct TcParams {
  AttnArgs a;
  float slope_log2[512];   // exact mode: log2(e) / sigma_h
  int num_items;
  int QT;                  // query tiles per (b, h)
};

// Sorted bin starts (and ends when not causal) of every row: [lists][s][BM].
__host__ __device__ constexpr uint32_t bp_bytes(int s, bool exact, bool causal) {
  return exact ? 0u : (uint32_t)(causal ? 1 : 2) * (uint32_t)s * BM * 4u;
}
// Bin records of the item's 128 rows, one ring slot per item: [2][s][4] x 16 B.
__host__ __device__ constexpr uint32_t stage_bytes(int s, bool exact) {
  return exact ? 0u : 2u * (uint32_t)s * kWordsPerTile * 16u;
}

__device__ __forceinline__ Item read_item(const Ctl* ctl, int slot) {
  const volatile int* v = reinterpret_cast<const volatile int*>(&ctl->ring[slot]);
  Item it;
  it.valid = v[0]; it.b = v[1]; it.h = v[2]; it.qt = v[3];
  it.kt_lo = v[4]; it.kt_hi = v[5];
  return it;
}

__device__ __forceinline__ BinRecord unpack_record(const uint4& rv) {
  BinRecord rc;
  rc.bits = rv.x;
  rc.prev = (int)rv.y;
  rc.next = (int)rv.z;
  rc.pad = 0;
  return rc;
}

template <bool EXACT, bool CAUSAL>
__global__ void __launch_bounds__(kThreads, 1)
attn_tc_kernel(const __grid_constant__ CUtensorMap tmQ,
               const __grid_constant__ CUtensorMap tmK,
               const __grid_constant__ CUtensorMap tmV,
               const __grid_constant__ TcParams p) {
  extern __shared__ uint8_t smem_raw[];
  const AttnArgs& a = p.a;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t raw_u32 = smem_u32(smem_raw);
  const uint32_t sbase = (raw_u32 + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_u32);
  const int s = a.s;
  int* bp = reinterpret_cast<int*>(smem + OFF_BP);
  uint4* stage = reinterpret_cast<uint4*>(smem + OFF_BP + bp_bytes(s, EXACT, CAUSAL));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + OFF_BP + bp_bytes(s, EXACT, CAUSAL) +
                                    stage_bytes(s, EXACT));
  auto bar = [&](int k) { return smem_u32(&ctl->bars[k]); };
  volatile int* abort = &ctl->abort;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_QFULL + k), 1);
      mbar_init(bar(B_QEMPTY + k), 1);
      mbar_init(bar(B_KFULL + k), 1);
      mbar_init(bar(B_KEMPTY + k), 1);
      mbar_init(bar(B_VFULL + k), 1);
      mbar_init(bar(B_VEMPTY + k), 1);
      mbar_init(bar(B_SFULL + k), 1);
      mbar_init(bar(B_IFULL + k), 1);
      mbar_init(bar(B_IEMPTY + k), 1 + BM);
    }
    mbar_init(bar(B_PFULL), BM);
    mbar_init(bar(B_PVDONE), 1);
    mbar_init(bar(B_DRAIN), 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == 5) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 4 && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const int n = a.n, Hq = a.Hq, Hkv = a.Hkv, B = a.B;
  const int QT = p.QT;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    int g = 0;
    int q_issued[2] = {0, 0}, k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
    bool ok = true;
    for (int seq = 0;; ++seq) {
      const int slot = seq & 1;
      const uint32_t use = (uint32_t)seq >> 1;
      int idx = 0;
      if (lane == 0) {
        ok = mbar_wait(bar(B_IEMPTY + slot), (use & 1u) ^ 1u, abort, lim);
        if (ok) idx = atomicAdd(a.queue, 1);
      }
      ok = __shfl_sync(FULL, (int)ok, 0) != 0;
      idx = __shfl_sync(FULL, idx, 0);
      if (!ok) break;
      if (idx >= p.num_items) {
        if (lane == 0) {
          ctl->ring[slot].valid = 0;
          mbar_arrive(bar(B_IFULL + slot));
        }
        break;
      }
      int b, h, qt;
      if (EXACT) {
        // longest rows first: query tiles in descending order
        qt = QT - 1 - idx / (B * Hq);
        const int rem = idx % (B * Hq);
        b = rem / Hq;
        h = rem % Hq;
      } else {
        // heads in descending expected work, then every (b, query tile)
        const int hh = idx / (B * QT);
        const int rem = idx % (B * QT);
        h = a.head_order[hh];
        b = rem / QT;
        qt = rem % QT;
      }
      const int i0 = qt * BM;
      int kt_lo, kt_hi;
      if (EXACT) {
        kt_lo = 0;
        kt_hi = CAUSAL ? qt + 1 : (n + BN - 1) / BN;
      } else {
        // stage the records of the tile's rows (4 words per hash) and find
        // the key envelope: lo_t(i) is non-decreasing in i, so the first row
        // bounds it from the left (the last row from the right)
        const int w0 = i0 >> 5;
        const int ilast = min(i0 + BM - 1, n - 1);
        int mylo = INT_MAX, myhi = 0;
        uint4* dst = stage + slot * s * kWordsPerTile;
        for (int e = lane; e < s * kWordsPerTile; e += 32) {
          const int t = e / kWordsPerTile, wq = e % kWordsPerTile;
          const int wd = min(w0 + wq, (int)a.W - 1);
          const uint4 rv = __ldg(reinterpret_cast<const uint4*>(a.rec) +
                                 ((int64_t)h * s + t) * a.W + wd);
          dst[e] = rv;
          const BinRecord rc = unpack_record(rv);
          if (wq == 0) mylo = min(mylo, bin_lo(rc, i0));
          if (!CAUSAL && wd == (ilast >> 5)) myhi = max(myhi, bin_hi(rc, ilast));
        }
        mylo = __reduce_min_sync(FULL, mylo);
        kt_lo = mylo / BN;
        if (CAUSAL) {
          kt_hi = qt + 1;
        } else {
          myhi = __reduce_max_sync(FULL, myhi);
          kt_hi = (myhi + BN - 1) / BN;
        }
        __syncwarp();
      }
      kt_lo = min(kt_lo, qt);
      kt_hi = max(kt_hi, kt_lo + 1);
      if (lane == 0) {
        volatile int* it = reinterpret_cast<volatile int*>(&ctl->ring[slot]);
        it[0] = 1; it[1] = b; it[2] = h; it[3] = qt; it[4] = kt_lo; it[5] = kt_hi;
        mbar_arrive(bar(B_IFULL + slot));
        const int qs = seq & 1;
        ok = mbar_wait(bar(B_QEMPTY + qs), (use & 1u) ^ 1u, abort, lim);
        if (ok) {
          const int qp = b * Hq + h;
          const uint32_t qdst = sbase + OFF_Q + qs * kTileBytes;
          mbar_arrive_expect_tx(bar(B_QFULL + qs), kTileBytes);
          tma_load_3d(qdst, &tmQ, bar(B_QFULL + qs), 0, i0, qp);
          tma_load_3d(qdst + kHalfBytes, &tmQ, bar(B_QFULL + qs), 64, i0, qp);
          ++q_issued[qs];
        }
        const int kvp = b * Hkv + h / (Hq / Hkv);
        for (int kt = kt_hi - 1; ok && kt >= kt_lo; --kt, ++g) {
          const int st = g & 1;
          const uint32_t u = (uint32_t)g >> 1;
          ok = mbar_wait(bar(B_KEMPTY + st), (u & 1u) ^ 1u, abort, lim);
          if (!ok) break;
          const uint32_t kdst = sbase + OFF_K + st * kTileBytes;
          mbar_arrive_expect_tx(bar(B_KFULL + st), kTileBytes);
          tma_load_3d(kdst, &tmK, bar(B_KFULL + st), 0, kt * BN, kvp);
          tma_load_3d(kdst + kHalfBytes, &tmK, bar(B_KFULL + st), 64, kt * BN, kvp);
          ++k_issued[st];
          ok = mbar_wait(bar(B_VEMPTY + st), (u & 1u) ^ 1u, abort, lim);
          if (!ok) break;
          const uint32_t vdst = sbase + OFF_V + st * kTileBytes;
          mbar_arrive_expect_tx(bar(B_VFULL + st), kTileBytes);
          tma_load_3d(vdst, &tmV, bar(B_VFULL + st), 0, kt * BN, kvp);
          tma_load_3d(vdst + kHalfBytes, &tmV, bar(B_VFULL + st), 64, kt * BN, kvp);
          ++v_issued[st];
        }
      }
      ok = __shfl_sync(FULL, (int)ok, 0) != 0;
      g = __shfl_sync(FULL, g, 0);
      if (!ok) break;
    }
    if (lane == 0) {
      if (!ok) {
        *abort = 1;
        atomicOr(a.err, 1);
      }
      // let every copy this warp started land before the CTA can exit
      for (int st = 0; st < 2; ++st) {
        if (q_issued[st])
          mbar_wait(bar(B_QFULL + st), (uint32_t)(q_issued[st] - 1) & 1u, nullptr, lim);
        if (k_issued[st])
          mbar_wait(bar(B_KFULL + st), (uint32_t)(k_issued[st] - 1) & 1u, nullptr, lim);
        if (v_issued[st])
          mbar_wait(bar(B_VFULL + st), (uint32_t)(v_issued[st] - 1) & 1u, nullptr, lim);
      }
    }
    __syncwarp();
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_bf16_f32(BM, HD, 0, 1);
      bool ok = true;
      int g = 0;
      auto issue_pv = [&](int gp, bool first) -> bool {
        const int st = gp & 1;
        const uint32_t u = (uint32_t)gp >> 1;
        if (!mbar_wait(bar(B_PFULL), (uint32_t)gp & 1u, abort, lim)) return false;
        if (!mbar_wait(bar(B_VFULL + st), u & 1u, abort, lim)) return false;
        tc_fence_after();
        const uint32_t vbase = sbase + OFF_V + st * kTileBytes;
        // keys 16kk..16kk+15 sit in chunk kk/2: P_hi in its first 16
        // columns, P_lo in the next 16, 8 packed columns per 16 keys
        const uint32_t pcol = tmem + st * BN;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = desc_sw128(vbase + kk * 2048, kHalfBytes, 1024);
          const uint32_t ac = pcol + (kk >> 1) * 32 + (kk & 1) * 8;
          mma_bf16_ts(tmem + kColO, ac, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
          mma_bf16_ts(tmem + kColO, ac + 16, bd, idesc_pv, 1u);
        }
        mma_commit(bar(B_PVDONE));
        mma_commit(bar(B_VEMPTY + st));
        return true;
      };
      for (int seq = 0; ok; ++seq) {
        const int slot = seq & 1;
        const uint32_t use = (uint32_t)seq >> 1;
        ok = mbar_wait(bar(B_IFULL + slot), use & 1u, abort, lim);
        if (!ok) break;
        const Item it = read_item(ctl, slot);
        if (!it.valid) break;
        const int ntiles = it.kt_hi - it.kt_lo;
        const int qs = seq & 1;
        ok = mbar_wait(bar(B_QFULL + qs), use & 1u, abort, lim);
        if (!ok) break;
        const uint32_t qbase = sbase + OFF_Q + qs * kTileBytes;
        for (int jj = 0; jj < ntiles; ++jj, ++g) {
          const int st = g & 1;
          const uint32_t u = (uint32_t)g >> 1;
          ok = mbar_wait(bar(B_KFULL + st), u & 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kbase = sbase + OFF_K + st * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            const uint64_t ad = desc_sw128(qbase + koff, 16, 1024);
            const uint64_t bd = desc_sw128(kbase + koff, 16, 1024);
            mma_bf16_ss(tmem + st * BN, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL + st));
          mma_commit(bar(B_KEMPTY + st));
          if (jj == ntiles - 1) mma_commit(bar(B_QEMPTY + qs));
          if (jj > 0) {
            ok = issue_pv(g - 1, jj == 1);
            if (!ok) break;
          }
        }
        if (!ok) break;
        ok = issue_pv(g - 1, ntiles == 1);
        if (!ok) break;
        mbar_arrive(bar(B_IEMPTY + slot));
      }
      if (!ok) {
        *abort = 1;
        atomicOr(a.err, 1);
      }
      // every MMA issued by this thread has completed once this arrives
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr, lim);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- softmax / epilogue
    const int r = threadIdx.x;   // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)(warp * 32) << 16;
    const float scale_log2 = 1.4426950408889634f * 0.08838834764831845f;  // log2(e)/sqrt(128)
    int* bpl = bp;                 // sorted bin starts of this row, [s][BM]
    int* bph = bp + s * BM;        // sorted bin ends (non-causal), [s][BM]
    bool ok = true;
    int g = 0;
    for (int seq = 0; ok; ++seq) {
      const int slot = seq & 1;
      const uint32_t use = (uint32_t)seq >> 1;
      ok = __all_sync(FULL, mbar_wait(bar(B_IFULL + slot), use & 1u, abort, lim));
      if (!ok) break;
      const Item it = read_item(ctl, slot);
      if (!it.valid) break;
      const int i0 = it.qt * BM;
      const int i = i0 + r;
      const bool row_ok = i < n;
      const int ii = row_ok ? i : n - 1;
      const int h = it.h;
      const int ntiles = it.kt_hi - it.kt_lo;
      // keys that take part: [vlo, vhi]
      int vlo = 0, vhi = CAUSAL ? ii : n - 1;
      int pl = s, ph = s, ql = s, qh = s;
      float slope = 0.f;
      if (EXACT) {
        slope = p.slope_log2[h];
      } else {
        // this row's bin starts (and ends) under every hash, sorted
        const uint4* rs = stage + slot * s * kWordsPerTile + ((ii >> 5) - (i0 >> 5));
        for (int t = 0; t < s; ++t) {
          const BinRecord rc = unpack_record(rs[t * kWordsPerTile]);
          const int lo = bin_lo(rc, ii);
          int k = t;
          while (k > 0) {
            const int prev = bpl[(k - 1) * BM + r];
            if (prev <= lo) break;
            bpl[k * BM + r] = prev;
            --k;
          }
          bpl[k * BM + r] = lo;
          if (!CAUSAL) {
            const int hi = bin_hi(rc, ii);
            int k2 = t;
            while (k2 > 0) {
              const int prev = bph[(k2 - 1) * BM + r];
              if (prev <= hi) break;
              bph[k2 * BM + r] = prev;
              --k2;
            }
            bph[k2 * BM + r] = hi;
          }
        }
        vlo = bpl[r];
        if (!CAUSAL) vhi = bph[(s - 1) * BM + r] - 1;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int jj = 0; jj < ntiles; ++jj, ++g) {
        const int st = g & 1;
        const uint32_t u = (uint32_t)g >> 1;
        const int jt = (it.kt_hi - 1 - jj) * BN;
        const uint32_t s_col = tmem + lane_base + st * BN;
        ok = __all_sync(FULL, mbar_wait(bar(B_SFULL + st), u & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();

        // pass 1: running max (log2 units) over the keys that take part
        float mt = -INFINITY;
#pragma unroll 1
        for (int q2 = 0; q2 < 2; ++q2) {
          uint32_t ra[32], rb2[32];
          tmem_ld32(s_col + q2 * 64, ra);
          tmem_ld32(s_col + q2 * 64 + 32, rb2);
          tmem_wait_ld();
#pragma unroll
          for (int half = 0; half < 2; ++half) {
            const uint32_t* rr = half ? rb2 : ra;
            const int jc = jt + q2 * 64 + half * 32;
            if (EXACT) {
              const float d0 = (float)(i - jc);
              if (CAUSAL) {
                const float base = -d0 * slope;
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  float x = fmaf(__uint_as_float(rr[e]), scale_log2, fmaf((float)e, slope, base));
                  if (jc + e > i) x = -INFINITY;
                  mt = fmaxf(mt, x);
                }
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) {
                  float x = fmaf(__uint_as_float(rr[e]), scale_log2,
                                 -fabsf(d0 - (float)e) * slope);
                  if (jc + e >= n) x = -INFINITY;
                  mt = fmaxf(mt, x);
                }
              }
            } else {
              const int ea = vlo - jc, eb = vhi - jc;
              if (__all_sync(FULL, ea <= 0 && eb >= 31)) {
#pragma unroll
                for (int e = 0; e < 32; ++e) mt = fmaxf(mt, __uint_as_float(rr[e]));
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (e >= ea && e <= eb) mt = fmaxf(mt, __uint_as_float(rr[e]));
              }
            }
          }
        }
        if (!EXACT) mt *= scale_log2;
        if (!row_ok) mt = -INFINITY;
        const float m_new = fmaxf(m_ref, mt);
        const bool resc = m_new > m_ref + kRescaleLog2;
        const float m_use = resc ? m_new : m_ref;
        const float alpha = resc ? ex2(m_ref - m_new) : 1.f;
        const float mu = (m_use == -INFINITY || !row_ok) ? 0.f : m_use;

        // pass 2: P = c 2^(x - m) = P_hi + P_lo (two bf16 terms) written over
        // the chunk's own score columns; chunks in descending key order so
        // that the breakpoint pointers only move down
        float lsum = 0.f;
#pragma unroll 1
        for (int q = 3; q >= 0; --q) {
          const int jc = jt + q * 32;
          uint32_t rr[32];
          tmem_ld32(s_col + q * 32, rr);
          float pv[32];
          if (EXACT) {
            tmem_wait_ld();
            const float d0 = (float)(i - jc);
#pragma unroll
            for (int e = 0; e < 32; ++e) {
              float x = CAUSAL
                  ? fmaf(__uint_as_float(rr[e]), scale_log2, fmaf((float)e, slope, -d0 * slope))
                  : fmaf(__uint_as_float(rr[e]), scale_log2, -fabsf(d0 - (float)e) * slope);
              if (CAUSAL ? (jc + e > i) : (jc + e >= n)) x = -INFINITY;
              pv[e] = ex2(x - mu);
            }
          } else {
            while (pl > 0 && bpl[(pl - 1) * BM + r] > jc) --pl;
            while (ph > pl && bpl[(ph - 1) * BM + r] > jc + 31) --ph;
            int base = pl;
            bool flat = ph == pl;
            if (!CAUSAL) {
              while (ql > 0 && bph[(ql - 1) * BM + r] > jc) --ql;
              while (qh > ql && bph[(qh - 1) * BM + r] > jc + 31) --qh;
              base -= ql;
              flat = flat && qh == ql;
            }
            const int ea = vlo - jc, eb = vhi - jc;
            const bool inside = ea <= 0 && eb >= 31 && row_ok;
            const bool outside = ea > 31 || eb < 0 || !row_ok;
            tmem_wait_ld();
            if (__all_sync(FULL, outside)) {
#pragma unroll
              for (int e = 0; e < 32; ++e) pv[e] = 0.f;
            } else if (__all_sync(FULL, (flat && inside) || outside)) {
              // one multiplicity for the whole chunk: log2(c) rides in the FMA
              const float off = outside ? -INFINITY : lg2((float)base) - mu;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                pv[e] = ex2(fmaf(__uint_as_float(rr[e]), scale_log2, off));
            } else {
              float cf[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) cf[e] = (float)base;
              // one ramp per distinct step position inside the chunk
              for (int k = pl; k < ph;) {
                const int bpos = bpl[k * BM + r];
                int k2 = k + 1;
                while (k2 < ph && bpl[k2 * BM + r] == bpos) ++k2;
                const int bo = bpos - jc;
                const float mult = (float)(k2 - k);
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (e >= bo) cf[e] += mult;
                k = k2;
              }
              if (!CAUSAL) {
                for (int k = ql; k < qh;) {
                  const int bpos = bph[k * BM + r];
                  int k2 = k + 1;
                  while (k2 < qh && bph[k2 * BM + r] == bpos) ++k2;
                  const int bo = bpos - jc;
                  const float mult = (float)(k2 - k);
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    if (e >= bo) cf[e] -= mult;
                  k = k2;
                }
              }
#pragma unroll
              for (int e = 0; e < 32; ++e) {
                const bool in = e >= ea && e <= eb && row_ok;
                pv[e] = in ? ex2(fmaf(__uint_as_float(rr[e]), scale_log2, -mu)) * cf[e] : 0.f;
              }
            }
          }
          uint32_t hi[16], lo[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            const float p0 = pv[2 * e2], p1 = pv[2 * e2 + 1];
            lsum += p0 + p1;
            const uint32_t hp = pack_bf16(p0, p1);
            hi[e2] = hp;
            lo[e2] = pack_bf16(p0 - __uint_as_float(hp << 16),
                               p1 - __uint_as_float(hp & 0xffff0000u));
          }
          tmem_st16(s_col + q * 32, hi);
          tmem_st16(s_col + q * 32 + 16, lo);
        }
        l = l * alpha + lsum;
        m_ref = m_use;

        // P(g) may be published once P V(g-1) has landed: this keeps every
        // barrier within one phase of its waiters, and a grown max rescales
        // O only after that product
        if (g > 0) {
          ok = __all_sync(FULL, mbar_wait(bar(B_PVDONE), (uint32_t)(g - 1) & 1u, abort, lim));
          if (!ok) break;
        }
        tc_fence_after();
        if (jj > 0 && __any_sync(FULL, resc)) {
          const float f = resc ? alpha : 1.f;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kColO + q * 32;
            tmem_ld32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(ta, o);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL));
      }
      if (!ok) break;

      // epilogue: O_i = acc_i / l_i
      ok = __all_sync(FULL, mbar_wait(bar(B_PVDONE), (uint32_t)(g - 1) & 1u, abort, lim));
      if (!ok) break;
      tc_fence_after();
      const float inv_l = l > 0.f ? 1.f / l : 0.f;
      uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.O) +
                                             (((int64_t)it.b * Hq + h) * n + ii) * HD);
#pragma unroll 1
      for (int q = 0; q < 4; ++q) {
        uint32_t o[32];
        tmem_ld32(tmem + lane_base + kColO + q * 32, o);
        tmem_wait_ld();
        uint32_t pk[16];
#pragma unroll
        for (int e2 = 0; e2 < 16; ++e2)
          pk[e2] = pack_bf16(__uint_as_float(o[2 * e2]) * inv_l,
                             __uint_as_float(o[2 * e2 + 1]) * inv_l);
        if (row_ok) {
#pragma unroll
          for (int v = 0; v < 4; ++v)
            orow[q * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_IEMPTY + slot));
    }
    if (!ok && lane == 0) {
      *abort = 1;
      atomicOr(a.err, 1);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
  if (threadIdx.x == 0) {
    // the last CTA to finish returns the queue slot to zero for the next call
    __threadfence();
    if (atomicAdd(a.queue + 1, 1) == (int)gridDim.x - 1) {
      atomicExch(a.queue, 0);
      atomicExch(a.queue + 1, 0);
      __threadfence();
    }
  }
}

// ------------------------------------------------------------------- host
typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t,
                                  void*, const cuuint64_t*, const cuuint64_t*,
                                  const cuuint32_t*, const cuuint32_t*,
                                  CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion,
                                  CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// [planes, n, 128] bf16 viewed as a 3-D tensor with 64 x 128 x 1 boxes and
// 128-byte swizzle; rows past n read as zeros.
bool make_map(CUtensorMap* map, const void* base, int64_t planes, int64_t n) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)HD, (cuuint64_t)n, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)HD * 2, (cuuint64_t)n * HD * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)BM, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool EXACT, bool CAUSAL>
cudaError_t launch_variant(const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const TcParams& p,
                           size_t smem, int grid, cudaStream_t st) {
  auto kern = attn_tc_kernel<EXACT, CAUSAL>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, smem, st>>>(mq, mk, mv, p);
  return cudaGetLastError();
}

}  // namespace

size_t attn_tc_smem_bytes(int s, int causal, int exact) {
  return 1024 + OFF_BP + bp_bytes(s, exact != 0, causal != 0) +
         stage_bytes(s, exact != 0) + sizeof(Ctl);
}

cudaError_t launch_attn_tc(const AttnArgs& a, const float* slopes_host,
                           int num_sms, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.Q, (int64_t)a.B * a.Hq, a.n) ||
      !make_map(&mk, a.K, (int64_t)a.B * a.Hkv, a.n) ||
      !make_map(&mv, a.V, (int64_t)a.B * a.Hkv, a.n))
    return cudaErrorInvalidValue;
  TcParams p;
  p.a = a;
  for (int h = 0; h < 512; ++h)
    p.slope_log2[h] = (slopes_host && h < a.Hq) ? slopes_host[h] : 0.f;
  p.QT = (a.n + BM - 1) / BM;
  p.num_items = a.B * a.Hq * p.QT;
  const int grid = p.num_items < num_sms ? p.num_items : num_sms;
  const size_t smem = attn_tc_smem_bytes(a.s, a.causal, a.exact);
  if (a.exact) {
    return a.causal ? launch_variant<true, true>(mq, mk, mv, p, smem, grid, st)
                    : launch_variant<true, false>(mq, mk, mv, p, smem, grid, st);
  }
  return a.causal ? launch_variant<false, true>(mq, mk, mv, p, smem, grid, st)
                  : launch_variant<false, false>(mq, mk, mv, p, smem, grid, st);
}

}  // namespace plsh
