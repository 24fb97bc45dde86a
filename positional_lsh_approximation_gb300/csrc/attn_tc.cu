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
// which gives the same sums as the per-sample loop.  For row i, c_i(j) is a
// step function of j that rises at the s bin starts lo_t(i) (and falls at the
// bin ends hi_t(i) when not causal); the row's thread keeps those starts
// sorted in shared memory and walks them while it sweeps the key tiles.
// c enters the exponent as log2(c), so a chunk of keys with a constant count
// costs one FMA per score.
//
// Exact ALiBi (the dense comparator) runs on the same pipeline with weight
// e^{S_ij - |i-j|/sigma_h} over every key tile.
//
// Pipeline (one persistent CTA per SM, 6 warps):
//   warp 4      producer: pops work items (b, h, 128-row query tile) from a
//               global queue ordered by expected cost, finds the item's key
//               envelope from the bin records, TMA-loads Q once and K/V tiles
//               (two stages each) from the diagonal tile downwards;
//   warp 5      one thread issues tcgen05.mma: S = Q K^T into one of two TMEM
//               score buffers, then O += P V into the TMEM accumulator;
//   warps 0-3   one thread per query row: tcgen05.ld of the score row,
//               weights and running max, lazy rescale of O in TMEM (only when
//               the max grows by more than 2^8), P = 2^(x - m) in bf16 written
//               to shared memory in the 128B-swizzled K-major layout, row sums
//               in fp32, and the final O / l epilogue.
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
constexpr uint32_t OFF_Q = 0;
constexpr uint32_t OFF_K = OFF_Q + kTileBytes;
constexpr uint32_t OFF_V = OFF_K + 2 * kTileBytes;
constexpr uint32_t OFF_P = OFF_V + 2 * kTileBytes;
constexpr uint32_t OFF_BP = OFF_P + kTileBytes;
constexpr uint32_t kTmemCols = 512;   // S0 | S1 | O | unused
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)
constexpr unsigned FULL = 0xffffffffu;

enum {
  B_QFULL = 0, B_QEMPTY, B_KFULL, B_KFULL1, B_KEMPTY, B_KEMPTY1, B_VFULL,
  B_VFULL1, B_VEMPTY, B_VEMPTY1, B_SFULL, B_SFULL1, B_SFREE, B_SFREE1, B_PFULL,
  B_PVDONE, B_IFULL, B_IFULL1, B_IEMPTY, B_IEMPTY1, B_DRAIN, NUM_BARS
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

__host__ __device__ constexpr uint32_t bp_bytes(int s, bool exact, bool causal) {
  return exact ? 0u : (uint32_t)(causal ? 1 : 2) * (uint32_t)s * BM * 4u;
}

__device__ __forceinline__ Item read_item(const Ctl* ctl, int slot) {
  const volatile int* v = reinterpret_cast<const volatile int*>(&ctl->ring[slot]);
  Item it;
  it.valid = v[0]; it.b = v[1]; it.h = v[2]; it.qt = v[3];
  it.kt_lo = v[4]; it.kt_hi = v[5];
  return it;
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
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + OFF_BP + bp_bytes(s, EXACT, CAUSAL));
  auto bar = [&](int k) { return smem_u32(&ctl->bars[k]); };
  volatile int* abort = &ctl->abort;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    mbar_init(bar(B_QFULL), 1);
    mbar_init(bar(B_QEMPTY), 1);
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_KFULL + k), 1);
      mbar_init(bar(B_KEMPTY + k), 1);
      mbar_init(bar(B_VFULL + k), 1);
      mbar_init(bar(B_VEMPTY + k), 1);
      mbar_init(bar(B_SFULL + k), 1);
      mbar_init(bar(B_SFREE + k), BM);
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
    int g = 0, q_issued = 0;
    int k_issued[2] = {0, 0}, v_issued[2] = {0, 0};
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
        // the tile's key envelope: bins are contiguous and lo_t(i) is
        // non-decreasing in i, so the first row bounds it from the left
        const int ilast = min(i0 + BM - 1, n - 1);
        int mylo = INT_MAX, myhi = 0;
        for (int t = lane; t < s; t += 32) {
          const int64_t rb = ((int64_t)h * s + t) * a.W;
          mylo = min(mylo, bin_lo(load_record(a.rec, rb + (i0 >> 5)), i0));
          if (!CAUSAL)
            myhi = max(myhi, bin_hi(load_record(a.rec, rb + (ilast >> 5)), ilast));
        }
        mylo = __reduce_min_sync(FULL, mylo);
        kt_lo = mylo / BN;
        if (CAUSAL) {
          kt_hi = qt + 1;
        } else {
          myhi = __reduce_max_sync(FULL, myhi);
          kt_hi = (myhi + BN - 1) / BN;
        }
      }
      kt_lo = min(kt_lo, qt);
      kt_hi = max(kt_hi, kt_lo + 1);
      if (lane == 0) {
        volatile int* it = reinterpret_cast<volatile int*>(&ctl->ring[slot]);
        it[0] = 1; it[1] = b; it[2] = h; it[3] = qt; it[4] = kt_lo; it[5] = kt_hi;
        mbar_arrive(bar(B_IFULL + slot));
        ok = mbar_wait(bar(B_QEMPTY), ((uint32_t)seq & 1u) ^ 1u, abort, lim);
        if (ok) {
          const int qp = b * Hq + h;
          mbar_arrive_expect_tx(bar(B_QFULL), kTileBytes);
          tma_load_3d(sbase + OFF_Q, &tmQ, bar(B_QFULL), 0, i0, qp);
          tma_load_3d(sbase + OFF_Q + kHalfBytes, &tmQ, bar(B_QFULL), 64, i0, qp);
          ++q_issued;
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
      if (q_issued) mbar_wait(bar(B_QFULL), (uint32_t)(q_issued - 1) & 1u, nullptr, lim);
      for (int st = 0; st < 2; ++st) {
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
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t ad = desc_sw128(sbase + OFF_P + (kk >> 2) * kHalfBytes +
                                             (kk & 3) * 32, 16, 1024);
          const uint64_t bd = desc_sw128(vbase + kk * 2048, kHalfBytes, 1024);
          mma_bf16_ss(tmem + kColO, ad, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
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
        ok = mbar_wait(bar(B_QFULL), (uint32_t)seq & 1u, abort, lim);
        if (!ok) break;
        for (int jj = 0; jj < ntiles; ++jj, ++g) {
          const int st = g & 1;
          const uint32_t u = (uint32_t)g >> 1;
          ok = mbar_wait(bar(B_KFULL + st), u & 1u, abort, lim);
          if (ok) ok = mbar_wait(bar(B_SFREE + st), (u & 1u) ^ 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
          const uint32_t kbase = sbase + OFF_K + st * kTileBytes;
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk) {
            const uint32_t koff = (kk >> 2) * kHalfBytes + (kk & 3) * 32;
            const uint64_t ad = desc_sw128(sbase + OFF_Q + koff, 16, 1024);
            const uint64_t bd = desc_sw128(kbase + koff, 16, 1024);
            mma_bf16_ss(tmem + st * BN, ad, bd, idesc_qk, kk > 0 ? 1u : 0u);
          }
          mma_commit(bar(B_SFULL + st));
          mma_commit(bar(B_KEMPTY + st));
          if (jj == ntiles - 1) mma_commit(bar(B_QEMPTY));
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
      int pl = s, ph = s, ql = s, qh = s;
      float slope = 0.f;
      if (EXACT) {
        slope = p.slope_log2[h];
      } else {
        // this row's bin starts (and ends) under every hash, sorted
        const int64_t rb = (int64_t)h * s * a.W + (ii >> 5);
        for (int t0 = 0; t0 < s; t0 += 4) {
          BinRecord rr[4];
#pragma unroll
          for (int q = 0; q < 4; ++q)
            if (t0 + q < s) rr[q] = load_record(a.rec, rb + (int64_t)(t0 + q) * a.W);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (t0 + q >= s) break;
            const int lo = bin_lo(rr[q], ii);
            int k = t0 + q;
            while (k > 0) {
              const int prev = bpl[(k - 1) * BM + r];
              if (prev <= lo) break;
              bpl[k * BM + r] = prev;
              --k;
            }
            bpl[k * BM + r] = lo;
            if (!CAUSAL) {
              const int hi = bin_hi(rr[q], ii);
              int k2 = t0 + q;
              while (k2 > 0) {
                const int prev = bph[(k2 - 1) * BM + r];
                if (prev <= hi) break;
                bph[k2 * BM + r] = prev;
                --k2;
              }
              bph[k2 * BM + r] = hi;
            }
          }
        }
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int jj = 0; jj < ntiles; ++jj, ++g) {
        const int st = g & 1;
        const uint32_t u = (uint32_t)g >> 1;
        const int jt = (it.kt_hi - 1 - jj) * BN;
        ok = __all_sync(FULL, mbar_wait(bar(B_SFULL + st), u & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();
        float x[BN];
        {
          uint32_t raw[32];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            tmem_ld32(tmem + lane_base + st * BN + q * 32, raw);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) x[q * 32 + e] = __uint_as_float(raw[e]);
          }
        }
        tc_fence_before();
        mbar_arrive(bar(B_SFREE + st));

        // pass 1: log2-domain weights x = S log2(e)/sqrt(d) + log2(c) (or the
        // ALiBi bias), -inf where the key does not take part; running max
        float mt = -INFINITY;
#pragma unroll
        for (int q = 3; q >= 0; --q) {
          const int jc = jt + q * 32;
          if (EXACT) {
            // bias -|i-j| slope with j = jc + e
            const float d0 = (float)(i - jc);
            const bool edge = CAUSAL ? (jc + 31 > i) : (jc + 31 >= n);
            if (CAUSAL) {
              const float base = -d0 * slope;
#pragma unroll
              for (int e = 0; e < 32; ++e)
                x[q * 32 + e] = fmaf(x[q * 32 + e], scale_log2, fmaf((float)e, slope, base));
              if (__any_sync(FULL, edge)) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (jc + e > i) x[q * 32 + e] = -INFINITY;
              }
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                x[q * 32 + e] = fmaf(x[q * 32 + e], scale_log2,
                                     -fabsf(d0 - (float)e) * slope);
              if (__any_sync(FULL, edge)) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (jc + e >= n) x[q * 32 + e] = -INFINITY;
              }
            }
          } else {
            while (pl > 0 && bpl[(pl - 1) * BM + r] > jc) --pl;
            while (ph > pl && bpl[(ph - 1) * BM + r] > jc + 31) --ph;
            int base = pl, nb = ph - pl;
            if (!CAUSAL) {
              while (ql > 0 && bph[(ql - 1) * BM + r] > jc) --ql;
              while (qh > ql && bph[(qh - 1) * BM + r] > jc + 31) --qh;
              base -= ql;
              nb += qh - ql;
            }
            const bool slow = nb > 0 || (CAUSAL && jc + 31 > i);
            if (__any_sync(FULL, slow)) {
              int c[32];
#pragma unroll
              for (int e = 0; e < 32; ++e) c[e] = base;
              for (int k = pl; k < ph; ++k) {
                const int bo = bpl[k * BM + r] - jc;
#pragma unroll
                for (int e = 0; e < 32; ++e) c[e] += (e >= bo) ? 1 : 0;
              }
              if (!CAUSAL) {
                for (int k = ql; k < qh; ++k) {
                  const int bo = bph[k * BM + r] - jc;
#pragma unroll
                  for (int e = 0; e < 32; ++e) c[e] -= (e >= bo) ? 1 : 0;
                }
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (jc + e > i) c[e] = 0;
              }
#pragma unroll
              for (int e = 0; e < 32; ++e)
                x[q * 32 + e] = c[e] > 0
                    ? fmaf(x[q * 32 + e], scale_log2, lg2((float)c[e]))
                    : -INFINITY;
            } else if (base > 0) {
              const float lc = lg2((float)base);
#pragma unroll
              for (int e = 0; e < 32; ++e)
                x[q * 32 + e] = fmaf(x[q * 32 + e], scale_log2, lc);
            } else {
#pragma unroll
              for (int e = 0; e < 32; ++e) x[q * 32 + e] = -INFINITY;
            }
          }
#pragma unroll
          for (int e = 0; e < 32; ++e) mt = fmaxf(mt, x[q * 32 + e]);
        }
        if (!row_ok) mt = -INFINITY;
        const float m_new = fmaxf(m_ref, mt);
        const bool resc = m_new > m_ref + kRescaleLog2;
        const float m_use = resc ? m_new : m_ref;
        const float alpha = resc ? ex2(m_ref - m_new) : 1.f;

        // the previous P V has finished: P's buffer and O may be touched
        if (g > 0) {
          ok = __all_sync(FULL, mbar_wait(bar(B_PVDONE), (uint32_t)(g - 1) & 1u, abort, lim));
          if (!ok) break;
        }
        tc_fence_after();
        if (jj > 0 && __any_sync(FULL, resc)) {
          const float f = resc ? alpha : 1.f;
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            const uint32_t ta = tmem + lane_base + kColO + q * 32;
            tmem_ld32(ta, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(ta, o);
          }
          tmem_wait_st();
        }

        // pass 2: P = 2^(x - m) in bf16, K-major 128B-swizzled rows
        const float mu = (m_use == -INFINITY || !row_ok) ? 0.f : m_use;
        float lsum = 0.f;
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint32_t pk[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2) {
            float p0 = ex2(x[q * 32 + 2 * e2] - mu);
            float p1 = ex2(x[q * 32 + 2 * e2 + 1] - mu);
            if (!row_ok) { p0 = 0.f; p1 = 0.f; }
            lsum += p0 + p1;
            pk[e2] = pack_bf16(p0, p1);
          }
          const uint32_t half_base = sbase + OFF_P + (q >> 1) * kHalfBytes + r * 128;
#pragma unroll
          for (int cc = 0; cc < 4; ++cc) {
            const int ch = (q & 1) * 4 + cc;
            st_shared_v4(half_base + ((uint32_t)(ch ^ (r & 7)) << 4), pk[4 * cc],
                         pk[4 * cc + 1], pk[4 * cc + 2], pk[4 * cc + 3]);
          }
        }
        l = l * alpha + lsum;
        m_ref = m_use;
        fence_proxy_async_smem();
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
#pragma unroll
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
  return 1024 + OFF_BP + bp_bytes(s, exact != 0, causal != 0) + sizeof(Ctl);
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
