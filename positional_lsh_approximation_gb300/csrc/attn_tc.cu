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
// bin ends hi_t(i) when not causal).  The row's thread holds those starts
// in registers (s <= 16; counted per 32-key chunk) or sorted in shared
// memory (walked by pointers); a chunk with no step takes log2(c) into the
// exponent's offset, a chunk with steps multiplies by the running count.
//
// Exact ALiBi (the dense comparator) runs on the same pipeline with weight
// e^{S_ij - |i-j|/sigma_h} over every key tile.
//
// One persistent CTA per SM, 12 warps, two 128-row query tiles A and B per
// work item (two heads of one KV group at the same rows, or two row tiles of
// one head), sharing every K/V tile:
//   warp 10     scheduler: pops items from a global queue (cost order),
//               stages the rows' bin records in shared memory, finds the key
//               envelope and publishes the item in a two-deep ring (one
//               item staged behind the one in progress);
//   warp 8      producer: TMA-loads the item's first K tile, then Q_A and
//               Q_B, then the other K/V tiles from the diagonal tile down
//               (a ring of three 32 KB slots);
//   warp 11     converter: turns each V tile from bf16 into f16 in place in
//               shared memory once it lands (exact within f16's range; a
//               value beyond it raises the range bit of the error flag);
//   warp 9      one thread issues tcgen05.mma in one stream across items,
//               PV_A(g-1) S_A(g) PV_B(g-1) S_B(g) ..., so that while one
//               warpgroup turns its scores into weights the tensor core works
//               for the other (tcgen05 MMAs of one thread execute in issue
//               order: the commit that follows S_X(g) also proves PV_X(g-1)
//               has landed);
//   warps 0-3   softmax of tile A, warps 4-7 softmax of tile B: one thread
//               per row, tcgen05.ld of the score row, running max over the
//               valid keys, lazy rescale of O in TMEM (only when the max grows
//               by more than 2^8), P = c 2^(x - m) rounded to f16 and
//               written back over score columns already consumed, fp32 row
//               sums, and the O / l epilogue (through shared memory into
//               whole-line stores).
//   O += P V runs on the tensor cores in f16 with A read from TMEM: f16 keeps
//   11 significant bits of each weight (bf16 only 8, whose 2^-9 relative
//   error per weight shows in rows whose few keys cancel), and every bf16
//   value of V within f16's range is an f16 value.
// TMEM columns: S_A | S_B | O_A | O_B.  Every wait on an mbarrier is bounded;
// on expiry the CTA raises the library error flag, drains its in-flight copies
// and MMAs, frees TMEM and exits.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
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
constexpr int kWarps = 12;
constexpr int kThreads = kWarps * 32;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kSchedWarp = 10;
constexpr int kConvWarp = 11;
constexpr int kRing = 2;                         // work items in flight
constexpr int kSlots = 3;                        // K/V tile ring depth
constexpr int kMaxSlots = 4;                     // barriers reserved for the ring
constexpr uint32_t kTileBytes = BM * HD * 2;     // 32 KB bf16 tile
constexpr uint32_t kHalfBytes = kTileBytes / 2;  // one 64-column TMA box
constexpr uint32_t OFF_Q = 0;                          // Q_A, Q_B
constexpr uint32_t OFF_KV = OFF_Q + 2 * kTileBytes;    // ring of `slots` tiles
constexpr uint32_t kTmemCols = 512;   // S_A | S_B | O_A | O_B; P over S
constexpr uint32_t kColP = 64;        // P (f16 pairs) in the upper half of S
constexpr uint32_t kColO = 256;
constexpr float kRescaleLog2 = 8.0f;  // lazy rescale threshold (factor 256)
constexpr float kGrowLog2 = 15.0f;    // largest weight 2^15 before a mid-tile rescale (f16 P)
constexpr unsigned FULL = 0xffffffffu;
constexpr int kWordsPerTile = BM / 32;
constexpr uint32_t kOutBytes = 8 * 32 * 64 * 2;   // O transpose: 32 rows x 64 bf16 per warp

enum {
  B_QFULL = 0, B_QFULL1, B_QEMPTY, B_QEMPTY1, B_KVFULL, B_KVFULL_END = B_KVFULL + kMaxSlots,
  B_KVEMPTY = B_KVFULL_END, B_KVEMPTY_END = B_KVEMPTY + kMaxSlots,
  B_SFULL = B_KVEMPTY_END, B_SFULL1, B_PFULL, B_PFULL1, B_ODONE, B_ODONE1,
  B_IFULL, B_IFULL_END = B_IFULL + kRing, B_IEMPTY = B_IFULL_END,
  B_IEMPTY_END = B_IEMPTY + kRing, B_DRAIN = B_IEMPTY_END,
  B_VREADY, B_VREADY_END = B_VREADY + kMaxSlots, NUM_BARS
};

// Error flag bits: 1 a wait ran out, 2 a value of V lies beyond f16's range.
constexpr int kErrTimeout = 1;
constexpr int kErrRange = 2;

struct Item {
  int valid, b, hA, hB, qtA, qtB, kt_lo, kt_hi;
  int ws;                    // workspace slot of a split part, -1 for a whole item
};

struct Ctl {
  uint64_t bars[NUM_BARS];
  Item ring[kRing];
  uint32_t tmem_base;
  int abort;
};

struct TcParams {
  AttnArgs a;
  float slope_log2[512];   // exact mode: log2(e) / sigma_h
  int QT;                  // query tiles per (b, h)
  int out_smem;            // 1: the epilogue transposes O through shared memory
};

// Sorted bin starts (and ends when not causal) of every row of both tiles:
// [tile][lists][s][BM] int32.
__host__ __device__ constexpr uint32_t bp_bytes(int s, bool exact, bool causal, int sreg) {
  return (exact || sreg > 0) ? 0u : 2u * (uint32_t)(causal ? 1 : 2) * (uint32_t)s * BM * 4u;
}
// Bin records of both tiles' rows, per item slot: [kRing][2 tiles][s][4] x 16 B.
__host__ __device__ constexpr uint32_t stage_bytes(int s, bool exact) {
  return exact ? 0u : 2u * kRing * (uint32_t)s * kWordsPerTile * 16u;
}

__device__ __forceinline__ Item read_item(const Ctl* ctl, int slot) {
  const volatile int* v = reinterpret_cast<const volatile int*>(&ctl->ring[slot]);
  Item it;
  it.valid = v[0]; it.b = v[1]; it.hA = v[2]; it.hB = v[3];
  it.qtA = v[4]; it.qtB = v[5]; it.kt_lo = v[6]; it.kt_hi = v[7];
  it.ws = v[8];
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

// Bit e set when key jc + e of a row whose keys are [jc + ea, jc + eb] takes
// part.
__device__ __forceinline__ uint32_t key_mask(int ea, int eb, bool row_ok) {
  if (!row_ok || ea > 31 || eb < 0 || ea > eb) return 0u;
  const uint32_t up = eb >= 31 ? 0xffffffffu : ((2u << eb) - 1u);
  const uint32_t dn = ea <= 0 ? 0xffffffffu : ~((1u << ea) - 1u);
  return up & dn;
}

// Adds one step at the positions of `m` to a five-plane binary counter.
__device__ __forceinline__ void plane_add(uint32_t (&pl)[5], uint32_t m) {
#pragma unroll
  for (int b = 0; b < 5; ++b) {
    const uint32_t c = pl[b] & m;
    pl[b] ^= m;
    m = c;
  }
}

// Multiplies the chunk's weights by the running count c(e): base plus the
// binary planes of step multiplicities at each key (up) minus those of bin
// ends (dn, non-causal only), L planes in use; four independent runs of
// eight keys.
template <int L, bool CAUSAL>
__device__ __forceinline__ void scale_by_planes(float (&pv)[32], int base,
                                                const uint32_t (&up)[5],
                                                const uint32_t (&dn)[5]) {
  float c[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t below = (1u << (8 * g)) - 1u;
    int cb = base;
#pragma unroll
    for (int b = 0; b < L; ++b) {
      cb += __popc(up[b] & below) << b;
      if (!CAUSAL) cb -= __popc(dn[b] & below) << b;
    }
    c[g] = (float)cb;
  }
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int e = 8 * g + k;
      float ce = 0.f;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int b = 0; b < L; ++b) {
          if (up[b] & (1u << (e + h))) c[g] += (float)(1 << b);
          if (!CAUSAL && (dn[b] & (1u << (e + h)))) c[g] -= (float)(1 << b);
        }
        if (h == 0) ce = c[g];
      }
      const uint64_t p2 = f2_mul(f2_pack(pv[e], pv[e + 1]), f2_pack(ce, c[g]));
      f2_unpack(p2, pv[e], pv[e + 1]);
    }
  }
}

// The same for chunks where no two starts (or ends) share a key: one bit
// per step, counted in four independent runs of eight keys.
template <bool CAUSAL>
__device__ __forceinline__ void scale_by_steps(float (&pv)[32], int base,
                                               uint32_t up, uint32_t dn) {
  float c[4];
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    const uint32_t below = (1u << (8 * g)) - 1u;
    int cb = base + __popc(up & below);
    if (!CAUSAL) cb -= __popc(dn & below);
    c[g] = (float)cb;
  }
#pragma unroll
  for (int k = 0; k < 8; k += 2) {
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      const int e = 8 * g + k;
      if (up & (1u << e)) c[g] += 1.f;
      if (!CAUSAL && (dn & (1u << e))) c[g] -= 1.f;
      const float ce = c[g];
      if (up & (2u << e)) c[g] += 1.f;
      if (!CAUSAL && (dn & (2u << e))) c[g] -= 1.f;
      const uint64_t p2 = f2_mul(f2_pack(pv[e], pv[e + 1]), f2_pack(ce, c[g]));
      f2_unpack(p2, pv[e], pv[e + 1]);
    }
  }
}

// SREG > 0: each row keeps its s <= SREG bin starts (and ends) in registers,
// unsorted, and counts them per chunk; SREG == 0: sorted lists in shared
// memory walked by pointers (any s).
template <bool EXACT, bool CAUSAL, int SREG>
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
  constexpr uint32_t nslots = kSlots;
  const uint32_t off_out = OFF_KV + nslots * kTileBytes;   // 8 warps x 4 KB
  const uint32_t off_bp = off_out + (p.out_smem ? kOutBytes : 0u);
  int* bp = reinterpret_cast<int*>(smem + off_bp);
  uint4* stage = reinterpret_cast<uint4*>(smem + off_bp + bp_bytes(s, EXACT, CAUSAL, SREG));
  Ctl* ctl = reinterpret_cast<Ctl*>(smem + off_bp + bp_bytes(s, EXACT, CAUSAL, SREG) +
                                    stage_bytes(s, EXACT));
  auto bar = [&](int k) { return smem_u32(&ctl->bars[k]); };
  volatile int* abort = &ctl->abort;
  const uint64_t lim = a.wait_ns;

  if (threadIdx.x == 0) {
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_QFULL + k), 1);
      mbar_init(bar(B_QEMPTY + k), 1);
    }
    for (int k = 0; k < kMaxSlots; ++k) {
      mbar_init(bar(B_KVFULL + k), 1);
      mbar_init(bar(B_KVEMPTY + k), 1);
      mbar_init(bar(B_VREADY + k), 1);
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar(B_SFULL + k), 1);
      mbar_init(bar(B_PFULL + k), BM);
      mbar_init(bar(B_ODONE + k), 1);
    }
    for (int k = 0; k < kRing; ++k) {
      mbar_init(bar(B_IFULL + k), 1);
      // released by the producer, the converter, the MMA thread and every
      // softmax thread
      mbar_init(bar(B_IEMPTY + k), 3 + 2 * BM);
    }
    mbar_init(bar(B_DRAIN), 1);
    ctl->abort = 0;
    fence_barrier_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(&ctl->tmem_base), kTmemCols);
    tmem_relinquish();
  }
  if (warp == kProducerWarp && lane == 0) {
    prefetch_tensormap(&tmQ);
    prefetch_tensormap(&tmK);
    prefetch_tensormap(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // launched as a programmatic dependent of the kernel before it (the
  // sampler): the set-up above overlaps its tail; nothing in global memory
  // is read or written before that kernel has completed
  grid_dep_wait();
  const uint32_t tmem = ctl->tmem_base;
  const int n = a.n, Hq = a.Hq, Hkv = a.Hkv;

  if (warp == kSchedWarp) {
    // ----------------------------------------------------------- scheduler
    // pops items, stages the rows' bin records, finds the key envelope and
    // publishes the item up to kRing - 1 items ahead of its consumers: one
    // item waits behind the one in progress (the least the MMA thread
    // allows: it sees the next item published before it issues an item's
    // last P V).  A deeper lookahead (two items) left the last CTA up to two
    // items behind the rest when the queue ran dry and was no faster before
    bool ok = true;
    for (int seq = 0; !a.stall; ++seq) {   // stall: fault injection
      const int slot = seq % kRing;
      const uint32_t use = (uint32_t)(seq / kRing);
      if (lane == 0) ok = mbar_wait(bar(B_IEMPTY + slot), (use & 1u) ^ 1u, abort, lim);
      ok = __shfl_sync(FULL, (int)ok, 0) != 0;
      if (!ok) break;
      // pop until an item with work (a split item's part past its key
      // envelope only marks its rows empty) or the end of the queue
      bool published = false, drained = false;
      while (!published) {
      int idx = 0;
      if (lane == 0) idx = atomicAdd(a.queue, 1);
      idx = __shfl_sync(FULL, idx, 0);
      if (idx >= a.num_items) {
        if (lane == 0) {
          ctl->ring[slot].valid = 0;
          mbar_arrive(bar(B_IFULL + slot));
        }
        drained = true;
        break;
      }
      const int4 e4 = __ldg(a.items + idx);
      const int b = e4.x, hA = e4.y & 0xffff, hB = (e4.y >> 16) & 0xffff;
      const int qtA = e4.z, qtB = e4.w;          // qtB < 0: tile B unused
      const int qmax = max(qtA, qtB);
      int kt_lo, kt_hi;
      if (EXACT) {
        kt_lo = 0;
        kt_hi = CAUSAL ? qmax + 1 : (n + BN - 1) / BN;
      } else {
        // records of both tiles' rows (4 words per hash); lo_t(i) is
        // non-decreasing in i, so a tile's first row bounds the envelope from
        // the left (its last row from the right)
        int mylo = INT_MAX, myhi = 0;
        const int per = s * kWordsPerTile;
        uint4 rv[4];
        int ecount = 0;
#pragma unroll 1
        for (int e0 = 0; e0 < 2 * per; e0 += 4 * 32) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * 32 + lane;
            if (e < 2 * per) {
              const int tile = e / per, el = e % per;
              const int qt = tile ? qtB : qtA;
              const int h = tile ? hB : hA;
              const int t = el / kWordsPerTile, wq = el % kWordsPerTile;
              const int wd = min((max(qt, 0) * BM >> 5) + wq, (int)a.W - 1);
              rv[u] = __ldg(reinterpret_cast<const uint4*>(a.rec) +
                            ((int64_t)h * s + t) * a.W + wd);
            }
          }
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            const int e = e0 + u * 32 + lane;
            if (e < 2 * per) {
              const int tile = e / per, el = e % per;
              const int qt = tile ? qtB : qtA;
              stage[(slot * 2 + tile) * per + el] = rv[u];
              if (qt < 0) continue;
              const int i0 = qt * BM;
              const int ilast = min(i0 + BM - 1, n - 1);
              const int wq = el % kWordsPerTile;
              const BinRecord rc = unpack_record(rv[u]);
              if (wq == 0) mylo = min(mylo, bin_lo(rc, i0));
              if (!CAUSAL && min((i0 >> 5) + wq, (int)a.W - 1) == (ilast >> 5))
                myhi = max(myhi, bin_hi(rc, ilast));
            }
          }
          ecount += 4 * 32;
        }
        mylo = __reduce_min_sync(FULL, mylo);
        kt_lo = mylo / BN;
        if (CAUSAL) {
          kt_hi = qmax + 1;
        } else {
          myhi = __reduce_max_sync(FULL, myhi);
          kt_hi = (myhi + BN - 1) / BN;
        }
        __syncwarp();
      }
      kt_lo = min(kt_lo, qmax);
      kt_hi = max(kt_hi, kt_lo + 1);
      int ws = -1;
      if (a.item_ext != nullptr) {
        // part x.x of x.y over the key tiles of the envelope
        const int4 x = __ldg(a.item_ext + idx);
        if (x.y > 1) {
          const int len = kt_hi - kt_lo;
          const int lo_p = kt_lo + (len * x.x) / x.y;
          const int hi_p = kt_lo + (len * (x.x + 1)) / x.y;
          ws = x.z;
          if (hi_p <= lo_p) {
            // no key tile: every row of the part has no weight
            float* wm = a.split_ws + (size_t)ws * kSplitSlotFloats + 2 * BM * kSplitRowFloats;
            for (int k = lane; k < 2 * BM; k += 32) {
              wm[k] = -INFINITY;        // max
              wm[2 * BM + k] = 0.f;     // row sum
            }
            __syncwarp();
            continue;
          }
          kt_lo = lo_p;
          kt_hi = hi_p;
        }
      }
      if (lane == 0) {
        volatile int* it = reinterpret_cast<volatile int*>(&ctl->ring[slot]);
        it[0] = 1; it[1] = b; it[2] = hA; it[3] = hB; it[4] = qtA; it[5] = qtB;
        it[6] = kt_lo; it[7] = kt_hi; it[8] = ws;
        mbar_arrive(bar(B_IFULL + slot));
      }
      __syncwarp();
      published = true;
      }
      if (drained) break;
    }
    if (!ok && lane == 0) {
      *abort = 1;
      atomicOr(a.err, kErrTimeout);
    }
    __syncwarp();
  } else if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      int ld = 0;                       // K/V loads issued (K and V alternate)
      int q_issued = 0;
      int kv_issued[kMaxSlots] = {0, 0, 0, 0};
      bool ok = true;
      for (int seq = 0; ok; ++seq) {
        const int slot = seq % kRing;
        const uint32_t use = (uint32_t)(seq / kRing);
        ok = mbar_wait(bar(B_IFULL + slot), use & 1u, abort, lim);
        if (!ok) break;
        const Item it = read_item(ctl, slot);
        if (!it.valid) break;
        // the item's first K tile goes first: it does not wait for the Q
        // buffers, which free only when the item before has issued its last S
        const int kvp = it.b * Hkv + it.hA / (Hq / Hkv);
        for (int kt = it.kt_hi - 1; ok && kt >= it.kt_lo; --kt) {
          for (int kv = 0; kv < 2 && ok; ++kv, ++ld) {
            const uint32_t sl = (uint32_t)ld % nslots;
            const uint32_t u = (uint32_t)ld / nslots;
            ok = mbar_wait(bar(B_KVEMPTY + sl), (u & 1u) ^ 1u, abort, lim);
            if (!ok) break;
            const uint32_t dst = sbase + OFF_KV + sl * kTileBytes;
            const CUtensorMap* m = kv ? &tmV : &tmK;
            mbar_arrive_expect_tx(bar(B_KVFULL + sl), kTileBytes);
            tma_load_3d(dst, m, bar(B_KVFULL + sl), 0, kt * BN, kvp);
            tma_load_3d(dst + kHalfBytes, m, bar(B_KVFULL + sl), 64, kt * BN, kvp);
            ++kv_issued[sl];
            if (kt == it.kt_hi - 1 && kv == 0) {
              for (int tile = 0; tile < 2 && ok; ++tile) {
                ok = mbar_wait(bar(B_QEMPTY + tile), ((uint32_t)seq & 1u) ^ 1u, abort, lim);
                if (!ok) break;
                // an unused tile B reloads A's rows so its scores stay finite
                const int qt = (tile && it.qtB >= 0) ? it.qtB : it.qtA;
                const int h = (tile && it.qtB >= 0) ? it.hB : it.hA;
                const uint32_t qdst = sbase + OFF_Q + tile * kTileBytes;
                mbar_arrive_expect_tx(bar(B_QFULL + tile), kTileBytes);
                tma_load_3d(qdst, &tmQ, bar(B_QFULL + tile), 0, qt * BM, it.b * Hq + h);
                tma_load_3d(qdst + kHalfBytes, &tmQ, bar(B_QFULL + tile), 64, qt * BM,
                            it.b * Hq + h);
              }
              if (ok) ++q_issued;
            }
          }
        }
        if (ok) mbar_arrive(bar(B_IEMPTY + slot));
      }
      if (!ok) {
        *abort = 1;
        atomicOr(a.err, kErrTimeout);
      }
      // let every copy this warp started land before the CTA can exit
      if (q_issued) {
        mbar_wait(bar(B_QFULL + 0), (uint32_t)(q_issued - 1) & 1u, nullptr, lim);
        mbar_wait(bar(B_QFULL + 1), (uint32_t)(q_issued - 1) & 1u, nullptr, lim);
      }
      for (uint32_t sl = 0; sl < nslots; ++sl)
        if (kv_issued[sl])
          mbar_wait(bar(B_KVFULL + sl), (uint32_t)(kv_issued[sl] - 1) & 1u, nullptr, lim);
    }
    __syncwarp();
  } else if (warp == kConvWarp) {
    // ----------------------------------------------------------- converter
    // follows the producer's load order (per item, tiles from the diagonal
    // down, K then V) and turns every V tile into f16 in place: the element
    // positions of the swizzled layout do not depend on the element type
    bool ok = true;
    int ld = 0;
    float vmax = 0.f;                   // largest |v| seen, as f32
    for (int seq = 0; ok; ++seq) {
      const int slot = seq % kRing;
      const uint32_t use = (uint32_t)(seq / kRing);
      ok = __all_sync(FULL, mbar_wait(bar(B_IFULL + slot), use & 1u, abort, lim));
      if (!ok) break;
      const Item it = read_item(ctl, slot);
      if (!it.valid) break;
      for (int kt = it.kt_hi - 1; kt >= it.kt_lo; --kt, ld += 2) {
        const int lv = ld + 1;
        const uint32_t sl = (uint32_t)lv % nslots;
        ok = __all_sync(FULL, mbar_wait(bar(B_KVFULL + sl), ((uint32_t)lv / nslots) & 1u, abort,
                                        lim));
        if (!ok) break;
        const uint32_t vb = sbase + OFF_KV + sl * kTileBytes + (uint32_t)lane * 16u;
#pragma unroll 4
        for (uint32_t c = 0; c < kTileBytes / 16u; c += 32) {
          const uint4 v = ld_shared_v4(vb + c * 16u);
          const float a0 = __uint_as_float(v.x << 16), a1 = __uint_as_float(v.x & 0xffff0000u);
          const float b0 = __uint_as_float(v.y << 16), b1 = __uint_as_float(v.y & 0xffff0000u);
          const float c0 = __uint_as_float(v.z << 16), c1 = __uint_as_float(v.z & 0xffff0000u);
          const float d0 = __uint_as_float(v.w << 16), d1 = __uint_as_float(v.w & 0xffff0000u);
          vmax = max3(vmax, fabsf(a0), fabsf(a1));
          vmax = max3(vmax, fabsf(b0), fabsf(b1));
          vmax = max3(vmax, fabsf(c0), fabsf(c1));
          vmax = max3(vmax, fabsf(d0), fabsf(d1));
          st_shared_v4(vb + c * 16u, pack_f16(a0, a1), pack_f16(b0, b1), pack_f16(c0, c1),
                       pack_f16(d0, d1));
        }
        // the tensor core reads the tile through the async proxy
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_VREADY + sl));
      }
      if (!ok) break;
      if (lane == 0) mbar_arrive(bar(B_IEMPTY + slot));
      __syncwarp();
    }
    // 65520 and above round to infinity in f16 (NaN inputs stay NaN)
    const bool range = __any_sync(FULL, vmax >= 65520.f);
    if (lane == 0) {
      if (!ok) {
        *abort = 1;
        atomicOr(a.err, kErrTimeout);
      }
      if (range) atomicOr(a.err, kErrRange);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issue
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_bf16_f32(BM, BN, 0, 0);
      constexpr uint32_t idesc_pv = idesc_f16_f32(BM, HD, 0, 1);
      bool ok = true;
      int ld = 0;        // K/V loads consumed so far (same numbering as producer)
      int gt = 0;        // tiles processed so far (both tiles advance together)
      auto wait_slot = [&](int l) -> bool {
        return mbar_wait(bar(B_KVFULL + (uint32_t)l % nslots), ((uint32_t)l / nslots) & 1u, abort,
                        lim);
      };
      // V load l (odd) sits in slot l % 3; that slot holds V on every other
      // use, so this is its (l / 6)-th V: the converter's phase
      static_assert(kSlots == 3, "V phases assume a ring of three slots");
      auto wait_v = [&](int l) -> bool {
        return mbar_wait(bar(B_VREADY + (uint32_t)l % nslots), ((uint32_t)l / 6u) & 1u, abort,
                        lim);
      };
      // descriptors of the tiles' first 16-column slices; a slice further
      // on adds its byte offset / 16 to the start-address field
      const uint64_t dq0 = desc_sw128(sbase + OFF_Q, 16, 1024);
      const uint64_t dk0 = desc_sw128(sbase + OFF_KV, 16, 1024);
      const uint64_t dv0 = desc_sw128(sbase + OFF_KV, kHalfBytes, 1024);
      auto issue_s = [&](int tile, int lk) {
        const uint64_t qd = desc_add(dq0, tile * (kTileBytes >> 4));
        const uint64_t kd = desc_add(dk0, ((uint32_t)lk % nslots) * (kTileBytes >> 4));
#pragma unroll
        for (int kk = 0; kk < HD / 16; ++kk) {
          const uint32_t koff = ((kk >> 2) * kHalfBytes + (kk & 3) * 32) >> 4;
          mma_bf16_ss(tmem + tile * BN, desc_add(qd, koff), desc_add(kd, koff), idesc_qk,
                      kk > 0 ? 1u : 0u);
        }
        mma_commit(bar(B_SFULL + tile));
      };
      auto issue_pv = [&](int tile, int lv, bool first) {
        const uint64_t vd = desc_add(dv0, ((uint32_t)lv % nslots) * (kTileBytes >> 4));
        // keys 16kk..16kk+15: 8 columns of f16 pairs at 8 kk past the
        // tile's P base
        const uint32_t pcol = tmem + tile * BN + kColP;
        const uint32_t ocol = tmem + kColO + tile * HD;
#pragma unroll
        for (int kk = 0; kk < BN / 16; ++kk) {
          const uint64_t bd = desc_add(vd, kk * (2048 >> 4));
          mma_f16kind_ts(ocol, pcol + kk * 8, bd, idesc_pv, (first && kk == 0) ? 0u : 1u);
        }
      };
      // one continuous stream of tiles across items: the head of an item
      // (its first S_A, S_B) is issued between the tail P Vs of the item
      // before, so that Q loads and epilogues overlap tensor work
      int seq = 0;
      ok = mbar_wait(bar(B_IFULL + 0), 0u, abort, lim);
      Item cur = ok ? read_item(ctl, 0) : Item{0, 0, 0, 0, 0, 0, 0, 0, -1};
      int T = cur.kt_hi - cur.kt_lo, jj = 0;
      bool have_prev = false;
      int prev_lv = 0, prev_slot = 0;
      bool prev_first = false, prev_last = false;
      while (ok && cur.valid) {
        const int lk = ld;                      // K of this tile; V is ld + 1
        if (have_prev) {
          ok = mbar_wait(bar(B_PFULL + 0), (uint32_t)(gt - 1) & 1u, abort, lim) &&
               wait_v(prev_lv);
          if (!ok) break;
          tc_fence_after();
          issue_pv(0, prev_lv, prev_first);
          if (prev_last) mma_commit(bar(B_ODONE + 0));
        }
        ok = wait_slot(lk);
        if (!ok) break;
        if (jj == 0) {
          ok = mbar_wait(bar(B_QFULL + 0), (uint32_t)seq & 1u, abort, lim);
          if (!ok) break;
        }
        tc_fence_after();
        issue_s(0, lk);
        if (jj == T - 1) mma_commit(bar(B_QEMPTY + 0));
        if (have_prev) {
          ok = mbar_wait(bar(B_PFULL + 1), (uint32_t)(gt - 1) & 1u, abort, lim);
          if (!ok) break;
          tc_fence_after();
          issue_pv(1, prev_lv, prev_first);
          mma_commit(bar(B_KVEMPTY + (uint32_t)prev_lv % nslots));
          if (prev_last) {
            mma_commit(bar(B_ODONE + 1));
            mbar_arrive(bar(B_IEMPTY + prev_slot));
          }
        }
        if (jj == 0) {
          ok = mbar_wait(bar(B_QFULL + 1), (uint32_t)seq & 1u, abort, lim);
          if (!ok) break;
        }
        tc_fence_after();
        issue_s(1, lk);
        mma_commit(bar(B_KVEMPTY + (uint32_t)lk % nslots));
        if (jj == T - 1) mma_commit(bar(B_QEMPTY + 1));
        have_prev = true;
        prev_lv = lk + 1;
        prev_first = jj == 0;
        prev_last = jj == T - 1;
        prev_slot = seq % kRing;
        ld += 2;
        ++gt;
        if (++jj == T) {
          ++seq;
          ok = mbar_wait(bar(B_IFULL + seq % kRing), (uint32_t)(seq / kRing) & 1u, abort, lim);
          if (!ok) break;
          cur = read_item(ctl, seq % kRing);
          T = cur.kt_hi - cur.kt_lo;
          jj = 0;
        }
      }
      if (ok && have_prev) {
        // tail of the last tile
        ok = mbar_wait(bar(B_PFULL + 0), (uint32_t)(gt - 1) & 1u, abort, lim) &&
             wait_v(prev_lv);
        if (ok) {
          tc_fence_after();
          issue_pv(0, prev_lv, prev_first);
          mma_commit(bar(B_ODONE + 0));
          ok = mbar_wait(bar(B_PFULL + 1), (uint32_t)(gt - 1) & 1u, abort, lim);
        }
        if (ok) {
          tc_fence_after();
          issue_pv(1, prev_lv, prev_first);
          mma_commit(bar(B_KVEMPTY + (uint32_t)prev_lv % nslots));
          mma_commit(bar(B_ODONE + 1));
          mbar_arrive(bar(B_IEMPTY + prev_slot));
        }
      }
      if (!ok) {
        *abort = 1;
        atomicOr(a.err, kErrTimeout);
      }
      // every MMA issued by this thread has completed once this arrives
      mma_commit(bar(B_DRAIN));
      mbar_wait(bar(B_DRAIN), 0, nullptr, lim);
    }
    __syncwarp();
  } else {
    // ----------------------------------------------------- softmax / epilogue
    const int tile = warp >> 2;                 // 0: tile A, 1: tile B
    const int r = threadIdx.x & (BM - 1);       // row within the tile == TMEM lane
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t s_col = tmem + lane_base + tile * BN;
    const uint32_t o_col = tmem + lane_base + kColO + tile * HD;
    // log2(e) / sqrt(d); d = 64 runs zero-padded to 128 columns
    const float scale_log2 = 1.4426950408889634f * (a.d == 64 ? 0.125f : 0.08838834764831845f);
    const uint64_t scale2 = f2_pack(scale_log2, scale_log2);
    const int nlists = CAUSAL ? 1 : 2;
    int* bpl = bp + tile * nlists * s * BM;      // sorted bin starts, [s][BM]
    int* bph = bpl + s * BM;                     // sorted bin ends (non-causal)
    bool ok = true;
    int g = 0;
    // with bin lists in shared memory the output of an item is written once
    // the next item is set up (the sort hides the item's last P V); with
    // starts in registers the set-up is short and the output goes first
    constexpr bool kDefer = SREG == 0;
    bool pend = false;
    float pend_l = 0.f, pend_m = 0.f;
    const uint32_t obuf = sbase + off_out + (uint32_t)warp * 4096u;
    // epilogue of item pseq: O_i = acc_i / l_i, then its item slot is released
    auto finish = [&](int pseq) -> bool {
      if (!__all_sync(FULL, mbar_wait(bar(B_ODONE + tile), (uint32_t)pseq & 1u, abort, lim)))
        return false;
      tc_fence_after();
      // the item stays in its ring slot until this thread releases it
      const int pslot = pseq % kRing;
      const Item pit = read_item(ctl, pslot);
      const int qt = tile ? pit.qtB : pit.qtA;
      const int h = tile ? pit.hB : pit.hA;
      const int i = max(qt, 0) * BM + r;
      const int64_t row0 = ((int64_t)pit.b * Hq + h) * n;
      if (pit.ws >= 0) {
        // a part of a split item: its unnormalised P V, max and row sum go
        // to its workspace slot, to be combined with the other parts
        float* w = a.split_ws + (size_t)pit.ws * kSplitSlotFloats;
        float4* acc = reinterpret_cast<float4*>(w + ((size_t)tile * BM + r) * kSplitRowFloats);
#pragma unroll 1
        for (int q2 = 0; q2 < 4; ++q2) {
          uint32_t o[32];
          tmem_ld32(o_col + q2 * 32, o);
          tmem_wait_ld();
#pragma unroll
          for (int v = 0; v < 8; ++v)
            acc[q2 * 8 + v] = make_float4(__uint_as_float(o[4 * v]), __uint_as_float(o[4 * v + 1]),
                                          __uint_as_float(o[4 * v + 2]),
                                          __uint_as_float(o[4 * v + 3]));
        }
        w[2 * BM * kSplitRowFloats + tile * BM + r] = pend_m;
        w[2 * BM * kSplitRowFloats + 2 * BM + tile * BM + r] = pend_l;
        tc_fence_before();
        mbar_arrive(bar(B_IEMPTY + pslot));
        pend = false;
        return true;
      }
      const float inv_l = pend_l > 0.f ? 1.f / pend_l : 0.f;
      if (a.stats != nullptr) {
        // m, l and Delta = sum_d (acc_d / l) dO_d for the backward pass (the
        // TMEM loads are warp-wide: every lane takes part, valid rows or not)
        const bool valid = qt >= 0 && i < n;
        const uint4* dorow = reinterpret_cast<const uint4*>(
            static_cast<const uint16_t*>(a.dO) + (row0 + (valid ? i : 0)) * HD);
        float dsum = 0.f;
#pragma unroll 1
        for (int q2 = 0; q2 < 4; ++q2) {
          uint32_t o[32];
          tmem_ld32(o_col + q2 * 32, o);
          tmem_wait_ld();
          if (valid) {
#pragma unroll
            for (int v = 0; v < 4; ++v) {
              const uint4 g = dorow[q2 * 4 + v];
              const uint32_t gw[4] = {g.x, g.y, g.z, g.w};
#pragma unroll
              for (int k = 0; k < 4; ++k) {
                dsum = fmaf(__uint_as_float(o[8 * v + 2 * k]), __uint_as_float(gw[k] << 16), dsum);
                dsum = fmaf(__uint_as_float(o[8 * v + 2 * k + 1]),
                            __uint_as_float(gw[k] & 0xffff0000u), dsum);
              }
            }
          }
        }
        if (valid) {
          float* st2 = a.stats + (row0 + i) * 2;
          st2[0] = pend_l > 0.f ? -(pend_m + lg2(pend_l)) : -INFINITY;
          st2[1] = dsum * inv_l;
        }
        if (a.O == nullptr) {
          tc_fence_before();
          mbar_arrive(bar(B_IEMPTY + pslot));
          pend = false;
          return true;
        }
      } else if (a.lse != nullptr && qt >= 0 && i < n) {
        a.lse[row0 + i] = pend_l > 0.f ? pend_m + lg2(pend_l) : -INFINITY;
      }
#pragma unroll 1
      for (int q2 = 0; q2 < a.d / 64; ++q2) {          // d = 64: the padding's half is not stored
        uint32_t o0[32], o1[32];
        tmem_ld32(o_col + q2 * 64, o0);
        tmem_ld32(o_col + q2 * 64 + 32, o1);
        tmem_wait_ld();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          const uint32_t* o = half ? o1 : o0;
          uint32_t pk[16];
#pragma unroll
          for (int e2 = 0; e2 < 16; ++e2)
            pk[e2] = pack_bf16(__uint_as_float(o[2 * e2]) * inv_l,
                               __uint_as_float(o[2 * e2 + 1]) * inv_l);
          if (p.out_smem) {
            // row-major 32 rows x 128 bytes, 16-byte chunks swizzled by row
#pragma unroll
            for (int v = 0; v < 4; ++v)
              st_shared_v4(obuf + lane * 128 + (((half * 4 + v) ^ (lane & 7)) << 4),
                           pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          } else if (qt >= 0 && i < n) {
            uint4* orow = reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.O) +
                                                   (row0 + i) * a.d + q2 * 64);
#pragma unroll
            for (int v = 0; v < 4; ++v)
              orow[half * 4 + v] = make_uint4(pk[4 * v], pk[4 * v + 1], pk[4 * v + 2], pk[4 * v + 3]);
          }
        }
        if (p.out_smem) {
          // read back transposed: eight lanes write one row's 128 bytes, so
          // every store instruction fills four whole lines
          __syncwarp();
          const int c = lane & 7;
#pragma unroll
          for (int k = 0; k < 8; ++k) {
            const int rr = 4 * k + (lane >> 3);
            const uint4 v = ld_shared_v4(obuf + rr * 128 + ((c ^ (rr & 7)) << 4));
            const int ir = max(qt, 0) * BM + (warp & 3) * 32 + rr;
            if (qt >= 0 && ir < n)
              reinterpret_cast<uint4*>(static_cast<uint16_t*>(a.O) + (row0 + ir) * a.d +
                                       q2 * 64)[c] = v;
          }
          __syncwarp();
        }
      }
      tc_fence_before();
      mbar_arrive(bar(B_IEMPTY + pslot));
      pend = false;
      return true;
    };
    for (int seq = 0; ok; ++seq) {
      const int slot = seq % kRing;
      const uint32_t use = (uint32_t)(seq / kRing);
      ok = __all_sync(FULL, mbar_wait(bar(B_IFULL + slot), use & 1u, abort, lim));
      if (!ok) break;
      const Item it = read_item(ctl, slot);
      if (!it.valid) {
        if (pend) ok = finish(seq - 1);
        break;
      }
      const int qt = tile ? it.qtB : it.qtA;
      const int h = tile ? it.hB : it.hA;
      const int i0 = max(qt, 0) * BM;
      const int i = i0 + r;
      const bool row_ok = qt >= 0 && i < n;
      const int ii = min(i, n - 1);
      const int ntiles = it.kt_hi - it.kt_lo;
      // keys that take part: [vlo, vhi]
      int vlo = 0, vhi = CAUSAL ? ii : n - 1;
      int pl = s, ph = s, ql = s, qh = s;
      float slope = 0.f;
      int lo_r[SREG > 0 ? SREG : 1], hi_r[SREG > 0 ? SREG : 1];
      int lomax = 0, himin = 0;
      if (EXACT) {
        slope = p.slope_log2[h];
      } else if (SREG > 0) {
        // this row's bin starts (and ends) under every hash, in registers
        const uint4* rs = stage + (slot * 2 + tile) * s * kWordsPerTile + ((ii >> 5) - (i0 >> 5));
        int lomin = INT_MAX, himax = 0;
        lomax = INT_MIN;
        himin = INT_MAX;
        // every record is loaded first (a clamped index, so that no load
        // waits behind a branch), then the bins are found
        uint4 rec_r[SREG > 0 ? SREG : 1];
        const uint32_t rs_addr = smem_u32(rs);
#pragma unroll
        for (int t = 0; t < (SREG > 0 ? SREG : 1); ++t)
          rec_r[t] = ld_shared_v4(rs_addr + (uint32_t)min(t, s - 1) * (kWordsPerTile * 16u));
#pragma unroll
        for (int t = 0; t < (SREG > 0 ? SREG : 1); ++t) {
          int lo = INT_MAX, hi = INT_MAX;
          if (t < s) {
            const BinRecord rc = unpack_record(rec_r[t]);
            lo = bin_lo(rc, ii);
            if (!CAUSAL) hi = bin_hi(rc, ii);
            lomin = min(lomin, lo);
            lomax = max(lomax, lo);
            himax = max(himax, hi);
            himin = min(himin, hi);
          }
          lo_r[t] = lo;
          hi_r[t] = hi;
        }
        vlo = lomin;
        if (!CAUSAL) vhi = himax - 1;
      } else if (qt >= 0) {
        // this row's bin starts (and ends) under every hash, sorted
        const uint4* rs = stage + (slot * 2 + tile) * s * kWordsPerTile + ((ii >> 5) - (i0 >> 5));
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
      // e * slope for e = 0..31 in packed pairs (exact mode bias)
      uint64_t eslope[16];
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2)
        eslope[e2] = f2_pack((float)(2 * e2) * slope, (float)(2 * e2 + 1) * slope);
      if (pend) {
        ok = finish(seq - 1);
        if (!ok) break;
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int jj = 0; jj < ntiles; ++jj, ++g) {
        const int jt = (it.kt_hi - 1 - jj) * BN;
        ok = __all_sync(FULL, mbar_wait(bar(B_SFULL + tile), (uint32_t)g & 1u, abort, lim));
        if (!ok) break;
        tc_fence_after();

        // exact ALiBi: after a row's first tile the weights are taken against
        // the running max as it stands and pass 2 watches for growth; the
        // first tile (or a warp with a row that has no max yet) finds the
        // tile's max first.  (The approximation keeps both passes: its masked
        // chunks skip most of pass 1 already, and the growth check costs it
        // registers.)
        const bool one_pass =
            EXACT && jj > 0 && !__any_sync(FULL, row_ok && m_ref == -INFINITY);
        float m_use = m_ref, alpha = 1.f;
        bool resc = false;
        if (!one_pass) {
          // pass 1: running max (log2 units) over the keys that take part
          float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
          for (int q2 = 0; q2 < 2; ++q2) {
            uint32_t vmh[2];
            uint32_t ra[32], rb2[32];
            if (EXACT) {
              tmem_ld32(s_col + q2 * 64, ra);
              tmem_ld32(s_col + q2 * 64 + 32, rb2);
            }
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const int jc = jt + q2 * 64 + half * 32;
              vmh[half] = EXACT ? key_mask(-1, CAUSAL ? i - jc : n - 1 - jc, row_ok)
                                : key_mask(vlo - jc, vhi - jc, row_ok);
            }
            if (!EXACT) {
              // 64 keys that no row of this warp takes: nothing to read
              if (!__any_sync(FULL, (vmh[0] | vmh[1]) != 0u)) continue;
              tmem_ld32(s_col + q2 * 64, ra);
              tmem_ld32(s_col + q2 * 64 + 32, rb2);
            }
            tmem_wait_ld();
#pragma unroll
            for (int half = 0; half < 2; ++half) {
              const uint32_t* rr = half ? rb2 : ra;
              const int jc = jt + q2 * 64 + half * 32;
              float xv[32];
              const uint32_t vm = vmh[half];
              if (EXACT) {
                const float d0 = (float)(i - jc);
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                  if (CAUSAL) {
                    const uint64_t b2 = f2_add(eslope[e >> 1], f2_pack(-d0 * slope, -d0 * slope));
                    f2_unpack(f2_fma(f2_pack(__uint_as_float(rr[e]), __uint_as_float(rr[e + 1])),
                                     scale2, b2), xv[e], xv[e + 1]);
                  } else {
                    xv[e] = fmaf(__uint_as_float(rr[e]), scale_log2, -fabsf(d0 - (float)e) * slope);
                    xv[e + 1] = fmaf(__uint_as_float(rr[e + 1]), scale_log2,
                                     -fabsf(d0 - (float)(e + 1)) * slope);
                  }
                }
              } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) xv[e] = __uint_as_float(rr[e]);
              }
              if (__any_sync(FULL, vm != 0xffffffffu)) {
#pragma unroll
                for (int e = 0; e < 32; ++e)
                  if (!(vm & (1u << e))) xv[e] = -INFINITY;
              }
#pragma unroll
              for (int e = 0; e < 32; e += 4) {
                mx0 = max3(mx0, xv[e], xv[e + 1]);
                mx1 = max3(mx1, xv[e + 2], xv[e + 3]);
              }
            }
          }
          float mt = fmaxf(mx0, mx1);
          if (!EXACT) mt *= scale_log2;
          if (!row_ok) mt = -INFINITY;
          const float m_new = fmaxf(m_ref, mt);
          resc = m_new > m_ref + kRescaleLog2;
          m_use = resc ? m_new : m_ref;
          alpha = resc ? ex2(m_ref - m_new) : 1.f;
        }
        float mu = (m_use == -INFINITY || !row_ok) ? 0.f : m_use;

        // a grown max rescales O; the commit behind S(g) proves P V(g-1) landed
        if (jj > 0 && __any_sync(FULL, resc)) {
          const float f = resc ? alpha : 1.f;
#pragma unroll 1
          for (int q = 0; q < 4; ++q) {
            uint32_t o[32];
            tmem_ld32(o_col + q * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
            tmem_st32(o_col + q * 32, o);
          }
        }

        // pass 2: P = c 2^(x - m) in f16 pairs, written over score columns
        // already consumed; chunks in descending key order so that the
        // breakpoint pointers only move down
        uint64_t lsum2 = f2_pack(0.f, 0.f);
#pragma unroll 1
        for (int q = 3; q >= 0; --q) {
          const int jc = jt + q * 32;
          uint32_t rr[32];
          uint32_t vm;
          if (EXACT) {
            tmem_ld32(s_col + q * 32, rr);
            vm = key_mask(-1, CAUSAL ? i - jc : n - 1 - jc, row_ok);
          } else {
            vm = key_mask(vlo - jc, vhi - jc, row_ok);
            if (!__any_sync(FULL, vm != 0u)) {
              // no key of the chunk takes part in a row of this warp
              const uint32_t z[16] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u,
                                      0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
              tmem_st16(s_col + kColP + q * 16, z);
              continue;
            }
            tmem_ld32(s_col + q * 32, rr);
          }
          int base = 0;
          bool flat = true, big = false, multi = true;
          uint32_t up[5] = {0u, 0u, 0u, 0u, 0u}, dn[5] = {0u, 0u, 0u, 0u, 0u};
          if (EXACT) {
          } else if (SREG > 0) {
            // rows past every bin start of the chunk (and before every end)
            // have c = s throughout
            const bool deep = lomax <= jc && (CAUSAL || himin > jc + 31);
            if (__all_sync(FULL, deep || vm == 0u)) {
              base = s;
            } else {
              // starts at or before jc count into base, starts inside the
              // chunk set their step bit; two accumulators for ILP (unused
              // registers hold INT_MAX and add nothing)
              const int jc1 = jc + 1;
              int c0 = 0, c1 = 0;
              uint32_t u0 = 0u, u1 = 0u, d0 = 0u, d1 = 0u, x0 = 0u, x1 = 0u;
#pragma unroll
              for (int t = 0; t < (SREG > 0 ? SREG : 1); t += 2) {
                if (t >= s) break;
                {
                  const int dm = lo_r[t] - jc1;
                  c0 -= dm >> 31;
                  const uint32_t bt = shl_clamp(2u, dm);
                  x0 |= u0 & bt;
                  u0 |= bt;
                }
                {
                  const int dm = lo_r[t + 1] - jc1;
                  c1 -= dm >> 31;
                  const uint32_t bt = shl_clamp(2u, dm);
                  x1 |= u1 & bt;
                  u1 |= bt;
                }
                if (!CAUSAL) {
                  const int da = hi_r[t] - jc1, db = hi_r[t + 1] - jc1;
                  c0 += da >> 31;
                  c1 += db >> 31;
                  const uint32_t ba = shl_clamp(2u, da), bb = shl_clamp(2u, db);
                  x0 |= d0 & ba;
                  d0 |= ba;
                  x1 |= d1 & bb;
                  d1 |= bb;
                }
              }
              base = c0 + c1;
              up[0] = u0 | u1;
              dn[0] = d0 | d1;
              uint32_t dup = x0 | x1 | (u0 & u1) | (d0 & d1);
              if (vm == 0u) { up[0] = 0u; dn[0] = 0u; dup = 0u; }
              flat = (up[0] | dn[0]) == 0u;
              multi = __any_sync(FULL, dup != 0u);
              if (multi) {
                // several starts share a key: binary planes of multiplicities
                up[0] = 0u;
                dn[0] = 0u;
                if (vm != 0u) {
#pragma unroll
                  for (int t = 0; t < (SREG > 0 ? SREG : 1); ++t) {
                    plane_add(up, shl_clamp(2u, lo_r[t] - jc1));
                    if (!CAUSAL) plane_add(dn, shl_clamp(2u, hi_r[t] - jc1));
                  }
                }
              }
            }
          } else {
            while (pl > 0 && bpl[(pl - 1) * BM + r] > jc) --pl;
            while (ph > pl && bpl[(ph - 1) * BM + r] > jc + 31) --ph;
            base = pl;
            flat = ph == pl;
            if (!CAUSAL) {
              while (ql > 0 && bph[(ql - 1) * BM + r] > jc) --ql;
              while (qh > ql && bph[(qh - 1) * BM + r] > jc + 31) --qh;
              base -= ql;
              flat = flat && qh == ql;
            }
            if (vm == 0u) flat = true;
            if (!flat) {
              // binary planes of the step multiplicities inside the chunk
              for (int k = pl; k < ph;) {
                const int bpos = bpl[k * BM + r];
                int k2 = k + 1;
                while (k2 < ph && bpl[k2 * BM + r] == bpos) ++k2;
                const uint32_t bit = 1u << (bpos - jc);
                const int m = k2 - k;
#pragma unroll
                for (int b = 0; b < 5; ++b)
                  if (m & (1 << b)) up[b] |= bit;
                big = big || m >= 32;
                k = k2;
              }
              if (!CAUSAL) {
                for (int k = ql; k < qh;) {
                  const int bpos = bph[k * BM + r];
                  int k2 = k + 1;
                  while (k2 < qh && bph[k2 * BM + r] == bpos) ++k2;
                  const uint32_t bit = 1u << (bpos - jc);
                  const int m = k2 - k;
#pragma unroll
                  for (int b = 0; b < 5; ++b)
                    if (m & (1 << b)) dn[b] |= bit;
                  big = big || m >= 32;
                  k = k2;
                }
              }
            }
          }
          tmem_wait_ld();
          uint32_t pk[16];
          {
            const bool all_flat = EXACT || __all_sync(FULL, flat);
            const float lgb = (!EXACT && all_flat) ? lg2((float)max(base, 1)) : 0.f;
            float off;
            if (EXACT) off = -(float)(i - jc) * slope - mu;
            else off = lgb - mu;
            float pv[32];
#pragma unroll
            for (int e = 0; e < 32; e += 2) {
              uint64_t b2 = f2_pack(off, off);
              if (EXACT && CAUSAL) b2 = f2_add(eslope[e >> 1], b2);
              uint64_t a2;
              if (EXACT && !CAUSAL) {
                const float d0 = (float)(i - jc);
                a2 = f2_pack(fmaf(__uint_as_float(rr[e]), scale_log2,
                                  -fabsf(d0 - (float)e) * slope - mu),
                             fmaf(__uint_as_float(rr[e + 1]), scale_log2,
                                  -fabsf(d0 - (float)(e + 1)) * slope - mu));
              } else {
                a2 = f2_fma(f2_pack(__uint_as_float(rr[e]), __uint_as_float(rr[e + 1])),
                            scale2, b2);
              }
              f2_unpack(a2, pv[e], pv[e + 1]);
            }
            if (__any_sync(FULL, vm != 0xffffffffu)) {
#pragma unroll
              for (int e = 0; e < 32; ++e)
                if (!(vm & (1u << e))) pv[e] = -INFINITY;
            }
            if (one_pass) {
              // the chunk's largest exponent: far above the running max (a
              // jump of the scores), O, l and the chunks of this tile written
              // so far are scaled down to the new max first, so that no
              // weight passes 2^15 (f16 holds up to 65504)
              float c0 = -INFINITY, c1 = -INFINITY;
#pragma unroll
              for (int e = 0; e < 32; e += 4) {
                c0 = max3(c0, pv[e], pv[e + 1]);
                c1 = max3(c1, pv[e + 2], pv[e + 3]);
              }
              const float cm = fmaxf(c0, c1);
              if (__any_sync(FULL, cm > kGrowLog2)) {
                const float d = cm > kGrowLog2 ? cm - lgb : 0.f;
                const float f = ex2(-d);
                mu += d;
                if (row_ok) m_use = mu;
#pragma unroll
                for (int e = 0; e < 32; ++e) pv[e] -= d;
                l *= f;
                lsum2 = f2_mul(lsum2, f2_pack(f, f));
#pragma unroll 1
                for (int q3 = 0; q3 < 4; ++q3) {
                  uint32_t o[32];
                  tmem_ld32(o_col + q3 * 32, o);
                  tmem_wait_ld();
#pragma unroll
                  for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * f);
                  tmem_st32(o_col + q3 * 32, o);
                }
#pragma unroll 1
                for (int q3 = 3; q3 > q; --q3) {
                  uint32_t w[16];
                  tmem_ld16(s_col + kColP + q3 * 16, w);
                  tmem_wait_ld();
#pragma unroll
                  for (int e = 0; e < 16; ++e) {
                    const float2 x = __half22float2(*reinterpret_cast<const __half2*>(&w[e]));
                    w[e] = pack_f16(x.x * f, x.y * f);
                  }
                  tmem_st16(s_col + kColP + q3 * 16, w);
                }
              }
            }
#pragma unroll
            for (int e = 0; e < 32; ++e) pv[e] = ex2(pv[e]);
            if (!EXACT && !all_flat) {
              // c_ij inside the chunk: a running count of the bin starts
              // (minus bin ends), one plane per bit of the multiplicities
              const float fb = (float)base;
              if (SREG == 0 && __any_sync(FULL, big)) {
                float cf[32];
#pragma unroll
                for (int e = 0; e < 32; ++e) cf[e] = fb;
                for (int k = pl; k < ph; ++k) {
                  const int bo = bpl[k * BM + r] - jc;
#pragma unroll
                  for (int e = 0; e < 32; ++e)
                    if (e >= bo) cf[e] += 1.f;
                }
                if (!CAUSAL) {
                  for (int k = ql; k < qh; ++k) {
                    const int bo = bph[k * BM + r] - jc;
#pragma unroll
                    for (int e = 0; e < 32; ++e)
                      if (e >= bo) cf[e] -= 1.f;
                  }
                }
#pragma unroll
                for (int e = 0; e < 32; ++e) pv[e] *= cf[e];
              } else if (!multi) {
                scale_by_steps<CAUSAL>(pv, base, up[0], dn[0]);
              } else if (__any_sync(FULL, (up[2] | up[3] | up[4] | dn[2] | dn[3] | dn[4]) != 0u)) {
                // a multiplicity never exceeds the number of register slots
                scale_by_planes<(SREG == 0 || SREG > 15) ? 5 : (SREG > 7 ? 4 : 3), CAUSAL>(
                    pv, base, up, dn);
              } else {
                scale_by_planes<2, CAUSAL>(pv, base, up, dn);
              }
            }
            // P rounded to f16 pairs; the row sum takes the fp32 values
#pragma unroll
            for (int e2 = 0; e2 < 16; ++e2) {
              lsum2 = f2_add(lsum2, f2_pack(pv[2 * e2], pv[2 * e2 + 1]));
              pk[e2] = pack_f16(pv[2 * e2], pv[2 * e2 + 1]);
            }
          }
          // chunks run in descending order, so P of chunk q lands on the
          // score columns of chunks q + 2 and q + 3, already consumed
          tmem_st16(s_col + kColP + q * 16, pk);
        }
        float ls0, ls1;
        f2_unpack(lsum2, ls0, ls1);
        l = l * alpha + (ls0 + ls1);
        m_ref = m_use;
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(bar(B_PFULL + tile));
      }
      if (!ok) break;

      // the output is written once the next item is set up (or at the end),
      // so that the item's last P V runs meanwhile
      pend = true;
      pend_l = l;
      pend_m = (row_ok && l > 0.f) ? m_ref : -INFINITY;
      if (!kDefer) {
        ok = finish(seq);
        if (!ok) break;
      }
    }
    if (!ok && lane == 0) {
      *abort = 1;
      atomicOr(a.err, kErrTimeout);
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
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

// ----------------------------------------------------------- split merge
// The parts of a split item cover disjoint key ranges of its rows' envelopes,
// each with its own running max m_p (log2 units) and row sum l_p:
//   O_i = sum_p 2^(m_p - m) acc_p / sum_p 2^(m_p - m) l_p,  m = max_p m_p,
// over the parts that saw a key of row i (l_p > 0).  A warp per row, a float4
// of the head dimension per lane.  Grid: (split items, 2 tiles, 16 row groups).
__global__ void __launch_bounds__(256)
split_merge_kernel(const int4* __restrict__ merge, const float* __restrict__ ws,
                   __nv_bfloat16* __restrict__ O, float* __restrict__ lse, int Hq, int n, int d) {
  const int item = blockIdx.x, tile = blockIdx.y;
  const int r = blockIdx.z * 8 + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  const int4 e = merge[2 * item], x = merge[2 * item + 1];
  const int qt = tile ? e.w : e.z;
  const int h = tile ? (e.y >> 16) & 0xffff : e.y & 0xffff;
  const int i = qt * BM + r;
  if (qt < 0 || i >= n) return;
  const int slot0 = x.x, parts = x.y;
  float m = -INFINITY;
  for (int p = 0; p < parts; ++p) {
    const float* w = ws + (size_t)(slot0 + p) * kSplitSlotFloats + 2 * BM * kSplitRowFloats;
    if (w[2 * BM + tile * BM + r] > 0.f) m = fmaxf(m, w[tile * BM + r]);
  }
  float l = 0.f;
  float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int p = 0; p < parts; ++p) {
    const float* w = ws + (size_t)(slot0 + p) * kSplitSlotFloats;
    const float* wm = w + 2 * BM * kSplitRowFloats;
    const float lp = wm[2 * BM + tile * BM + r];
    if (!(lp > 0.f)) continue;
    const float f = exp2f(wm[tile * BM + r] - m);
    l = fmaf(f, lp, l);
    const float4 a4 =
        reinterpret_cast<const float4*>(w + ((size_t)tile * BM + r) * kSplitRowFloats)[lane];
    o.x = fmaf(f, a4.x, o.x);
    o.y = fmaf(f, a4.y, o.y);
    o.z = fmaf(f, a4.z, o.z);
    o.w = fmaf(f, a4.w, o.w);
  }
  const float inv = l > 0.f ? 1.f / l : 0.f;
  if (4 * lane < d) {                                    // d = 64: the padding is not stored
    __nv_bfloat162* out =
        reinterpret_cast<__nv_bfloat162*>(O + (((int64_t)e.x * Hq + h) * n + i) * d) + 2 * lane;
    out[0] = __floats2bfloat162_rn(o.x * inv, o.y * inv);
    out[1] = __floats2bfloat162_rn(o.z * inv, o.w * inv);
  }
  if (lse != nullptr && lane == 0)
    lse[((int64_t)e.x * Hq + h) * n + i] = l > 0.f ? m + __log2f(l) : -INFINITY;
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

// [planes, n, d] bf16 (d = 64 or 128) viewed as a 3-D tensor with 64 x rows
// x 1 boxes and 128-byte swizzle; rows past n, and with d = 64 the columns
// past 64 (the second box of a tile), read as zeros, so that a d = 64 tile
// enters the kernel zero-padded to 128 columns.
bool make_map(CUtensorMap* map, const void* base, int64_t planes, int64_t n, int box_rows,
              int d) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)n, (cuuint64_t)planes};
  const cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)n * d * 2};
  const cuuint32_t box[3] = {64, (cuuint32_t)box_rows, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base),
            dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool EXACT, bool CAUSAL, int SREG>
cudaError_t launch_variant(const CUtensorMap& mq, const CUtensorMap& mk,
                           const CUtensorMap& mv, const TcParams& p,
                           size_t smem, int grid, cudaStream_t st) {
  auto kern = attn_tc_kernel<EXACT, CAUSAL, SREG>;
  cudaError_t e = set_smem_limit(reinterpret_cast<const void*>(kern), (int)smem);
  if (e != cudaSuccess) return e;
  // programmatic stream serialization: the CTAs may start (and set up
  // shared memory, barriers and TMEM) while the previous kernel finishes
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, mq, mk, mv, p);
}

// Register slots for the rows' bin starts (and, without the causal mask,
// ends): the smallest compiled size that holds s, so that no slot is padding
// the per-chunk count walks over; sorted lists in shared memory beyond.
int sreg_for(int s, int causal, int exact) {
  if (exact) return 0;
  if (causal) {
    for (int r : {4, 8, 10, 12, 16})
      if (s <= r) return r;
    return 0;
  }
  for (int r : {8, 16})
    if (s <= r) return r;
  return 0;
}

constexpr size_t kSmemLimit = 232448;   // opt-in dynamic shared memory per CTA

size_t smem_for(int slots, bool out, int s, int causal, int exact) {
  const int sreg = sreg_for(s, causal, exact);
  return 1024 + OFF_KV + (size_t)slots * kTileBytes + (out ? kOutBytes : 0) +
         bp_bytes(s, exact != 0, causal != 0, sreg) + stage_bytes(s, exact != 0) +
         sizeof(Ctl);
}

// The output staging buffer when the per-row bin lists leave room for it
// (else the epilogue stores its rows directly).
bool out_staged(int s, int causal, int exact) {
  return smem_for(kSlots, true, s, causal, exact) <= kSmemLimit;
}
}  // namespace

bool make_tile_map_bf16(CUtensorMap* map, const void* base, int64_t planes, int64_t n) {
  return make_map(map, base, planes, n, BM, HD);
}

bool make_rows_map_bf16(CUtensorMap* map, const void* base, int64_t planes, int64_t n,
                        int box_rows, int d) {
  return make_map(map, base, planes, n, box_rows, d);
}

size_t attn_tc_smem_bytes(int s, int causal, int exact) {
  return smem_for(kSlots, out_staged(s, causal, exact), s, causal, exact);
}

cudaError_t launch_split_merge(const int4* merge, int count, const float* ws, void* O, float* lse,
                               int Hq, int n, int d, cudaStream_t st) {
  if (count <= 0) return cudaSuccess;
  split_merge_kernel<<<dim3((unsigned)count, 2, BM / 8), 256, 0, st>>>(
      merge, ws, static_cast<__nv_bfloat16*>(O), lse, Hq, n, d);
  return cudaGetLastError();
}

cudaError_t launch_attn_tc(const AttnArgs& a, const float* slopes_host,
                           int num_sms, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, a.Q, (int64_t)a.B * a.Hq, a.n, BM, a.d) ||
      !make_map(&mk, a.K, (int64_t)a.B * a.Hkv, a.n, BN, a.d) ||
      !make_map(&mv, a.V, (int64_t)a.B * a.Hkv, a.n, BN, a.d))
    return cudaErrorInvalidValue;
  TcParams p;
  p.a = a;
  for (int h = 0; h < 512; ++h)
    p.slope_log2[h] = (slopes_host && h < a.Hq) ? slopes_host[h] : 0.f;
  p.QT = (a.n + BM - 1) / BM;
  p.out_smem = out_staged(a.s, a.causal, a.exact) ? 1 : 0;
  const int grid = a.num_items < num_sms ? a.num_items : num_sms;
  const size_t smem = attn_tc_smem_bytes(a.s, a.causal, a.exact);
  if (a.exact) {
    return a.causal ? launch_variant<true, true, 0>(mq, mk, mv, p, smem, grid, st)
                    : launch_variant<true, false, 0>(mq, mk, mv, p, smem, grid, st);
  }
  switch (a.causal ? sreg_for(a.s, 1, 0) : -sreg_for(a.s, 0, 0)) {
    case 4: return launch_variant<false, true, 4>(mq, mk, mv, p, smem, grid, st);
    case 8: return launch_variant<false, true, 8>(mq, mk, mv, p, smem, grid, st);
    case 10: return launch_variant<false, true, 10>(mq, mk, mv, p, smem, grid, st);
    case 12: return launch_variant<false, true, 12>(mq, mk, mv, p, smem, grid, st);
    case 16: return launch_variant<false, true, 16>(mq, mk, mv, p, smem, grid, st);
    case -8: return launch_variant<false, false, 8>(mq, mk, mv, p, smem, grid, st);
    case -16: return launch_variant<false, false, 16>(mq, mk, mv, p, smem, grid, st);
    default: break;
  }
  return a.causal ? launch_variant<false, true, 0>(mq, mk, mv, p, smem, grid, st)
                  : launch_variant<false, false, 0>(mq, mk, mv, p, smem, grid, st);
}

}  // namespace plsh
