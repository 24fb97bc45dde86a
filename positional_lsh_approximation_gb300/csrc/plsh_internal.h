// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <map>
#include <mutex>
#include <string>
#include <utility>
#include <vector>

#include "../../include/plsh.h"

namespace plsh {

// A kernel's dynamic shared-memory limit, set in the device's context the
// first time a size is asked for (the attribute persists), so that repeated
// launches skip the driver call.
inline cudaError_t set_smem_limit(const void* kern, int bytes) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lk(mu);
  int& have = done[std::make_pair(dev, kern)];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}


// One record per (hash, 32-position word): which positions of the word open a
// bin, the last bin start at or before the word's first position, and the
// first bin start after the word (n when none).
struct __align__(16) BinRecord {
  uint32_t bits;
  int32_t prev;
  int32_t next;
  int32_t pad;
};

constexpr int kMaxS = 64;
constexpr int kMaxExactHeads = 512;
constexpr uint64_t kDefaultWaitNs = 2000000000ull;

// Work-item table of the tensor-core kernel for one problem shape and head
// order, kept on the device once built.  Items whose key envelope is long are
// split into parts over the key range: each part has an entry in `ext`
// {part, parts, workspace slot, 0} (no `ext` when nothing is split), writes
// its partial rows (unnormalised P V, max, row sum) to its workspace slot, and
// `merge` lists the split items {b, hA | hB << 16, qtA, qtB}, {first slot,
// parts, 0, 0} for the kernel that combines the parts into O.
struct ItemTable {
  std::vector<int4> host;
  std::vector<int4> ext;
  std::vector<int4> merge;
  int4* dev = nullptr;
  int4* dev_ext = nullptr;
  int4* dev_merge = nullptr;
  float* ws = nullptr;
  uint64_t last_use = 0;
  // device memory is stream-ordered: allocated and uploaded on `home`
  // (`ready` recorded behind the upload), freed behind the events that the
  // calls using it recorded on their streams; `pins` counts the calls between
  // lookup and launch, which keep the table from being evicted
  cudaStream_t home = nullptr;
  cudaEvent_t ready = nullptr;
  int pins = 0;
  std::vector<std::pair<cudaStream_t, cudaEvent_t>> uses;
};
// floats of one split part's workspace slot: both tiles' rows of P V, then
// their maxima, then their row sums
constexpr int kSplitRowFloats = 128;
constexpr size_t kSplitSlotFloats = 2 * 128 * (kSplitRowFloats + 2);
constexpr int kMaxSplitParts = 16;

// Per-device library state.
constexpr int kMaxHostChunks = 4;    // query-row chunks of the host-buffer entry point
struct DeviceCtx {
  int device = -1;
  int num_sms = 0;
  int* d_err = nullptr;        // device error flag (bit 0: wait timeout)
  int split_parts = 0;         // 0: automatic, 1: never split, >= 2: every item in that many parts
  int* d_queue = nullptr;      // kQueueSlots x {next item, finished CTAs}
  uint64_t slot_counter = 0;
  uint64_t wait_ns = kDefaultWaitNs;
  std::map<std::string, ItemTable> tables;
  uint64_t table_clock = 0;
  // staging of the host-buffer entry point: device copies of Q, K, V, O,
  // one stream per copy direction and the events that chain the chunks
  void* stage[4] = {nullptr, nullptr, nullptr, nullptr};
  size_t stage_bytes[4] = {0, 0, 0, 0};
  cudaStream_t h2d = nullptr, d2h = nullptr;
  cudaEvent_t ev[2 + 2 * kMaxHostChunks] = {};
  // per-chunk partial results of the decode step (m, l, P V), grown on demand
  float* decode_work = nullptr;
  size_t decode_work_bytes = 0;
  cudaEvent_t decode_ev = nullptr;   // last stream use of decode_work
  // scratch of the backward pass (row statistics, fp32 dQ accumulator),
  // grown on demand and kept between calls
  float* bwd_work = nullptr;
  size_t bwd_work_bytes = 0;
  cudaEvent_t bwd_ev = nullptr;      // last stream use of bwd_work
};
constexpr size_t kMaxTables = 16;
constexpr int kQueueSlots = 1024;

}  // namespace plsh

struct plsh_bins {
  int device;
  int64_t n;
  int32_t H, s;
  int64_t W;                      // words per hash = ceil(n / 32)
  double* d_sigma = nullptr;      // [H]
  double* d_w = nullptr;          // [H*s]
  double* d_u = nullptr;          // [H*s]
  plsh::BinRecord* d_rec = nullptr;  // [H*s][W]
  int32_t* d_head_order = nullptr;   // [H]
  std::vector<double> sigma_host;    // per-head scale (drawn or estimated)
  std::vector<int32_t> head_order;   // heads by expected work, descending
  bool sigma_on_device = false;      // d_sigma / d_head_order hold sigma_host
};

namespace plsh {

// sampler.cu
cudaError_t launch_sample(plsh_bins* b, uint64_t seed, cudaStream_t st);
cudaError_t launch_bins_from_starts(plsh_bins* b, const int32_t* d_starts,
                                    const int64_t* d_offsets, int64_t total,
                                    cudaStream_t st);

// Arguments common to the attention kernels.
struct AttnArgs {
  const void* Q;
  const void* K;
  const void* V;
  void* O;
  int B, Hq, Hkv, n, d;
  int causal;
  int exact;                       // 1: exact ALiBi, 0: Positional LSH
  const BinRecord* rec;            // [Hq*s][W] (approximate mode)
  int s;
  int64_t W;
  // tensor-core path: work items, each two 128-row query tiles that share
  // one KV head, {b, hA | hB << 16, qtA, qtB (-1: none)}, in cost order
  const int4* items;
  int num_items;
  const int4* item_ext;            // split parts {part, parts, slot, 0}, or null
  float* split_ws;                 // workspace slots of split parts
  // row statistics mode (the backward pass's first step): with stats set,
  // every row's -lse (lse = m + log2 l, the base-2 log-sum-exp of the scaled
  // scores with their multiplicities; m the running max, l the row sum) and
  // Delta = sum_d O_d dO_d (O = acc / l in fp32) go to stats[row][2], with
  // dO [B, Hq, n, 128] bf16; O itself is written only when O != null
  float* stats;
  const void* dO;
  // with lse set (and no stats), every row's lse goes to lse[row] beside O
  float* lse;
  int* err;
  int* queue;                      // {next item, finished CTAs}
  uint64_t wait_ns;
  int stall;                       // fault injection: the scheduler publishes no item
};

// decode.cu: one query position against the cached keys.  A CTA serves up
// to eight query heads of one KV group (a warp each) over one of S shares of
// the union of their key envelopes; S is chosen for about three CTAs per SM
// (at most 64).
inline int decode_heads(int G) { return G < 8 ? G : 8; }
// useful: shares worth having, from the widest envelope expected (at most 64)
inline int decode_splits(int B, int Hq, int Hkv, int num_sms, int useful) {
  const int G = Hq / Hkv;
  const int64_t ctas = (int64_t)B * Hkv * ((G + decode_heads(G) - 1) / decode_heads(G));
  const int64_t want = 12LL * num_sms;
  const int64_t cap = useful < 1 ? 1 : (useful > 64 ? 64 : useful);
  const int64_t sp = (want + ctas - 1) / ctas;
  return (int)(sp < 1 ? 1 : (sp > cap ? cap : sp));
}
// the envelope of a row at pos under bins of scale sigma reaches about
// 1.2 sigma keys back (the widest of the s bins around pos); a share of the
// split takes about 64 keys of it
inline int decode_useful_splits(double sigma_max, int pos) {
  const double keys = 1.2 * sigma_max + 128.0;
  const double lim = pos + 1.0 < keys ? pos + 1.0 : keys;
  const double sp = lim / 64.0 + 1.0;
  return sp > 64.0 ? 64 : (int)sp;
}
inline size_t decode_work_floats(int B, int Hq, int Hkv, int d, int num_sms, int useful) {
  return (size_t)B * Hq * decode_splits(B, Hq, Hkv, num_sms, useful) * (size_t)(d + 2);
}
struct DecodeArgs {
  const void* q;         // [B, Hq, 1, d]
  const void* K;         // [B, Hkv, n, d]
  const void* V;
  void* o;               // [B, Hq, 1, d]
  const BinRecord* rec;  // [Hq*s][W]
  int B, Hq, Hkv, n, d, s;
  int64_t W;
  int pos;
  int dtype;             // PLSH_BF16 or PLSH_F32
  int num_sms;
  int useful_splits;     // decode_useful_splits of the widest bins
  const double* sigma;   // host [Hq] scales of the heads' bins, or null if unknown
  float* work;           // decode_work_floats(B, Hq, Hkv, d, num_sms, useful_splits)
  int* err;              // device error flag (bit 0: a bounded wait ran out)
  uint64_t wait_ns;
};
cudaError_t launch_decode(const DecodeArgs& a, cudaStream_t st);

// attn_simt.cu (CUDA cores, any dtype, d in {64, 128})
// slopes_host: exact mode, [Hq] log2(e)/sigma_h (at most kMaxExactHeads)
cudaError_t launch_attn_simt(const AttnArgs& a, const float* slopes_host,
                             int dtype, cudaStream_t st);
// attn_tc.cu (tcgen05 tensor cores, bf16, d = 128)
cudaError_t launch_attn_tc(const AttnArgs& a, const float* slopes_host,
                           int num_sms, cudaStream_t st);
// combines the parts of `count` split items (entries of `merge`, two int4
// each) into O (bf16 [B, Hq, n, 128])
cudaError_t launch_split_merge(const int4* merge, int count, const float* ws, void* O, float* lse,
                               int Hq, int n, int d, cudaStream_t st);
size_t attn_tc_smem_bytes(int s, int causal, int exact);
// [planes, n, 128] bf16 as a TMA tensor map with 64 x 128 x 1 boxes, 128-byte
// swizzle, rows past n reading as zeros (attn_tc.cu)
bool make_tile_map_bf16(CUtensorMap* map, const void* base, int64_t planes, int64_t n);
// [planes, n, d] bf16 (d = 64 or 128) as a 3-D tensor map of 64-value x
// box_rows x 1 tiles with 128-byte swizzle (rows past n read as zeros)
bool make_rows_map_bf16(CUtensorMap* map, const void* base, int64_t planes, int64_t n,
                        int box_rows, int d);

// bwd_tc.cu: gradients on the tensor cores (bf16, d = 128, s <= 16) from the
// rows' statistics [B * Hq * n][2] (-lse, Delta); dq_acc is fp32 scratch of
// B * Hq * n * 128 floats, cleared by the call when clear_acc is set (else
// already zero)
constexpr int kBwdTcMaxS = 16;
constexpr int kBwdTcMaxGroup = 64;
size_t bwd_tc_smem_bytes();
cudaError_t launch_attn_bwd_tc(const void* Q, const void* K, const void* V, const void* dO,
                               void* dQ, void* dK, void* dV, const float* stats, float* dq_acc,
                               bool clear_acc, const plsh_bins* bn, int B, int Hq, int Hkv, int n,
                               int causal, int* queue, int* err, uint64_t wait_ns, int num_sms,
                               cudaStream_t st);
// the rows' statistics from a saved O and lse ([rows] base-2 log-sum-exp):
// stats[row] = (-lse, dO . O), and dq_acc's rows cleared (rows = B * Hq * n,
// O and dO [rows][128] bf16)
cudaError_t launch_bwd_delta(const void* O, const void* dO, const float* lse, float* stats,
                             float* dq_acc, int64_t rows, cudaStream_t st);

}  // namespace plsh
