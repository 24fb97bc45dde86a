// C ABI entry points (include/plsh.h): validation, handles, dispatch.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <algorithm>
#include <atomic>
#include <mutex>
#include <numeric>
#include <string>
#include <vector>

#include "plsh_internal.h"

namespace {

thread_local std::string g_last_error;

plsh_status fail(plsh_status st, const std::string& msg) {
  g_last_error = msg;
  return st;
}

plsh_status cuda_fail(cudaError_t e, const char* what) {
  return fail(PLSH_ERR_CUDA, std::string(what) + ": " + cudaGetErrorString(e));
}

#define PLSH_TRY_CUDA(expr, what)                      \
  do {                                                 \
    cudaError_t e_ = (expr);                           \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

constexpr int kMaxDevices = 64;
std::mutex g_ctx_mu;
// held while a call enqueues work on a per-device scratch buffer
std::mutex g_bwd_mu, g_decode_mu;

bool fault_oom();

// A per-device scratch buffer of at least `bytes`, ordered after its last
// use on any stream: the calling stream first waits for the event recorded
// after that use; a buffer too small is then replaced in stream order on the
// calling stream (freed, allocated from the device's stream-ordered pool and
// zeroed there), so that growing it stalls neither the host nor other
// streams.  The caller holds the buffer's mutex and records *ev on its stream
// after its launches.
plsh_status scratch_acquire(float** buf, size_t* have, cudaEvent_t* ev, size_t bytes,
                            cudaStream_t cs, const char* what) {
  if (*ev == nullptr) PLSH_TRY_CUDA(cudaEventCreateWithFlags(ev, cudaEventDisableTiming), what);
  PLSH_TRY_CUDA(cudaStreamWaitEvent(cs, *ev, 0), what);
  if (*have < bytes) {
    if (*buf != nullptr) PLSH_TRY_CUDA(cudaFreeAsync(*buf, cs), what);
    *buf = nullptr;
    *have = 0;
    if (fault_oom()) return fail(PLSH_ERR_NOMEM, std::string(what) + ": injected allocation failure");
    const cudaError_t e = cudaMallocAsync((void**)buf, bytes, cs);
    if (e == cudaErrorMemoryAllocation) {
      cudaGetLastError();
      *buf = nullptr;
      return fail(PLSH_ERR_NOMEM, std::string(what) + ": out of device memory");
    }
    PLSH_TRY_CUDA(e, what);
    // zeroed once, so that counters kept in it start from a known state
    PLSH_TRY_CUDA(cudaMemsetAsync(*buf, 0, bytes, cs), what);
    *have = bytes;
  }
  return PLSH_OK;
}
plsh::DeviceCtx g_ctx[kMaxDevices];

// Fault injection for the tests, from the environment: PLSH_FAULT=oom fails
// every device allocation; PLSH_FAULT=stall makes the next tensor-core
// attention publish no work item, so every device-side wait runs out (with
// nothing in flight) and the error flag reports PLSH_ERR_TIMEOUT.
bool fault_is(const char* what) {
  const char* f = getenv("PLSH_FAULT");
  return f != nullptr && strcmp(f, what) == 0;
}
bool fault_oom() { return fault_is("oom"); }

plsh_status dev_alloc(void** p, size_t bytes, const char* what) {
  if (fault_oom()) return fail(PLSH_ERR_NOMEM, std::string(what) + ": injected allocation failure");
  cudaError_t e = cudaMalloc(p, bytes == 0 ? 16 : bytes);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    return fail(PLSH_ERR_NOMEM, std::string(what) + ": out of device memory");
  }
  if (e != cudaSuccess) return cuda_fail(e, what);
  return PLSH_OK;
}

// The same, ordered on `st` (no implicit synchronisation; free with
// cudaFreeAsync).
plsh_status dev_alloc_async(void** p, size_t bytes, cudaStream_t st, const char* what) {
  *p = nullptr;
  if (fault_oom()) return fail(PLSH_ERR_NOMEM, std::string(what) + ": injected allocation failure");
  cudaError_t e = cudaMallocAsync(p, bytes == 0 ? 16 : bytes, st);
  if (e == cudaErrorMemoryAllocation) {
    cudaGetLastError();
    *p = nullptr;
    return fail(PLSH_ERR_NOMEM, std::string(what) + ": out of device memory");
  }
  if (e != cudaSuccess) return cuda_fail(e, what);
  return PLSH_OK;
}

// Context of the current device, created on first use.
plsh_status current_ctx(plsh::DeviceCtx** out) {
  int dev = -1;
  PLSH_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PLSH_ERR_UNSUPPORTED, "device index out of range");
  std::lock_guard<std::mutex> lk(g_ctx_mu);
  plsh::DeviceCtx& c = g_ctx[dev];
  if (c.device < 0) {
    int sms = 0;
    PLSH_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                  "cudaDeviceGetAttribute");
    int* err = nullptr;
    int* queue = nullptr;
    plsh_status st = dev_alloc((void**)&err, sizeof(int), "error flag");
    if (st != PLSH_OK) return st;
    st = dev_alloc((void**)&queue, sizeof(int) * 2 * plsh::kQueueSlots, "work queues");
    if (st != PLSH_OK) {
      cudaFree(err);
      return st;
    }
    PLSH_TRY_CUDA(cudaMemset(err, 0, sizeof(int)), "cudaMemset");
    PLSH_TRY_CUDA(cudaMemset(queue, 0, sizeof(int) * 2 * plsh::kQueueSlots), "cudaMemset");
    PLSH_TRY_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
    c.num_sms = sms;
    c.d_err = err;
    c.d_queue = queue;
    c.device = dev;
  }
  *out = &c;
  return PLSH_OK;
}

plsh_status check_sigma(const double* sigma, int32_t H) {
  if (sigma == nullptr) return fail(PLSH_ERR_INVALID, "sigma_h is NULL");
  for (int32_t h = 0; h < H; ++h) {
    const double v = sigma[h];
    if (!(v > 0.0) || !(v <= 1e15) || !isfinite(v))
      return fail(PLSH_ERR_INVALID, "sigma_h[" + std::to_string(h) +
                                        "] must be finite and in (0, 1e15]");
  }
  return PLSH_OK;
}

void order_heads(plsh_bins* b) {
  b->head_order.resize(b->H);
  std::iota(b->head_order.begin(), b->head_order.end(), 0);
  std::stable_sort(b->head_order.begin(), b->head_order.end(),
                   [&](int x, int y) { return b->sigma_host[x] > b->sigma_host[y]; });
}

void free_bins(plsh_bins* b) {
  if (!b) return;
  int prev = -1;
  cudaGetDevice(&prev);
  cudaSetDevice(b->device);
  cudaDeviceSynchronize();
  cudaFree(b->d_sigma);
  cudaFree(b->d_w);
  cudaFree(b->d_u);
  cudaFree(b->d_rec);
  cudaFree(b->d_head_order);
  if (prev >= 0) cudaSetDevice(prev);
  delete b;
}

plsh_status new_bins(int64_t n, int32_t H, int32_t s, plsh_bins** out) {
  int dev = -1;
  PLSH_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  plsh_bins* b = new (std::nothrow) plsh_bins();
  if (!b) return fail(PLSH_ERR_NOMEM, "host allocation");
  b->device = dev;
  b->n = n;
  b->H = H;
  b->s = s;
  b->W = (n + 31) / 32;
  const size_t HS = (size_t)H * s;
  plsh_status st;
  if ((st = dev_alloc((void**)&b->d_sigma, sizeof(double) * H, "sigma")) != PLSH_OK ||
      (st = dev_alloc((void**)&b->d_w, sizeof(double) * HS, "draws")) != PLSH_OK ||
      (st = dev_alloc((void**)&b->d_u, sizeof(double) * HS, "draws")) != PLSH_OK ||
      (st = dev_alloc((void**)&b->d_rec, sizeof(plsh::BinRecord) * HS * b->W, "bin records")) != PLSH_OK ||
      (st = dev_alloc((void**)&b->d_head_order, sizeof(int32_t) * H, "head order")) != PLSH_OK) {
    free_bins(b);
    return st;
  }
  *out = b;
  return PLSH_OK;
}

plsh_status check_bins_device(const plsh_bins* b) {
  int dev = -1;
  PLSH_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev != b->device) return fail(PLSH_ERR_INVALID, "bins handle lives on another device");
  return PLSH_OK;
}

plsh_status resample(plsh_bins* b, const double* sigma, uint64_t seed, cudaStream_t st) {
  // sigma and the head order live on the device; they are uploaded again only
  // when sigma changes (a redraw with new seeds alone launches one kernel)
  if (!b->sigma_on_device || !std::equal(sigma, sigma + b->H, b->sigma_host.begin())) {
    b->sigma_host.assign(sigma, sigma + b->H);
    order_heads(b);
    PLSH_TRY_CUDA(cudaMemcpyAsync(b->d_sigma, sigma, sizeof(double) * b->H,
                                  cudaMemcpyHostToDevice, st), "copy sigma");
    PLSH_TRY_CUDA(cudaMemcpyAsync(b->d_head_order, b->head_order.data(),
                                  sizeof(int32_t) * b->H, cudaMemcpyHostToDevice, st),
                  "copy head order");
    b->sigma_on_device = true;
  }
  PLSH_TRY_CUDA(plsh::launch_sample(b, seed, st), "sampler launch");
  return PLSH_OK;
}

// Host copy of the records -> (offsets, starts).  Synchronises `st`.
plsh_status records_to_host(const plsh_bins* b, cudaStream_t st,
                            std::vector<int64_t>* offsets, std::vector<int32_t>* starts) {
  const size_t HS = (size_t)b->H * b->s;
  std::vector<plsh::BinRecord> rec(HS * b->W);
  PLSH_TRY_CUDA(cudaMemcpyAsync(rec.data(), b->d_rec, sizeof(plsh::BinRecord) * rec.size(),
                                cudaMemcpyDeviceToHost, st), "copy records");
  PLSH_TRY_CUDA(cudaStreamSynchronize(st), "cudaStreamSynchronize");
  offsets->assign(HS + 1, 0);
  starts->clear();
  for (size_t hs = 0; hs < HS; ++hs) {
    (*offsets)[hs] = (int64_t)starts->size();
    for (int64_t w = 0; w < b->W; ++w) {
      uint32_t bits = rec[hs * b->W + w].bits;
      while (bits) {
        const int r = __builtin_ctz(bits);
        starts->push_back((int32_t)(w * 32 + r));
        bits &= bits - 1;
      }
    }
    starts->push_back((int32_t)b->n);
  }
  (*offsets)[HS] = (int64_t)starts->size();
  return PLSH_OK;
}

plsh_status check_tensor(const plsh_tensor* t, const char* name) {
  if (t == nullptr) return fail(PLSH_ERR_INVALID, std::string(name) + " is NULL");
  if (t->data == nullptr) return fail(PLSH_ERR_INVALID, std::string(name) + "->data is NULL");
  if (((uintptr_t)t->data & 15u) != 0)
    return fail(PLSH_ERR_INVALID, std::string(name) + "->data must be 16-byte aligned");
  if (t->dtype != PLSH_F32 && t->dtype != PLSH_BF16)
    return fail(PLSH_ERR_INVALID, std::string(name) + ": dtype must be PLSH_F32 or PLSH_BF16");
  if (t->B < 1 || t->H < 1 || t->n < 1 || t->d < 1)
    return fail(PLSH_ERR_INVALID, std::string(name) + ": every dimension must be >= 1");
  return PLSH_OK;
}

plsh_status check_qkvo(const plsh_tensor* Q, const plsh_tensor* K, const plsh_tensor* V,
                       const plsh_tensor* O) {
  plsh_status st;
  if ((st = check_tensor(Q, "Q")) != PLSH_OK || (st = check_tensor(K, "K")) != PLSH_OK ||
      (st = check_tensor(V, "V")) != PLSH_OK || (st = check_tensor(O, "O")) != PLSH_OK)
    return st;
  if (K->dtype != Q->dtype || V->dtype != Q->dtype || O->dtype != Q->dtype)
    return fail(PLSH_ERR_INVALID, "Q, K, V and O must share one dtype");
  if (Q->d != 64 && Q->d != 128) return fail(PLSH_ERR_INVALID, "head dim d must be 64 or 128");
  if (K->B != Q->B || K->n != Q->n || K->d != Q->d)
    return fail(PLSH_ERR_INVALID, "K must be [B, Hkv, n, d] with Q's B, n, d");
  if (V->B != K->B || V->H != K->H || V->n != K->n || V->d != K->d)
    return fail(PLSH_ERR_INVALID, "V must have K's shape");
  if (O->B != Q->B || O->H != Q->H || O->n != Q->n || O->d != Q->d)
    return fail(PLSH_ERR_INVALID, "O must have Q's shape");
  if (Q->H % K->H != 0) return fail(PLSH_ERR_INVALID, "Hq must be a multiple of Hkv");
  if (Q->n >= ((int64_t)1 << 31)) return fail(PLSH_ERR_INVALID, "n must be < 2^31");
  const int64_t tiles = Q->B * Q->H * ((Q->n + 127) / 128);
  if (Q->B * Q->H >= ((int64_t)1 << 31) || tiles >= ((int64_t)1 << 31))
    return fail(PLSH_ERR_INVALID, "B * Hq * ceil(n/128) must be < 2^31");
  return PLSH_OK;
}

// Expected key tiles of an item: the exact kernel takes every key tile up to
// the diagonal (every key tile without the causal mask); the approximation
// the diagonal tile plus its rows' look-back, about 1.5 sigma (1 + 0.7 ln s)
// keys (the mean age of the Gamma(2, sigma) bin that holds a row is 1.5 sigma;
// the largest of s such ages grows like ln s; the factor 0.7 matches the
// envelopes measured at s = 10).
double expected_tiles(bool exact, bool causal, int QT, int qt, double sigma, int s) {
  if (exact) return causal ? qt + 1 : QT;
  const double back = 1.5 * sigma * (1.0 + 0.7 * log((double)std::max(s, 1)));
  const double t = 1.0 + ceil(back / 128.0);
  return causal ? std::min((double)(qt + 1), t) : std::min((double)QT, 2.0 * t - 1.0);
}

struct ItemList {
  std::vector<int4> items, ext, merge;
};

// Items of the tensor-core kernel: two 128-row query tiles sharing one KV
// head.  Heads of a KV group pair up (sorted by sigma so that paired heads
// have similar key envelopes); an odd group's last head pairs its own row
// tiles.  Ordered by expected cost, largest first, so that the dynamic queue
// balances like longest-processing-time scheduling: the key tiles the item
// is expected to run (the diagonal tile plus the look-back of its heads'
// widest bins, clipped at the sequence start), then sigma and row tile.
//
// Key-range split: with split_parts = 0 an item whose expected key tiles
// exceed half the per-SM share of the whole call (at least 2) is cut into
// parts of at most that size, so that the longest-first queue can even the
// SMs out (pieces of a whole share would still leave one SM with a piece plus
// an item); with
// split_parts >= 2 every item is cut into that many parts; 1 never splits.
// The parts of an item follow it in the order and cover consecutive key
// ranges of its envelope.
ItemList build_items(int B, int Hq, int Hkv, int QT, int qt0, int qt1, bool exact, bool causal,
                     int s, int num_sms, int split_parts, const std::vector<double>& sigma) {
  const int G = Hq / Hkv;
  std::vector<int4> items;
  std::vector<double> cost, tiles;
  items.reserve((size_t)B * Hq * (qt1 - qt0) / 2 + B * Hkv);
  for (int b = 0; b < B; ++b) {
    for (int kvh = 0; kvh < Hkv; ++kvh) {
      std::vector<int> heads(G);
      std::iota(heads.begin(), heads.end(), kvh * G);
      if (!exact)
        std::stable_sort(heads.begin(), heads.end(),
                         [&](int x, int y) { return sigma[x] > sigma[y]; });
      for (int pr = 0; pr + 1 < G; pr += 2) {
        const int hA = heads[pr], hB = heads[pr + 1];
        const double sg = exact ? 0.0 : std::max(sigma[hA], sigma[hB]);
        for (int qt = qt0; qt < qt1; ++qt) {
          items.push_back(make_int4(b, hA | (hB << 16), qt, qt));
          cost.push_back(exact ? (double)qt : sg * 1e6 + qt);
          tiles.push_back(expected_tiles(exact, causal, QT, qt, sg, s));
        }
      }
      if (G % 2) {
        const int hL = heads[G - 1];
        const double sg = exact ? 0.0 : sigma[hL];
        for (int qt = qt0; qt < qt1; qt += 2) {
          const int qtB = qt + 1 < qt1 ? qt + 1 : -1;
          items.push_back(make_int4(b, hL | (hL << 16), qt, qtB));
          cost.push_back(exact ? (double)std::max(qt, qtB) : sg * 1e6 + qt);
          tiles.push_back(expected_tiles(exact, causal, QT, std::max(qt, qtB), sg, s) + 1.0);
        }
      }
    }
  }
  // parts per item
  std::vector<int> parts(items.size(), 1);
  if (split_parts >= 2) {
    std::fill(parts.begin(), parts.end(), std::min(split_parts, plsh::kMaxSplitParts));
  } else if (split_parts == 0 && num_sms > 0) {
    double total = 0.0;
    for (double t : tiles) total += t;
    const double cap = std::max(2.0, ceil(0.5 * total / num_sms));
    for (size_t k = 0; k < items.size(); ++k)
      if (tiles[k] > cap)
        parts[k] = (int)std::min((double)plsh::kMaxSplitParts, ceil(tiles[k] / cap));
  }
  std::vector<size_t> order(items.size());
  std::iota(order.begin(), order.end(), 0);
  // longest first by the expected key tiles of a part, then by sigma and
  // row tile
  std::stable_sort(order.begin(), order.end(), [&](size_t x, size_t y) {
    const double tx = tiles[x] / parts[x], ty = tiles[y] / parts[y];
    if (tx != ty) return tx > ty;
    return cost[x] > cost[y];
  });
  ItemList out;
  bool any_split = false;
  for (int pc : parts) any_split = any_split || pc > 1;
  int slot = 0;
  for (size_t k = 0; k < order.size(); ++k) {
    const int4 it = items[order[k]];
    const int pc = parts[order[k]];
    if (pc > 1) {
      out.merge.push_back(it);
      out.merge.push_back(make_int4(slot, pc, 0, 0));
    }
    for (int p = 0; p < pc; ++p) {
      out.items.push_back(it);
      if (any_split) out.ext.push_back(make_int4(p, pc, pc > 1 ? slot + p : -1, 0));
    }
    if (pc > 1) slot += pc;
  }
  return out;
}

// Device copy of the item table for this shape and head order (built and
// uploaded on first use, then reused), with the split parts' extra entries,
// merge list and workspace when some item is split.
struct TableRef {
  const int4* items = nullptr;
  int count = 0;
  const int4* ext = nullptr;
  const int4* merge = nullptr;
  int merges = 0;
  float* ws = nullptr;
  plsh::ItemTable* table = nullptr;   // pinned until table_release
};

// Frees a table's device memory on `st` once the work of every call that
// used it is done (stream-ordered: the host does not wait).
void free_table(plsh::ItemTable& t, cudaStream_t st) {
  for (auto& u : t.uses) {
    cudaStreamWaitEvent(st, u.second, 0);
    cudaEventDestroy(u.second);
  }
  t.uses.clear();
  if (t.ready != nullptr) {
    cudaStreamWaitEvent(st, t.ready, 0);
    cudaEventDestroy(t.ready);
    t.ready = nullptr;
  }
  for (void* q : {(void*)t.dev, (void*)t.dev_ext, (void*)t.dev_merge, (void*)t.ws})
    if (q != nullptr) cudaFreeAsync(q, st);
  t.dev = nullptr;
  t.dev_ext = nullptr;
  t.dev_merge = nullptr;
  t.ws = nullptr;
}

// Ends a call's hold on its table: an event behind the call's work on `st`
// (one per stream that used the table; beyond eight streams the oldest
// entry is taken over once its work is done) and the pin released.
void table_release(TableRef& tab, cudaStream_t st, bool used) {
  if (tab.table == nullptr) return;
  std::lock_guard<std::mutex> lk(g_ctx_mu);
  plsh::ItemTable& t = *tab.table;
  if (used) {
    cudaEvent_t ev = nullptr;
    for (auto& u : t.uses)
      if (u.first == st) ev = u.second;
    if (ev == nullptr) {
      if (t.uses.size() >= 8) {
        cudaEventSynchronize(t.uses.front().second);
        ev = t.uses.front().second;
        t.uses.erase(t.uses.begin());
      } else if (cudaEventCreateWithFlags(&ev, cudaEventDisableTiming) != cudaSuccess) {
        ev = nullptr;
      }
      if (ev != nullptr) t.uses.emplace_back(st, ev);
    }
    if (ev == nullptr || cudaEventRecord(ev, st) != cudaSuccess) {
      // no event to order the free behind: keep the table from eviction
      t.pins += 1;
    }
  }
  t.pins -= 1;
  tab.table = nullptr;
}

// Releases a call's table hold on every path out of the call.
struct TableHold {
  TableRef* tab;
  cudaStream_t st;
  bool used = false;
  ~TableHold() { table_release(*tab, st, used); }
};

plsh_status item_table(plsh::DeviceCtx* ctx, int B, int Hq, int Hkv, int QT, int qt0, int qt1,
                       bool exact, bool causal, int s, const std::vector<double>& sigma,
                       int split_parts, cudaStream_t st, TableRef* out) {
  // the table depends on the shape, the range of query tiles, the split
  // setting and, for the approximate kernel, on the order of sigma inside
  // each KV group and across heads (and on s and sigma through the split)
  std::string key = std::to_string(exact) + ":" + std::to_string(causal) + ":" +
                    std::to_string(B) + ":" + std::to_string(Hq) + ":" + std::to_string(Hkv) +
                    ":" + std::to_string(QT) + ":" + std::to_string(qt0) + "-" +
                    std::to_string(qt1) + ":split" + std::to_string(split_parts);
  if (!exact) {
    std::vector<int> rank(Hq);
    std::iota(rank.begin(), rank.end(), 0);
    std::stable_sort(rank.begin(), rank.end(),
                     [&](int x, int y) { return sigma[x] > sigma[y]; });
    key += ":s" + std::to_string(s) + ":";
    for (int h : rank) key += std::to_string(h) + ",";
    if (split_parts == 0) {
      // the automatic split follows the scales themselves
      char buf[32];
      for (double v : sigma) {
        snprintf(buf, sizeof buf, "%.6g,", v);
        key += buf;
      }
    }
  }
  std::lock_guard<std::mutex> lk(g_ctx_mu);
  auto it = ctx->tables.find(key);
  if (it == ctx->tables.end()) {
    if (ctx->tables.size() >= plsh::kMaxTables) {
      // the least recently used table that no call holds, freed behind the
      // work that used it (if every table is held, the cache grows instead)
      auto victim = ctx->tables.end();
      for (auto jt = ctx->tables.begin(); jt != ctx->tables.end(); ++jt)
        if (jt->second.pins == 0 &&
            (victim == ctx->tables.end() || jt->second.last_use < victim->second.last_use))
          victim = jt;
      if (victim != ctx->tables.end()) {
        free_table(victim->second, st);
        ctx->tables.erase(victim);
      }
    }
    plsh::ItemTable t;
    ItemList lst = build_items(B, Hq, Hkv, QT, qt0, qt1, exact, causal, s, ctx->num_sms,
                               split_parts, sigma);
    t.host = std::move(lst.items);
    t.ext = std::move(lst.ext);
    t.merge = std::move(lst.merge);
    t.home = st;
    int slots = 0;
    for (size_t k = 1; k < t.merge.size(); k += 2) slots += t.merge[k].y;
    plsh_status s1 = dev_alloc_async((void**)&t.dev, sizeof(int4) * t.host.size(), st,
                                     "item table");
    if (s1 == PLSH_OK && !t.ext.empty())
      s1 = dev_alloc_async((void**)&t.dev_ext, sizeof(int4) * t.ext.size(), st, "item table");
    if (s1 == PLSH_OK && !t.merge.empty())
      s1 = dev_alloc_async((void**)&t.dev_merge, sizeof(int4) * t.merge.size(), st, "item table");
    if (s1 == PLSH_OK && slots > 0)
      s1 = dev_alloc_async((void**)&t.ws, sizeof(float) * plsh::kSplitSlotFloats * slots, st,
                           "split workspace");
    if (s1 != PLSH_OK) {
      free_table(t, st);
      return s1;
    }
    cudaError_t e = cudaMemcpyAsync(t.dev, t.host.data(), sizeof(int4) * t.host.size(),
                                    cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !t.ext.empty())
      e = cudaMemcpyAsync(t.dev_ext, t.ext.data(), sizeof(int4) * t.ext.size(),
                          cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess && !t.merge.empty())
      e = cudaMemcpyAsync(t.dev_merge, t.merge.data(), sizeof(int4) * t.merge.size(),
                          cudaMemcpyHostToDevice, st);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&t.ready, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventRecord(t.ready, st);
    if (e != cudaSuccess) {
      free_table(t, st);
      return cuda_fail(e, "item table upload");
    }
    it = ctx->tables.emplace(key, std::move(t)).first;
  } else if (it->second.home != st && it->second.ready != nullptr) {
    // another stream built the table: order this call behind its upload
    PLSH_TRY_CUDA(cudaStreamWaitEvent(st, it->second.ready, 0), "stream wait");
  }
  it->second.last_use = ++ctx->table_clock;
  out->items = it->second.dev;
  out->count = (int)it->second.host.size();
  out->ext = it->second.dev_ext;
  out->merge = it->second.dev_merge;
  out->merges = (int)it->second.merge.size() / 2;
  out->ws = it->second.ws;
  it->second.pins += 1;
  out->table = &it->second;
  return PLSH_OK;
}

enum class Path { Auto, Simt, Tc };

Path path_override();

// The tensor-core backward serves bf16 with d = 128, s <= 16 and at most 64
// query heads per KV head (and a forward statistics pass on the tensor-core
// kernel); everything else takes the CUDA-core backward.
bool bwd_tc_ok(const plsh_tensor* Q, const plsh_tensor* K, const plsh_bins* bins, int causal) {
  return path_override() != Path::Simt && Q->dtype == PLSH_BF16 && Q->d == 128 &&
         bins->s <= plsh::kBwdTcMaxS && Q->H / K->H <= plsh::kBwdTcMaxGroup &&
         plsh::attn_tc_smem_bytes(bins->s, causal, 0) <= 232448;
}

// The tensor-core kernel serves bf16 with d = 128 and s within its shared
// memory; everything else takes the CUDA-core kernel.
bool tc_path_ok(int dtype, int64_t d, int s, int causal, int exact) {
  return dtype == PLSH_BF16 && (d == 128 || d == 64) &&
         plsh::attn_tc_smem_bytes(s, causal, exact) <= 232448;
}

// Status of the device error word: bit 0 a bounded wait ran out, bit 1 a
// value of V beyond f16's range on the tensor-core path.
plsh_status device_flag_status(int flag) {
  if (flag & 1) return fail(PLSH_ERR_TIMEOUT, "a device-side wait ran out of time");
  if (flag & 2)
    return fail(PLSH_ERR_RANGE, "V holds a value beyond +-65504, which the tensor-core path "
                                "takes in f16 (scale V down by a power of two: O scales with it)");
  return PLSH_OK;
}

Path path_override() {
  const char* p = getenv("PLSH_PATH");
  if (p == nullptr) return Path::Auto;
  if (strcmp(p, "simt") == 0) return Path::Simt;
  if (strcmp(p, "tc") == 0) return Path::Tc;
  return Path::Auto;
}

plsh_status run_attention(const plsh_tensor* Q, const plsh_tensor* K, const plsh_tensor* V,
                          plsh_tensor* O, int causal, const plsh_bins* bins,
                          const float* slopes, cudaStream_t st, int qt0 = 0, int qt1 = -1,
                          float* lse = nullptr) {
  plsh::DeviceCtx* ctx = nullptr;
  plsh_status s0 = current_ctx(&ctx);
  if (s0 != PLSH_OK) return s0;
  plsh::AttnArgs a;
  memset(&a, 0, sizeof a);
  a.Q = Q->data;
  a.K = K->data;
  a.V = V->data;
  a.O = O->data;
  a.B = (int)Q->B;
  a.Hq = (int)Q->H;
  a.Hkv = (int)K->H;
  a.n = (int)Q->n;
  a.d = (int)Q->d;
  a.causal = causal ? 1 : 0;
  a.exact = bins == nullptr ? 1 : 0;
  if (bins) {
    a.rec = bins->d_rec;
    a.s = bins->s;
    a.W = bins->W;
  }
  a.err = ctx->d_err;
  a.wait_ns = ctx->wait_ns;
  a.stall = fault_is("stall") ? 1 : 0;
  {
    std::lock_guard<std::mutex> lk(g_ctx_mu);
    a.queue = ctx->d_queue + 2 * (ctx->slot_counter++ % plsh::kQueueSlots);
  }
  const bool tc_ok = tc_path_ok(Q->dtype, Q->d, a.s, a.causal, a.exact);
  Path path = path_override();
  if (path == Path::Auto) path = tc_ok ? Path::Tc : Path::Simt;
  if (path == Path::Tc && !tc_ok)
    return fail(PLSH_ERR_UNSUPPORTED, "tensor-core path needs bf16, d = 128 and s within "
                                      "its shared-memory budget");
  if (lse != nullptr && path != Path::Tc)
    return fail(PLSH_ERR_UNSUPPORTED, "the log-sum-exp output is written by the tensor-core "
                                      "path only (bf16, d = 128)");
  a.lse = lse;
  TableRef tab;
  TableHold hold{&tab, st};
  if (path == Path::Tc) {
    const int QT = (int)((Q->n + 127) / 128);
    plsh_status s1 = item_table(ctx, a.B, a.Hq, a.Hkv, QT, qt0, qt1 < 0 ? QT : qt1, a.exact != 0,
                                a.causal != 0, a.s,
                                bins ? bins->sigma_host : std::vector<double>(),
                                ctx->split_parts, st, &tab);
    if (s1 != PLSH_OK) return s1;
    a.items = tab.items;
    a.num_items = tab.count;
    a.item_ext = tab.ext;
    a.split_ws = tab.ws;
  }
  hold.used = true;
  cudaError_t e = path == Path::Tc ? plsh::launch_attn_tc(a, slopes, ctx->num_sms, st)
                                   : plsh::launch_attn_simt(a, slopes, Q->dtype, st);
  if (e != cudaSuccess) return cuda_fail(e, "attention launch");
  if (path == Path::Tc && tab.merges > 0) {
    e = plsh::launch_split_merge(tab.merge, tab.merges, tab.ws, a.O, a.lse, a.Hq, a.n, a.d, st);
    if (e != cudaSuccess) return cuda_fail(e, "split merge launch");
  }
  return PLSH_OK;
}

}  // namespace

// ------------------------------------------------------- allocation-free path
// plsh_alibi_attn_noalloc keeps its scratch (work-queue counters and the
// work-item table of the tensor-core kernel) in this fixed device array
// instead of library-allocated memory.  Element 0 holds {next item, finished
// CTAs, device error flag, unused}; elements 1.. hold the items.  Every call
// on a device uses the same array.
constexpr int kNoAllocMaxItems = 65536;
static __device__ __align__(256) int4 g_noalloc_scratch[1 + kNoAllocMaxItems];

// Device address of g_noalloc_scratch per device, resolved once per device.
int4* g_noalloc_addr[kMaxDevices] = {};
std::mutex g_noalloc_mu;

constexpr int kNoAllocMaxUnits = 512;

// Wait limit of the allocation-free path per device (set with
// plsh_set_wait_limit_ns; kept apart from the per-device context, whose
// creation allocates).
std::atomic<uint64_t> g_noalloc_wait_ns[kMaxDevices];

// Work units in cost order: a pair of heads of one KV group (every row tile
// is an item), or the last head of an odd group (pairs of its row tiles).
// Consecutive units of equal cost form a run whose items interleave.
struct NoAllocUnits {
  int count;
  int unit[kNoAllocMaxUnits];   // hA | hB << 10 | leftover << 20 | run start << 21
};

// One thread per work item: writes the item table the tensor-core kernel
// reads, in the order of the ordinary entry point's table: runs in cost
// order; inside a run, row tiles from the last (the most keys under the
// causal mask) down, then batch elements, then units.  Thread 0 also clears
// the queue counters (not the error word, which persists until read).
__global__ void noalloc_items_kernel(int4* scratch, const __grid_constant__ NoAllocUnits u,
                                     int B, int QT, int num_items) {
  const int idx = blockIdx.x * blockDim.x + threadIdx.x;
  if (idx == 0) {
    reinterpret_cast<int*>(scratch)[0] = 0;
    reinterpret_cast<int*>(scratch)[1] = 0;
  }
  if (idx >= num_items) return;
  int off = idx;
  for (int k = 0; k < u.count;) {
    int R = 1;
    while (k + R < u.count && !((u.unit[k + R] >> 21) & 1)) ++R;
    const bool leftover = (u.unit[k] >> 20) & 1;
    const int levels = leftover ? (QT + 1) / 2 : QT;
    if (off < R * B * levels) {
      const int lvl = off / (R * B), rem = off % (R * B);
      const int b = rem / R, code = u.unit[k + rem % R];
      const int q = levels - 1 - lvl;
      const int hA = code & 1023, hB = (code >> 10) & 1023;
      const int qtA = leftover ? 2 * q : q;
      const int qtB = leftover ? (2 * q + 1 < QT ? 2 * q + 1 : -1) : q;
      scratch[1 + idx] = make_int4(b, hA | (hB << 16), qtA, qtB);
      return;
    }
    off -= R * B * levels;
    k += R;
  }
}

namespace plsh {
// sampler.cu: fixed blocks, width d_w[hs] and offset d_u[hs] (integers) for
// every hash (declared here: only the entry point below launches it)
cudaError_t launch_bins_fixed(plsh_bins* b, cudaStream_t st);
// bias.cu: ||L* - M~|| in max and spectral norm for one head
cudaError_t bias_error(const plsh_bins* bn, double sigma, int h, int iters, uint64_t seed,
                       double* max_abs, double* spectral, cudaStream_t st);
// bwd.cu: gradients of the approximation
cudaError_t launch_attn_bwd(const void* Q, const void* K, const void* V, const void* dO, void* dQ,
                            void* dK, void* dV, float* stats, const plsh_bins* bn, int B, int Hq,
                            int Hkv, int n, int d, int causal, int dtype, cudaStream_t st);
}  // namespace plsh

extern "C" {

plsh_status plsh_sample_bins(int64_t n, const double* sigma_h, int32_t H, int32_t s,
                             uint64_t seed, void* stream, plsh_bins** out) {
  if (out == nullptr) return fail(PLSH_ERR_INVALID, "out is NULL");
  if (n < 1 || n >= ((int64_t)1 << 31)) return fail(PLSH_ERR_INVALID, "n must be in [1, 2^31)");
  if (H < 1) return fail(PLSH_ERR_INVALID, "H must be >= 1");
  if (s < 1 || s > plsh::kMaxS) return fail(PLSH_ERR_INVALID, "s must be in [1, 64]");
  plsh_status st = check_sigma(sigma_h, H);
  if (st != PLSH_OK) return st;
  plsh::DeviceCtx* ctx = nullptr;
  if ((st = current_ctx(&ctx)) != PLSH_OK) return st;
  plsh_bins* b = nullptr;
  if ((st = new_bins(n, H, s, &b)) != PLSH_OK) return st;
  if ((st = resample(b, sigma_h, seed, (cudaStream_t)stream)) != PLSH_OK) {
    free_bins(b);
    return st;
  }
  *out = b;
  return PLSH_OK;
}

plsh_status plsh_bins_resample(plsh_bins* bins, const double* sigma_h, uint64_t seed,
                               void* stream) {
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  plsh_status st = check_sigma(sigma_h, bins->H);
  if (st != PLSH_OK) return st;
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  return resample(bins, sigma_h, seed, (cudaStream_t)stream);
}

plsh_status plsh_bins_from_host(int64_t n, int32_t H, int32_t s, const int64_t* offsets,
                                const int32_t* starts, void* stream, plsh_bins** out) {
  if (out == nullptr || offsets == nullptr || starts == nullptr)
    return fail(PLSH_ERR_INVALID, "NULL argument");
  if (n < 1 || n >= ((int64_t)1 << 31)) return fail(PLSH_ERR_INVALID, "n must be in [1, 2^31)");
  if (H < 1) return fail(PLSH_ERR_INVALID, "H must be >= 1");
  if (s < 1 || s > plsh::kMaxS) return fail(PLSH_ERR_INVALID, "s must be in [1, 64]");
  const int64_t HS = (int64_t)H * s;
  if (offsets[0] != 0) return fail(PLSH_ERR_INVALID, "offsets[0] must be 0");
  std::vector<double> sigma_est(H, 0.0);
  for (int64_t hs = 0; hs < HS; ++hs) {
    const int64_t o0 = offsets[hs], o1 = offsets[hs + 1];
    if (o1 - o0 < 2 || o1 - o0 > n + 1)
      return fail(PLSH_ERR_INVALID, "hash " + std::to_string(hs) + ": needs 2..n+1 entries");
    if (starts[o0] != 0) return fail(PLSH_ERR_INVALID, "hash " + std::to_string(hs) + ": first start must be 0");
    if (starts[o1 - 1] != n) return fail(PLSH_ERR_INVALID, "hash " + std::to_string(hs) + ": last entry must be n");
    for (int64_t e = o0 + 1; e < o1; ++e)
      if (starts[e] <= starts[e - 1])
        return fail(PLSH_ERR_INVALID, "hash " + std::to_string(hs) + ": starts must strictly increase");
    // mean bin width of a Gamma(2, sigma) draw is 2 sigma: a cost estimate
    sigma_est[hs / s] += (double)n / (double)(o1 - o0 - 1) / (2.0 * s);
  }
  const int64_t total = offsets[HS];
  plsh::DeviceCtx* ctx = nullptr;
  plsh_status st = current_ctx(&ctx);
  if (st != PLSH_OK) return st;
  plsh_bins* b = nullptr;
  if ((st = new_bins(n, H, s, &b)) != PLSH_OK) return st;
  b->sigma_host = sigma_est;
  order_heads(b);
  cudaStream_t cs = (cudaStream_t)stream;
  int32_t* d_starts = nullptr;
  int64_t* d_off = nullptr;
  if ((st = dev_alloc((void**)&d_starts, sizeof(int32_t) * total, "starts upload")) != PLSH_OK ||
      (st = dev_alloc((void**)&d_off, sizeof(int64_t) * (HS + 1), "offsets upload")) != PLSH_OK) {
    cudaFree(d_starts);
    free_bins(b);
    return st;
  }
  cudaError_t e = cudaMemcpyAsync(d_starts, starts, sizeof(int32_t) * total, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(d_off, offsets, sizeof(int64_t) * (HS + 1), cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(b->d_head_order, b->head_order.data(), sizeof(int32_t) * H, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemsetAsync(b->d_w, 0, sizeof(double) * HS, cs);
  if (e == cudaSuccess) e = cudaMemsetAsync(b->d_u, 0, sizeof(double) * HS, cs);
  if (e == cudaSuccess) e = plsh::launch_bins_from_starts(b, d_starts, d_off, total, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  cudaFree(d_starts);
  cudaFree(d_off);
  if (e != cudaSuccess) {
    free_bins(b);
    return cuda_fail(e, "bins upload");
  }
  *out = b;
  return PLSH_OK;
}

plsh_status plsh_bins_fixed(int64_t n, const int32_t* width_h, int32_t H, int32_t s,
                            void* stream, plsh_bins** out) {
  if (out == nullptr || width_h == nullptr) return fail(PLSH_ERR_INVALID, "NULL argument");
  if (n < 1 || n >= ((int64_t)1 << 31)) return fail(PLSH_ERR_INVALID, "n must be in [1, 2^31)");
  if (H < 1) return fail(PLSH_ERR_INVALID, "H must be >= 1");
  if (s < 1 || s > plsh::kMaxS) return fail(PLSH_ERR_INVALID, "s must be in [1, 64]");
  for (int32_t h = 0; h < H; ++h)
    if (width_h[h] < 1) return fail(PLSH_ERR_INVALID, "width_h[" + std::to_string(h) + "] must be >= 1");
  const int64_t HS = (int64_t)H * s;
  std::vector<double> w(HS), u(HS), sigma_est(H);
  for (int32_t h = 0; h < H; ++h) {
    // s grids shifted evenly across one block; blocks of width w cost like
    // random bins of mean width 2 sigma
    sigma_est[h] = 0.5 * width_h[h];
    for (int32_t t = 0; t < s; ++t) {
      w[(int64_t)h * s + t] = (double)width_h[h];
      u[(int64_t)h * s + t] = (double)((int64_t)t * width_h[h] / s);
    }
  }
  plsh::DeviceCtx* ctx = nullptr;
  plsh_status st = current_ctx(&ctx);
  if (st != PLSH_OK) return st;
  plsh_bins* b = nullptr;
  if ((st = new_bins(n, H, s, &b)) != PLSH_OK) return st;
  b->sigma_host = sigma_est;
  order_heads(b);
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = cudaMemcpyAsync(b->d_w, w.data(), sizeof(double) * HS, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(b->d_u, u.data(), sizeof(double) * HS, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaMemcpyAsync(b->d_head_order, b->head_order.data(), sizeof(int32_t) * H, cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = plsh::launch_bins_fixed(b, cs);
  // the host arrays above go out of scope: wait for the copies
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) {
    free_bins(b);
    return cuda_fail(e, "fixed bins");
  }
  *out = b;
  return PLSH_OK;
}

// The backward pass; O and lse (the forward's output and log-sum-exp) are
// null when the row statistics are to be recomputed.
plsh_status backward_impl(const plsh_tensor* Q, const plsh_tensor* K, const plsh_tensor* V,
                          const plsh_tensor* O, const float* lse, const plsh_tensor* dO,
                          const plsh_bins* bins, int32_t causal, plsh_tensor* dQ,
                          plsh_tensor* dK, plsh_tensor* dV, void* stream) {
  plsh_status st = check_qkvo(Q, K, V, dO);
  if (st != PLSH_OK) return st;
  if (O != nullptr) {
    if ((st = check_tensor(O, "O")) != PLSH_OK) return st;
    if (O->dtype != Q->dtype || O->B != Q->B || O->H != Q->H || O->n != Q->n || O->d != Q->d)
      return fail(PLSH_ERR_INVALID, "O must have Q's shape and dtype");
    if (lse == nullptr) return fail(PLSH_ERR_INVALID, "lse is NULL");
  }
  if ((st = check_tensor(dQ, "dQ")) != PLSH_OK || (st = check_tensor(dK, "dK")) != PLSH_OK ||
      (st = check_tensor(dV, "dV")) != PLSH_OK)
    return st;
  if (dQ->dtype != Q->dtype || dK->dtype != Q->dtype || dV->dtype != Q->dtype)
    return fail(PLSH_ERR_INVALID, "dQ, dK and dV must have Q's dtype");
  if (dQ->B != Q->B || dQ->H != Q->H || dQ->n != Q->n || dQ->d != Q->d)
    return fail(PLSH_ERR_INVALID, "dQ must have Q's shape");
  if (dK->B != K->B || dK->H != K->H || dK->n != K->n || dK->d != K->d ||
      dV->B != K->B || dV->H != K->H || dV->n != K->n || dV->d != K->d)
    return fail(PLSH_ERR_INVALID, "dK and dV must have K's shape");
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (bins->n != Q->n) return fail(PLSH_ERR_INVALID, "bins were drawn for another n");
  if (bins->H != Q->H) return fail(PLSH_ERR_INVALID, "bins were drawn for another number of heads");
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  cudaStream_t cs = (cudaStream_t)stream;
  float* stats = nullptr;
  const size_t bytes = sizeof(float) * 3 * (size_t)Q->B * Q->H * Q->n;
  const bool tc = bwd_tc_ok(Q, K, bins, causal ? 1 : 0);
  if (O != nullptr && !tc)
    return fail(PLSH_ERR_UNSUPPORTED, "the backward pass from a saved O and log-sum-exp runs on "
                                      "the tensor cores only (bf16, d = 128, s <= 16)");
  if (tc) {
    // tensor cores: the rows' -lse and Delta = dO . O (from the saved O and
    // lse, or from the forward kernel in its row statistics mode), then the
    // backward kernel
    plsh::DeviceCtx* ctx = nullptr;
    if ((st = current_ctx(&ctx)) != PLSH_OK) return st;
    const size_t stat_floats = (2 * (size_t)Q->B * Q->H * Q->n + 63) & ~(size_t)63;
    const size_t acc_bytes = sizeof(float) * (size_t)Q->B * Q->H * Q->n * Q->d;
    std::lock_guard<std::mutex> bk(g_bwd_mu);
    if ((st = scratch_acquire(&ctx->bwd_work, &ctx->bwd_work_bytes, &ctx->bwd_ev,
                              sizeof(float) * stat_floats + acc_bytes, cs, "backward scratch")) !=
        PLSH_OK)
      return st;
    stats = ctx->bwd_work;
    float* dq_acc = ctx->bwd_work + stat_floats;
    cudaError_t e = cudaSuccess;
    plsh::AttnArgs a;
    memset(&a, 0, sizeof a);
    a.Q = Q->data;
    a.K = K->data;
    a.V = V->data;
    a.O = nullptr;
    a.B = (int)Q->B;
    a.Hq = (int)Q->H;
    a.Hkv = (int)K->H;
    a.n = (int)Q->n;
    a.d = (int)Q->d;
    a.causal = causal ? 1 : 0;
    a.rec = bins->d_rec;
    a.s = bins->s;
    a.W = bins->W;
    a.err = ctx->d_err;
    a.wait_ns = ctx->wait_ns;
    a.stats = stats;
    a.dO = dO->data;
    {
      std::lock_guard<std::mutex> lk(g_ctx_mu);
      a.queue = ctx->d_queue + 2 * (ctx->slot_counter++ % plsh::kQueueSlots);
    }
    int* bq = nullptr;
    {
      std::lock_guard<std::mutex> lk(g_ctx_mu);
      bq = ctx->d_queue + 2 * (ctx->slot_counter++ % plsh::kQueueSlots);
    }
    const int QT = (int)((Q->n + 127) / 128);
    TableRef tab;
    TableHold hold{&tab, cs};
    hold.used = true;
    plsh_status s1 = item_table(ctx, a.B, a.Hq, a.Hkv, QT, 0, QT, false, a.causal != 0, a.s,
                                bins->sigma_host, 1, cs, &tab);
    if (s1 == PLSH_OK) {
      a.items = tab.items;
      a.num_items = tab.count;
      if (O != nullptr)
        e = plsh::launch_bwd_delta(O->data, dO->data, lse, stats, dq_acc,
                                   (int64_t)a.B * a.Hq * a.n, cs);
      else
        e = plsh::launch_attn_tc(a, nullptr, ctx->num_sms, cs);
      if (e == cudaSuccess)
        e = plsh::launch_attn_bwd_tc(Q->data, K->data, V->data, dO->data, dQ->data, dK->data,
                                     dV->data, stats, dq_acc, O == nullptr, bins, a.B, a.Hq,
                                     a.Hkv, a.n, a.causal, bq, ctx->d_err, ctx->wait_ns,
                                     ctx->num_sms, cs);
    }
    const cudaError_t er = cudaEventRecord(ctx->bwd_ev, cs);
    if (s1 != PLSH_OK) return s1;
    if (e == cudaSuccess) e = er;
    PLSH_TRY_CUDA(e, "backward launch");
    return PLSH_OK;
  }
  plsh::DeviceCtx* ctx = nullptr;
  if ((st = current_ctx(&ctx)) != PLSH_OK) return st;
  std::lock_guard<std::mutex> bk(g_bwd_mu);
  if ((st = scratch_acquire(&ctx->bwd_work, &ctx->bwd_work_bytes, &ctx->bwd_ev, bytes, cs,
                            "backward scratch")) != PLSH_OK)
    return st;
  stats = ctx->bwd_work;
  cudaError_t e = plsh::launch_attn_bwd(Q->data, K->data, V->data, dO->data, dQ->data, dK->data,
                                        dV->data, stats, bins, (int)Q->B, (int)Q->H, (int)K->H,
                                        (int)Q->n, (int)Q->d, causal ? 1 : 0, Q->dtype, cs);
  const cudaError_t er = cudaEventRecord(ctx->bwd_ev, cs);
  if (e == cudaSuccess) e = er;
  PLSH_TRY_CUDA(e, "backward launch");
  return PLSH_OK;
}

plsh_status plsh_alibi_attn_backward(const plsh_tensor* Q, const plsh_tensor* K,
                                     const plsh_tensor* V, const plsh_tensor* dO,
                                     const plsh_bins* bins, int32_t causal, plsh_tensor* dQ,
                                     plsh_tensor* dK, plsh_tensor* dV, void* stream) {
  return backward_impl(Q, K, V, nullptr, nullptr, dO, bins, causal, dQ, dK, dV, stream);
}

plsh_status plsh_alibi_attn_backward_lse(const plsh_tensor* Q, const plsh_tensor* K,
                                         const plsh_tensor* V, const plsh_tensor* O,
                                         const float* lse, const plsh_tensor* dO,
                                         const plsh_bins* bins, int32_t causal, plsh_tensor* dQ,
                                         plsh_tensor* dK, plsh_tensor* dV, void* stream) {
  if (O == nullptr) return fail(PLSH_ERR_INVALID, "O is NULL");
  return backward_impl(Q, K, V, O, lse, dO, bins, causal, dQ, dK, dV, stream);
}

plsh_status plsh_bias_error(const plsh_bins* bins, double sigma, int32_t h,
                            int32_t lanczos_iters, uint64_t seed, double* max_abs,
                            double* spectral, void* stream) {
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (max_abs == nullptr && spectral == nullptr)
    return fail(PLSH_ERR_INVALID, "nothing to compute: max_abs and spectral are NULL");
  if (!(sigma > 0.0) || !isfinite(sigma)) return fail(PLSH_ERR_INVALID, "sigma must be finite and > 0");
  if (h < 0 || h >= bins->H) return fail(PLSH_ERR_INVALID, "h must be in [0, H)");
  if (spectral != nullptr && (lanczos_iters < 2 || lanczos_iters > 1000))
    return fail(PLSH_ERR_INVALID, "lanczos_iters must be in [2, 1000]");
  plsh_status st = check_bins_device(bins);
  if (st != PLSH_OK) return st;
  PLSH_TRY_CUDA(plsh::bias_error(bins, sigma, h, lanczos_iters, seed, max_abs, spectral,
                                 (cudaStream_t)stream),
                "bias error");
  return PLSH_OK;
}

plsh_status plsh_bins_share_groups(const plsh_bins* src, int32_t Hq, void* stream,
                                   plsh_bins** out) {
  if (src == nullptr || out == nullptr) return fail(PLSH_ERR_INVALID, "NULL argument");
  if (Hq < 1 || Hq % src->H != 0)
    return fail(PLSH_ERR_INVALID, "Hq must be a positive multiple of the source's heads");
  plsh_status st = check_bins_device(src);
  if (st != PLSH_OK) return st;
  plsh_bins* b = nullptr;
  if ((st = new_bins(src->n, Hq, src->s, &b)) != PLSH_OK) return st;
  const int32_t group = Hq / src->H;
  const int64_t s = src->s;
  b->sigma_host.resize(Hq);
  for (int32_t h = 0; h < Hq; ++h) b->sigma_host[h] = src->sigma_host[h / group];
  order_heads(b);
  cudaStream_t cs = (cudaStream_t)stream;
  cudaError_t e = cudaSuccess;
  // head h takes every record, draw and scale of head h / group of src
  for (int32_t h = 0; h < Hq && e == cudaSuccess; ++h) {
    const int32_t g = h / group;
    e = cudaMemcpyAsync(b->d_rec + (int64_t)h * s * b->W, src->d_rec + (int64_t)g * s * src->W,
                        sizeof(plsh::BinRecord) * s * src->W, cudaMemcpyDeviceToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(b->d_w + h * s, src->d_w + g * s, sizeof(double) * s,
                          cudaMemcpyDeviceToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(b->d_u + h * s, src->d_u + g * s, sizeof(double) * s,
                          cudaMemcpyDeviceToDevice, cs);
    if (e == cudaSuccess)
      e = cudaMemcpyAsync(b->d_sigma + h, src->d_sigma + g, sizeof(double),
                          cudaMemcpyDeviceToDevice, cs);
  }
  if (e == cudaSuccess)
    e = cudaMemcpyAsync(b->d_head_order, b->head_order.data(), sizeof(int32_t) * Hq,
                        cudaMemcpyHostToDevice, cs);
  if (e == cudaSuccess) e = cudaStreamSynchronize(cs);
  if (e != cudaSuccess) {
    free_bins(b);
    return cuda_fail(e, "shared bins");
  }
  b->sigma_on_device = true;
  *out = b;
  return PLSH_OK;
}

plsh_status plsh_bins_info(const plsh_bins* bins, int64_t* n, int32_t* H, int32_t* s,
                           int64_t* n_entries, void* stream) {
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (n) *n = bins->n;
  if (H) *H = bins->H;
  if (s) *s = bins->s;
  if (n_entries) {
    plsh_status st = check_bins_device(bins);
    if (st != PLSH_OK) return st;
    std::vector<int64_t> off;
    std::vector<int32_t> starts;
    if ((st = records_to_host(bins, (cudaStream_t)stream, &off, &starts)) != PLSH_OK) return st;
    *n_entries = (int64_t)starts.size();
  }
  return PLSH_OK;
}

plsh_status plsh_bins_to_host(const plsh_bins* bins, int64_t* offsets, int32_t* starts,
                              int64_t cap, void* stream) {
  if (bins == nullptr || offsets == nullptr || starts == nullptr)
    return fail(PLSH_ERR_INVALID, "NULL argument");
  plsh_status st = check_bins_device(bins);
  if (st != PLSH_OK) return st;
  std::vector<int64_t> off;
  std::vector<int32_t> st_list;
  if ((st = records_to_host(bins, (cudaStream_t)stream, &off, &st_list)) != PLSH_OK) return st;
  if ((int64_t)st_list.size() > cap)
    return fail(PLSH_ERR_INVALID, "starts buffer too small: need " + std::to_string(st_list.size()));
  memcpy(offsets, off.data(), sizeof(int64_t) * off.size());
  memcpy(starts, st_list.data(), sizeof(int32_t) * st_list.size());
  return PLSH_OK;
}

plsh_status plsh_bins_draws(const plsh_bins* bins, double* w, double* u, void* stream) {
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  plsh_status st = check_bins_device(bins);
  if (st != PLSH_OK) return st;
  const size_t HS = (size_t)bins->H * bins->s;
  cudaStream_t cs = (cudaStream_t)stream;
  if (w) PLSH_TRY_CUDA(cudaMemcpyAsync(w, bins->d_w, sizeof(double) * HS, cudaMemcpyDeviceToHost, cs), "copy w");
  if (u) PLSH_TRY_CUDA(cudaMemcpyAsync(u, bins->d_u, sizeof(double) * HS, cudaMemcpyDeviceToHost, cs), "copy u");
  PLSH_TRY_CUDA(cudaStreamSynchronize(cs), "cudaStreamSynchronize");
  return PLSH_OK;
}

void plsh_bins_free(plsh_bins* bins) { free_bins(bins); }

plsh_status plsh_alibi_attn(const plsh_tensor* Q, const plsh_tensor* K, const plsh_tensor* V,
                            const plsh_bins* bins, int32_t causal, plsh_tensor* O,
                            void* stream) {
  plsh_status st = check_qkvo(Q, K, V, O);
  if (st != PLSH_OK) return st;
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (bins->n != Q->n) return fail(PLSH_ERR_INVALID, "bins were drawn for another n");
  if (bins->H != Q->H) return fail(PLSH_ERR_INVALID, "bins were drawn for another number of heads");
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  return run_attention(Q, K, V, O, causal, bins, nullptr, (cudaStream_t)stream);
}

plsh_status plsh_alibi_attn_lse(const plsh_tensor* Q, const plsh_tensor* K, const plsh_tensor* V,
                                const plsh_bins* bins, int32_t causal, plsh_tensor* O, float* lse,
                                void* stream) {
  plsh_status st = check_qkvo(Q, K, V, O);
  if (st != PLSH_OK) return st;
  if (lse == nullptr) return fail(PLSH_ERR_INVALID, "lse is NULL");
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (bins->n != Q->n) return fail(PLSH_ERR_INVALID, "bins were drawn for another n");
  if (bins->H != Q->H) return fail(PLSH_ERR_INVALID, "bins were drawn for another number of heads");
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  return run_attention(Q, K, V, O, causal, bins, nullptr, (cudaStream_t)stream, 0, -1, lse);
}

plsh_status plsh_alibi_attn_host(const plsh_tensor* Q, const plsh_tensor* K,
                                 const plsh_tensor* V, const plsh_bins* bins, int32_t causal,
                                 plsh_tensor* O, void* stream) {
  plsh_status st = check_qkvo(Q, K, V, O);
  if (st != PLSH_OK) return st;
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (bins->n != Q->n) return fail(PLSH_ERR_INVALID, "bins were drawn for another n");
  if (bins->H != Q->H) return fail(PLSH_ERR_INVALID, "bins were drawn for another number of heads");
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  plsh::DeviceCtx* ctx = nullptr;
  if ((st = current_ctx(&ctx)) != PLSH_OK) return st;
  cudaStream_t cs = (cudaStream_t)stream;
  const size_t esz = Q->dtype == PLSH_BF16 ? 2 : 4;
  const int64_t n = Q->n, d = Q->d;
  const size_t row = (size_t)d * esz;                       // bytes of one token row
  const size_t bytes[4] = {(size_t)(Q->B * Q->H * n) * row, (size_t)(K->B * K->H * n) * row,
                           (size_t)(V->B * V->H * n) * row, (size_t)(O->B * O->H * n) * row};
  {
    std::lock_guard<std::mutex> lk(g_ctx_mu);
    if (ctx->h2d == nullptr) {
      PLSH_TRY_CUDA(cudaStreamCreateWithFlags(&ctx->h2d, cudaStreamNonBlocking), "copy stream");
      PLSH_TRY_CUDA(cudaStreamCreateWithFlags(&ctx->d2h, cudaStreamNonBlocking), "copy stream");
      for (cudaEvent_t& e : ctx->ev)
        PLSH_TRY_CUDA(cudaEventCreateWithFlags(&e, cudaEventDisableTiming), "event");
    }
    // this call follows the previous one (its last copy out recorded ev[1];
    // an event never recorded is no wait): the staging buffers are free
    // then, and grow in stream order without synchronising the device
    PLSH_TRY_CUDA(cudaStreamWaitEvent(cs, ctx->ev[1], 0), "stream wait");
    for (int k = 0; k < 4; ++k) {
      if (ctx->stage_bytes[k] >= bytes[k]) continue;
      if (ctx->stage[k] != nullptr) PLSH_TRY_CUDA(cudaFreeAsync(ctx->stage[k], cs), "host staging");
      ctx->stage[k] = nullptr;
      ctx->stage_bytes[k] = 0;
      if ((st = dev_alloc_async(&ctx->stage[k], bytes[k], cs, "host staging")) != PLSH_OK)
        return st;
      ctx->stage_bytes[k] = bytes[k];
    }
  }
  plsh_tensor dQ = *Q, dK = *K, dV = *V, dO = *O;
  dQ.data = ctx->stage[0];
  dK.data = ctx->stage[1];
  dV.data = ctx->stage[2];
  dO.data = ctx->stage[3];
  // query rows in up to kMaxHostChunks chunks on the tensor-core path (one
  // otherwise): the copies of chunk c + 1 in and chunk c - 1 out overlap the
  // kernel on chunk c; without the causal mask every chunk needs all keys
  const int QT = (int)((n + 127) / 128);
  const bool tc = tc_path_ok(Q->dtype, Q->d, bins->s, causal ? 1 : 0, 0) &&
                  path_override() != Path::Simt;
  const int nchunk = tc ? std::min(plsh::kMaxHostChunks, QT) : 1;
  const int tpc = (QT + nchunk - 1) / nchunk;
  const bool kv_chunked = causal && nchunk > 1;
  cudaEvent_t ev_start = ctx->ev[0], ev_done = ctx->ev[1];
  // the staging buffers are free once everything queued on the stream is
  PLSH_TRY_CUDA(cudaEventRecord(ev_start, cs), "event");
  PLSH_TRY_CUDA(cudaStreamWaitEvent(ctx->h2d, ev_start, 0), "stream wait");
  PLSH_TRY_CUDA(cudaStreamWaitEvent(ctx->d2h, ev_start, 0), "stream wait");
  auto rows_copy = [&](void* dst, const void* src, int64_t heads, int64_t r0, int64_t r1,
                       cudaMemcpyKind kind, cudaStream_t s2) -> cudaError_t {
    // rows [r0, r1) of every (b, h): one strided copy
    const size_t pitch = (size_t)n * row;
    return cudaMemcpy2DAsync(static_cast<char*>(dst) + r0 * row, pitch,
                             static_cast<const char*>(src) + r0 * row, pitch,
                             (size_t)(r1 - r0) * row, (size_t)heads, kind, s2);
  };
  if (!kv_chunked) {
    PLSH_TRY_CUDA(cudaMemcpyAsync(dK.data, K->data, bytes[1], cudaMemcpyHostToDevice, ctx->h2d),
                  "copy K");
    PLSH_TRY_CUDA(cudaMemcpyAsync(dV.data, V->data, bytes[2], cudaMemcpyHostToDevice, ctx->h2d),
                  "copy V");
  }
  for (int c = 0; c < nchunk; ++c) {
    const int qt0 = c * tpc, qt1 = std::min(QT, (c + 1) * tpc);
    if (qt0 >= qt1) break;
    const int64_t r0 = (int64_t)qt0 * 128, r1 = std::min(n, (int64_t)qt1 * 128);
    cudaEvent_t ev_in = ctx->ev[2 + 2 * c], ev_out = ctx->ev[3 + 2 * c];
    PLSH_TRY_CUDA(rows_copy(dQ.data, Q->data, Q->B * Q->H, r0, r1, cudaMemcpyHostToDevice,
                            ctx->h2d), "copy Q rows");
    if (kv_chunked) {
      PLSH_TRY_CUDA(rows_copy(dK.data, K->data, K->B * K->H, r0, r1, cudaMemcpyHostToDevice,
                              ctx->h2d), "copy K rows");
      PLSH_TRY_CUDA(rows_copy(dV.data, V->data, V->B * V->H, r0, r1, cudaMemcpyHostToDevice,
                              ctx->h2d), "copy V rows");
    }
    PLSH_TRY_CUDA(cudaEventRecord(ev_in, ctx->h2d), "event");
    PLSH_TRY_CUDA(cudaStreamWaitEvent(cs, ev_in, 0), "stream wait");
    if ((st = run_attention(&dQ, &dK, &dV, &dO, causal, bins, nullptr, cs,
                            tc ? qt0 : 0, tc ? qt1 : -1)) != PLSH_OK)
      return st;
    PLSH_TRY_CUDA(cudaEventRecord(ev_out, cs), "event");
    PLSH_TRY_CUDA(cudaStreamWaitEvent(ctx->d2h, ev_out, 0), "stream wait");
    PLSH_TRY_CUDA(rows_copy(O->data, dO.data, O->B * O->H, r0, r1, cudaMemcpyDeviceToHost,
                            ctx->d2h), "copy O rows");
  }
  // the caller's stream continues once O is on the host
  PLSH_TRY_CUDA(cudaEventRecord(ev_done, ctx->d2h), "event");
  PLSH_TRY_CUDA(cudaStreamWaitEvent(cs, ev_done, 0), "stream wait");
  return PLSH_OK;
}

plsh_status plsh_alibi_decode(const plsh_tensor* q, const plsh_tensor* K, const plsh_tensor* V,
                              const plsh_bins* bins, int64_t pos, plsh_tensor* o, void* stream) {
  plsh_status st;
  if ((st = check_tensor(q, "q")) != PLSH_OK || (st = check_tensor(K, "K")) != PLSH_OK ||
      (st = check_tensor(V, "V")) != PLSH_OK || (st = check_tensor(o, "o")) != PLSH_OK)
    return st;
  if (K->dtype != q->dtype || V->dtype != q->dtype || o->dtype != q->dtype)
    return fail(PLSH_ERR_INVALID, "q, K, V and o must share one dtype");
  if (q->d != 64 && q->d != 128) return fail(PLSH_ERR_INVALID, "head dim d must be 64 or 128");
  if (q->n != 1) return fail(PLSH_ERR_INVALID, "q must be [B, Hq, 1, d]");
  if (o->B != q->B || o->H != q->H || o->n != 1 || o->d != q->d)
    return fail(PLSH_ERR_INVALID, "o must have q's shape");
  if (K->B != q->B || K->d != q->d)
    return fail(PLSH_ERR_INVALID, "K must be [B, Hkv, n, d] with q's B and d");
  if (V->B != K->B || V->H != K->H || V->n != K->n || V->d != K->d)
    return fail(PLSH_ERR_INVALID, "V must have K's shape");
  if (q->H % K->H != 0) return fail(PLSH_ERR_INVALID, "Hq must be a multiple of Hkv");
  if (K->n >= ((int64_t)1 << 31)) return fail(PLSH_ERR_INVALID, "n must be < 2^31");
  if (q->B * q->H > 65535) return fail(PLSH_ERR_UNSUPPORTED, "B * Hq must be <= 65535");
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (bins->n != K->n) return fail(PLSH_ERR_INVALID, "bins were drawn for another n");
  if (bins->H != q->H) return fail(PLSH_ERR_INVALID, "bins were drawn for another number of heads");
  if (pos < 0 || pos >= K->n) return fail(PLSH_ERR_INVALID, "pos must be in [0, n)");
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  plsh::DeviceCtx* ctx = nullptr;
  if ((st = current_ctx(&ctx)) != PLSH_OK) return st;
  double sigma_max = 1e30;                 // unknown scales: any envelope
  if (bins->sigma_host.size() == (size_t)q->H) {
    sigma_max = 0.0;
    for (double sg : bins->sigma_host) sigma_max = sg > sigma_max ? sg : sigma_max;
  }
  const int useful = plsh::decode_useful_splits(sigma_max, (int)pos);
  const size_t bytes =
      sizeof(float) * plsh::decode_work_floats((int)q->B, (int)q->H, (int)K->H, (int)q->d,
                                               ctx->num_sms, useful);
  std::lock_guard<std::mutex> dk(g_decode_mu);
  if ((st = scratch_acquire(&ctx->decode_work, &ctx->decode_work_bytes, &ctx->decode_ev, bytes,
                            (cudaStream_t)stream, "decode partials")) != PLSH_OK)
    return st;
  float* work = ctx->decode_work;
  plsh::DecodeArgs a;
  a.q = q->data;
  a.K = K->data;
  a.V = V->data;
  a.o = o->data;
  a.rec = bins->d_rec;
  a.B = (int)q->B;
  a.Hq = (int)q->H;
  a.Hkv = (int)K->H;
  a.n = (int)K->n;
  a.d = (int)q->d;
  a.s = bins->s;
  a.W = bins->W;
  a.pos = (int)pos;
  a.dtype = q->dtype;
  a.num_sms = ctx->num_sms;
  a.useful_splits = useful;
  a.sigma = (int64_t)bins->sigma_host.size() == q->H ? bins->sigma_host.data() : nullptr;
  a.work = work;
  a.err = ctx->d_err;
  a.wait_ns = ctx->wait_ns;
  cudaError_t e = plsh::launch_decode(a, (cudaStream_t)stream);
  const cudaError_t er = cudaEventRecord(ctx->decode_ev, (cudaStream_t)stream);
  if (e == cudaSuccess) e = er;
  PLSH_TRY_CUDA(e, "decode launch");
  return PLSH_OK;
}

plsh_status plsh_alibi_exact(const plsh_tensor* Q, const plsh_tensor* K, const plsh_tensor* V,
                             const double* sigma_h, int32_t causal, plsh_tensor* O,
                             void* stream) {
  plsh_status st = check_qkvo(Q, K, V, O);
  if (st != PLSH_OK) return st;
  if (Q->H > plsh::kMaxExactHeads) return fail(PLSH_ERR_UNSUPPORTED, "exact path serves at most 512 heads");
  if ((st = check_sigma(sigma_h, (int32_t)Q->H)) != PLSH_OK) return st;
  std::vector<float> slopes(Q->H);
  for (int64_t h = 0; h < Q->H; ++h) slopes[h] = (float)(1.4426950408889634 / sigma_h[h]);
  return run_attention(Q, K, V, O, causal, nullptr, slopes.data(), (cudaStream_t)stream);
}

plsh_status plsh_stream_status(void* stream) {
  plsh::DeviceCtx* ctx = nullptr;
  plsh_status st = current_ctx(&ctx);
  if (st != PLSH_OK) return st;
  PLSH_TRY_CUDA(cudaStreamSynchronize((cudaStream_t)stream), "cudaStreamSynchronize");
  PLSH_TRY_CUDA(cudaGetLastError(), "pending CUDA error");
  int flag = 0;
  PLSH_TRY_CUDA(cudaMemcpy(&flag, ctx->d_err, sizeof(int), cudaMemcpyDeviceToHost), "read error flag");
  if (flag != 0) {
    PLSH_TRY_CUDA(cudaMemset(ctx->d_err, 0, sizeof(int)), "clear error flag");
    PLSH_TRY_CUDA(cudaDeviceSynchronize(), "cudaDeviceSynchronize");
  }
  return device_flag_status(flag);
}

plsh_status plsh_set_split_parts(int32_t parts) {
  if (parts < 0 || parts > plsh::kMaxSplitParts)
    return fail(PLSH_ERR_INVALID, "parts must be in [0, " + std::to_string(plsh::kMaxSplitParts) + "]");
  plsh::DeviceCtx* ctx = nullptr;
  plsh_status st = current_ctx(&ctx);
  if (st != PLSH_OK) return st;
  ctx->split_parts = parts;
  return PLSH_OK;
}

plsh_status plsh_set_wait_limit_ns(uint64_t ns) {
  plsh::DeviceCtx* ctx = nullptr;
  plsh_status st = current_ctx(&ctx);
  if (st != PLSH_OK) return st;
  ctx->wait_ns = ns == 0 ? plsh::kDefaultWaitNs : ns;
  g_noalloc_wait_ns[ctx->device].store(ctx->wait_ns, std::memory_order_relaxed);
  return PLSH_OK;
}

const char* plsh_status_string(plsh_status status) {
  switch (status) {
    case PLSH_OK: return "ok";
    case PLSH_ERR_INVALID: return "invalid argument";
    case PLSH_ERR_CUDA: return "CUDA error";
    case PLSH_ERR_NOMEM: return "out of memory";
    case PLSH_ERR_TIMEOUT: return "device wait timed out";
    case PLSH_ERR_UNSUPPORTED: return "unsupported";
    case PLSH_ERR_RANGE: return "input value out of range";
  }
  return "unknown status";
}

const char* plsh_last_error(void) { return g_last_error.c_str(); }

// Allocation-free variant of plsh_alibi_attn (see include/plsh.h).
plsh_status plsh_alibi_attn_noalloc(const plsh_tensor* Q, const plsh_tensor* K,
                                    const plsh_tensor* V, const plsh_bins* bins,
                                    int32_t causal, plsh_tensor* O, void* stream) {
  plsh_status st = check_qkvo(Q, K, V, O);
  if (st != PLSH_OK) return st;
  if (bins == nullptr) return fail(PLSH_ERR_INVALID, "bins is NULL");
  if (bins->n != Q->n) return fail(PLSH_ERR_INVALID, "bins were drawn for another n");
  if (bins->H != Q->H) return fail(PLSH_ERR_INVALID, "bins were drawn for another number of heads");
  if ((st = check_bins_device(bins)) != PLSH_OK) return st;
  if (Q->d != 128 || !tc_path_ok(Q->dtype, Q->d, bins->s, causal ? 1 : 0, 0))
    return fail(PLSH_ERR_UNSUPPORTED, "allocation-free path: needs bf16, d = 128 and s within "
                                      "the tensor-core kernel's shared-memory budget");
  const int B = (int)Q->B, Hq = (int)Q->H, Hkv = (int)K->H;
  const int QT = (int)((Q->n + 127) / 128);
  const int G = Hq / Hkv;
  if (Hq > 1023 || Hkv * (G / 2 + G % 2) > kNoAllocMaxUnits)
    return fail(PLSH_ERR_UNSUPPORTED, "allocation-free path: at most 1023 query heads and " +
                                          std::to_string(kNoAllocMaxUnits) + " work units");
  // units in cost order, built on the stack
  NoAllocUnits u;
  u.count = 0;
  double key[kNoAllocMaxUnits];
  int64_t num_items = 0;
  for (int kvh = 0; kvh < Hkv; ++kvh) {
    int heads[1024];
    for (int gi = 0; gi < G; ++gi) heads[gi] = kvh * G + gi;
    for (int a = 1; a < G; ++a) {          // by sigma, descending (stable)
      const int h = heads[a];
      int b2 = a;
      while (b2 > 0 && bins->sigma_host[heads[b2 - 1]] < bins->sigma_host[h]) {
        heads[b2] = heads[b2 - 1];
        --b2;
      }
      heads[b2] = h;
    }
    for (int pr = 0; pr + 1 < G; pr += 2) {
      u.unit[u.count] = heads[pr] | (heads[pr + 1] << 10);
      key[u.count] = std::max(bins->sigma_host[heads[pr]], bins->sigma_host[heads[pr + 1]]);
      ++u.count;
      num_items += (int64_t)B * QT;
    }
    if (G % 2) {
      u.unit[u.count] = heads[G - 1] | (heads[G - 1] << 10) | (1 << 20);
      key[u.count] = bins->sigma_host[heads[G - 1]];
      ++u.count;
      num_items += (int64_t)B * ((QT + 1) / 2);
    }
  }
  for (int a = 1; a < u.count; ++a) {      // units by cost, descending (stable)
    const int cu = u.unit[a];
    const double ck = key[a];
    int b2 = a;
    while (b2 > 0 && key[b2 - 1] < ck) {
      u.unit[b2] = u.unit[b2 - 1];
      key[b2] = key[b2 - 1];
      --b2;
    }
    u.unit[b2] = cu;
    key[b2] = ck;
  }
  for (int a = 0; a < u.count; ++a)        // runs of equal cost and unit kind
    if (a == 0 || key[a] != key[a - 1] || ((u.unit[a] ^ u.unit[a - 1]) >> 20 & 1))
      u.unit[a] |= 1 << 21;
  if (num_items > kNoAllocMaxItems)
    return fail(PLSH_ERR_UNSUPPORTED,
                "allocation-free path: " + std::to_string(num_items) + " work items exceed its " +
                    std::to_string(kNoAllocMaxItems) + "-item scratch area");
  int dev = -1;
  PLSH_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PLSH_ERR_UNSUPPORTED, "device index out of range");
  int4* scratch = nullptr;
  {
    // set-up, once per device with that device current: the array's host
    // name is not a device address, so resolve it here
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (g_noalloc_addr[dev] == nullptr) {
      void* ptr = nullptr;
      PLSH_TRY_CUDA(cudaGetSymbolAddress(&ptr, g_noalloc_scratch), "cudaGetSymbolAddress");
      g_noalloc_addr[dev] = static_cast<int4*>(ptr);
    }
    scratch = g_noalloc_addr[dev];
  }
  int sms = 0;
  PLSH_TRY_CUDA(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev),
                "cudaDeviceGetAttribute");
  cudaStream_t cs = (cudaStream_t)stream;
  noalloc_items_kernel<<<(unsigned)((num_items + 255) / 256), 256, 0, cs>>>(
      scratch, u, B, QT, (int)num_items);
  PLSH_TRY_CUDA(cudaGetLastError(), "item table launch");
  plsh::AttnArgs a;
  memset(&a, 0, sizeof a);
  a.Q = Q->data;
  a.K = K->data;
  a.V = V->data;
  a.O = O->data;
  a.B = B;
  a.Hq = Hq;
  a.Hkv = Hkv;
  a.n = (int)Q->n;
  a.d = (int)Q->d;
  a.causal = causal ? 1 : 0;
  a.exact = 0;
  a.rec = bins->d_rec;
  a.s = bins->s;
  a.W = bins->W;
  a.items = scratch + 1;
  a.num_items = (int)num_items;
  a.queue = reinterpret_cast<int*>(scratch);
  a.err = reinterpret_cast<int*>(scratch) + 2;
  const uint64_t wl = g_noalloc_wait_ns[dev].load(std::memory_order_relaxed);
  a.wait_ns = wl == 0 ? plsh::kDefaultWaitNs : wl;
  a.stall = fault_is("stall") ? 1 : 0;
  PLSH_TRY_CUDA(plsh::launch_attn_tc(a, nullptr, sms, cs), "attention launch");
  return PLSH_OK;
}

plsh_status plsh_noalloc_status(void* stream) {
  int dev = -1;
  PLSH_TRY_CUDA(cudaGetDevice(&dev), "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return fail(PLSH_ERR_UNSUPPORTED, "device index out of range");
  cudaStream_t cs = (cudaStream_t)stream;
  PLSH_TRY_CUDA(cudaStreamSynchronize(cs), "cudaStreamSynchronize");
  PLSH_TRY_CUDA(cudaGetLastError(), "pending CUDA error");
  // the error word is the third int of the array's first element
  int word = 0;
  const size_t at = 2 * sizeof(int);
  PLSH_TRY_CUDA(cudaMemcpyFromSymbolAsync(&word, g_noalloc_scratch, sizeof(int), at,
                                          cudaMemcpyDeviceToHost, cs), "read error word");
  PLSH_TRY_CUDA(cudaStreamSynchronize(cs), "cudaStreamSynchronize");
  if (word != 0) {
    const int zero = 0;
    PLSH_TRY_CUDA(cudaMemcpyToSymbolAsync(g_noalloc_scratch, &zero, sizeof(int), at,
                                          cudaMemcpyHostToDevice, cs), "clear error word");
    PLSH_TRY_CUDA(cudaStreamSynchronize(cs), "cudaStreamSynchronize");
  }
  return device_flag_status(word);
}

plsh_status plsh_attn_path(const plsh_tensor* Q, const plsh_bins* bins, int32_t causal,
                           int32_t* path) {
  if (Q == nullptr || path == nullptr) return fail(PLSH_ERR_INVALID, "NULL argument");
  *path = tc_path_ok(Q->dtype, Q->d, bins ? bins->s : 0, causal ? 1 : 0, bins ? 0 : 1) &&
                  path_override() != Path::Simt
              ? PLSH_PATH_TENSOR_CORES
              : PLSH_PATH_CUDA_CORES;
  return PLSH_OK;
}

}  // extern "C"
