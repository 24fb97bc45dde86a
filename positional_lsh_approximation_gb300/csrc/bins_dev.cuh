// Bin of a position from the per-word records (see sampler.cu).
#pragma once

#include <stdint.h>

#include "plsh_internal.h"

namespace plsh {

// Start of the bin that contains position i (i lies in word wd = i >> 5, bit
// r = i & 31): the highest set bit at or below r, else the record's prev.
__device__ __forceinline__ int bin_lo(const BinRecord& rec, int i) {
  const int r = i & 31;
  const uint32_t le = rec.bits & (0xffffffffu >> (31 - r));
  return le ? ((i & ~31) + 31 - __clz(le)) : rec.prev;
}

// End (exclusive) of the bin that contains position i: the lowest set bit
// above r, else the record's next (n at the end of the sequence).
__device__ __forceinline__ int bin_hi(const BinRecord& rec, int i) {
  const int r = i & 31;
  const uint32_t gt = r == 31 ? 0u : (rec.bits & (0xfffffffeu << r));
  return gt ? ((i & ~31) + __ffs(gt) - 1) : rec.next;
}

__device__ __forceinline__ BinRecord load_record(const BinRecord* rec,
                                                 int64_t idx) {
  const uint4 v = __ldg(reinterpret_cast<const uint4*>(rec) + idx);
  BinRecord r;
  r.bits = v.x;
  r.prev = (int32_t)v.y;
  r.next = (int32_t)v.z;
  r.pad = 0;
  return r;
}

}  // namespace plsh
