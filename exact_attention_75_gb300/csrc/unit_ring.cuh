// Run-time hand-out of work units in the persistent backward kernels.
//
// Each CTA's producer takes its next unit from a counter in global memory
// (zeroed by the D pass before the kernel starts) with an atomic add and
// publishes it through a ring of kUnitSlots entries in shared memory.  The
// issuer, the relay and the 8 compute warps read each entry and release it
// with one arrival each; an entry of -1 ends the CTA's work.  Every wait is
// bounded (Watchdog).
#pragma once

#include <cstdint>

#include "sm103_ptx.cuh"

namespace attn {

constexpr int kUnitSlots = 4;
constexpr int kUnitReaders = 10;  // issuer + relay + 8 compute warps

// Producer side (one thread): once entry un's slot has been released, takes
// the next unit from the counter and publishes it (-1 once the counter has
// passed num_units).  Returns the unit, or -1 with ok false when the wait ran
// out.
__device__ __forceinline__ int publish_unit(volatile int* ring, uint32_t full0, uint32_t empty0,
                                            uint32_t un, int* counter, int num_units,
                                            const Watchdog& wd, bool& ok, int site) {
  const uint32_t us = un % kUnitSlots;
  ok = mbar_wait(empty0 + 8u * us, ((un / kUnitSlots) & 1) ^ 1, wd, site);
  if (!ok) return -1;
  int u = atomicAdd(counter, 1);
  if (u >= num_units) u = -1;
  ring[us] = u;
  mbar_arrive(full0 + 8u * us);
  return u;
}

// Reader side (every lane of a warp): waits for entry un, reads it and
// releases it with one arrival for the warp.  Returns -1 with ok false when
// the wait ran out.
__device__ __forceinline__ int take_unit(volatile int* ring, uint32_t full0, uint32_t empty0,
                                         uint32_t un, const Watchdog& wd, bool& ok, int site) {
  const uint32_t us = un % kUnitSlots;
  ok = mbar_wait(full0 + 8u * us, (un / kUnitSlots) & 1, wd, site);
  const int u = ok ? ring[us] : -1;
  __syncwarp();
  if (ok && (threadIdx.x & 31) == 0) mbar_arrive(empty0 + 8u * us);
  return u;
}

// The same for the relay / issuer pair: the relay has waited for entry un and
// met the issuer at their named barrier, so both read it and release it.
__device__ __forceinline__ int read_unit(volatile int* ring, uint32_t empty0, uint32_t un) {
  const uint32_t us = un % kUnitSlots;
  const int u = ring[us];
  __syncwarp();
  if ((threadIdx.x & 31) == 0) mbar_arrive(empty0 + 8u * us);
  return u;
}

// Decodes unit u of an order that hands out all units of one block of
// head_block heads before the next block's (the last block may hold fewer
// heads).  Within a block the length class varies slowest (class 0 = the
// longest units, so longest first), then the head, then an inner index
// (inner_n values per head and class, e.g. output column halves).
struct BlockedUnit {
  int head;   // head index over all blocks
  int cls;    // length class within the head (0 = longest)
  int inner;  // index below the head (e.g. an output column half), 0 if none
};

__device__ __forceinline__ BlockedUnit blocked_unit(int u, int heads, int head_block,
                                                    int per_head, int inner_n) {
  const int per_blk = head_block * per_head * inner_n;
  const int blk = u / per_blk;
  const int r = u - blk * per_blk;
  const int h0 = blk * head_block;
  const int hb = min(head_block, heads - h0);
  BlockedUnit b;
  b.cls = r / (hb * inner_n);
  const int rr = r - b.cls * hb * inner_n;
  const int hh = rr / inner_n;
  b.head = h0 + hh;
  b.inner = rr - hh * inner_n;
  return b;
}

}  // namespace attn
