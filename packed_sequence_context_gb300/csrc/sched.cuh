// Dynamic hand-out of work items inside a persistent attention kernel.
//
// Every CTA starts with item blockIdx.x and then claims the next free item
// from a per-launch counter in global memory (zeroed by the planner of the
// same call), so a CTA that drew short items simply takes more of them: the
// makespan is the greedy list-scheduling one, whatever the item order.  That
// frees the order to serve locality (see q_item / the dK/dV item map: items
// that reuse the same keys and values, or queries and output gradients, run
// side by side while those stay in L2).
//
// Inside the CTA one thread (the producer's lane 0) claims the items and
// publishes them, in claim order, through a ring of kItemSlots shared-memory
// slots; every other role reads slot k before it starts its k-th item and
// releases the slot at once (it keeps the index in a register), so the
// producer is never held back by a role that is still working on an earlier
// item.  A claimed index >= n_items is published as the end marker.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace thd {

constexpr int kItemSlots = 8;

struct ItemRing {
  uint64_t full[kItemSlots];   // slot written (one arrival: the producer)
  uint64_t empty[kItemSlots];  // slot read by every consumer role
  int item[kItemSlots];
};

// One thread, before the CTA-wide barrier that precedes the roles.
__device__ inline void item_ring_init(ItemRing* r, uint32_t consumer_arrivals) {
  for (int s = 0; s < kItemSlots; ++s) {
    mbar_init(&r->full[s], 1);
    mbar_init(&r->empty[s], consumer_arrivals);
  }
}

// The CTA's first item, and the next one it claims.
__device__ inline int item_first() { return (int)blockIdx.x; }
__device__ inline int item_claim(int32_t* counter) { return (int)gridDim.x + atomicAdd(counter, 1); }

// Producer (one thread): publish this CTA's k-th item (or the end marker).
// Returns false when the CTA is aborting.  Slot k % kItemSlots is reused
// once every consumer has read its previous content, so the barrier is never
// two phases behind this wait.
__device__ inline bool item_publish(ItemRing* r, uint32_t k, int w, volatile int* abort_flag) {
  const uint32_t s = k % kItemSlots;
  if (!mbar_wait(&r->empty[s], ((k / kItemSlots) & 1u) ^ 1u, abort_flag)) return false;
  *reinterpret_cast<volatile int*>(&r->item[s]) = w;
  mbar_arrive(&r->full[s]);  // release: the slot's value is visible to whoever observes the phase
  return true;
}

// Consumer: this CTA's k-th item into w; false when the CTA is aborting.
__device__ inline bool item_take(ItemRing* r, uint32_t k, int& w, volatile int* abort_flag) {
  const uint32_t s = k % kItemSlots;
  if (!mbar_wait(&r->full[s], (k / kItemSlots) & 1u, abort_flag)) return false;
  w = *reinterpret_cast<volatile int*>(&r->item[s]);
  return true;
}

// Whole-warp consumer: every lane calls it; the decision is warp-uniform and
// lane 0 releases the slot for the warp (one arrival per warp).
__device__ inline bool item_take_warp(ItemRing* r, uint32_t k, int& w, volatile int* abort_flag) {
  int v = 0;
  const bool got = __all_sync(0xffffffffu, item_take(r, k, v, abort_flag));
  if (!got) return false;
  w = __shfl_sync(0xffffffffu, v, 0);
  if ((threadIdx.x & 31) == 0) mbar_arrive(&r->empty[k % kItemSlots]);
  return true;
}

// Single-thread consumer: read and release.
__device__ inline bool item_take_one(ItemRing* r, uint32_t k, int& w, volatile int* abort_flag) {
  if (!item_take(r, k, w, abort_flag)) return false;
  mbar_arrive(&r->empty[k % kItemSlots]);
  return true;
}

}  // namespace thd
