// Work-counter slots for the kernels that hand out their work dynamically
// (the forward postmix claims tiles, the KV remap claims chunks).
//
// A launch works from one slot: {owner, next, done}. Its thread blocks take
// the slot when it is free (owner 0) or already held by their own launch:
// owner is the launch's grid id (%gridid, unique per launch in the context,
// graph replays included) plus one. A block that finds the slot held by
// another launch still in flight claims nothing from it and reports a fault,
// so two launches never share a counter. The last block of the owning launch
// returns next and done to zero and then frees the slot.
//
// The host hands out slots in turn: eager launches take the first
// kEagerSlots, launches made while the stream is being captured into a CUDA
// graph take the other kCaptureSlots (a captured launch keeps its slot on
// every replay, so it must not share one with eager launches).
#pragma once

#include <cstdint>

namespace invrope {

struct SchedSlot {
  unsigned long long owner;  // 0 = free, else the owning launch's grid id + 1
  unsigned int next;         // next work item to claim (beyond the static first ones)
  unsigned int done;         // thread blocks of the owner that have finished
};

constexpr int kEagerSlots = 256;
constexpr int kCaptureSlots = 256;
constexpr int kSchedSlots = kEagerSlots + kCaptureSlots;

__device__ __forceinline__ unsigned long long launch_tag() {
  unsigned long long g;
  asm volatile("mov.u64 %0, %%gridid;" : "=l"(g));
  return g + 1ull;
}

// True when this launch owns the slot (this block took it, or another block
// of the same launch did); false when another launch holds it.
__device__ __forceinline__ bool sched_acquire(SchedSlot* s, unsigned long long tag) {
  unsigned long long o = *reinterpret_cast<volatile unsigned long long*>(&s->owner);
  if (o != tag) o = atomicCAS(&s->owner, 0ull, tag);
  return o == 0ull || o == tag;
}

// Once per block that acquired the slot, after its last claim: the last of the
// launch's nblocks blocks returns the counters to zero and frees the slot.
// Each block's claims are performed before its done count (fence), so the
// last block sees no claim still in flight and resets with plain stores,
// ordered before the slot is freed.
__device__ __forceinline__ void sched_release(SchedSlot* s, unsigned int nblocks) {
  __threadfence();
  if (atomicAdd(&s->done, 1u) == nblocks - 1u) {
    *reinterpret_cast<volatile unsigned int*>(&s->next) = 0u;
    *reinterpret_cast<volatile unsigned int*>(&s->done) = 0u;
    __threadfence();
    *reinterpret_cast<volatile unsigned long long*>(&s->owner) = 0ull;
  }
}

}  // namespace invrope
