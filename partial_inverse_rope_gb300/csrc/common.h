// Host-side helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include <mutex>

#include "invrope.h"
#include "sched.cuh"

namespace invrope {

struct DeviceInfo {
  int device = -1;
  int sms = 0;
  int major = 0;
  int minor = 0;
  size_t max_smem_optin = 0;
};

// Cached attributes of the current device; returns INVROPE_OK or an error status.
int current_device(DeviceInfo* out);

// Remember a CUDA error for invrope_last_cuda_error() and map it to a status.
int cuda_fail(cudaError_t err);

// Check the last launch on this thread.
int check_launch();

// [a, a+na) and [b, b+nb) overlap (byte ranges, both non-empty).
inline bool overlaps(const void* a, size_t na, const void* b, size_t nb) {
  if (na == 0 || nb == 0) return false;
  const uintptr_t a0 = reinterpret_cast<uintptr_t>(a), b0 = reinterpret_cast<uintptr_t>(b);
  return a0 < b0 + nb && b0 < a0 + na;
}

inline bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Host-side hand-out of the work-counter slots of one __device__ SchedSlot
// array (see sched.cuh), per device. `symbol` is the array's host-side
// stand-in; its device address is looked up once per device.
struct SlotRing {
  std::mutex mu;
  SchedSlot* base[64] = {};
  unsigned int eager[64] = {};
  unsigned int capture[64] = {};
};

// The slot of the next launch on `stream` (an eager slot, or a capture slot
// while the stream is being captured into a graph).
int slot_take(SlotRing& ring, const void* symbol, int device, cudaStream_t stream, SchedSlot** out);

// The slot the next eager launch will take, without taking it.
int slot_peek_eager(SlotRing& ring, const void* symbol, int device, SchedSlot** out);

// Zero every slot of the array on `device` (nothing may be running on it).
int slot_reset_all(SlotRing& ring, const void* symbol, int device);

// Read and clear the remap kernel's fault word on the current device.
int take_remap_fault(unsigned int* code);

// Reset the forward's and the remap's slot arrays on `device`.
int reset_postmix_sched(int device);
int reset_remap_sched(int device);

// Write `owner` into the owner word of the slot the next eager forward
// (which = 0) or remap (which = 1) launch will take.
int occupy_postmix_slot(int device, unsigned long long owner);
int occupy_remap_slot(int device, unsigned long long owner);

}  // namespace invrope
