// Host-side helpers shared by the library's translation units.
#pragma once

#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "invrope.h"

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

}  // namespace invrope
