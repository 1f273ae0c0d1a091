// Backward of the fused inverse-RoPE + VHA postmix for callers that cannot
// allocate device memory: the per-CTA dM partials live in a fixed scratch
// array that belongs to this library instead of a caller-provided workspace.
//
// Who needs it: code that is not allowed to call cudaMalloc (or any
// allocating library routine) on its call path and has no workspace to hand
// in -- e.g. a host runtime whose device memory is planned once up front, or
// a plugin interface that passes only input and output buffers. cudaMalloc
// can also synchronise the device, which such callers must avoid.
//
// The array is a file-scope __device__ object, so every device on which this
// library's module is loaded holds it until the process exits. In host code
// its name is only a host-side stand-in; the device address is looked up
// once per device with cudaGetSymbolAddress and passed to the kernels.
#include <cuda_runtime.h>

#include <mutex>

#include "common.h"

// One fp32 [nh, nh] dM partial per CTA of the backward kernel.
static __device__ __align__(256) unsigned char g_noalloc_scratch[INVROPE_NOALLOC_SCRATCH_BYTES];

namespace invrope {
namespace {

std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device (set up once per
// device, with that device current). Returns INVROPE_OK or an error status.
int scratch_for_current_device(void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= 64) return INVROPE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* ptr = nullptr;
    err = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
    if (err != cudaSuccess) return cuda_fail(err);
    if (!ptr) return INVROPE_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return INVROPE_OK;
}

}  // namespace
}  // namespace invrope

extern "C" int invrope_postmix_bwd_noalloc(const void* dY, const void* O, const float* M, void* dO, float* dM,
                                           int64_t sq, int nh, int nope, int pe, int64_t pos0, double theta,
                                           struct CUstream_st* stream) {
  using namespace invrope;
  DeviceInfo dev;
  int st = current_device(&dev);
  if (st != INVROPE_OK) return st;
  // 0 means the shape itself is invalid: let the regular entry point report why.
  const size_t need = invrope_postmix_bwd_workspace_bytes(sq, nh, nope, pe);
  if (need > INVROPE_NOALLOC_SCRATCH_BYTES) return INVROPE_ERR_WORKSPACE;
  void* scratch = nullptr;
  if ((st = scratch_for_current_device(&scratch)) != INVROPE_OK) return st;
  // Every partial the reduction reads is written by the same launch first, so
  // whatever an earlier call left in the array does not matter.
  return invrope_postmix_bwd(dY, O, M, dO, dM, scratch, INVROPE_NOALLOC_SCRATCH_BYTES, sq, nh, nope, pe, pos0,
                             theta, stream);
}
