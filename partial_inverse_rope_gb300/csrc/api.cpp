// Status strings, error bookkeeping, the device-attribute cache and the
// host-side work-counter slot hand-out of the C ABI.
#include <mutex>

#include "common.h"

namespace invrope {

namespace {
thread_local int g_last_cuda_error = 0;
std::mutex g_dev_mu;
DeviceInfo g_dev_cache[64];
}  // namespace

int cuda_fail(cudaError_t err) {
  g_last_cuda_error = static_cast<int>(err);
  return INVROPE_ERR_CUDA;
}

int check_launch() {
  const cudaError_t err = cudaGetLastError();
  if (err != cudaSuccess) return cuda_fail(err);
  return INVROPE_OK;
}

int current_device(DeviceInfo* out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return cuda_fail(err);
  if (dev < 0 || dev >= 64) return INVROPE_ERR_DEVICE;
  std::lock_guard<std::mutex> lock(g_dev_mu);
  DeviceInfo& d = g_dev_cache[dev];
  if (d.device != dev) {
    DeviceInfo n;
    n.device = dev;
    int v = 0;
    if ((err = cudaDeviceGetAttribute(&n.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&n.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&n.minor, cudaDevAttrComputeCapabilityMinor, dev)) != cudaSuccess ||
        (err = cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev)) != cudaSuccess)
      return cuda_fail(err);
    n.max_smem_optin = static_cast<size_t>(v);
    d = n;
  }
  *out = d;
  if (!(d.major == 10 && d.minor == 3)) return INVROPE_ERR_DEVICE;
  return INVROPE_OK;
}

namespace {
int slot_base(SlotRing& ring, const void* symbol, int device) {
  if (device < 0 || device >= 64) return INVROPE_ERR_DEVICE;
  if (!ring.base[device]) {
    void* ptr = nullptr;
    const cudaError_t err = cudaGetSymbolAddress(&ptr, symbol);
    if (err != cudaSuccess) return cuda_fail(err);
    ring.base[device] = static_cast<SchedSlot*>(ptr);
  }
  return INVROPE_OK;
}
}  // namespace

int slot_take(SlotRing& ring, const void* symbol, int device, cudaStream_t stream, SchedSlot** out) {
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  const cudaError_t err = cudaStreamIsCapturing(stream, &cap);
  if (err != cudaSuccess) return cuda_fail(err);
  std::lock_guard<std::mutex> lock(ring.mu);
  const int st = slot_base(ring, symbol, device);
  if (st != INVROPE_OK) return st;
  if (cap == cudaStreamCaptureStatusNone)
    *out = ring.base[device] + (ring.eager[device]++ % kEagerSlots);
  else
    *out = ring.base[device] + kEagerSlots + (ring.capture[device]++ % kCaptureSlots);
  return INVROPE_OK;
}

int slot_peek_eager(SlotRing& ring, const void* symbol, int device, SchedSlot** out) {
  std::lock_guard<std::mutex> lock(ring.mu);
  const int st = slot_base(ring, symbol, device);
  if (st != INVROPE_OK) return st;
  *out = ring.base[device] + (ring.eager[device] % kEagerSlots);
  return INVROPE_OK;
}

int slot_reset_all(SlotRing& ring, const void* symbol, int device) {
  std::lock_guard<std::mutex> lock(ring.mu);
  const int st = slot_base(ring, symbol, device);
  if (st != INVROPE_OK) return st;
  const cudaError_t err = cudaMemset(ring.base[device], 0, sizeof(SchedSlot) * kSchedSlots);
  if (err != cudaSuccess) return cuda_fail(err);
  return INVROPE_OK;
}

}  // namespace invrope

extern "C" {

const char* invrope_status_string(int status) {
  switch (status) {
    case INVROPE_OK: return "INVROPE_OK";
    case INVROPE_ERR_INVALID_ARG: return "INVROPE_ERR_INVALID_ARG: invalid argument";
    case INVROPE_ERR_UNSUPPORTED: return "INVROPE_ERR_UNSUPPORTED: shape not covered by the kernels";
    case INVROPE_ERR_WORKSPACE: return "INVROPE_ERR_WORKSPACE: workspace missing or too small";
    case INVROPE_ERR_CUDA: return "INVROPE_ERR_CUDA: CUDA runtime or launch error";
    case INVROPE_ERR_DEVICE: return "INVROPE_ERR_DEVICE: current device is not compute capability 10.3";
    default: return "INVROPE_ERR_UNKNOWN";
  }
}

int invrope_last_cuda_error(void) { return invrope::g_last_cuda_error; }

int invrope_debug_occupy_next_slot(int which, unsigned long long owner) {
  int dev = 0;
  const cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return invrope::cuda_fail(err);
  if (which == 0) return invrope::occupy_postmix_slot(dev, owner);
  if (which == 1) return invrope::occupy_remap_slot(dev, owner);
  return INVROPE_ERR_INVALID_ARG;
}

}  // extern "C"
