// Status strings, error bookkeeping and the device-attribute cache of the C ABI.
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

}  // extern "C"
