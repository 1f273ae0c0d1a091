// Per-batch-local -> flat-global sparse-attention KV column remap on GB300.
//
// PaddleFleet PR #1772, "Fuse HCA inverse RoPE into the VHA postmix, and the
// sparse-attention KV index remap", English description item 2 and Chinese
// description section 2: out = idx + b * seqlen_kv over the [b*sq, topk]
// table, padding (negative entries) kept, in one pass instead of the eager
// chain of seven elementwise kernels.
//
// The table is streamed once as a flat array. Batch b owns the contiguous
// element range [b*sq*topk, (b+1)*sq*topk), so a thread block that walks a
// chunk of the flat array finds its batch with one division per chunk and
// at most one boundary inside it. 16-byte vectors when the layout allows.
// Chunks are handed out dynamically (a per-launch counter slot, sched.cuh):
// SMs differ in the memory bandwidth they get, and a fixed split would wait on
// the slowest.
// int32 and int64 tables (the int64 one for callers that index past 2^31).
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "common.h"
#include "sched.cuh"

namespace invrope {

// The remap's own fault word (each translation unit's device code is linked
// separately): invrope_take_device_fault() reads and clears it together with
// the postmix kernels' word.
__device__ unsigned int g_remap_fault = 0;

// Dynamic chunk scheduling: one work-counter slot per launch (sched.cuh).
__device__ SchedSlot g_remap_sched[kSchedSlots];

namespace {

constexpr int kThreads = 256;
constexpr int kPer = 8;                         // vectors per thread per chunk
constexpr int kChunk = kThreads * kPer;         // vectors per chunk

// Entry types: int32 (offset added mod 2^32) and int64 (mod 2^64).
__device__ __forceinline__ int32_t remap1(int32_t v, uint64_t off) {
  return v < 0 ? v : static_cast<int32_t>(static_cast<uint32_t>(v) + static_cast<uint32_t>(off));
}
__device__ __forceinline__ long long remap1(long long v, uint64_t off) {
  return v < 0 ? v : static_cast<long long>(static_cast<uint64_t>(v) + off);
}

__device__ __forceinline__ int4 load_vec(const int4* p) { return __ldcs(p); }
__device__ __forceinline__ int load_vec(const int* p) { return __ldcs(p); }
__device__ __forceinline__ longlong2 load_vec(const longlong2* p) { return __ldcs(p); }
__device__ __forceinline__ long long load_vec(const long long* p) { return __ldcs(p); }
__device__ __forceinline__ void store_vec(int4* p, int4 v) { __stcs(p, v); }
__device__ __forceinline__ void store_vec(int* p, int v) { __stcs(p, v); }
__device__ __forceinline__ void store_vec(longlong2* p, longlong2 v) { __stcs(p, v); }
__device__ __forceinline__ void store_vec(long long* p, long long v) { __stcs(p, v); }

__device__ __forceinline__ int4 remap_vec(int4 v, uint64_t off) {
  v.x = remap1(v.x, off);
  v.y = remap1(v.y, off);
  v.z = remap1(v.z, off);
  v.w = remap1(v.w, off);
  return v;
}
__device__ __forceinline__ int remap_vec(int v, uint64_t off) { return remap1(v, off); }
__device__ __forceinline__ longlong2 remap_vec(longlong2 v, uint64_t off) {
  v.x = remap1(v.x, off);
  v.y = remap1(v.y, off);
  return v;
}
__device__ __forceinline__ long long remap_vec(long long v, uint64_t off) { return remap1(v, off); }

// V = a 16-byte vector (int4: 4 int32 entries, longlong2: 2 int64 entries) or
// one entry. seg = entries of one batch in units of V.
// kOneBoundary: seg >= kChunk, so a chunk crosses at most one batch boundary.
template <typename V, bool kOneBoundary>
__global__ void __launch_bounds__(kThreads) kv_remap_kernel(const V* in, V* out, int64_t n, int64_t seg,
                                                            uint64_t seqlen_kv, SchedSlot* sched) {
  __shared__ int64_t next_chunk;
  const int64_t nchunks = (n + kChunk - 1) / kChunk;
  // Thread 0 takes the launch's counter slot along with its first claim. A
  // block that finds the slot held by another launch still in flight does its
  // static first chunk, claims nothing and records a fault. A launch with no
  // more chunks than blocks has no slot (sched == nullptr) and claims nothing.
  bool mine = false;
  // first chunk = block index; each later one is claimed while the current one streams
  for (int64_t ch = blockIdx.x; ch < nchunks;) {
    if (threadIdx.x == 0) {
      if (sched != nullptr && ch == static_cast<int64_t>(blockIdx.x)) {
        mine = sched_acquire(sched, launch_tag());
        if (!mine) atomicCAS(&g_remap_fault, 0u, static_cast<unsigned>(INVROPE_FAULT_SCHED_BUSY_REMAP));
      }
      next_chunk = mine ? static_cast<int64_t>(gridDim.x) + static_cast<int64_t>(atomicAdd(&sched->next, 1u))
                        : nchunks;
    }
    const int64_t v0 = ch * kChunk;
    const int64_t b0 = v0 / seg;
    const int64_t boundary = (b0 + 1) * seg;
    V x[kPer];
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int64_t v = v0 + k * kThreads + threadIdx.x;
      if (v < n) x[k] = load_vec(in + v);
    }
#pragma unroll
    for (int k = 0; k < kPer; ++k) {
      const int64_t v = v0 + k * kThreads + threadIdx.x;
      if (v < n) {
        const int64_t b = kOneBoundary ? b0 + (v >= boundary ? 1 : 0) : v / seg;
        store_vec(out + v, remap_vec(x[k], static_cast<uint64_t>(b) * seqlen_kv));
      }
    }
    __syncthreads();  // next_chunk is visible
    ch = next_chunk;
    __syncthreads();  // and read by all before thread 0 claims again
  }
  if (threadIdx.x == 0 && mine) sched_release(sched, gridDim.x);
}

SlotRing g_remap_ring;

template <typename V>
int launch(const void* in, void* out, int64_t n, int64_t seg, uint64_t skv, const DeviceInfo& dev,
           cudaStream_t s) {
  const int64_t nchunks = (n + kChunk - 1) / kChunk;
  const int64_t slots = static_cast<int64_t>(dev.sms) * 8;
  const int64_t grid = nchunks < slots ? nchunks : slots;
  // a work-counter slot only when there is something to claim beyond the
  // first chunk of each block
  SchedSlot* sched = nullptr;
  if (nchunks > grid) {
    const int st = slot_take(g_remap_ring, &g_remap_sched, dev.device, s, &sched);
    if (st != INVROPE_OK) return st;
  }
  if (seg >= kChunk)
    kv_remap_kernel<V, true><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
        static_cast<const V*>(in), static_cast<V*>(out), n, seg, skv, sched);
  else
    kv_remap_kernel<V, false><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(
        static_cast<const V*>(in), static_cast<V*>(out), n, seg, skv, sched);
  return check_launch();
}

// Argument checks common to both entry types; returns the entry count in *n.
int check_remap(const void* idx, const void* out, int64_t rows, int topk, int64_t sq, int64_t seqlen_kv,
                size_t esize, int64_t* n) {
  if (rows < 0 || topk < 0 || sq < 1 || seqlen_kv < 0) return INVROPE_ERR_INVALID_ARG;
  if (rows % sq != 0) return INVROPE_ERR_INVALID_ARG;
  *n = rows * static_cast<int64_t>(topk);
  if (*n == 0) return INVROPE_OK;
  if (!idx || !out || !aligned(idx, esize) || !aligned(out, esize)) return INVROPE_ERR_INVALID_ARG;
  const size_t bytes = static_cast<size_t>(*n) * esize;
  if (idx != out && overlaps(idx, bytes, out, bytes)) return INVROPE_ERR_INVALID_ARG;
  return INVROPE_OK;
}

}  // namespace

int take_remap_fault(unsigned int* code) {
  cudaError_t err = cudaMemcpyFromSymbol(code, g_remap_fault, sizeof(*code));
  if (err != cudaSuccess) return cuda_fail(err);
  const unsigned int zero = 0;
  if ((err = cudaMemcpyToSymbol(g_remap_fault, &zero, sizeof(zero))) != cudaSuccess) return cuda_fail(err);
  return INVROPE_OK;
}

int reset_remap_sched(int device) { return slot_reset_all(g_remap_ring, &g_remap_sched, device); }

int occupy_remap_slot(int device, unsigned long long owner) {
  SchedSlot* s = nullptr;
  const int st = slot_peek_eager(g_remap_ring, &g_remap_sched, device, &s);
  if (st != INVROPE_OK) return st;
  const cudaError_t err = cudaMemcpy(&s->owner, &owner, sizeof(owner), cudaMemcpyHostToDevice);
  return err == cudaSuccess ? INVROPE_OK : cuda_fail(err);
}

}  // namespace invrope

using namespace invrope;

extern "C" int kv_idx_local_to_global(const int32_t* idx, int32_t* out, int64_t rows, int topk, int64_t sq,
                                      int64_t seqlen_kv, struct CUstream_st* stream) {
  int64_t n = 0;
  int st = check_remap(idx, out, rows, topk, sq, seqlen_kv, 4, &n);
  if (st != INVROPE_OK) return st;
  const int64_t nb = rows / sq;
  if (nb > 0 && seqlen_kv > (int64_t(1) << 31) / nb) return INVROPE_ERR_INVALID_ARG;  // b*seqlen_kv <= 2^31
  if (n == 0) return INVROPE_OK;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != INVROPE_OK) return st;
  const int64_t seg = sq * topk;  // entries per batch
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint64_t skv = static_cast<uint64_t>(seqlen_kv);
  if (aligned(idx, 16) && aligned(out, 16) && seg % 4 == 0)
    return launch<int4>(idx, out, n / 4, seg / 4, skv, dev, s);
  return launch<int>(idx, out, n, seg, skv, dev, s);
}

extern "C" int kv_idx_local_to_global_i64(const int64_t* idx, int64_t* out, int64_t rows, int topk, int64_t sq,
                                          int64_t seqlen_kv, struct CUstream_st* stream) {
  int64_t n = 0;
  int st = check_remap(idx, out, rows, topk, sq, seqlen_kv, 8, &n);
  if (st != INVROPE_OK) return st;
  const int64_t nb = rows / sq;
  // b * seqlen_kv <= 2^63: every in-range index maps into int64
  if (nb > 0 && static_cast<uint64_t>(seqlen_kv) > (uint64_t(1) << 63) / static_cast<uint64_t>(nb))
    return INVROPE_ERR_INVALID_ARG;
  if (n == 0) return INVROPE_OK;
  DeviceInfo dev;
  if ((st = current_device(&dev)) != INVROPE_OK) return st;
  const int64_t seg = sq * topk;
  const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const uint64_t skv = static_cast<uint64_t>(seqlen_kv);
  if (aligned(idx, 16) && aligned(out, 16) && seg % 2 == 0)
    return launch<longlong2>(idx, out, n / 2, seg / 2, skv, dev, s);
  return launch<long long>(idx, out, n, seg, skv, dev, s);
}
