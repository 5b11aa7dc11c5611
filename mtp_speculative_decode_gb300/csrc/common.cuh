// Shared device/host helpers of libmtpsd (internal header).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>

#include "../../include/mtpsd.h"

#define MTPSD_HD __host__ __device__ __forceinline__

namespace mtpsd {

// Thread-local error message for mtpsd_last_error().
void set_error(const char* fmt, ...);

inline int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return MTPSD_ECUDA;
  }
  return MTPSD_OK;
}

__device__ __forceinline__ void flag_status(int32_t* st, int32_t bit) {
  if (st) atomicOr(st, bit);
}

// Request owning query row r: the b with row_offsets[b] <= r < row_offsets[b+1].
__device__ __forceinline__ int request_of_row(const uint32_t* row_offsets, int B, uint32_t r) {
  int lo = 0, hi = B;  // answer in [lo, hi)
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (row_offsets[mid] <= r) lo = mid; else hi = mid;
  }
  return lo;
}

// The same search by a whole warp (all 32 lanes call it): each round loads 32 evenly spaced offsets
// at once and keeps the last one <= r, so B <= 32 takes one round of loads and B <= 1024 two,
// instead of log2(B) dependent loads.
__device__ __forceinline__ int request_of_row_warp(const uint32_t* row_offsets, int B, uint32_t r) {
  const int lane = threadIdx.x & 31;
  int lo = 0, n = B;  // answer in [lo, lo + n): row_offsets[lo] <= r
  while (n > 1) {
    const int step = (n + 31) >> 5;
    const int c = lo + lane * step;
    const bool le = c < lo + n && row_offsets[c] <= r;
    const unsigned m = __ballot_sync(0xffffffffu, le) | 1u;   // lane 0 (c = lo) holds by the invariant
    const int k = 31 - __clz((int)m);
    const int c_k = lo + k * step;
    n = min(step, lo + n - c_k);
    lo = c_k;
  }
  return lo;
}

// Pool slot of position s of request b in a paged cache (block table bt [B, stride], pages of
// 2^shift tokens), or -1 when s is negative, lies past the table's width or its page entry is negative.
__device__ __forceinline__ int64_t paged_slot(const int32_t* bt, int32_t stride, int32_t shift, int b, int64_t s) {
  if (s < 0) return -1;
  const int64_t pg = s >> shift;
  if (pg >= stride) return -1;
  const int32_t e = __ldg(bt + (int64_t)b * stride + pg);
  if (e < 0) return -1;
  return ((int64_t)e << shift) | (s & ((1LL << shift) - 1));
}

MTPSD_HD int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

// Programmatic dependent launch.  Every kernel of the library is launched with launch_k(), which lets
// it start while the previous kernel on the stream finishes; it calls griddep_wait() before its first
// access to global memory (this waits until the previous grid has completed and its writes are
// visible) and griddep_launch_dependents() right after, so the next kernel's blocks may be scheduled
// as soon as this one's have all started.  Outside such a launch both are no-ops.
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                            Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Device facts and once-per-device set-up, keyed by the current device ordinal, so a process that
// drives several GPUs gets each one's own values.  Thread-safe: the caches are atomics, and two threads
// that race only repeat an idempotent query or attribute call.
constexpr int kMaxCachedDevices = 64;

inline int current_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = 0;
  return dev;
}

inline int device_attr_cached(std::atomic<int>* cache, cudaDeviceAttr attr, int fallback) {
  const int dev = current_device();
  if (dev >= 0 && dev < kMaxCachedDevices) {
    const int v = cache[dev].load(std::memory_order_relaxed);
    if (v) return v;
  }
  int v = 0;
  if (cudaDeviceGetAttribute(&v, attr, dev) != cudaSuccess || v <= 0) v = fallback;
  if (dev >= 0 && dev < kMaxCachedDevices) cache[dev].store(v, std::memory_order_relaxed);
  return v;
}

inline int num_sms() {
  static std::atomic<int> cache[kMaxCachedDevices];
  return device_attr_cached(cache, cudaDevAttrMultiProcessorCount, 148);
}

inline int cc_major() {
  static std::atomic<int> cache[kMaxCachedDevices];
  return device_attr_cached(cache, cudaDevAttrComputeCapabilityMajor, -1);
}

// Raises a kernel's dynamic shared-memory limit on the current device, once per device (done: one
// bit per device ordinal, owned by the caller for that kernel).  False when the call failed.
template <typename Kernel>
inline bool set_smem_limit_once(Kernel kernel, int bytes, std::atomic<uint64_t>& done) {
  const int dev = current_device();
  const bool cacheable = dev >= 0 && dev < kMaxCachedDevices;
  const uint64_t bit = cacheable ? (1ull << dev) : 0;
  if (cacheable && (done.load(std::memory_order_acquire) & bit)) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) return false;
  if (cacheable) done.fetch_or(bit, std::memory_order_acq_rel);
  return true;
}

// Order-preserving map of a float to uint32 (larger float -> larger key).
__device__ __forceinline__ uint32_t float_key(float f) {
  uint32_t u = __float_as_uint(f == 0.f ? 0.f : f);   // -0 and +0 compare equal
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  uint32_t u = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(u);
}

}  // namespace mtpsd
