// Measurement and failure-detection kernels: the copy roofline probe and a
// look-back wait on a word that nothing sets.
#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace lsdrs {

namespace {

constexpr int kCopyThreads = 512;

__global__ void __launch_bounds__(kCopyThreads) copy_kernel(uint4* __restrict__ dst,
                                                            const uint4* __restrict__ src,
                                                            size_t n16) {
  const size_t stride = static_cast<size_t>(gridDim.x) * kCopyThreads;
  size_t i = static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x;
  for (; i + 3 * stride < n16; i += 4 * stride) {
    uint4 a0 = __ldcs(src + i);
    uint4 a1 = __ldcs(src + i + stride);
    uint4 a2 = __ldcs(src + i + 2 * stride);
    uint4 a3 = __ldcs(src + i + 3 * stride);
    __stcs(dst + i, a0);
    __stcs(dst + i + stride, a1);
    __stcs(dst + i + 2 * stride, a2);
    __stcs(dst + i + 3 * stride, a3);
  }
  for (; i < n16; i += stride) __stcs(dst + i, __ldcs(src + i));
}

// Same bounded wait as the scatter kernels use (see onesweep.cuh).
__global__ void timeout_probe_kernel(uint32_t* word, uint32_t* error, uint64_t timeout_ns) {
  uint32_t v = ld_relaxed(word);
  if (v != 0) return;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  for (;;) {
    v = ld_relaxed(word);
    if (v != 0) return;
    if ((++spins & 63u) == 0) {
      if (ld_relaxed(error) != kErrNone) return;
      if (global_timer_ns() - t0 > timeout_ns) {
        atomicCAS(error, kErrNone, kErrLookback);
        return;
      }
    }
  }
}

}  // namespace

int device_sm_count() {
  constexpr int kMaxDevices = 64;
  static std::atomic<int> cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
  if (dev < kMaxDevices) {
    const int c = cache[dev].load(std::memory_order_relaxed);
    if (c > 0) return c;
  }
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 1;
  if (dev < kMaxDevices) cache[dev].store(sms, std::memory_order_relaxed);
  return sms;
}

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  const int sms = device_sm_count();
  const size_t n16 = bytes / 16;
  size_t want = (n16 + kCopyThreads * 4 - 1) / (kCopyThreads * 4);
  size_t grid = static_cast<size_t>(sms) * 4;
  if (want < grid) grid = want > 0 ? want : 1;
  copy_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, s>>>(
      static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
  return cudaGetLastError();
}

// The finishing step of a sort (see FinishArgs), grid-stride, in the widest
// units that the pointers' alignment and the size allow (16, 4 or 2 bytes:
// every key and payload size is a multiple of 2).
template <class U>
__device__ __forceinline__ void copy_units(void* dst, const void* src, size_t units) {
  U* d = static_cast<U*>(dst);
  const U* s = static_cast<const U*>(src);
  const size_t stride = static_cast<size_t>(gridDim.x) * kCopyThreads;
  for (size_t i = static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x; i < units;
       i += stride)
    __stcs(d + i, __ldcs(s + i));
}

__device__ __forceinline__ void copy_bytes(void* dst, const void* src, size_t bytes) {
  const uintptr_t a = reinterpret_cast<uintptr_t>(dst) | reinterpret_cast<uintptr_t>(src) | bytes;
  if ((a & 15) == 0)
    copy_units<uint4>(dst, src, bytes / 16);
  else if ((a & 3) == 0)
    copy_units<uint32_t>(dst, src, bytes / 4);
  else
    copy_units<unsigned short>(dst, src, bytes / 2);
}

__global__ void __launch_bounds__(kCopyThreads) finish_kernel(FinishArgs f) {
  grid_dependency_sync();
  const uint32_t m = *f.passes_run;
  const void* ksrc = nullptr;
  const void* vsrc = nullptr;
  if (m == 0) {
    ksrc = f.keys_in;
    vsrc = f.vals_in;
    if (f.idx_out != nullptr) {
      const size_t n = static_cast<size_t>(f.rows) * static_cast<size_t>(f.cols);
      const size_t stride = static_cast<size_t>(gridDim.x) * kCopyThreads;
      for (size_t i = static_cast<size_t>(blockIdx.x) * kCopyThreads + threadIdx.x; i < n;
           i += stride)
        f.idx_out[i] = static_cast<int64_t>(i % static_cast<size_t>(f.cols));
    }
  } else if (f.in_place && (m & 1u)) {
    ksrc = f.keys_alt;
    vsrc = f.vals_alt;
  }
  if (ksrc != nullptr && ksrc != f.keys_out) copy_bytes(f.keys_out, ksrc, f.keys_bytes);
  if (vsrc != nullptr && vsrc != f.vals_out && f.vals_bytes)
    copy_bytes(f.vals_out, vsrc, f.vals_bytes);
}

cudaError_t launch_finish(const FinishArgs& f, cudaStream_t s) {
  if (f.keys_bytes % 2 || f.vals_bytes % 2) return cudaErrorInvalidValue;
  const size_t units = (f.keys_bytes > f.vals_bytes ? f.keys_bytes : f.vals_bytes) / 16;
  size_t grid = (units + kCopyThreads - 1) / kCopyThreads;
  const size_t cap = 4 * static_cast<size_t>(device_sm_count());
  if (grid > cap) grid = cap;
  if (grid == 0) grid = 1;
  return launch_kernel(finish_kernel, static_cast<unsigned>(grid), kCopyThreads, 0, s, f);
}

cudaError_t launch_timeout_probe(uint32_t* word, uint32_t* error, uint64_t timeout_ns,
                                 cudaStream_t s) {
  timeout_probe_kernel<<<1, 1, 0, s>>>(word, error, timeout_ns);
  return cudaGetLastError();
}

}  // namespace lsdrs
