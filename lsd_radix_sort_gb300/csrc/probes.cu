// Measurement and failure-detection kernels: the copy roofline probe and a
// look-back wait on a word that nothing sets.
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

cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const size_t n16 = bytes / 16;
  size_t want = (n16 + kCopyThreads * 4 - 1) / (kCopyThreads * 4);
  size_t grid = static_cast<size_t>(sms) * 4;
  if (want < grid) grid = want > 0 ? want : 1;
  copy_kernel<<<static_cast<unsigned>(grid), kCopyThreads, 0, s>>>(
      static_cast<uint4*>(dst), static_cast<const uint4*>(src), n16);
  return cudaGetLastError();
}

cudaError_t launch_timeout_probe(uint32_t* word, uint32_t* error, uint64_t timeout_ns,
                                 cudaStream_t s) {
  timeout_probe_kernel<<<1, 1, 0, s>>>(word, error, timeout_ns);
  return cudaGetLastError();
}

}  // namespace lsdrs
