// Shared device helpers for the sm_103a radix-sort kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lsdrs.h"

namespace lsdrs {

constexpr int kWarp = 32;
constexpr unsigned kFull = 0xFFFFFFFFu;

// Look-back status word: [P:1][A:1][value:30].  A = the tile's own digit
// count is published; P = the inclusive prefix over the row's tiles up to
// this one is published.  Zero means "nothing yet".
constexpr uint32_t kFlagA = 1u << 30;
constexpr uint32_t kFlagP = 1u << 31;
constexpr uint32_t kValueMask = kFlagA - 1u;
constexpr uint64_t kMaxRowLen = kValueMask;  // counts must fit in 30 bits

// Device error word values (mirrors rs_status).
constexpr uint32_t kErrNone = 0;
constexpr uint32_t kErrLookback = RS_ERR_LOOKBACK_TIMEOUT;

__device__ __forceinline__ uint32_t lanemask_lt() {
  uint32_t m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}

__device__ __forceinline__ uint32_t lane_id() {
  uint32_t l;
  asm("mov.u32 %0, %%laneid;" : "=r"(l));
  return l;
}

__device__ __forceinline__ uint64_t global_timer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Relaxed, GPU-scope accesses for the look-back words: the flag and the
// value share one 32-bit word, so no further ordering is needed.
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(uint32_t* p, uint32_t v) {
  asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Streaming loads of data read exactly once per pass.
template <typename T>
__device__ __forceinline__ T ld_stream(const T* p) {
  return __ldcs(p);
}

__host__ __device__ constexpr inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

}  // namespace lsdrs
