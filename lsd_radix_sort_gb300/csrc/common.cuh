// Shared device helpers for the sm_103a radix-sort kernels.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

#include "../../include/lsdrs.h"

// Programmatic dependent launch between the kernels of one sort: each
// kernel is launched with programmatic stream serialisation, so the next
// kernel of the stream may be scheduled while this one drains; every kernel
// waits for its predecessors' completion and memory before its first global
// access (griddepcontrol.wait), so the order of memory operations is that of
// plain stream order.  0 launches plainly (A/B builds).
#ifndef LSDRS_PDL
#define LSDRS_PDL 1
#endif

// Bounds-checked build (LSDRS_CHECKED=1): every shared and global index of
// the scatter, histogram and small-sort kernels is tested before the access;
// a failed test is recorded in the scratch header and the access is skipped.
#ifndef LSDRS_CHECKED
#define LSDRS_CHECKED 0
#endif

namespace lsdrs {

constexpr int kWarp = 32;

// First statement of every kernel of a sort: wait for the grids this one
// depends on (a no-op when launched without the attribute), then let the
// next grid of the stream be scheduled.
__device__ __forceinline__ void grid_dependency_sync() {
#if LSDRS_PDL
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
#endif
}

// Host: launch `kern` with programmatic stream serialisation (LSDRS_PDL),
// else with a plain launch.  Returns the launch error.
template <class... KArgs, class... Args>
cudaError_t launch_kernel(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                          cudaStream_t s, Args&&... args) {
#if LSDRS_PDL
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
#else
  kern<<<grid, block, smem, s>>>(static_cast<KArgs>(args)...);
  return cudaGetLastError();
#endif
}
constexpr unsigned kFull = 0xFFFFFFFFu;

// Look-back status word: [P:1][A:1][value] in 32 bits (30-bit value) or 64
// bits (62-bit value).  A = the tile's own digit count is published; P = the
// inclusive prefix over the row's tiles up to this one is published.  Zero
// means "nothing yet".  Flag and value share one word, so one relaxed load
// sees a consistent pair.
template <class SW>
struct LookbackWord {
  static constexpr SW kFlagA = SW(1) << (8 * sizeof(SW) - 2);
  static constexpr SW kFlagP = SW(1) << (8 * sizeof(SW) - 1);
  static constexpr SW kValueMask = kFlagA - 1;
};
constexpr uint32_t kFlagA = LookbackWord<uint32_t>::kFlagA;
constexpr uint32_t kFlagP = LookbackWord<uint32_t>::kFlagP;
constexpr uint32_t kValueMask = LookbackWord<uint32_t>::kValueMask;

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

// 64-bit look-back words (flat sorts of 2^30 keys or more).
__device__ __forceinline__ uint64_t ld_relaxed(const uint64_t* p) {
  uint64_t v;
  asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_relaxed(uint64_t* p, uint64_t v) {
  asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Streaming loads of data read exactly once per pass.
template <typename T>
__device__ __forceinline__ T ld_stream(const T* p) {
  return __ldcs(p);
}

// A hint that the 128-byte line at global address p will be read soon:
// fetch it into L2 (no fault, no result).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile(
      "{\n\t.reg .u64 g;\n\tcvta.to.global.u64 g, %0;\n\tprefetch.global.L2 [g];\n\t}" ::"l"(p));
}

// ---- mbarrier + 1-D bulk copy (TMA) helpers -------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
               : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
               "r"(bytes)
               : "memory");
}

// Global -> shared copy of `bytes` (multiple of 16, both ends 16-byte
// aligned); completion is signalled on `bar` as transaction bytes.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes,
                                              uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
          "r"(smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Limit on the second wait for a bulk copy whose first wait timed out: the
// copy writes the CTA's shared memory, so the CTA waits for it (boundedly)
// before going on.
constexpr uint64_t kCopyDrainNs = 1000000000ull;

// Wait for phase `parity` of `bar` to complete, giving up after timeout_ns.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity,
                                                  uint64_t timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (;;) {
    if (mbar_try_wait(bar, parity)) return true;
    if (global_timer_ns() - t0 > timeout_ns) return false;
  }
}

// Scratch-header words of a bounds-checked build: the number of index tests
// that failed and the site (a small code per access) of the first one.
constexpr int kHdrViolations = 192;

// Index test of a bounds-checked build: true when `ok`; otherwise counts
// the failure in the scratch header and returns false, so that the caller
// skips the access.  Always true in other builds.
__device__ __forceinline__ bool in_bounds(bool ok, uint32_t* header, uint32_t site) {
#if LSDRS_CHECKED
  if (!ok) {
    atomicAdd(header + kHdrViolations, 1u);
    atomicCAS(header + kHdrViolations + 1, 0u, site);
  }
  return ok;
#else
  (void)header;
  (void)site;
  return true;
#endif
}

__host__ __device__ constexpr inline size_t align_up(size_t x, size_t a) {
  return (x + a - 1) / a * a;
}

}  // namespace lsdrs
