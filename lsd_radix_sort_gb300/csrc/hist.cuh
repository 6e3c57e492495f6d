// K-HIST: digit histograms of every pass from one read of the keys.
//
// A pass only reorders keys, so the count of each digit of pass p is the
// same in the unsorted input as in pass p's input; one read of the keys
// therefore yields the histograms of all passes (FlagTree PR #1084,
// section 2: "compute_global_hist_kernel" fills a (passes, 2^b) table per
// row in one sweep).  Counting uses shared-memory counters private to the
// CTA ("privatized" histograms, CUDA Handbook ch. 16 section 16.3, named in
// the Radix Sort section as usable without modification), replicated over
// lane columns so that a warp's increments never serialise on one counter,
// whatever the key distribution.
// Each CTA writes its partial counts to its own slot; K-SCAN adds the slots
// and scans (DSA CUDA from First Principles, section 13.1: the base of digit
// d is the exclusive prefix sum of the counts of the digits below it).
#pragma once
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "keys.cuh"

namespace lsdrs {

// Counter columns per digit: lane l counts into column l % kCols.  With 32
// columns every lane of a warp owns its own column and bank, so a warp's 32
// increments never collide, whatever the digits are (constant input included).
// 16 columns when 32 would not fit in shared memory (64-bit keys, 8-bit digits).
// Row-wise 16-bit sorts count each row in its own CTA (a row of a few tens
// of thousands of keys): threads and counter columns for those (build-time).
#ifndef LSDRS_HIST_F16_THREADS
#define LSDRS_HIST_F16_THREADS 512
#endif
#ifndef LSDRS_HIST_F16_COLS
#define LSDRS_HIST_F16_COLS 32
#endif
#ifndef LSDRS_HIST_F16_UNROLL
#define LSDRS_HIST_F16_UNROLL 4
#endif
#ifndef LSDRS_HIST_F16_MINB
#define LSDRS_HIST_F16_MINB 3
#endif

template <class KeyOp, int BITS>
struct HistCfg {
  static constexpr bool kRows = std::is_same<KeyOp, KeyF16Bits>::value;
  static constexpr int kThreads = kRows ? LSDRS_HIST_F16_THREADS : kHistThreads;
  static constexpr int kRadix = 1 << BITS;
  static constexpr int kMaxPasses = (KeyOp::kBits + BITS - 1) / BITS;
  static constexpr int kCols =
      kRows ? LSDRS_HIST_F16_COLS
            : (static_cast<size_t>(kMaxPasses) * kRadix * 32 * sizeof(uint32_t) <= 128 * 1024 ? 32
                                                                                             : 16);
  static constexpr int kVec = 16 / sizeof(typename KeyOp::T);
  static constexpr int kUnroll = kRows ? LSDRS_HIST_F16_UNROLL : 4;
  static constexpr int kMinBlocks = kRows ? LSDRS_HIST_F16_MINB : 1;
  static size_t smem_bytes(int passes) {
    return static_cast<size_t>(passes) * kRadix * kCols * sizeof(uint32_t);
  }
};

// Per-thread view of the counters: shift and mask of every pass held in
// registers; ALL = every pass of the key type is present (the usual case),
// which drops the per-pass bound test.  BYTES = 8-bit digits covering the
// whole key from bit 0, so that pass p's digit is byte p of T(k): the key is
// transformed once and each digit is one byte permute, which keeps the
// counting loop short enough to run at the speed of the key reads.
template <class KeyOp, int BITS, bool ALL, bool BYTES = false>
struct KeyCounter {
  static_assert(!BYTES || (ALL && BITS == 8), "byte digits cover every pass");
  using Cfg = HistCfg<KeyOp, BITS>;
  static constexpr int R = Cfg::kRadix;
  static constexpr int C = Cfg::kCols;
  static constexpr int MP = Cfg::kMaxPasses;
  // many narrow passes (digits of 1-3 bits) would not fit in registers:
  // those compute shift and mask per key instead
  static constexpr bool kHeld = MP <= 16;
  static constexpr int MH = kHeld ? MP : 1;
  uint32_t* col;
  uint32_t* hdr;  // scratch header (bounds-checked builds record failures there)
  int begin_bit, passes;
  uint32_t last_mask;
  KeyXform xf;
  int shift[MH];
  uint32_t mask[MH];

  __device__ __forceinline__ KeyCounter(uint32_t* c, uint32_t* h, int b, int np, uint32_t lm,
                                        const KeyXform& x)
      : col(c), hdr(h), begin_bit(b), passes(np), last_mask(lm), xf(x) {
#pragma unroll
    for (int p = 0; p < MH; ++p) {
      shift[p] = b + p * BITS;
      mask[p] = p == np - 1 ? lm : static_cast<uint32_t>(R - 1);
    }
  }
  // The keys of one 16-byte load.  For 16-bit float keys with byte digits
  // (the row-wise sorts) two keys are transformed at once per 32-bit word:
  // T(u) = u ^ pos ^ (sign(u) ? pos ^ neg : 0) in each half, the sign bits
  // taken to bits 0 and 16 and multiplied by pos ^ neg (below 2^16, so the
  // halves never carry into each other).
  __device__ __forceinline__ void add_vec(const uint4& b) const {
    if constexpr (BYTES && std::is_same<KeyOp, KeyF16Bits>::value) {
      const uint32_t pos = static_cast<uint32_t>(xf.pos) & 0xFFFFu;
      const uint32_t diff = (static_cast<uint32_t>(xf.pos) ^ static_cast<uint32_t>(xf.neg)) & 0xFFFFu;
      const uint32_t pos2 = pos * 0x10001u;
      const uint32_t w4[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint32_t w = w4[q];
        const uint32_t t = w ^ pos2 ^ (((w >> 15) & 0x00010001u) * diff);
#pragma unroll
        for (int h = 0; h < 2; ++h) {      // key h of the word
#pragma unroll
          for (int p = 0; p < 2; ++p) {    // its two byte digits
            const uint32_t d = __byte_perm(t, 0u, 0x4440u + 2 * h + p);
            if (in_bounds(d < R, hdr, 10)) atomicAdd(col + (p * R + d) * C, 1u);
          }
        }
      }
    } else {
      const typename KeyOp::T* ks = reinterpret_cast<const typename KeyOp::T*>(&b);
#pragma unroll
      for (int e = 0; e < 16 / static_cast<int>(sizeof(typename KeyOp::T)); ++e) add(ks[e]);
    }
  }
  __device__ __forceinline__ void add(typename KeyOp::T k) const {
    if constexpr (BYTES) {
      const auto t = KeyOp::encode(k, xf);
#pragma unroll
      for (int p = 0; p < MP; ++p) {
        const uint32_t w = static_cast<uint32_t>(t >> (32 * (p / 4)));
        const uint32_t d = __byte_perm(w, 0u, 0x4440u + (p & 3));
        if (in_bounds(d < R, hdr, 10)) atomicAdd(col + (p * R + d) * C, 1u);
      }
    } else if constexpr (kHeld) {
#pragma unroll
      for (int p = 0; p < MP; ++p) {
        if (ALL || p < passes) {
          const uint32_t d = KeyOp::digit(k, shift[p], mask[p], xf);
          if (in_bounds(d < R && p < passes, hdr, 11)) atomicAdd(col + (p * R + d) * C, 1u);
        }
      }
    } else {
      for (int p = 0; p < passes; ++p) {
        const uint32_t m = p == passes - 1 ? last_mask : static_cast<uint32_t>(R - 1);
        const uint32_t d = KeyOp::digit(k, begin_bit + p * BITS, m, xf);
        if (in_bounds(d < R, hdr, 12)) atomicAdd(col + (p * R + d) * C, 1u);
      }
    }
  }
};

// Counts keys [begin, end) of one row slice: a scalar head up to 16-byte
// alignment, a vectorised body (U 16-byte loads in flight per thread) and a
// scalar tail.
template <class KeyOp, int BITS, bool ALL, bool BYTES>
__device__ __forceinline__ void count_range(const typename KeyOp::T* base, int64_t begin,
                                            int64_t end, int64_t cols,
                                            const KeyCounter<KeyOp, BITS, ALL, BYTES>& c) {
  using T = typename KeyOp::T;
  using Cfg = HistCfg<KeyOp, BITS>;
  constexpr int V = Cfg::kVec;
  constexpr int U = Cfg::kUnroll;
  const int tid = threadIdx.x;
  const uintptr_t addr = reinterpret_cast<uintptr_t>(base + begin);
  int64_t head = static_cast<int64_t>(((16 - (addr & 15)) & 15) / sizeof(T));
  if (head > end - begin) head = end - begin;
  const int64_t body_begin = begin + head;
  const int64_t nvec = (end - body_begin) / V;
  const int64_t body_end = body_begin + nvec * V;
  if (tid < head && in_bounds(begin + tid < cols, c.hdr, 13)) c.add(base[begin + tid]);
  if (tid < end - body_end && in_bounds(body_end + tid < cols, c.hdr, 14))
    c.add(base[body_end + tid]);
  const uint4* vp = reinterpret_cast<const uint4*>(base + body_begin);
  int64_t v = tid;
  for (; v + (U - 1) * Cfg::kThreads < nvec; v += U * Cfg::kThreads) {
    uint4 buf[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      buf[u] = in_bounds(body_begin + (v + u * Cfg::kThreads + 1) * V <= cols, c.hdr, 15)
                   ? __ldcs(vp + v + u * Cfg::kThreads)
                   : make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
    for (int u = 0; u < U; ++u) c.add_vec(buf[u]);
  }
  for (; v < nvec; v += Cfg::kThreads) {
    if (!in_bounds(body_begin + (v + 1) * V <= cols, c.hdr, 16)) continue;
    c.add_vec(__ldcs(vp + v));
  }
}

template <class KeyOp, int BITS>
__global__ void __launch_bounds__(HistCfg<KeyOp, BITS>::kThreads, HistCfg<KeyOp, BITS>::kMinBlocks)
    upfront_hist_kernel(HistArgs a) {
  using T = typename KeyOp::T;
  using Cfg = HistCfg<KeyOp, BITS>;
  constexpr int R = Cfg::kRadix;
  constexpr int C = Cfg::kCols;
  extern __shared__ __align__(16) uint32_t cnt[];
  grid_dependency_sync();

  const int tid = threadIdx.x;
  const int nb = a.passes * R;
  for (int i = tid; i < nb * C; i += Cfg::kThreads) cnt[i] = 0;

  // Zero the look-back words and counters the sweeps start from.
  {
    const size_t stride = static_cast<size_t>(gridDim.x) * Cfg::kThreads;
    for (size_t i = static_cast<size_t>(blockIdx.x) * Cfg::kThreads + tid; i < a.zero_words;
         i += stride)
      if (i < kHdrViolations || i >= kHdrViolations + 2) a.zero_ptr[i] = 0;
  }
  __syncthreads();

  // block -> (row, chunk of the row); 32-bit arithmetic (grids fit it)
  const uint32_t row32 = blockIdx.x / static_cast<uint32_t>(a.chunks_per_row);
  const int64_t row = row32;
  const int64_t chunk = blockIdx.x - row32 * static_cast<uint32_t>(a.chunks_per_row);
  const int64_t begin = chunk * a.chunk_len;
  const int64_t end = begin + a.chunk_len < a.cols ? begin + a.chunk_len : a.cols;
  const T* base = static_cast<const T*>(a.keys) + row * a.cols;
  uint32_t* col = cnt + (tid & (C - 1));
  if (begin < end) {
    if (BITS == 8 && a.passes == Cfg::kMaxPasses && a.begin_bit == 0 && a.last_mask == 0xFFu) {
      const KeyCounter<KeyOp, BITS, true, BITS == 8> c(col, a.zero_ptr, a.begin_bit, a.passes,
                                                       a.last_mask, a.xf);
      count_range(base, begin, end, a.cols, c);
    } else if (a.passes == Cfg::kMaxPasses) {
      const KeyCounter<KeyOp, BITS, true> c(col, a.zero_ptr, a.begin_bit, a.passes, a.last_mask,
                                            a.xf);
      count_range(base, begin, end, a.cols, c);
    } else {
      const KeyCounter<KeyOp, BITS, false> c(col, a.zero_ptr, a.begin_bit, a.passes, a.last_mask,
                                             a.xf);
      count_range(base, begin, end, a.cols, c);
    }
  }
  __syncthreads();

  if constexpr (Cfg::kRows && BITS == 8 && Cfg::kThreads % R == 0) {
    if (a.fused_scan && nb <= Cfg::kThreads) {
      // The row's totals (one CTA per row: the CTA's counts) and their
      // exclusive scan over the digits of each pass: thread t holds digit
      // t % R of pass t / R, and the R threads of a pass are whole warps.
      const int lane = tid & 31, warp = tid >> 5;
      const int p = tid / R, d = tid % R;
      uint32_t total = 0;
      if (tid < nb) {
#pragma unroll
        for (int k = 0; k < C; ++k) total += cnt[tid * C + (k + tid) % C];
      }
      uint32_t incl = total;
#pragma unroll
      for (int o = 1; o < kWarp; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += y;
      }
      __shared__ uint32_t warp_sums[Cfg::kThreads / kWarp];
      if (lane == kWarp - 1) warp_sums[warp] = incl;
      __syncthreads();
      uint32_t excl = incl - total;
      for (int w = p * (R / kWarp); w < warp; ++w) excl += warp_sums[w];
      if (tid < nb) {
        const int64_t o = (row * a.passes + p) * R + d;
        a.bases[o] = excl;
        if (a.hist_out) a.hist_out[o] = total;
        if (a.bases_out) a.bases_out[o] = excl;
      }
      // every pass runs (this CTA zeroed the header word above)
      if (blockIdx.x == 0 && tid == 0) a.zero_ptr[kHdrPassesRun] = static_cast<uint32_t>(a.passes);
      return;
    }
  }

  uint32_t* slot = a.slots + static_cast<int64_t>(blockIdx.x) * nb;
  for (int b = tid; b < nb; b += Cfg::kThreads) {
    uint32_t s = 0;
#pragma unroll
    for (int k = 0; k < C; ++k) s += cnt[b * C + (k + b) % C];
    slot[b] = s;
  }
}

template <class KeyOp, int BITS>
cudaError_t launch_hist_t(const HistArgs& a, int grid, cudaStream_t s) {
  using Cfg = HistCfg<KeyOp, BITS>;
  const size_t smem = Cfg::smem_bytes(a.passes);
  auto kern = upfront_hist_kernel<KeyOp, BITS>;
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, grid, Cfg::kThreads, smem, s, a);
}

template <class KeyOp>
cudaError_t launch_hist_k(int bits, const HistArgs& a, int grid, cudaStream_t s) {
  switch (bits) {
    case 1: return launch_hist_t<KeyOp, 1>(a, grid, s);
    case 2: return launch_hist_t<KeyOp, 2>(a, grid, s);
    case 3: return launch_hist_t<KeyOp, 3>(a, grid, s);
    case 4: return launch_hist_t<KeyOp, 4>(a, grid, s);
    case 5: return launch_hist_t<KeyOp, 5>(a, grid, s);
    case 6: return launch_hist_t<KeyOp, 6>(a, grid, s);
    case 7: return launch_hist_t<KeyOp, 7>(a, grid, s);
    case 8: return launch_hist_t<KeyOp, 8>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsdrs
