// K-SMALL: a whole sort of at most one tile of keys (a small flat sort, or
// each row of a row-wise sort whose rows fit in a tile) in one CTA, every
// pass in shared memory: no upfront histogram, no scan kernel, no look-back
// (the tile is the whole row, so its digit starts are the bucket bases),
// one launch for the whole sort.
//
// Per pass (CUDA Handbook ch. 16, Listing 16-8, on one tile): the warp
// ranking and digit scan of the onesweep kernel give every key its
// position in the pass's stable order; keys and payloads are scattered to
// those positions in shared memory and read back warp-striped, which is the
// next pass's input order.  Lanes past the end of the row take the highest
// digit in every pass, so they stay behind every real key.
#include "onesweep.cuh"

namespace lsdrs {

namespace {

template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS>
struct SmallSmem {
  using T = typename KeyOp::T;
  static constexpr int kTile = THREADS * ITEMS;
  static constexpr int W = THREADS / kWarp;
  alignas(16) T stage[kTile];
  alignas(16) uint32_t vals[VK != kValNone ? kTile : 4];
  uint32_t warp_cnt[W][1 << BITS];
  uint32_t warp_tot[W];
};

template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS>
__global__ void __launch_bounds__(THREADS) small_sort_kernel(SmallArgs a) {
  using T = typename KeyOp::T;
  using S = SmallSmem<KeyOp, BITS, VK, THREADS, ITEMS>;
  constexpr int R = 1 << BITS;
  constexpr int W = THREADS / kWarp;
  constexpr int WKEYS = kWarp * ITEMS;
  constexpr bool kVals = VK != kValNone;
  static_assert(R <= THREADS, "one thread per digit");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  grid_dependency_sync();

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t row = blockIdx.x;
  const int valid = static_cast<int>(a.cols);
  const int wpos = warp * WKEYS + lane;  // tile position of item 0
  const uint32_t lt = lanemask_lt();
  if (blockIdx.x == 0 && tid == 0) {
    a.header[kHdrError] = kErrNone;
    a.header[kHdrPassesRun] = static_cast<uint32_t>(a.passes);
  }

  T keys[ITEMS];
  uint32_t vals[ITEMS];
  {
    const T* src = static_cast<const T*>(a.keys_in) + row * a.cols;
    const uint32_t* vsrc = static_cast<const uint32_t*>(a.vals_in) + row * a.cols;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int p = wpos + i * kWarp;
      keys[i] = (p < valid && in_bounds(p < S::kTile, a.header, 20)) ? src[p] : T(0);
      vals[i] = VK == kValIdx ? static_cast<uint32_t>(p) : ((kVals && p < valid) ? vsrc[p] : 0u);
    }
  }

  for (int q = 0; q < a.passes; ++q) {
    const int shift = a.begin_bit + q * BITS;
    const uint32_t mask = q == a.passes - 1 ? a.last_mask : static_cast<uint32_t>(R - 1);
    for (int i = tid; i < W * R; i += THREADS) (&s.warp_cnt[0][0])[i] = 0;
    __syncthreads();

    // rank within the warp
    uint32_t dig[ITEMS], rank[ITEMS];
    uint32_t* wc = s.warp_cnt[warp];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const uint32_t d = wpos + i * kWarp < valid ? KeyOp::digit(keys[i], shift, mask, a.xf)
                                                  : static_cast<uint32_t>(R - 1);
      const uint32_t peers = digit_peers<BITS>(d);
      const bool d_ok = in_bounds(d < R, a.header, 21);
      const uint32_t before = d_ok ? wc[d] : 0u;
      __syncwarp();
      if (d_ok) wc[d] = before + __popc(peers);
      __syncwarp();
      dig[i] = d;
      rank[i] = before + __popc(peers & lt);
    }
    __syncthreads();

    // warp offsets and digit starts (the tile is the whole row)
    uint32_t total = 0;
    if (tid < R) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const uint32_t c = s.warp_cnt[w][tid];
        s.warp_cnt[w][tid] = total;
        total += c;
      }
    }
    uint32_t incl = total;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == kWarp - 1) s.warp_tot[warp] = incl;
    __syncthreads();
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w + 1 < W; ++w)
      if (w < warp) before += s.warp_tot[w];
    if (tid < R) {
      const uint32_t start = before + incl - total;
#pragma unroll
      for (int w = 0; w < W; ++w) s.warp_cnt[w][tid] += start;
    }
    __syncthreads();

    // scatter to this pass's order, then read back warp-striped
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      if (!in_bounds(dig[i] < R, a.header, 22)) continue;
      const uint32_t pos = s.warp_cnt[warp][dig[i]] + rank[i];
      if (!in_bounds(pos < S::kTile, a.header, 23)) continue;
      s.stage[pos] = keys[i];
      if (kVals) s.vals[pos] = vals[i];
    }
    __syncthreads();
    if (q + 1 < a.passes) {
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        keys[i] = s.stage[wpos + i * kWarp];
        if (kVals) vals[i] = s.vals[wpos + i * kWarp];
      }
      __syncthreads();
    }
  }

  // the stage holds the row in sorted order
  T* kout = static_cast<T*>(a.keys_out) + row * a.cols;
  for (int j = tid; j < valid; j += THREADS) {
    kout[j] = s.stage[j];
    if (VK == kValU32) static_cast<uint32_t*>(a.vals_out)[row * a.cols + j] = s.vals[j];
    if (VK == kValIdx)
      static_cast<int64_t*>(a.vals_out)[row * a.cols + j] = static_cast<int64_t>(s.vals[j]);
  }
}

template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS>
cudaError_t launch_small_t(const SmallArgs& a, cudaStream_t s) {
  auto kern = small_sort_kernel<KeyOp, BITS, VK, THREADS, ITEMS>;
  const size_t smem = sizeof(SmallSmem<KeyOp, BITS, VK, THREADS, ITEMS>);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, static_cast<unsigned>(a.rows), THREADS, smem, s, a);
}

// Three tile sizes: 1,024 keys (256 threads x 4), 4,096 (512 x 8) and 8,192
// (1,024 x 8; more items per thread would not fit the registers).
template <class KeyOp, int BITS, int VK>
cudaError_t launch_small_b(const SmallArgs& a, cudaStream_t s) {
  if (a.cols <= 1024) return launch_small_t<KeyOp, BITS, VK, 256, 4>(a, s);
  if (a.cols <= 4096) return launch_small_t<KeyOp, BITS, VK, 512, 8>(a, s);
  return launch_small_t<KeyOp, BITS, VK, 1024, 8>(a, s);
}

template <class KeyOp, int VK>
cudaError_t launch_small_k(int bits, const SmallArgs& a, cudaStream_t s) {
  if (bits == 8) return launch_small_b<KeyOp, 8, VK>(a, s);
  if (bits == 4) return launch_small_b<KeyOp, 4, VK>(a, s);
  return cudaErrorInvalidValue;
}

template <class KeyOp>
cudaError_t launch_small_v(ValKind v, int bits, const SmallArgs& a, cudaStream_t s) {
  if (v == kValNone) return launch_small_k<KeyOp, kValNone>(bits, a, s);
  if (v == kValU32) return launch_small_k<KeyOp, kValU32>(bits, a, s);
  return cudaErrorInvalidValue;
}

}  // namespace

bool small_sort_fits(KeyKind k, ValKind v, int bits, int64_t cols) {
  if (cols > kSmallMaxKeys || (bits != 4 && bits != 8)) return false;
  if (k == kKeyF16) return v == kValIdx && bits == 8;
  return v != kValIdx;
}

cudaError_t launch_small(KeyKind k, ValKind v, int bits, const SmallArgs& a, cudaStream_t s) {
  if (a.rows == 0) return cudaSuccess;
  switch (k) {
    case kKeyU32: return launch_small_v<KeyU32>(v, bits, a, s);
    case kKeyX32: return launch_small_v<KeyX32>(v, bits, a, s);
    case kKeyU64: return launch_small_v<KeyU64>(v, bits, a, s);
    case kKeyX64: return launch_small_v<KeyX64>(v, bits, a, s);
    case kKeyF16:
      if (v != kValIdx || bits != 8) return cudaErrorInvalidValue;
      return launch_small_b<KeyF16Bits, 8, kValIdx>(a, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
