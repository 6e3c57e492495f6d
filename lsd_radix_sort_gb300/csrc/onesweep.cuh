// K-SWEEP: one stable scatter pass of LSD radix sort ("onesweep").
//
// What a pass computes (CUDA Handbook ch. 16, Listing 16-8 step 3; DSA CUDA
// from First Principles section 13.2): the key at input position i with
// digit d goes to
//     base[d] + #{ j < i : digit(j) == d },
// where base[d] is the exclusive scan of the digit counts (from K-SCAN).
//
// How one CTA computes it for a tile of THREADS * ITEMS consecutive keys:
//  1. The tile index comes from an atomic counter, so tiles start in index
//     order and every tile a CTA waits on belongs to a CTA that is already
//     running (forward progress of the look-back).
//  2. Keys are loaded warp-striped: warp w owns a contiguous run of 32*ITEMS
//     keys and its item i covers keys 32*i .. 32*i+31 of that run, one per
//     lane, so (warp, item, lane) order is input order.
//  3. Rank within the warp: for each item, the lanes holding the same digit
//     are found by one ballot per digit bit; a lane's rank is the number of
//     such peers in lower lanes plus the warp's running count of that digit
//     (a per-warp shared-memory counter that the lowest peer advances).
//     This is the per-digit exclusive scan of the indicator "digit == d"
//     (section 13.2's rank within digit), done for all digits at once.
//  4. A per-digit scan over the warps gives each warp's offset and the
//     tile's digit counts; the counts are published at once for later tiles
//     (decoupled look-back, flag A), then a scan over the digits gives each
//     digit's start inside the tile.
//  5. Keys are placed in shared memory in tile-sorted order.
//  6. Look-back: for each digit, the counts of earlier tiles of the row are
//     summed walking backwards until a tile that has published its inclusive
//     prefix (flag P); this tile then publishes its own inclusive prefix.
//     The precomputed alternative (per-tile offsets from a separate pass,
//     FlagTree PR #1084 section 2) needs a second read of the keys; the
//     look-back needs none.  Every wait is bounded in time.
//  7. Thread j writes staged key j to base[d] + prefix[d] + (j - start[d]):
//     every digit's keys leave as one contiguous run ("100 Days of GPU",
//     day 35: after the local sort the write out is one run per digit).
//     Payloads follow through the same staging buffer.
// Lanes past the end of the last tile take the highest digit, rank after
// every real key of the tile, are not counted in the published counts and
// are not stored (the page's sentinel padding, without the padding).
#pragma once
#include "common.cuh"
#include "kernels.h"
#include "keys.cuh"

namespace lsdrs {

// Lanes of the warp whose digit equals this lane's digit.
template <int BITS>
__device__ __forceinline__ uint32_t digit_peers(uint32_t d) {
  uint32_t peers = kFull;
#pragma unroll
  for (int b = 0; b < BITS; ++b) {
    const bool bit = (d >> b) & 1u;
    const uint32_t votes = __ballot_sync(kFull, bit);
    peers &= bit ? votes : ~votes;
  }
  return peers;
}

// Bounded wait for a non-zero look-back word.  On timeout, or when another
// tile has already reported an error, records the error and returns a word
// with flag P and value 0 so that the walk ends.
__device__ __forceinline__ uint32_t wait_status(const uint32_t* p, uint32_t* error,
                                                uint64_t timeout_ns) {
  uint32_t v = ld_relaxed(p);
  if (v != 0) return v;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  for (;;) {
    v = ld_relaxed(p);
    if (v != 0) return v;
    if ((++spins & 63u) == 0) {
      if (ld_relaxed(error) != kErrNone) return kFlagP;
      if (global_timer_ns() - t0 > timeout_ns) {
        atomicCAS(error, kErrNone, kErrLookback);
        return kFlagP;
      }
    }
  }
}

template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS>
struct SweepSmem {
  using T = typename KeyOp::T;
  static constexpr int kRadix = 1 << BITS;
  static constexpr int kWarps = THREADS / kWarp;
  static constexpr int kTile = THREADS * ITEMS;
  using V = uint32_t;  // staged payload word (u32 or int32 index)
  static constexpr size_t kStageBytes =
      (VK != kValNone && sizeof(V) > sizeof(T)) ? kTile * sizeof(V) : kTile * sizeof(T);
  alignas(16) unsigned char stage[kStageBytes];
  uint32_t warp_cnt[kWarps][kRadix];
  uint32_t tile_start[kRadix];
  uint32_t g_off[kRadix];
  uint32_t tile_id;
  uint32_t abort;
};

template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS, int MINB>
__global__ void __launch_bounds__(THREADS, MINB) onesweep_kernel(SweepArgs a) {
  using T = typename KeyOp::T;
  using S = SweepSmem<KeyOp, BITS, VK, THREADS, ITEMS>;
  constexpr int R = S::kRadix;
  constexpr int W = S::kWarps;
  constexpr int TILE = S::kTile;
  constexpr int WKEYS = kWarp * ITEMS;
  static_assert(R <= THREADS, "one thread per digit");

  extern __shared__ __align__(16) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  T* stage_keys = reinterpret_cast<T*>(s.stage);
  uint32_t* stage_vals = reinterpret_cast<uint32_t*>(s.stage);

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  if (tid == 0) {
    s.tile_id = atomicAdd(a.tile_counter, 1u);
    s.abort = ld_relaxed(a.error) != kErrNone;
  }
  for (int i = tid; i < W * R; i += THREADS) (&s.warp_cnt[0][0])[i] = 0;
  __syncthreads();

  const int64_t tile = s.tile_id;
  const int64_t row = tile / a.tiles_per_row;
  const int64_t t = tile - row * a.tiles_per_row;
  const int64_t row_base = row * a.cols;
  const int64_t tile_begin = t * TILE;
  const int valid = static_cast<int>(a.cols - tile_begin < TILE ? a.cols - tile_begin : TILE);
  uint32_t* status_tile = a.status + tile * R;

  if (s.abort) {  // an earlier tile failed: release successors and stop
    if (tid < R) st_relaxed(status_tile + tid, kFlagP);
    if (a.status_zero != nullptr && tid < R) a.status_zero[tile * R + tid] = 0;
    return;
  }

  // ---- 2. load (warp-striped) -------------------------------------------
  const int wpos = warp * WKEYS + lane;  // tile position of item 0
  const T* kin = static_cast<const T*>(a.keys_in) + row_base + tile_begin + wpos;
  T keys[ITEMS];
  if (valid == TILE) {
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) keys[i] = ld_stream(kin + i * kWarp);
  } else {
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      keys[i] = (wpos + i * kWarp < valid) ? ld_stream(kin + i * kWarp) : T(0);
  }
  uint32_t vals[VK == kValNone ? 1 : ITEMS];
  if constexpr (VK != kValNone) {
    if (VK == kValIdx && a.vals_in == nullptr) {
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) vals[i] = static_cast<uint32_t>(tile_begin + wpos + i * kWarp);
    } else {
      const uint32_t* vin = static_cast<const uint32_t*>(a.vals_in) + row_base + tile_begin + wpos;
      if (valid == TILE) {
#pragma unroll
        for (int i = 0; i < ITEMS; ++i) vals[i] = ld_stream(vin + i * kWarp);
      } else {
#pragma unroll
        for (int i = 0; i < ITEMS; ++i)
          vals[i] = (wpos + i * kWarp < valid) ? ld_stream(vin + i * kWarp) : 0u;
      }
    }
  }

  // ---- 3. rank within the warp ------------------------------------------
  // packed[i] = digit << 16 | rank of the item among the warp's keys of
  // that digit.
  uint32_t packed[ITEMS];
  uint32_t* wc = s.warp_cnt[warp];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const uint32_t d = (wpos + i * kWarp < valid) ? KeyOp::digit(keys[i], a.shift, a.mask, a.flip)
                                                  : static_cast<uint32_t>(R - 1);
    const uint32_t peers = digit_peers<BITS>(d);
    const int leader = __ffs(peers) - 1;
    uint32_t before = 0;
    if (lane == leader) {
      before = wc[d];
      wc[d] = before + __popc(peers);
    }
    before = __shfl_sync(kFull, before, leader);
    __syncwarp();
    packed[i] = (d << 16) | (before + __popc(peers & lanemask_lt()));
  }
  __syncthreads();

  // ---- 4. warp offsets, tile counts, publish, digit starts --------------
  uint32_t my_count = 0;  // this tile's count of digit tid (without padding)
  if (tid < R) {
    uint32_t sum = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) {
      const uint32_t c = s.warp_cnt[w][tid];
      s.warp_cnt[w][tid] = sum;
      sum += c;
    }
    s.tile_start[tid] = sum;
    my_count = (tid == R - 1) ? sum - static_cast<uint32_t>(TILE - valid) : sum;
    st_relaxed(status_tile + tid, (t == 0 ? kFlagP : kFlagA) | my_count);
  }
  __syncthreads();
  if (warp == 0) {  // exclusive scan of tile_start over the digits
    constexpr int PER = (R + kWarp - 1) / kWarp;
    uint32_t v[PER];
    uint32_t local = 0;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int d = lane * PER + k;
      v[k] = d < R ? s.tile_start[d] : 0u;
      local += v[k];
    }
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    uint32_t run = incl - local;
#pragma unroll
    for (int k = 0; k < PER; ++k) {
      const int d = lane * PER + k;
      if (d < R) s.tile_start[d] = run;
      run += v[k];
    }
  }
  __syncthreads();

  // ---- 5. stage keys in tile-sorted order -------------------------------
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const uint32_t d = packed[i] >> 16;
    const uint32_t pos = s.tile_start[d] + s.warp_cnt[warp][d] + (packed[i] & 0xFFFFu);
    stage_keys[pos] = keys[i];
    packed[i] = pos;  // keep the staging slot for the payload
  }

  // ---- 6. decoupled look-back -------------------------------------------
  if (tid < R) {
    uint32_t excl = 0;
    if (t > 0) {
      const uint32_t* p = status_tile - R + tid;
      for (;;) {
        const uint32_t v = wait_status(p, a.error, a.timeout_ns);
        excl += v & kValueMask;
        if (v & kFlagP) break;
        p -= R;
      }
      st_relaxed(status_tile + tid, kFlagP | (excl + my_count));
    }
    s.g_off[tid] = a.bases[row * a.bases_row_stride + tid] + excl - s.tile_start[tid];
  }
  __syncthreads();

  // ---- 7. contiguous per-digit runs out ---------------------------------
  T* kout = static_cast<T*>(a.keys_out) + row_base;
  uint32_t dst[VK == kValNone ? 1 : ITEMS];
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int j = i * THREADS + tid;
    if (j < valid) {
      const T k = stage_keys[j];
      const uint32_t d = KeyOp::digit(k, a.shift, a.mask, a.flip);
      const uint32_t g = s.g_off[d] + static_cast<uint32_t>(j);
      kout[g] = k;
      if constexpr (VK != kValNone) dst[i] = g;
    }
  }
  if constexpr (VK != kValNone) {
    __syncthreads();
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) stage_vals[packed[i]] = vals[i];
    __syncthreads();
    if (VK == kValIdx && a.wide_out) {
      int64_t* vout = static_cast<int64_t*>(a.vals_out) + row_base;
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        const int j = i * THREADS + tid;
        if (j < valid) vout[dst[i]] = static_cast<int64_t>(static_cast<int32_t>(stage_vals[j]));
      }
    } else {
      uint32_t* vout = static_cast<uint32_t*>(a.vals_out) + row_base;
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        const int j = i * THREADS + tid;
        if (j < valid) vout[dst[i]] = stage_vals[j];
      }
    }
  }

  if (a.status_zero != nullptr && tid < R) a.status_zero[tile * R + tid] = 0;
}

template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS, int MINB>
cudaError_t launch_sweep_t(const SweepArgs& a, int64_t grid, cudaStream_t s) {
  using S = SweepSmem<KeyOp, BITS, VK, THREADS, ITEMS>;
  auto kern = onesweep_kernel<KeyOp, BITS, VK, THREADS, ITEMS, MINB>;
  const size_t smem = sizeof(S);
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  kern<<<static_cast<unsigned>(grid), THREADS, smem, s>>>(a);
  return cudaGetLastError();
}

template <class KeyOp, int VK, int THREADS, int ITEMS, int MINB>
cudaError_t launch_sweep_bits(int bits, const SweepArgs& a, int64_t grid, cudaStream_t s) {
  switch (bits) {
    case 1: return launch_sweep_t<KeyOp, 1, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 2: return launch_sweep_t<KeyOp, 2, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 3: return launch_sweep_t<KeyOp, 3, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 4: return launch_sweep_t<KeyOp, 4, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 5: return launch_sweep_t<KeyOp, 5, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 6: return launch_sweep_t<KeyOp, 6, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 7: return launch_sweep_t<KeyOp, 7, VK, THREADS, ITEMS, MINB>(a, grid, s);
    case 8: return launch_sweep_t<KeyOp, 8, VK, THREADS, ITEMS, MINB>(a, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsdrs
