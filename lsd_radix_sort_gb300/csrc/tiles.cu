// Precomputed tile offsets: the alternative to the decoupled look-back for
// row-wise sorts (FlagTree PR #1084, section 2, "precompute each tile": a
// histogram kernel counts every digit of every tile of a pass's input, the
// counts are scanned over the tiles of each row, and the scatter then reads
// its tile's offsets instead of waiting on its predecessors).  It reads the
// keys once more per pass, which the look-back does not.
//
// K-TCOUNT: one CTA per tile; per-warp shared-memory counters (a warp's
//           increments of one digit serialise only within the warp), summed
//           into counts[tile][d].
// K-TSCAN:  one CTA per row, thread d walks the row's tiles in order and
//           replaces each count by the digit's base plus the counts of the
//           earlier tiles (the tile's first output position of digit d).
#include "common.cuh"
#include "kernels.h"
#include "keys.cuh"

namespace lsdrs {

namespace {

constexpr int kCountThreads = 256;

template <class KeyOp, int BITS>
__global__ void __launch_bounds__(kCountThreads) tile_count_kernel(TileCountArgs a) {
  using T = typename KeyOp::T;
  constexpr int R = 1 << BITS;
  constexpr int W = kCountThreads / kWarp;
  __shared__ uint32_t cnt[W][R];
  grid_dependency_sync();
  const int tid = threadIdx.x;
  for (int i = tid; i < W * R; i += kCountThreads) (&cnt[0][0])[i] = 0;
  __syncthreads();
  const int64_t tile = blockIdx.x;
  const int64_t row = tile / a.tiles_per_row;
  const int64_t begin = (tile - row * a.tiles_per_row) * a.tile;
  const int64_t left = a.cols - begin;
  const int valid = static_cast<int>(left < a.tile ? left : a.tile);
  const T* src = static_cast<const T*>(a.keys) + row * a.cols + begin;
  uint32_t* wc = cnt[tid / kWarp];
  for (int i = tid; i < valid; i += kCountThreads)
    atomicAdd(wc + KeyOp::digit(ld_stream(src + i), a.shift, a.mask, a.xf), 1u);
  __syncthreads();
  for (int d = tid; d < R; d += kCountThreads) {
    uint32_t sum = 0;
#pragma unroll
    for (int w = 0; w < W; ++w) sum += cnt[w][d];
    a.offsets[tile * R + d] = sum;
  }
}

template <int R>
__global__ void __launch_bounds__(R < kWarp ? kWarp : R) tile_scan_kernel(TileCountArgs a) {
  grid_dependency_sync();
  const int d = threadIdx.x;
  if (d >= R) return;
  const int64_t row = blockIdx.x;
  uint32_t run = a.bases[row * a.bases_row_stride + d];
  uint32_t* c = a.offsets + row * a.tiles_per_row * R + d;
  for (int64_t t = 0; t < a.tiles_per_row; ++t) {
    const uint32_t v = c[t * R];
    c[t * R] = run;
    run += v;
  }
}

}  // namespace

cudaError_t launch_tile_counts_f16(const TileCountArgs& a, cudaStream_t s) {
  const int64_t tiles = a.rows * a.tiles_per_row;
  if (tiles == 0) return cudaSuccess;
  cudaError_t e = launch_kernel(tile_count_kernel<KeyF16Bits, 8>, static_cast<unsigned>(tiles),
                                kCountThreads, 0, s, a);
  if (e != cudaSuccess) return e;
  return launch_kernel(tile_scan_kernel<256>, static_cast<unsigned>(a.rows), 256, 0, s, a);
}

}  // namespace lsdrs
