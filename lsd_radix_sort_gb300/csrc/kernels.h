// Launch interface between the C ABI (api.cu) and the kernel translation
// units.  Host-side structs only; no templates cross this boundary.
#pragma once
#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace lsdrs {

// Unsigned ascending keys (u32, u64), any other 32- or 64-bit key (signed,
// float, or descending: transformed on the fly), and 16-bit float rows.
enum KeyKind { kKeyU32 = 0, kKeyU64 = 1, kKeyF16 = 2, kKeyX32 = 3, kKeyX64 = 4 };

// The order-preserving map of a key to its unsigned sort key:
// T(k) = k ^ (top bit of k set ? neg : pos) (see keys.cuh).
struct KeyXform {
  uint64_t pos, neg;
};
// Payload carried with the keys: none, a u32 array, or a column index that
// is generated in the first pass, kept as int32 and widened to int64 by the
// last pass.
enum ValKind { kValNone = 0, kValU32 = 1, kValIdx = 2 };

// Threads per CTA and keys per thread of the onesweep kernel, per
// (key, payload) combination.  The tile is THREADS * ITEMS keys.
struct SweepShape {
  int threads;
  int items;
  int min_blocks;  // resident CTAs per SM the register budget is sized for
  int window;      // look-back words read per round trip
  constexpr int tile() const { return threads * items; }
};
// Shapes may be overridden at build time for tuning sweeps, e.g.
// -DLSDRS_U32P_T=256 -DLSDRS_U32P_I=16 -DLSDRS_U32P_B=4 -DLSDRS_U32P_W=4
// (threads, items per thread, CTAs per SM, look-back window); the defaults
// are the fastest measured on GB300 for 2^28-key sorts.
#ifndef LSDRS_U32K_T
#define LSDRS_U32K_T 256
#define LSDRS_U32K_I 28
#define LSDRS_U32K_B 4
#endif
#ifndef LSDRS_U32K_W
#define LSDRS_U32K_W 8
#endif
#ifndef LSDRS_U32P_T
#define LSDRS_U32P_T 256
#define LSDRS_U32P_I 23
#define LSDRS_U32P_B 4
#endif
#ifndef LSDRS_U32P_W
#define LSDRS_U32P_W 4
#endif
#ifndef LSDRS_U64K_T
#define LSDRS_U64K_T 256
#define LSDRS_U64K_I 16
#define LSDRS_U64K_B 3
#endif
#ifndef LSDRS_U64K_W
#define LSDRS_U64K_W 4
#endif
#ifndef LSDRS_U64P_T
#define LSDRS_U64P_T 256
#define LSDRS_U64P_I 18
#define LSDRS_U64P_B 3
#endif
#ifndef LSDRS_U64P_W
#define LSDRS_U64P_W 4
#endif
#ifndef LSDRS_F16_T
#define LSDRS_F16_T 256
#define LSDRS_F16_I 16
#define LSDRS_F16_B 4
#endif
#ifndef LSDRS_F16_W
#define LSDRS_F16_W 4
#endif
constexpr SweepShape kShapeU32Keys{LSDRS_U32K_T, LSDRS_U32K_I, LSDRS_U32K_B, LSDRS_U32K_W};
constexpr SweepShape kShapeU32Pairs{LSDRS_U32P_T, LSDRS_U32P_I, LSDRS_U32P_B, LSDRS_U32P_W};
constexpr SweepShape kShapeU64Keys{LSDRS_U64K_T, LSDRS_U64K_I, LSDRS_U64K_B, LSDRS_U64K_W};
constexpr SweepShape kShapeU64Pairs{LSDRS_U64P_T, LSDRS_U64P_I, LSDRS_U64P_B, LSDRS_U64P_W};
constexpr SweepShape kShapeF16Idx{LSDRS_F16_T, LSDRS_F16_I, LSDRS_F16_B, LSDRS_F16_W};
constexpr SweepShape sweep_shape(KeyKind k, ValKind v) {
  return (k == kKeyU32 || k == kKeyX32) ? (v == kValNone ? kShapeU32Keys : kShapeU32Pairs)
       : (k == kKeyU64 || k == kKeyX64) ? (v == kValNone ? kShapeU64Keys : kShapeU64Pairs)
                      : kShapeF16Idx;
}

constexpr int kHistThreads = 1024;
constexpr int kHistTargetCtas = 608;   // 152 SMs x 4 resident CTAs
constexpr int64_t kHistMinChunk = 4096;
constexpr int kScanThreads = 256;

struct HistArgs {
  const void* keys;
  int64_t rows, cols;
  int chunks_per_row;
  int64_t chunk_len;
  int begin_bit, passes;
  uint32_t last_mask;      // digit mask of the last (possibly narrower) pass
  KeyXform xf;             // key transform
  uint32_t* slots;         // [rows][chunks_per_row][passes][radix] counts
  uint32_t* zero_ptr;      // words zeroed by the grid before any sweep
  size_t zero_words;
};

struct ScanArgs {
  const uint32_t* slots;
  int64_t rows;
  int chunks_per_row;
  int passes;
  int radix;
  uint32_t* hist_out;      // optional [rows][passes][radix] totals
  uint32_t* bases;         // [rows][passes][radix] exclusive scans
};

struct SweepArgs {
  const void* keys_in;
  void* keys_out;
  const void* vals_in;     // null with kValIdx: generate column indices
  void* vals_out;
  int64_t rows, cols;
  int64_t tiles_per_row;
  int64_t full_per_row;    // tiles of a row that hold a whole tile of keys
  int full_tile;           // keys per full tile (set by the pass launcher)
  int shift;
  uint32_t mask;
  KeyXform xf;             // key transform
  int wide_out;            // kValIdx: write int64 indices
  const uint32_t* bases;   // bases of this pass for row 0
  int64_t bases_row_stride;
  uint32_t* status;        // [rows * tiles_per_row][radix] look-back words
  uint32_t* status_zero;   // next pass's look-back words, zeroed here
  uint32_t* tile_counter;
  uint32_t* error;
  uint64_t timeout_ns;
};

cudaError_t launch_hist(KeyKind k, int bits, const HistArgs& a, int grid, cudaStream_t s);
cudaError_t launch_hist_x(KeyKind k, int bits, const HistArgs& a, int grid, cudaStream_t s);
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);
// One scatter pass: a kernel over the full tiles, then one over each row's
// partial tile; *launched receives the number of kernels launched (0-2).
cudaError_t launch_sweep_u32(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_u64(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_x32(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_x64(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_f16(const SweepArgs& a, int* launched, cudaStream_t s);
cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s);
cudaError_t launch_timeout_probe(uint32_t* word, uint32_t* error, uint64_t timeout_ns,
                                 cudaStream_t s);

}  // namespace lsdrs
