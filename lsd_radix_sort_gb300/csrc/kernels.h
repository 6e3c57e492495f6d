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
// kValPack16: row-wise 16-bit sorts of rows of at most 65,536 columns whose
// column index rides in the low half of a packed 32-bit word (KeyF16Packed):
// the first pass reads 16-bit keys and generates the index, the last writes
// the values and int64 indices, the passes between move packed words.
enum ValKind { kValNone = 0, kValU32 = 1, kValIdx = 2, kValPack16 = 3 };
constexpr int64_t kPackMaxCols = 65536;

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
#define LSDRS_U32K_I 30
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
#define LSDRS_U64K_I 22
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
#define LSDRS_F16_I 24
#define LSDRS_F16_B 4
#endif
#ifndef LSDRS_F16_W
#define LSDRS_F16_W 4
#endif
#ifndef LSDRS_F16P_T
#define LSDRS_F16P_T 256
#define LSDRS_F16P_I 32
#define LSDRS_F16P_B 4
#endif
#ifndef LSDRS_F16P_W
#define LSDRS_F16P_W 4
#endif
constexpr SweepShape kShapeU32Keys{LSDRS_U32K_T, LSDRS_U32K_I, LSDRS_U32K_B, LSDRS_U32K_W};
constexpr SweepShape kShapeU32Pairs{LSDRS_U32P_T, LSDRS_U32P_I, LSDRS_U32P_B, LSDRS_U32P_W};
constexpr SweepShape kShapeU64Keys{LSDRS_U64K_T, LSDRS_U64K_I, LSDRS_U64K_B, LSDRS_U64K_W};
constexpr SweepShape kShapeU64Pairs{LSDRS_U64P_T, LSDRS_U64P_I, LSDRS_U64P_B, LSDRS_U64P_W};
constexpr SweepShape kShapeF16Idx{LSDRS_F16_T, LSDRS_F16_I, LSDRS_F16_B, LSDRS_F16_W};
constexpr SweepShape kShapeF16Packed{LSDRS_F16P_T, LSDRS_F16P_I, LSDRS_F16P_B, LSDRS_F16P_W};
// Flat u32 sorts of at most kMidMaxKeys keys take smaller tiles: each pass
// is a fraction of one wave of CTAs, so a tile's serial chain (load, rank,
// look-back, write) sets the pass time, and a shorter tile shortens it
// (measured: 2^16 keys 34.2 -> 32.1 us, 2^16 pairs 38.0 -> 35.0 us per
// sort launched on a stream); from 2^20 keys on the larger tiles are faster.
#ifndef LSDRS_MID_MAX_KEYS
#define LSDRS_MID_MAX_KEYS (1 << 18)
#endif
constexpr int64_t kMidMaxKeys = LSDRS_MID_MAX_KEYS;
constexpr SweepShape kShapeU32KeysMid{256, 14, 4, 8};
constexpr SweepShape kShapeU32PairsMid{256, 12, 4, 4};
constexpr bool mid_tiles(KeyKind k, ValKind v, int64_t rows, int64_t cols) {
  return k == kKeyU32 && v != kValIdx && rows == 1 && cols <= kMidMaxKeys;
}
constexpr SweepShape sweep_shape(KeyKind k, ValKind v, int64_t rows, int64_t cols) {
  return mid_tiles(k, v, rows, cols)     ? (v == kValNone ? kShapeU32KeysMid : kShapeU32PairsMid)
       : (k == kKeyU32 || k == kKeyX32) ? (v == kValNone ? kShapeU32Keys : kShapeU32Pairs)
       : (k == kKeyU64 || k == kKeyX64) ? (v == kValNone ? kShapeU64Keys : kShapeU64Pairs)
       : v == kValPack16                ? kShapeF16Packed
                                        : kShapeF16Idx;
}

constexpr int kHistThreads = 1024;
// K-HIST grid: one 1,024-thread CTA fits an SM (its counters take up to
// 128 KB of shared memory), so a flat sort takes one wave, one CTA per SM of
// the device (device_sm_count): no wave tail.  Scratch is sized for at most
// kMaxHistCtas chunks, which covers any current part.
constexpr int kMaxHistCtas = 256;
constexpr int64_t kHistMinChunk = 4096;
constexpr int kScanThreads = 256;

// Look-back words.  A 32-bit word holds [P:1][A:1][count:30], so it serves
// every chain of fewer than 2^30 keys: every row of a row-wise sort and flat
// sorts below 2^30 keys.  A flat sort of 2^30 keys or more uses 64-bit words,
// [P:1][A:1][count:62].
constexpr int64_t kMaxNarrowKeys = (int64_t(1) << 30) - 1;

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
  // Row-wise 16-bit sorts counted one CTA per row on the static schedule:
  // the CTA scans its own counts into `bases` (and the optional copies), so
  // no K-SCAN runs.  `zero_ptr` is the scratch header.
  int fused_scan;
  uint32_t* bases;         // [rows][passes][radix] exclusive scans
  uint32_t* hist_out;      // optional [rows][passes][radix] totals
  uint32_t* bases_out;     // optional [rows][passes][radix] exclusive scans
};

// Scratch header (u32 words): the device error word, one tile counter per
// pass, and the pass schedule that K-SCAN derives from the histograms.
constexpr int kHdrError = 0;
constexpr int kHdrTileCounter = 1;     // + pass
constexpr int kHdrScanDone = 65;       // K-SCAN CTAs finished
constexpr int kHdrPassesRun = 66;      // passes the schedule executes
constexpr int kHdrNontrivial = 128;    // + pass: some row has two digits in it
constexpr int kHdrProbeWord = 96;      // a word nothing sets, for the timeout probe
constexpr int kMaxPasses = 64;
// Words kHdrViolations.. (common.cuh): bounds-checked builds' failed index
// tests; K-HIST's zeroing skips them, radix_sort_checked_violations reads
// and clears them.

// Buffers a pass reads or writes: the caller's input, the scratch
// ping-pong buffer, the caller's output.
enum PassBuf : uint32_t { kBufIn = 0, kBufAlt = 1, kBufOut = 2 };

// The schedule.  A pass in which every row's keys share one digit is the
// identity permutation (a stable scatter of one bucket) and is skipped; the
// others alternate between the buffers so that the last one run writes the
// caller's output (an in-place sort with an odd number of passes run ends
// in the scratch buffer and is copied back).  K-SCAN writes each pass's
// entry into the top byte of the pass's tile counter, so the atomic that
// hands a CTA its tile also hands it the schedule: tile = value & kTileMask,
// code = value >> kCodeShift.
constexpr int kCodeShift = 24;
constexpr uint32_t kTileMask = (1u << kCodeShift) - 1;
constexpr uint32_t kCodeSrc = 0x03;    // PassBuf of the keys (and u32 payloads) read
constexpr uint32_t kCodeDst = 0x0C;    // PassBuf written, << 2
constexpr uint32_t kCodeOdd = 0x10;    // odd index among the passes run: look-back array 1
constexpr uint32_t kCodeFirst = 0x20;  // first pass run
constexpr uint32_t kCodeLast = 0x40;   // last pass run
constexpr uint32_t kCodeSkip = 0x80;   // identity pass: not run

struct ScanArgs {
  const uint32_t* slots;
  int64_t rows;
  int64_t cols;
  int chunks_per_row;
  int passes;
  int radix;
  uint32_t* hist_out;      // optional [rows][passes][radix] totals
  uint32_t* bases_out;     // optional [rows][passes][radix] exclusive scans
  uint32_t* bases;         // [rows][passes][radix] exclusive scans (scratch)
  uint32_t* header;        // scratch header: nontrivial flags, schedule
  int in_place;            // the sort reads and writes the same buffer
  int dynamic;             // write the schedule codes into the tile counters
};

// The schedule code of pass k of m run (host and K-SCAN use the same rule):
// pass 0 reads the input; in place, the passes alternate starting with the
// scratch buffer, otherwise they end on the output.
inline __host__ __device__ uint32_t pass_code(uint32_t k, uint32_t m, uint32_t src,
                                              bool in_place) {
  const bool to_out = in_place ? (k % 2 == 1) : ((m - 1 - k) % 2 == 0);
  const uint32_t dst = to_out ? kBufOut : kBufAlt;
  return src | (dst << 2) | ((k & 1) ? kCodeOdd : 0u) | (k == 0 ? kCodeFirst : 0u) |
         (k + 1 == m ? kCodeLast : 0u);
}

struct SweepArgs {
  // buffers by PassBuf: the caller's input, the scratch buffer, the output
  // (kValIdx: vals[kBufIn] is unused, indices are generated by the first
  // pass run; vals[kBufAlt] holds int32 indices, vals[kBufOut] int64)
  const void* keys[3];
  const void* vals[3];
  int64_t rows, cols;
  int64_t tiles_per_row;
  int64_t full_per_row;    // tiles of a row that hold a whole tile of keys
  int shift;
  uint32_t mask;
  uint32_t byte_sel;       // whole-byte digits: 0x4440 | byte index within a 32-bit word
  int byte_hi;             //   and whether that word is the high half of a 64-bit key
  KeyXform xf;             // key transform
  const uint32_t* bases;   // bases of this pass for row 0
  int64_t bases_row_stride;
  void* status_arr[2];     // look-back words [rows * full_per_row][radix], by parity
                           // (u32, or u64 for flat sorts of 2^30 keys or more)
  uint32_t* tile_counter;  // (schedule code << kCodeShift, when dynamic) | tiles handed out:
                           // ids below rows * full_per_row are full tiles, then one
                           // partial tile per row when cols is not a whole number of tiles
  int wide;                // 64-bit look-back words (flat sorts of 2^30 keys or more)
  int packed;              // row-wise: keys and columns packed in 32-bit words (kValPack16)
  int dynamic;             // the schedule comes from K-SCAN (pass skipping on)
  uint32_t code;           // otherwise: this pass's code, from the host, and
  const void* pass_keys_in;   // the buffers and look-back words it selects
  void* pass_keys_out;
  const void* pass_vals_in;
  void* pass_vals_out;
  void* pass_status;
  void* pass_status_zero;
  const uint32_t* offsets; // [rows * tiles_per_row][radix] precomputed output offsets, or null
  uint32_t* error;
  uint64_t timeout_ns;
  uint32_t prefetch_tiles;  // tiles ahead whose keys a tile prefetches into L2
                            // (about the CTAs resident at once; 0: none)
#ifndef LSDRS_PREFETCH_AHEAD_PCT
#define LSDRS_PREFETCH_AHEAD_PCT 35
#endif
};

cudaError_t launch_hist(KeyKind k, int bits, const HistArgs& a, int grid, cudaStream_t s);
cudaError_t launch_hist_x(KeyKind k, int bits, const HistArgs& a, int grid, cudaStream_t s);
cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s);
// One scatter pass: one kernel over every full tile and then each row's
// partial tile (tile ids in that order); *launched receives the number of
// kernels launched (0 or 1).
cudaError_t launch_sweep_u32(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_u32_mid(ValKind v, int bits, const SweepArgs& a, int* launched,
                                 cudaStream_t s);
cudaError_t launch_sweep_u64(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_x32(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_x64(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s);
cudaError_t launch_sweep_f16(const SweepArgs& a, int* launched, cudaStream_t s);
// The same with 64-bit look-back words (flat sorts of 2^30 keys or more).
cudaError_t launch_sweep_u32_wide(ValKind v, int bits, const SweepArgs& a, int* launched,
                                  cudaStream_t s);
cudaError_t launch_sweep_u64_wide(ValKind v, int bits, const SweepArgs& a, int* launched,
                                  cudaStream_t s);
cudaError_t launch_sweep_x32_wide(ValKind v, int bits, const SweepArgs& a, int* launched,
                                  cudaStream_t s);
cudaError_t launch_sweep_x64_wide(ValKind v, int bits, const SweepArgs& a, int* launched,
                                  cudaStream_t s);

// Precomputed tile offsets (row-wise sorts, instead of the look-back): per
// pass, the digit counts of every tile of the pass's input, then per row and
// digit an exclusive scan over the row's tiles plus the digit's base.
struct TileCountArgs {
  const void* keys;        // the pass's input keys
  int64_t rows, cols, tiles_per_row;
  int tile;                // keys per tile (the sweep's)
  int shift;
  uint32_t mask;
  KeyXform xf;
  const uint32_t* bases;   // this pass's bases of row 0
  int64_t bases_row_stride;
  uint32_t* offsets;       // [rows * tiles_per_row][radix]: counts, then offsets
};
cudaError_t launch_tile_counts_f16(const TileCountArgs& a, cudaStream_t s);

// A sort whose rows (one row for a flat sort) hold at most kSmallMaxKeys
// keys: one CTA per row does every pass in shared memory, one launch.
constexpr int64_t kSmallMaxKeys = 8192;
struct SmallArgs {
  const void* keys_in;
  void* keys_out;
  const void* vals_in;     // u32 payloads (kValU32) or unused
  void* vals_out;          // u32 payloads, or int64 column indices (kValIdx)
  int64_t rows, cols;
  int begin_bit, passes;
  uint32_t last_mask;
  KeyXform xf;
  uint32_t* header;        // scratch header: error word and passes run
};
bool small_sort_fits(KeyKind k, ValKind v, int bits, int64_t cols);
cudaError_t launch_small(KeyKind k, ValKind v, int bits, const SmallArgs& a, cudaStream_t s);
cudaError_t launch_copy(void* dst, const void* src, size_t bytes, cudaStream_t s);
// After the passes: when no pass ran (every pass was the identity) copy the
// input to the output, and write column indices as the identity; when an
// in-place sort ran an odd number of passes, copy the scratch buffers back.
// Decided on the device from the schedule; otherwise nothing is done.
struct FinishArgs {
  const uint32_t* passes_run;
  int in_place;
  const void* keys_in;
  const void* keys_alt;
  void* keys_out;
  size_t keys_bytes;       // multiple of 2
  const void* vals_in;     // u32 payloads (or null)
  const void* vals_alt;
  void* vals_out;
  size_t vals_bytes;       // multiple of 2; 0 without u32 payloads
  int64_t* idx_out;        // column indices (row-wise sort) or null
  int64_t rows, cols;
};
cudaError_t launch_finish(const FinishArgs& f, cudaStream_t s);
// Streaming multiprocessors of the current device (queried once per device).
int device_sm_count();
cudaError_t launch_timeout_probe(uint32_t* word, uint32_t* error, uint64_t timeout_ns,
                                 cudaStream_t s);

}  // namespace lsdrs
