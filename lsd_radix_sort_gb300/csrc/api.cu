// The C ABI (include/lsdrs.h): argument checks, the scratch layout, the pass
// schedule and the launches.  Everything here runs on the host; each sort
// enqueues K-HIST, K-SCAN and one K-SWEEP per pass on the caller's stream.
#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>
#include <vector>

#include "common.cuh"
#include "kernels.h"

using namespace lsdrs;

namespace {

std::atomic<uint64_t> g_launches{0};

// Default and largest limit on one look-back or copy wait inside a kernel.
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;
constexpr uint64_t kMaxTimeoutNs = 60000000000ull;

// ---------------------------------------------------------------- profiling
struct ProfRec {
  int kernel;
  uint64_t units;
  cudaEvent_t start, stop;
};
std::mutex g_prof_mu;
bool g_prof_on = false;
std::vector<ProfRec> g_prof;

// Runs `launch` bracketed by profiling events when enabled.
template <class F>
cudaError_t timed_launch(int kernel, uint64_t units, cudaStream_t s, F&& launch) {
  ProfRec r{kernel, units, nullptr, nullptr};
  bool prof;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    prof = g_prof_on;
  }
  if (prof) {
    if (cudaEventCreate(&r.start) != cudaSuccess || cudaEventCreate(&r.stop) != cudaSuccess)
      return cudaErrorUnknown;
    cudaEventRecord(r.start, s);
  }
  int launched = 1;
  cudaError_t e = launch(&launched);
  g_launches.fetch_add(static_cast<uint64_t>(launched), std::memory_order_relaxed);
  if (prof) {
    cudaEventRecord(r.stop, s);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    g_prof.push_back(r);
  }
  return e;
}

// Per-call options (rs_options), resolved against the defaults.
struct Options {
  bool pass_skipping = false;
  bool tile_offsets = false;
  bool small_sort = true;
  uint64_t timeout_ns = kDefaultTimeoutNs;
};

constexpr unsigned kKnownFlags = RS_OPT_PASS_SKIPPING | RS_OPT_TILE_OFFSETS | RS_OPT_NO_SMALL_SORT;

bool resolve_options(const rs_options* o, Options* out) {
  Options r;
  if (o != nullptr) {
    if (o->flags & ~kKnownFlags) return false;
    r.pass_skipping = (o->flags & RS_OPT_PASS_SKIPPING) != 0;
    r.tile_offsets = (o->flags & RS_OPT_TILE_OFFSETS) != 0;
    r.small_sort = (o->flags & RS_OPT_NO_SMALL_SORT) == 0;
    if (o->lookback_timeout_ns != 0) {
      if (o->lookback_timeout_ns > kMaxTimeoutNs) return false;
      r.timeout_ns = o->lookback_timeout_ns;
    }
  }
  *out = r;
  return true;
}

// -------------------------------------------------------------------- plan
// Scratch layout (offsets in bytes from `temp`, each 256-byte aligned):
//   header   : device error word, tile counters, pass schedule (kernels.h)
//   status0  : look-back words of even passes  [tiles][radix] u32 (u64 from 2^30 keys)
//   status1  : look-back words of odd passes   [tiles][radix]
//   bases    : [rows][passes][radix] u32
//   slots    : [rows][hist chunks][passes][radix] u32 partial histograms
//   alt_keys : ping-pong key buffer
//   alt_vals : ping-pong payload buffer (u32 / int32 indices)
// header and status0 are contiguous: K-HIST zeroes them in one range.
constexpr size_t kHeaderBytes = 1024;
static_assert((kHdrNontrivial + kMaxPasses) * 4 <= kHeaderBytes, "header layout");

struct Plan {
  KeyKind key;
  ValKind val;
  int key_bytes;
  int64_t rows, cols;
  int begin_bit, end_bit, bits, passes, radix;
  uint32_t last_mask;
  int tile;
  int64_t tiles_per_row, tiles;
  int status_word;           // bytes per look-back word: 4, or 8 from 2^30 keys
  int64_t max_chunks;        // histogram slots reserved per row
  // set per call by configure(): histogram chunks for the device's SMs
  int chunks_per_row;
  int64_t chunk_len;
  size_t off_status0, off_status1, off_bases, off_slots, off_tile_offsets, off_alt_keys,
      off_alt_vals, total;
};

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

rs_status make_plan(KeyKind key, ValKind val, int64_t rows, int64_t cols, int begin_bit,
                    int end_bit, int bits, Plan* out) {
  Plan p{};
  p.key = key;
  p.val = val;
  p.key_bytes = (key == kKeyU32 || key == kKeyX32) ? 4 : (key == kKeyU64 || key == kKeyX64) ? 8 : 2;
  const int kbits = p.key_bytes * 8;
  if (rows < 0 || cols < 0) return RS_ERR_INVALID;
  // a flat sort (one row) may hold up to RS_MAX_KEYS keys; a row of a
  // row-wise sort up to RS_MAX_ROW_KEYS (its column indices are int32 inside)
  const bool flat = rows == 1 && val != kValIdx;
  if (static_cast<uint64_t>(cols) > (flat ? RS_MAX_KEYS : RS_MAX_ROW_KEYS)) return RS_ERR_INVALID;
  // every row is at least one tile, and tile ids are 24 bits (this also keeps
  // rows * tiles_per_row and rows * cols far from overflowing)
  if (rows > static_cast<int64_t>(kTileMask)) return RS_ERR_INVALID;
  if (begin_bit < 0 || end_bit > kbits || begin_bit >= end_bit) return RS_ERR_INVALID;
  if (bits < 1 || bits > 8) return RS_ERR_INVALID;
  p.rows = rows;
  p.cols = cols;
  p.begin_bit = begin_bit;
  p.end_bit = end_bit;
  p.bits = bits;
  p.passes = (end_bit - begin_bit + bits - 1) / bits;
  if (p.passes > kMaxPasses) return RS_ERR_INVALID;
  p.radix = 1 << bits;
  const int last_w = end_bit - (begin_bit + (p.passes - 1) * bits);
  p.last_mask = (1u << last_w) - 1u;
  p.tile = sweep_shape(key, val, rows, cols).tile();
  p.tiles_per_row = cdiv(cols, p.tile);
  p.tiles = rows * p.tiles_per_row;
  if (p.tiles > static_cast<int64_t>(kTileMask)) return RS_ERR_INVALID;  // tile ids: 24 bits
  // A look-back count reaches the row length: 32-bit words hold 30 bits.
  p.status_word = cols > kMaxNarrowKeys ? 8 : 4;
  // histogram slots for the chunks of any device configure() may see
  p.max_chunks = rows > 0 ? cdiv(kMaxHistCtas, rows) : 1;

  const size_t status_bytes =
      align_up(static_cast<size_t>(p.tiles) * p.radix * p.status_word, 256);
  const size_t n = static_cast<size_t>(rows) * static_cast<size_t>(cols);
  const size_t pr = static_cast<size_t>(p.passes) * p.radix * 4;
  size_t off = kHeaderBytes;
  p.off_status0 = off;
  off += status_bytes;
  p.off_status1 = off;
  off += status_bytes;
  p.off_bases = off;
  off += align_up(static_cast<size_t>(rows) * pr, 256);
  p.off_slots = off;
  off += align_up(static_cast<size_t>(rows) * p.max_chunks * pr, 256);
  p.off_tile_offsets = off;  // row-wise sorts: precomputed tile offsets of one pass
  if (val == kValIdx) off += align_up(static_cast<size_t>(p.tiles) * p.radix * 4, 256);
  p.off_alt_keys = off;
  off += align_up(n * p.key_bytes, 256);
  p.off_alt_vals = off;
  if (val != kValNone) off += align_up(n * 4, 256);
  p.total = off;
  *out = p;
  return RS_OK;
}

// Per call: the K-HIST chunks, one CTA per SM of the device (at most
// kMaxHistCtas), each at least kHistMinChunk keys.
void configure(Plan* p) {
  const int64_t sms = std::min<int64_t>(device_sm_count(), kMaxHistCtas);
  int64_t want = p->rows > 0 ? cdiv(sms, p->rows) : 1;
  want = std::min<int64_t>(want, std::max<int64_t>(1, cdiv(p->cols, kHistMinChunk)));
  want = std::max<int64_t>(want, 1);
  p->chunks_per_row = static_cast<int>(want);
  p->chunk_len = static_cast<int64_t>(
      align_up(static_cast<size_t>(std::max<int64_t>(1, cdiv(p->cols, want))), 64));
}

inline unsigned char* at(void* temp, size_t off) { return static_cast<unsigned char*>(temp) + off; }

bool overlap(const void* a, size_t an, const void* b, size_t bn) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + bn && y < x + an;
}

// Enqueue K-HIST and K-SCAN.  hist_out / bases_out: optional copies of the
// rows' totals and bases ([rows][passes][radix]).
rs_status run_front(const Plan& p, const void* keys, const KeyXform& xf, void* temp,
                    uint32_t* hist_out, uint32_t* bases_out, bool in_place, bool dynamic,
                    cudaStream_t s) {
  HistArgs h{};
  h.keys = keys;
  h.rows = p.rows;
  h.cols = p.cols;
  h.chunks_per_row = p.chunks_per_row;
  h.chunk_len = p.chunk_len;
  h.begin_bit = p.begin_bit;
  h.passes = p.passes;
  h.last_mask = p.last_mask;
  h.xf = xf;
  h.slots = reinterpret_cast<uint32_t*>(at(temp, p.off_slots));
  h.zero_ptr = reinterpret_cast<uint32_t*>(temp);
  h.zero_words = (p.off_status1) / 4;  // header + status0
  const int64_t hgrid = p.rows * p.chunks_per_row;
  const uint64_t n = static_cast<uint64_t>(p.rows) * p.cols;
  // 16-bit rows counted one CTA per row, static schedule: K-HIST scans
  h.fused_scan = p.key == kKeyF16 && p.bits == 8 && p.chunks_per_row == 1 && !dynamic;
  h.bases = reinterpret_cast<uint32_t*>(at(temp, p.off_bases));
  h.hist_out = hist_out;
  h.bases_out = bases_out;
  cudaError_t e = timed_launch(0, n, s, [&](int*) {
    return launch_hist(p.key, p.bits, h, static_cast<int>(hgrid), s);
  });
  if (e != cudaSuccess) return RS_ERR_CUDA;
  if (h.fused_scan) return RS_OK;
  ScanArgs c{};
  c.slots = h.slots;
  c.rows = p.rows;
  c.chunks_per_row = p.chunks_per_row;
  c.passes = p.passes;
  c.radix = p.radix;
  c.hist_out = hist_out;
  c.bases_out = bases_out;
  c.bases = reinterpret_cast<uint32_t*>(at(temp, p.off_bases));
  c.header = reinterpret_cast<uint32_t*>(temp);
  c.cols = p.cols;
  c.in_place = in_place ? 1 : 0;
  c.dynamic = dynamic ? 1 : 0;
  e = timed_launch(1, static_cast<uint64_t>(p.rows) * p.passes * p.radix, s,
                   [&](int*) { return launch_scan(c, s); });
  return e == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

cudaError_t sweep(const Plan& p, const SweepArgs& a, int* launched, cudaStream_t s) {
  if (a.wide) {
    switch (p.key) {
      case kKeyU32: return launch_sweep_u32_wide(p.val, p.bits, a, launched, s);
      case kKeyU64: return launch_sweep_u64_wide(p.val, p.bits, a, launched, s);
      case kKeyX32: return launch_sweep_x32_wide(p.val, p.bits, a, launched, s);
      case kKeyX64: return launch_sweep_x64_wide(p.val, p.bits, a, launched, s);
      default: return cudaErrorInvalidValue;  // rows stay below 2^30 keys
    }
  }
  switch (p.key) {
    case kKeyU32: return launch_sweep_u32(p.val, p.bits, a, launched, s);
    case kKeyU64: return launch_sweep_u64(p.val, p.bits, a, launched, s);
    case kKeyF16: return launch_sweep_f16(a, launched, s);
    case kKeyX32: return launch_sweep_x32(p.val, p.bits, a, launched, s);
    case kKeyX64: return launch_sweep_x64(p.val, p.bits, a, launched, s);
  }
  return cudaErrorInvalidValue;
}

// A whole sort: front stages, then one sweep per pass.  The pass that
// writes `keys_out` last is chosen by parity so that no copy is needed,
// except for an in-place sort with an odd number of passes.
rs_status run_sort(Plan p, const void* keys_in, void* keys_out, const void* vals_in,
                   void* vals_out, const KeyXform& xf, void* temp, size_t temp_bytes,
                   const Options& opt, cudaStream_t s) {
  const size_t n = static_cast<size_t>(p.rows) * static_cast<size_t>(p.cols);
  if (n == 0) return RS_OK;
  if (temp == nullptr) return RS_ERR_INVALID;
  if (temp_bytes < p.total) return RS_ERR_TEMP_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(temp) % 256 != 0) return RS_ERR_INVALID;
  const size_t kb = static_cast<size_t>(p.key_bytes) * n;
  const size_t vb_in = 4 * n;
  const size_t vb_out = (p.val == kValIdx ? 8 : 4) * n;
  if (!keys_in || !keys_out) return RS_ERR_INVALID;
  if (p.val == kValU32 && (!vals_in || !vals_out)) return RS_ERR_INVALID;
  if (p.val == kValIdx && !vals_out) return RS_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(keys_in) % p.key_bytes ||
      reinterpret_cast<uintptr_t>(keys_out) % p.key_bytes)
    return RS_ERR_INVALID;
  if (keys_in != keys_out && overlap(keys_in, kb, keys_out, kb)) return RS_ERR_INVALID;
  if (overlap(temp, p.total, keys_out, kb) || overlap(temp, p.total, keys_in, kb))
    return RS_ERR_INVALID;
  bool in_place = keys_in == keys_out;
  if (p.val == kValU32) {
    if (reinterpret_cast<uintptr_t>(vals_in) % 4 || reinterpret_cast<uintptr_t>(vals_out) % 4)
      return RS_ERR_INVALID;
    if (vals_in != vals_out && overlap(vals_in, vb_in, vals_out, vb_out)) return RS_ERR_INVALID;
    if (overlap(keys_out, kb, vals_out, vb_out) || overlap(temp, p.total, vals_out, vb_out))
      return RS_ERR_INVALID;
    in_place = in_place || vals_in == vals_out;
  }
  if (p.val == kValIdx) {
    if (reinterpret_cast<uintptr_t>(vals_out) % 8) return RS_ERR_INVALID;
    if (overlap(keys_out, kb, vals_out, vb_out) || overlap(keys_in, kb, vals_out, vb_out) ||
        overlap(temp, p.total, vals_out, vb_out))
      return RS_ERR_INVALID;
  }

  if (p.val == kValIdx && p.passes > 2) return RS_ERR_INVALID;  // 16-bit keys: two passes

  // rows of at most one small tile: the whole sort in one kernel
  if (opt.small_sort && small_sort_fits(p.key, p.val, p.bits, p.cols)) {
    SmallArgs sa{};
    sa.keys_in = keys_in;
    sa.keys_out = keys_out;
    sa.vals_in = vals_in;
    sa.vals_out = vals_out;
    sa.rows = p.rows;
    sa.cols = p.cols;
    sa.begin_bit = p.begin_bit;
    sa.passes = p.passes;
    sa.last_mask = p.last_mask;
    sa.xf = xf;
    sa.header = reinterpret_cast<uint32_t*>(temp);
    cudaError_t e = timed_launch(7, n, s, [&](int*) {
      return launch_small(p.key, p.val, p.bits, sa, s);
    });
    return e == cudaSuccess ? RS_OK : RS_ERR_CUDA;
  }

  // row-wise sorts may take precomputed tile offsets instead of the
  // look-back; that mode keeps the static schedule (every pass runs)
  const bool precomputed = p.val == kValIdx && opt.tile_offsets;
  const bool dynamic = !precomputed && opt.pass_skipping;
  // Row-wise sorts of rows of at most 65,536 columns on the static schedule
  // carry each key's column in the low half of a 32-bit word between the
  // passes (the packed words use the payload ping-pong buffer), so each pass
  // stages one word per key; their tile is the packed kernel's.
  const bool packed = p.val == kValIdx && !precomputed && !dynamic && p.cols <= kPackMaxCols;
  if (packed) {
    // The scratch is planned for the unpacked tile; the packed tile is at
    // least as large (checked at compile time), so its look-back words fit.
    static_assert(kShapeF16Packed.tile() >= kShapeF16Idx.tile(),
                  "packed row tiles must not outnumber the planned tiles");
    const int64_t planned = p.tiles;
    p.tile = kShapeF16Packed.tile();
    p.tiles_per_row = cdiv(p.cols, p.tile);
    p.tiles = p.rows * p.tiles_per_row;
    if (p.tiles > planned) return RS_ERR_INVALID;
  }
  configure(&p);
  rs_status st = run_front(p, keys_in, xf, temp, nullptr, nullptr, in_place, dynamic, s);
  if (st != RS_OK) return st;

  // With pass skipping, K-SCAN has written the schedule (which passes run,
  // from which buffer to which) and every pass is launched, a skipped one
  // returning at once.  Otherwise every pass runs on the host's schedule.
  uint32_t* header = reinterpret_cast<uint32_t*>(temp);
  void* alt_keys = at(temp, p.off_alt_keys);
  void* alt_vals = at(temp, p.off_alt_vals);
  const uint32_t* bases = reinterpret_cast<const uint32_t*>(at(temp, p.off_bases));
  SweepArgs a{};
  a.keys[kBufIn] = keys_in;
  a.keys[kBufAlt] = packed ? alt_vals : alt_keys;
  a.packed = packed ? 1 : 0;
  a.keys[kBufOut] = keys_out;
  a.vals[kBufIn] = p.val == kValU32 ? vals_in : nullptr;
  a.vals[kBufAlt] = p.val == kValNone ? nullptr : alt_vals;
  a.vals[kBufOut] = vals_out;
  a.status_arr[0] = at(temp, p.off_status0);
  a.status_arr[1] = at(temp, p.off_status1);
  a.wide = p.status_word == 8 ? 1 : 0;
  a.rows = p.rows;
  a.cols = p.cols;
  a.tiles_per_row = p.tiles_per_row;
  a.full_per_row = p.cols / p.tile;
  a.xf = xf;
  a.bases_row_stride = static_cast<int64_t>(p.passes) * p.radix;
  a.error = header + kHdrError;
  a.timeout_ns = opt.timeout_ns;
  // flat sorts: prefetch, per tile, the keys of the tile taken about one
  // resident grid (LSDRS_PREFETCH_AHEAD_PCT percent of it) later
  a.prefetch_tiles =
      p.rows == 1 ? static_cast<uint32_t>(device_sm_count() *
                                          sweep_shape(p.key, p.val, p.rows, p.cols).min_blocks *
                                          LSDRS_PREFETCH_AHEAD_PCT / 100)
                  : 0u;
  a.dynamic = dynamic ? 1 : 0;
  uint32_t prev = kBufIn;
  for (int q = 0; q < p.passes; ++q) {
    const bool last = q == p.passes - 1;
    a.code = pass_code(q, p.passes, prev, in_place);
    prev = (a.code & kCodeDst) >> 2;
    // the static schedule's buffers, as kernel arguments
    const uint32_t src = a.code & kCodeSrc, dst = (a.code & kCodeDst) >> 2;
    a.pass_keys_in = a.keys[src];
    a.pass_keys_out = const_cast<void*>(a.keys[dst]);
    if (packed) {
      a.pass_vals_in = nullptr;  // the columns travel inside the key words
      a.pass_vals_out = last ? vals_out : nullptr;
    } else if (p.val == kValIdx) {
      a.pass_vals_in = q == 0 ? nullptr : alt_vals;
      a.pass_vals_out = last ? vals_out : alt_vals;
    } else {
      a.pass_vals_in = a.vals[src];
      a.pass_vals_out = const_cast<void*>(a.vals[dst]);
    }
    a.pass_status = a.status_arr[q & 1];
    a.pass_status_zero = last ? nullptr : a.status_arr[(q + 1) & 1];
    a.shift = p.begin_bit + q * p.bits;
    a.mask = last ? p.last_mask : static_cast<uint32_t>(p.radix - 1);
    a.byte_sel = 0x4440u | static_cast<uint32_t>((a.shift >> 3) & 3);
    a.byte_hi = (a.shift >> 3) >= 4 ? 1 : 0;
    a.bases = bases + static_cast<size_t>(q) * p.radix;
    a.tile_counter = header + kHdrTileCounter + q;
    if (precomputed) {
      TileCountArgs tc{};
      tc.keys = a.pass_keys_in;
      tc.rows = p.rows;
      tc.cols = p.cols;
      tc.tiles_per_row = p.tiles_per_row;
      tc.tile = p.tile;
      tc.shift = a.shift;
      tc.mask = a.mask;
      tc.xf = xf;
      tc.bases = a.bases;
      tc.bases_row_stride = a.bases_row_stride;
      tc.offsets = reinterpret_cast<uint32_t*>(at(temp, p.off_tile_offsets));
      a.offsets = tc.offsets;
      cudaError_t e = timed_launch(6, n, s, [&](int* k) {
        *k = 2;
        return launch_tile_counts_f16(tc, s);
      });
      if (e != cudaSuccess) return RS_ERR_CUDA;
    }
    cudaError_t e = timed_launch(2, n, s, [&](int* k) { return sweep(p, a, k, s); });
    if (e != cudaSuccess) return RS_ERR_CUDA;
  }
  // no pass run, or an odd number run in place: copy (decided on the device)
  FinishArgs f{};
  f.passes_run = header + kHdrPassesRun;
  f.in_place = in_place ? 1 : 0;
  f.keys_in = keys_in;
  f.keys_alt = alt_keys;
  f.keys_out = keys_out;
  f.keys_bytes = kb;
  if (p.val == kValU32) {
    f.vals_in = vals_in;
    f.vals_alt = alt_vals;
    f.vals_out = vals_out;
    f.vals_bytes = vb_out;
  }
  if (p.val == kValIdx) f.idx_out = static_cast<int64_t*>(vals_out);
  f.rows = p.rows;
  f.cols = p.cols;
  // (the static schedule needs it only in place with an odd number of passes)
  if (dynamic || (in_place && p.passes % 2 == 1)) {
    cudaError_t e = timed_launch(5, n, s, [&](int*) { return launch_finish(f, s); });
    if (e != cudaSuccess) return RS_ERR_CUDA;
  }
  return RS_OK;
}

rs_status flat_sort(KeyKind key, const KeyXform& xf, ValKind val, const void* ki, void* ko,
                    const void* vi, void* vo, size_t n, int begin_bit, int end_bit, int bits,
                    void* temp, size_t temp_bytes, const rs_options* opts, void* stream) {
  if (n > RS_MAX_KEYS) return RS_ERR_INVALID;
  Options o;
  if (!resolve_options(opts, &o)) return RS_ERR_INVALID;
  Plan p;
  rs_status st = make_plan(key, val, 1, static_cast<int64_t>(n), begin_bit, end_bit, bits, &p);
  if (st != RS_OK) return st;
  return run_sort(p, ki, ko, vi, vo, xf, temp, temp_bytes, o, static_cast<cudaStream_t>(stream));
}

// The key kind and transform of a typed global sort (see keys.cuh): unsigned
// ascending keys take the identity kernels, everything else the transformed
// ones.
bool typed_key(rs_key_type type, int descending, KeyKind* kind, KeyXform* xf) {
  if (descending != 0 && descending != 1) return false;
  const bool wide = type == RS_KEY_U64 || type == RS_KEY_I64 || type == RS_KEY_F64;
  const uint64_t ones = wide ? ~0ull : 0xFFFFFFFFull;
  const uint64_t sign = wide ? (1ull << 63) : (1ull << 31);
  uint64_t pos, neg;
  switch (type) {
    case RS_KEY_U32: case RS_KEY_U64: pos = neg = 0; break;
    case RS_KEY_I32: case RS_KEY_I64: pos = neg = sign; break;
    case RS_KEY_F32: case RS_KEY_F64: pos = sign; neg = ones; break;
    default: return false;
  }
  if (descending) {
    pos ^= ones;
    neg ^= ones;
  }
  xf->pos = pos;
  xf->neg = neg;
  const bool identity = pos == 0 && neg == 0;
  *kind = wide ? (identity ? kKeyU64 : kKeyX64) : (identity ? kKeyU32 : kKeyX32);
  return true;
}

}  // namespace

extern "C" {

rs_status radix_sort_keys_temp_bytes(size_t n, int key_bytes, int value_bytes, int begin_bit,
                                     int end_bit, int digit_bits, size_t* bytes) {
  if (!bytes || n > RS_MAX_KEYS) return RS_ERR_INVALID;
  if (key_bytes != 4 && key_bytes != 8) return RS_ERR_INVALID;
  if (value_bytes != 0 && value_bytes != 4) return RS_ERR_INVALID;
  Plan p;
  rs_status st = make_plan(key_bytes == 4 ? kKeyU32 : kKeyU64, value_bytes ? kValU32 : kValNone,
                           1, static_cast<int64_t>(n), begin_bit, end_bit, digit_bits, &p);
  if (st != RS_OK) return st;
  *bytes = p.total;
  return RS_OK;
}

rs_status radix_sort_keys_u32(const uint32_t* keys_in, uint32_t* keys_out, size_t n,
                              int begin_bit, int end_bit, int digit_bits, void* temp,
                              size_t temp_bytes, void* stream) {
  return flat_sort(kKeyU32, KeyXform{0, 0}, kValNone, keys_in, keys_out, nullptr, nullptr, n,
                   begin_bit, end_bit, digit_bits, temp, temp_bytes, nullptr, stream);
}

rs_status radix_sort_keys_u64(const uint64_t* keys_in, uint64_t* keys_out, size_t n,
                              int begin_bit, int end_bit, int digit_bits, void* temp,
                              size_t temp_bytes, void* stream) {
  return flat_sort(kKeyU64, KeyXform{0, 0}, kValNone, keys_in, keys_out, nullptr, nullptr, n,
                   begin_bit, end_bit, digit_bits, temp, temp_bytes, nullptr, stream);
}

rs_status radix_sort_pairs_u32(const uint32_t* keys_in, uint32_t* keys_out,
                               const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                               int begin_bit, int end_bit, int digit_bits, void* temp,
                               size_t temp_bytes, void* stream) {
  return flat_sort(kKeyU32, KeyXform{0, 0}, kValU32, keys_in, keys_out, vals_in, vals_out, n,
                   begin_bit, end_bit, digit_bits, temp, temp_bytes, nullptr, stream);
}

rs_status radix_sort_pairs_u64(const uint64_t* keys_in, uint64_t* keys_out,
                               const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                               int begin_bit, int end_bit, int digit_bits, void* temp,
                               size_t temp_bytes, void* stream) {
  return flat_sort(kKeyU64, KeyXform{0, 0}, kValU32, keys_in, keys_out, vals_in, vals_out, n,
                   begin_bit, end_bit, digit_bits, temp, temp_bytes, nullptr, stream);
}

rs_status radix_sort_keys_typed(rs_key_type type, int descending, const void* keys_in,
                                void* keys_out, size_t n, int begin_bit, int end_bit,
                                int digit_bits, void* temp, size_t temp_bytes,
                                const rs_options* opts, void* stream) {
  KeyKind kind;
  KeyXform xf;
  if (!typed_key(type, descending, &kind, &xf)) return RS_ERR_INVALID;
  return flat_sort(kind, xf, kValNone, keys_in, keys_out, nullptr, nullptr, n, begin_bit, end_bit,
                   digit_bits, temp, temp_bytes, opts, stream);
}

rs_status radix_sort_pairs_typed(rs_key_type type, int descending, const void* keys_in,
                                 void* keys_out, const uint32_t* vals_in, uint32_t* vals_out,
                                 size_t n, int begin_bit, int end_bit, int digit_bits, void* temp,
                                 size_t temp_bytes, const rs_options* opts, void* stream) {
  KeyKind kind;
  KeyXform xf;
  if (!typed_key(type, descending, &kind, &xf)) return RS_ERR_INVALID;
  return flat_sort(kind, xf, kValU32, keys_in, keys_out, vals_in, vals_out, n, begin_bit, end_bit,
                   digit_bits, temp, temp_bytes, opts, stream);
}

rs_status radix_segmented_sort_temp_bytes(int64_t rows, int64_t cols, size_t* bytes) {
  if (!bytes) return RS_ERR_INVALID;
  Plan p;
  rs_status st = make_plan(kKeyF16, kValIdx, rows, cols, 0, 16, 8, &p);
  if (st != RS_OK) return st;
  *bytes = p.total;
  return RS_OK;
}

rs_status radix_segmented_sort_f16_ex(const uint16_t* in, uint16_t* vals_out, int64_t* idx_out,
                                      int64_t rows, int64_t cols, rs_float_kind kind,
                                      int descending, void* temp, size_t temp_bytes,
                                      const rs_options* opts, void* stream) {
  if (kind != RS_F16 && kind != RS_BF16) return RS_ERR_INVALID;
  if (descending != 0 && descending != 1) return RS_ERR_INVALID;
  Options o;
  if (!resolve_options(opts, &o)) return RS_ERR_INVALID;
  Plan p;
  rs_status st = make_plan(kKeyF16, kValIdx, rows, cols, 0, 16, 8, &p);
  if (st != RS_OK) return st;
  // 16-bit float bijection; descending complements it
  const uint64_t flip = descending ? 0xFFFFu : 0u;
  return run_sort(p, in, vals_out, nullptr, idx_out, KeyXform{0x8000u ^ flip, 0xFFFFu ^ flip},
                  temp, temp_bytes, o, static_cast<cudaStream_t>(stream));
}

rs_status radix_segmented_sort_f16(const uint16_t* in, uint16_t* vals_out, int64_t* idx_out,
                                   int64_t rows, int64_t cols, rs_float_kind kind,
                                   int descending, void* temp, size_t temp_bytes,
                                   void* stream) {
  return radix_segmented_sort_f16_ex(in, vals_out, idx_out, rows, cols, kind, descending, temp,
                                     temp_bytes, nullptr, stream);
}

rs_status radix_sort_histograms(const void* keys, int key_bytes, size_t n, int begin_bit,
                                int end_bit, int digit_bits, uint32_t* hist_out,
                                uint32_t* bases_out, void* temp, size_t temp_bytes,
                                void* stream) {
  if (key_bytes != 4 && key_bytes != 8) return RS_ERR_INVALID;
  if (n > RS_MAX_KEYS) return RS_ERR_INVALID;
  Plan p;
  rs_status st = make_plan(key_bytes == 4 ? kKeyU32 : kKeyU64, kValNone, 1,
                           static_cast<int64_t>(n), begin_bit, end_bit, digit_bits, &p);
  if (st != RS_OK) return st;
  if (!hist_out || !bases_out || !temp) return RS_ERR_INVALID;
  if (n > 0 && !keys) return RS_ERR_INVALID;
  if (temp_bytes < p.total) return RS_ERR_TEMP_TOO_SMALL;
  if (reinterpret_cast<uintptr_t>(temp) % 256 != 0) return RS_ERR_INVALID;
  configure(&p);
  return run_front(p, keys, KeyXform{0, 0}, temp, hist_out, bases_out, false, false,
                   static_cast<cudaStream_t>(stream));
}

rs_status radix_sort_device_status(const void* temp, void* stream) {
  if (!temp) return RS_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, temp, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
  return word == kErrNone ? RS_OK : static_cast<rs_status>(word);
}

int rs_checked_build(void) { return LSDRS_CHECKED; }

rs_status radix_sort_checked_violations(void* temp, void* stream, uint32_t* count,
                                        uint32_t* first_site) {
  if (!temp || !count || !first_site) return RS_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t* w = static_cast<uint32_t*>(temp) + kHdrViolations;
  uint32_t h[2] = {0, 0};
  if (cudaMemcpyAsync(h, w, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RS_ERR_CUDA;
  if (cudaMemsetAsync(w, 0, sizeof(h), s) != cudaSuccess) return RS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
  *count = h[0];
  *first_site = h[1];
  return RS_OK;
}

rs_status radix_sort_passes_run(const void* temp, int* passes, void* stream) {
  if (!temp || !passes) return RS_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, static_cast<const uint32_t*>(temp) + kHdrPassesRun, 4,
                      cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
  *passes = static_cast<int>(word);
  return RS_OK;
}

const char* rs_status_string(rs_status status) {
  switch (status) {
    case RS_OK: return "RS_OK";
    case RS_ERR_INVALID: return "RS_ERR_INVALID";
    case RS_ERR_TEMP_TOO_SMALL: return "RS_ERR_TEMP_TOO_SMALL";
    case RS_ERR_CUDA: return "RS_ERR_CUDA";
    case RS_ERR_LOOKBACK_TIMEOUT: return "RS_ERR_LOOKBACK_TIMEOUT";
  }
  return "RS_UNKNOWN";
}

rs_status rs_lookback_timeout_probe(uint32_t* word, uint64_t timeout_ns, void* stream,
                                    rs_status* result) {
  if (!word || !result || timeout_ns == 0 || timeout_ns > kMaxTimeoutNs) return RS_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(word, 0, 8, s) != cudaSuccess) return RS_ERR_CUDA;
  cudaError_t e = timed_launch(4, 1, s, [&](int*) {
    return launch_timeout_probe(word, word + 1, timeout_ns, s);
  });
  if (e != cudaSuccess) return RS_ERR_CUDA;
  uint32_t err = 0;
  if (cudaMemcpyAsync(&err, word + 1, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
  *result = err == kErrNone ? RS_OK : static_cast<rs_status>(err);
  return RS_OK;
}

rs_status rs_copy_probe(void* dst, const void* src, size_t bytes, void* stream) {
  if (!dst || !src || bytes % 16 != 0) return RS_ERR_INVALID;
  if (reinterpret_cast<uintptr_t>(dst) % 16 || reinterpret_cast<uintptr_t>(src) % 16)
    return RS_ERR_INVALID;
  if (bytes == 0) return RS_OK;
  if (overlap(dst, bytes, src, bytes)) return RS_ERR_INVALID;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = timed_launch(3, bytes, s, [&](int*) { return launch_copy(dst, src, bytes, s); });
  return e == cudaSuccess ? RS_OK : RS_ERR_CUDA;
}

rs_status rs_profile_enable(int enable) {
  std::lock_guard<std::mutex> lk(g_prof_mu);
  g_prof_on = enable != 0;
  return RS_OK;
}

int rs_profile_read(rs_kernel_time* out, int max) {
  std::vector<ProfRec> recs;
  {
    std::lock_guard<std::mutex> lk(g_prof_mu);
    recs.swap(g_prof);
  }
  int w = 0;
  for (ProfRec& r : recs) {
    float ms = -1.0f;
    if (cudaEventSynchronize(r.stop) == cudaSuccess) cudaEventElapsedTime(&ms, r.start, r.stop);
    if (out && w < max) out[w++] = rs_kernel_time{r.kernel, ms, r.units};
    cudaEventDestroy(r.start);
    cudaEventDestroy(r.stop);
  }
  return w;
}

uint64_t rs_launch_count_reset(void) { return g_launches.exchange(0); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Key-value sort that allocates nothing.
//
// Some callers cannot allocate device memory where they sort: callers whose
// device memory is owned by a pool they may not grow, or plugins and
// callbacks that are handed only the buffers they work on and have no
// allocator of their own.  For them the scratch of the sort lives in one
// fixed array in this library's device image.  The array is created when the
// library's device code is loaded and stays until the process exits, on
// every GPU that loads the library, so it is kept small: sorts of at most
// kNoAllocMaxKeys keys.
// ---------------------------------------------------------------------------
namespace {
constexpr size_t kNoAllocMaxKeys = size_t(1) << 18;     // 262,144 keys
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB per GPU
constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};
}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

namespace {
// The host-side name of the array is not a device address: its address on
// the current device is looked up once per device, with that device current.
rs_status noalloc_scratch(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return RS_ERR_CUDA;
  if (dev < 0 || dev >= kNoAllocMaxDevices) return RS_ERR_INVALID;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (g_noalloc_addr[dev] == nullptr) {
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || addr == nullptr)
      return RS_ERR_CUDA;
    g_noalloc_addr[dev] = addr;
  }
  *out = g_noalloc_addr[dev];
  return RS_OK;
}
}  // namespace

extern "C" rs_status radix_sort_pairs_u32_noalloc(const uint32_t* keys_in, uint32_t* keys_out,
                                                  const uint32_t* vals_in, uint32_t* vals_out,
                                                  size_t n, int begin_bit, int end_bit,
                                                  int digit_bits, void* stream) {
  if (n > kNoAllocMaxKeys) return RS_ERR_INVALID;
  Plan p;
  rs_status st = make_plan(kKeyU32, kValU32, 1, static_cast<int64_t>(n), begin_bit, end_bit,
                           digit_bits, &p);
  if (st != RS_OK) return st;
  if (p.total > kNoAllocScratchBytes) return RS_ERR_INVALID;
  if (n == 0) return RS_OK;
  void* scratch = nullptr;
  st = noalloc_scratch(&scratch);
  if (st != RS_OK) return st;
  // The sort's first kernel zeroes every part of the scratch that must start
  // at zero, so what an earlier call left there does not matter.
  return run_sort(p, keys_in, keys_out, vals_in, vals_out, KeyXform{0, 0}, scratch,
                  kNoAllocScratchBytes, Options{}, static_cast<cudaStream_t>(stream));
}

extern "C" rs_status rs_noalloc_timeout_probe(uint64_t timeout_ns, void* stream,
                                             rs_status* result) {
  if (!result || timeout_ns == 0 || timeout_ns > kMaxTimeoutNs) return RS_ERR_INVALID;
  void* scratch = nullptr;
  rs_status st = noalloc_scratch(&scratch);
  if (st != RS_OK) return st;
  uint32_t* hdr = static_cast<uint32_t*>(scratch);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(hdr + kHdrProbeWord, 0, 4, s) != cudaSuccess ||
      cudaMemsetAsync(hdr + kHdrError, 0, 4, s) != cudaSuccess)
    return RS_ERR_CUDA;
  cudaError_t e = timed_launch(4, 1, s, [&](int*) {
    return launch_timeout_probe(hdr + kHdrProbeWord, hdr + kHdrError, timeout_ns, s);
  });
  if (e != cudaSuccess) return RS_ERR_CUDA;
  uint32_t err = 0;
  if (cudaMemcpyAsync(&err, hdr + kHdrError, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
  *result = err == kErrNone ? RS_OK : static_cast<rs_status>(err);
  return RS_OK;
}

extern "C" rs_status radix_sort_pairs_u32_noalloc_status(void* stream) {
  void* scratch = nullptr;
  rs_status st = noalloc_scratch(&scratch);
  if (st != RS_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  uint32_t word = 0;
  if (cudaMemcpyAsync(&word, scratch, 4, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return RS_ERR_CUDA;
  if (cudaStreamSynchronize(s) != cudaSuccess) return RS_ERR_CUDA;
  return word == kErrNone ? RS_OK : static_cast<rs_status>(word);
}
