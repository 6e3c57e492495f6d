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
//     running (forward progress of the look-back).  With pass skipping the
//     counter's top byte also carries the pass's schedule (which buffers it
//     reads and writes, or that it is skipped), written there by K-SCAN.
//  2. The tile's payloads are requested at once with one bulk (TMA) copy into
//     shared memory; they are not needed before step 5.  Keys are loaded
//     warp-striped into registers: warp w owns a contiguous run of 32*ITEMS
//     keys and its item i covers keys 32*i .. 32*i+31 of that run, one per
//     lane, so (warp, item, lane) order is input order.
//  3. Rank within the warp: for each item, the lanes holding the same digit
//     are found by one ballot per digit bit; a lane's rank is the number of
//     such peers in lower lanes plus the warp's running count of that digit
//     (a per-warp shared-memory counter that the peers advance together).
//     This is the per-digit exclusive scan of the indicator "digit == d"
//     (section 13.2's rank within digit), done for all digits at once.
//  4. A per-digit scan over the warps gives each warp's offset and the
//     tile's digit counts; the counts are published at once for later tiles
//     (decoupled look-back, flag A), then a block-wide scan over the digits
//     gives each digit's start inside the tile.
//  5. Keys, then payloads, are placed in shared memory in tile-sorted order.
//  6. Look-back: for each digit, the counts of earlier tiles of the row are
//     summed walking backwards, a window of tiles per memory round trip,
//     until a tile that has published its inclusive prefix (flag P); this
//     tile then publishes its own inclusive prefix.  Every wait is bounded
//     in time.  Row-wise sorts may instead take offsets precomputed before
//     the pass from per-tile counts (FlagTree PR #1084 section 2; tiles.cu),
//     at the cost of a second read of the keys.
//  7. Thread j writes staged key j to base[d] + prefix[d] + (j - start[d]):
//     every digit's keys leave as one contiguous run ("100 Days of GPU",
//     day 35: after the local sort the write out is one run per digit).
//     Payloads follow through the same staging buffer.
// The last, partial tile of each row takes a tile id after every full tile
// of the pass (nothing waits on it; it waits only on full tiles of its row,
// which have smaller ids), so it runs in the same launch on a separate code
// path: the full-tile path has no bounds checks.  In a partial tile, lanes
// past the end of the row take the highest digit, rank after every real key
// of the tile, are not counted in the published counts and are not stored
// (the page's sentinel padding, without the padding).
#pragma once
#include <type_traits>

#include "common.cuh"
#include "kernels.h"
#include "keys.cuh"

// Tuning knobs (build-time): a sleep between polls of a word that is not
// ready, the hardware match instruction instead of per-bit ballots, the bulk
// copies of payloads and of keys, and look-back statistics for measurement
// builds.
#ifndef LSDRS_SPIN_SLEEP_NS
#define LSDRS_SPIN_SLEEP_NS 0
#endif
#ifndef LSDRS_MATCH_ANY
#define LSDRS_MATCH_ANY 0
#endif
#ifndef LSDRS_VALS_TMA
#define LSDRS_VALS_TMA 1
#endif
// Keys by bulk copy: measured 1-2% slower than per-lane loads on GB300
// (1.075 vs 1.060 ms per 2^28 key-value pass, 0.765 vs 0.749 keys only):
// the keys are ranked as soon as they arrive, and one copy per tile makes
// every warp wait for the whole tile.
#ifndef LSDRS_KEYS_TMA
#define LSDRS_KEYS_TMA 0
#endif
#ifndef LSDRS_STATS
#define LSDRS_STATS 0
#endif
// L2 prefetch of the keys of a tile that a CTA will take later (a third of
// a resident grid ahead: LSDRS_PREFETCH_AHEAD_PCT of the CTAs resident at
// once), so that the tile's first loads hit L2: 1 for keys-only sorts, 2
// also for key-value sorts (their keys only: the payloads come by bulk copy,
// and prefetching them too measured slower), 0 never.  Measured at 2^28
// (ms per sort, none / one grid ahead / a third ahead): u32 pairs 4.448 /
// 4.345 / 4.320, u32 keys 3.176 / 3.140 / 3.139, u64 pairs 12.62 / 12.46 /
// 12.41, u64 keys 9.78 / 9.57 / 9.53; 1.5 and 2 grids ahead were slower
// than none.
#ifndef LSDRS_L2_PREFETCH
#define LSDRS_L2_PREFETCH 2
#endif
// Whole-byte digits by one byte permute (8-bit digits starting at a multiple
// of 8) instead of shift and mask.
#ifndef LSDRS_BYTE_DIGITS
#define LSDRS_BYTE_DIGITS 1
#endif

namespace lsdrs {

// Header words of the scratch buffer that measurement builds accumulate
// look-back statistics into (look-back round trips, polls of unready words),
// and, with LSDRS_STATS >= 2, per-phase cycle sums of thread 0 as 64-bit
// counters from word kPhaseWord on.
constexpr int kStatsWord = 100;
constexpr int kPhaseWord = 104;
#if LSDRS_STATS >= 2
#define LSDRS_PHASE(k)                                                                   \
  do {                                                                                   \
    if (threadIdx.x == 0) {                                                              \
      const long long now_ = clock64();                                                  \
      atomicAdd(reinterpret_cast<unsigned long long*>(a.error + kPhaseWord) + (k),       \
                static_cast<unsigned long long>(now_ - phase_t_));                       \
      phase_t_ = now_;                                                                   \
    }                                                                                    \
  } while (0)
#else
#define LSDRS_PHASE(k) \
  do {                 \
  } while (0)
#endif

// A store of the pass's output: evict-first (streaming) when
// LSDRS_STREAM_STORES, so that the output, which the next pass reads only
// after the whole pass, does not push the prefetched keys out of L2.
#ifndef LSDRS_STREAM_STORES
#define LSDRS_STREAM_STORES 1
#endif
template <class V>
__device__ __forceinline__ void out_store(V* p, V v) {
  if constexpr (LSDRS_STREAM_STORES && (sizeof(V) == 4 || sizeof(V) == 8)) {
    if constexpr (sizeof(V) == 4)
      __stcs(reinterpret_cast<unsigned int*>(p), static_cast<unsigned int>(v));
    else
      __stcs(reinterpret_cast<unsigned long long*>(p), static_cast<unsigned long long>(v));
  } else {
    *p = v;
  }
}

// This pass's digit of key k: one byte permute when the digit is a whole
// byte of the transformed key (BYTE), else shift and mask.
template <class KeyOp, bool BYTE>
__device__ __forceinline__ uint32_t pass_digit(typename KeyOp::T k, const SweepArgs& a) {
  if constexpr (BYTE)
    return KeyOp::digit_byte(k, a.byte_sel, a.byte_hi != 0, a.xf);
  else
    return KeyOp::digit(k, a.shift, a.mask, a.xf);
}

// Lanes of the warp whose digit equals this lane's digit.
template <int BITS>
__device__ __forceinline__ uint32_t digit_peers(uint32_t d) {
#if LSDRS_MATCH_ANY
  return __match_any_sync(kFull, d);
#else
  uint32_t peers = kFull;
#pragma unroll
  for (int b = 0; b < BITS; ++b) {
    // Vote on bit b; lanes whose bit is clear keep the complement of the
    // votes.  Written with the predicate explicit, the test, the vote and
    // the conditional complement stay about three instructions per bit.
    uint32_t agree;
    asm("{\n\t.reg .pred p;\n\t.reg .b32 t;\n\t"
        "and.b32 t, %1, %2;\n\t"
        "setp.ne.u32 p, t, 0;\n\t"
        "vote.sync.ballot.b32 %0, p, 0xffffffff;\n\t"
        "@!p not.b32 %0, %0;\n\t}"
        : "=r"(agree)
        : "r"(d), "r"(1u << b));
    peers &= agree;
  }
  return peers;
#endif
}

// Bounded wait for a non-zero look-back word (SW: uint32_t or uint64_t).
// On timeout, or when another tile has already reported an error, records
// the error and returns a word with flag P and value 0 so that the walk ends.
template <class SW>
__device__ __forceinline__ SW wait_status(const SW* p, uint32_t* error, uint64_t timeout_ns,
                                          uint32_t& polls) {
  SW v = ld_relaxed(p);
  if (v != 0) return v;
  const uint64_t t0 = global_timer_ns();
  uint32_t spins = 0;
  for (;;) {
#if LSDRS_SPIN_SLEEP_NS > 0
    __nanosleep(LSDRS_SPIN_SLEEP_NS);
#endif
    v = ld_relaxed(p);
    ++spins;
    if (v != 0) break;
    if ((spins & 63u) == 0) {
      if (ld_relaxed(error) != kErrNone) {
        v = LookbackWord<SW>::kFlagP;
        break;
      }
      if (global_timer_ns() - t0 > timeout_ns) {
        atomicCAS(error, kErrNone, kErrLookback);
        v = LookbackWord<SW>::kFlagP;
        break;
      }
    }
  }
  polls += spins;
  return v;
}

// Exclusive prefix of one digit over tiles [0, t) of a row.  `col` points at
// this digit's word of the row's tile 0; tile k's word is col[k * R].  Each
// round trip loads the words of WIN predecessors at once (for the 32 digits
// of a warp these are coalesced 128-byte rows) and consumes them up to the
// first inclusive prefix, or up to the first word not yet published, on
// which it then waits.
template <int R, int WIN, class SW>
__device__ __forceinline__ SW look_back(const SW* col, int64_t t, uint32_t* error,
                                        uint64_t timeout_ns, uint32_t& trips, uint32_t& polls) {
  static_assert(WIN >= 1 && WIN <= 32, "window of 1..32 tiles");
  using LW = LookbackWord<SW>;
  // Raw words are summed: the flag bits sit above the value field and the
  // true sum of the counts stays below its capacity (2^30 or 2^62), so
  // masking once at the end is exact.
  SW raw = 0;
  int pt = static_cast<int>(t) - 1;  // newest predecessor not yet consumed
  for (;;) {
    const SW* p = col + static_cast<int64_t>(pt) * R;  // word of tile pt
    SW v[WIN];
    if (pt >= WIN - 1) {
#pragma unroll
      for (int k = 0; k < WIN; ++k)
        v[k] = in_bounds(pt - k >= 0, error, 8) ? ld_relaxed(p - k * R) : LW::kFlagP;
    } else {
#pragma unroll
      for (int k = 0; k < WIN; ++k) v[k] = k <= pt ? ld_relaxed(p - k * R) : LW::kFlagP;
    }
    ++trips;
    // consume the window in order up to the first inclusive prefix (done),
    // or up to the first word not yet published (wait for it)
    int k = 0;
#pragma unroll
    for (; k < WIN; ++k) {
      if (v[k] == 0) break;
      raw += v[k];
      if (static_cast<std::make_signed_t<SW>>(v[k]) < 0) return raw & LW::kValueMask;  // flag P
    }
    if (k < WIN) {
      const SW w = wait_status(p - k * R, error, timeout_ns, polls);
      raw += w;
      if (w & LW::kFlagP) return raw & LW::kValueMask;
      pt -= k + 1;
    } else {
      pt -= WIN;
    }
  }
}

// Shared-memory arrays every tile needs besides its key/payload buffers.
template <int W, int R>
struct TileScratch {
  alignas(16) uint32_t warp_cnt[W][R];  // per-warp digit counters, then per-warp offsets
  uint32_t warp_tot[W];     // per-warp sums of the digit-count scan
  uint32_t g_off[R];        // output position of staged slot j is g_off[d] + j
  uint32_t code;            // this pass's schedule code (kCode* bits)
  uint32_t skip_stores;     // a copy into this tile's shared memory timed out
};

// This pass's buffers and look-back arrays, picked from the kernel
// parameters by the schedule entry (so that the compiler still sees global
// pointers).
template <class P>
__device__ __forceinline__ P pick_buf(const P (&b)[3], uint32_t i) {
  return i == kBufIn ? b[0] : (i == kBufAlt ? b[1] : b[2]);
}

template <bool DYN>
struct PassBufs {
  uint32_t code;
  const SweepArgs& a;
  __device__ __forceinline__ bool first() const { return code & kCodeFirst; }
  __device__ __forceinline__ bool last() const { return code & kCodeLast; }
  __device__ __forceinline__ uint32_t src() const { return code & kCodeSrc; }
  __device__ __forceinline__ uint32_t dst() const { return (code & kCodeDst) >> 2; }
  __device__ __forceinline__ const void* keys_in() const {
    return DYN ? pick_buf(a.keys, src()) : a.pass_keys_in;
  }
  __device__ __forceinline__ void* keys_out() const {
    return DYN ? const_cast<void*>(pick_buf(a.keys, dst())) : a.pass_keys_out;
  }
  // column indices (kValIdx): int32 in the scratch buffer, int64 at the end;
  // the first pass run generates them
  template <int VK>
  __device__ __forceinline__ const void* vals_in() const {
    if (!DYN) return a.pass_vals_in;
    if (VK == kValIdx) return first() ? nullptr : a.vals[kBufAlt];
    return pick_buf(a.vals, src());
  }
  template <int VK>
  __device__ __forceinline__ void* vals_out() const {
    if (!DYN) return a.pass_vals_out;
    if (VK == kValIdx) return const_cast<void*>(last() ? a.vals[kBufOut] : a.vals[kBufAlt]);
    return const_cast<void*>(pick_buf(a.vals, dst()));
  }
  __device__ __forceinline__ void* status() const {
    return DYN ? a.status_arr[(code & kCodeOdd) ? 1 : 0] : a.pass_status;
  }
  __device__ __forceinline__ void* status_zero() const {
    if (!DYN) return a.pass_status_zero;
    return last() ? nullptr : a.status_arr[(code & kCodeOdd) ? 0 : 1];
  }
};

// Where a tile's keys and payloads are read from and staged to.  The key
// source is global and the payloads are in shared memory, both by tile
// position (the item at tile position p is key_src[p], vals[p]).
template <class KeyOp>
struct TileIo {
  const typename KeyOp::T* key_src;  // global
  typename KeyOp::T* stage_keys;     // shared, TILE keys
  uint32_t* vals;                    // shared, TILE words: payloads in, then their stage
  uint64_t* val_bar;                 // non-null: a bulk copy into vals completes on it
  uint64_t* key_bar;                 // non-null: the keys come by a bulk copy into the
                                     // stage, which completes on it
  bool vals_in;                      // payloads were loaded (else indices are generated)
};

// One tile: rank, publish, look back, stage, write.  Called by every thread
// of the CTA; begins and ends with all threads converged.  The tile is tile
// t of its row; status_row points at the row's first look-back word (SW:
// 32- or 64-bit words).
template <bool FULL, bool DYN, bool PRE, class KeyOp, int BITS, int VK, int THREADS, int ITEMS,
          int WIN, bool BYTE, class SW>
__device__ __forceinline__ void sweep_tile(const SweepArgs& a,
                                           TileScratch<THREADS / kWarp, (1 << BITS)>& s,
                                           const TileIo<KeyOp>& io, SW* status_row, int64_t row,
                                           int64_t t, int64_t tile_begin, int valid) {
  using LW = LookbackWord<SW>;
  using T = typename KeyOp::T;
  constexpr int R = 1 << BITS;
  constexpr int W = THREADS / kWarp;
  constexpr int TILE = THREADS * ITEMS;
  constexpr int WKEYS = kWarp * ITEMS;
  constexpr bool kVals = VK == kValU32 || VK == kValIdx;  // a payload array travels
  constexpr bool kPack = VK == kValPack16;                // column index inside the key word
  // Keys whose transform is applied once (signed, float, descending): the
  // registers and ping-pong buffers hold T(k), whose digits are DK's.
  using DK = typename KeyOp::Stored;
  constexpr bool kEnc = !std::is_same<DK, KeyOp>::value;
  const PassBufs<DYN> pass{DYN ? s.code : a.code, a};

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int64_t row_base = row * a.cols;
  SW* status_tile = status_row + t * R;
  const int wpos = warp * WKEYS + lane;  // tile position of item 0
  uint32_t trips = 0, polls = 0;
#if LSDRS_STATS >= 2
  long long phase_t_ = clock64();
#endif

  T keys[ITEMS];
  if (FULL && io.key_bar != nullptr) {
    // The tile's keys were bulk-copied into the stage buffer (16-byte
    // transfers, waited for by the caller); each thread reads its items
    // warp-striped from there.
    if (kPack && pass.first()) {
      const uint16_t* st16 = reinterpret_cast<const uint16_t*>(io.stage_keys);
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) {
        const int p = wpos + i * kWarp;
        keys[i] = KeyF16Packed::pack(st16[p], static_cast<uint32_t>(tile_begin + p), a.xf);
      }
    } else {
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) keys[i] = io.stage_keys[wpos + i * kWarp];
    }
  } else if (kPack && pass.first()) {
    // the row's 16-bit keys, transformed and packed with their columns
    const uint16_t* src16 = reinterpret_cast<const uint16_t*>(io.key_src);
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int p = wpos + i * kWarp;
      keys[i] = ((FULL || p < valid) &&
                 in_bounds(p < valid && tile_begin + p < a.cols, a.error, 1))
                    ? KeyF16Packed::pack(src16[p], static_cast<uint32_t>(tile_begin + p), a.xf)
                    : T(0);
    }
  } else {
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      keys[i] = ((FULL || wpos + i * kWarp < valid) &&
                 in_bounds(wpos + i * kWarp < valid && tile_begin + wpos + i * kWarp < a.cols,
                           a.error, 1))
                    ? io.key_src[wpos + i * kWarp]
                    : T(0);
  }
  if constexpr (kEnc) {
    if (pass.first()) {
#pragma unroll
      for (int i = 0; i < ITEMS; ++i) keys[i] = static_cast<T>(KeyOp::encode(keys[i], a.xf));
    }
  }

  // ---- 3. rank within the warp ------------------------------------------
  // The rank of item i among the warp's keys of its digit (below
  // 32 * ITEMS < 2^16) is kept in half i % 2 of packed[i / 2]; the digit
  // is taken from the key again when it is needed.  Two ranks per register
  // keep the tile's state in registers.
  constexpr int NP = (ITEMS + 1) / 2;
  uint32_t packed[NP];
  uint32_t* wc = s.warp_cnt[warp];
  const uint32_t lt = lanemask_lt();
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    uint32_t d = pass_digit<DK, BYTE>(keys[i], a);
    if (!FULL && wpos + i * kWarp >= valid) d = R - 1;
    const uint32_t peers = digit_peers<BITS>(d);
    // Every peer lane reads the warp's count of its digit (one word per
    // digit, so a broadcast) and, after a warp barrier, stores the advanced
    // count: the peers write the same value to the same word.
    const bool d_ok = in_bounds(d < R, a.error, 2);
    const uint32_t before = d_ok ? wc[d] : 0u;
    __syncwarp();
    if (d_ok) wc[d] = before + __popc(peers);
    __syncwarp();
    const uint32_t rank = before + __popc(peers & lt);
    if (i & 1)
      packed[i >> 1] |= rank << 16;
    else
      packed[i >> 1] = rank;
  }
  __syncthreads();
  LSDRS_PHASE(0);  // loads + ranking

  // ---- 4. tile counts, publish, digit starts, warp offsets --------------
  // Thread d turns the warps' counts of digit d into exclusive prefixes over
  // the warps and publishes their sum; a block-wide exclusive scan of the
  // sums gives digit d's start in the tile, which is then added to the
  // prefixes: warp w's first slot for d (staging reads one word per key;
  // thread d walks column d, so the column accesses are conflict-free).
  uint32_t my_count = 0;  // this tile's count of digit tid (without padding)
  uint32_t start = 0;     // first slot of digit tid in the tile
  {
    uint32_t total = 0;
    if (tid < R) {
#pragma unroll
      for (int w = 0; w < W; ++w) {
        const uint32_t c = s.warp_cnt[w][tid];
        s.warp_cnt[w][tid] = total;
        total += c;
      }
      my_count = (!FULL && tid == R - 1) ? total - static_cast<uint32_t>(TILE - valid) : total;
      // a partial tile is the last of its row: nothing waits on it
      if (FULL && !PRE)
        st_relaxed(status_tile + tid, (t == 0 ? LW::kFlagP : LW::kFlagA) | SW(my_count));
    }
    uint32_t incl = total;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFull, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == kWarp - 1) s.warp_tot[warp] = incl;
    __syncthreads();
    LSDRS_PHASE(1);  // counts + publish
    uint32_t before = 0;
#pragma unroll
    for (int w = 0; w + 1 < W; ++w)
      if (w < warp) before += s.warp_tot[w];
    start = before + incl - total;
    if (tid < R) {
#pragma unroll
      for (int w = 0; w < W; ++w) s.warp_cnt[w][tid] += start;
    }
  }
  __syncthreads();
  LSDRS_PHASE(2);  // digit scan

  // ---- 5. stage keys, then payloads, in tile-sorted order ---------------
  auto half = [](uint32_t w, int i) -> uint32_t { return (i & 1) ? (w >> 16) : (w & 0xFFFFu); };
  auto item_digit = [&](int i) -> uint32_t {
    if (!FULL && wpos + i * kWarp >= valid) return R - 1;
    return pass_digit<DK, BYTE>(keys[i], a);
  };
  // Two items at a time: their warp offsets are packed like their ranks,
  // so one add gives both staging slots (each below TILE < 2^16, so the low
  // half never carries), and packed[] then holds the slots for the payloads.
#pragma unroll
  for (int k = 0; k < NP; ++k) {
    const int i0 = 2 * k, i1 = 2 * k + 1;
    const uint32_t d0 = item_digit(i0);
    const uint32_t d1 = i1 < ITEMS ? item_digit(i1) : 0u;
    const uint32_t o0 = in_bounds(d0 < R, a.error, 2) ? s.warp_cnt[warp][d0] : 0u;
    const uint32_t o1 = (i1 < ITEMS && in_bounds(d1 < R, a.error, 2)) ? s.warp_cnt[warp][d1] : 0u;
    const uint32_t pos = packed[k] + __byte_perm(o0, o1, 0x5410);
    if (in_bounds((pos & 0xFFFFu) < TILE, a.error, 3)) io.stage_keys[pos & 0xFFFFu] = keys[i0];
    if (i1 < ITEMS && in_bounds((pos >> 16) < TILE, a.error, 3))
      io.stage_keys[pos >> 16] = keys[i1];
    packed[k] = pos;
  }
  if constexpr (kVals) {
    if (io.val_bar != nullptr && !mbar_wait_bounded(io.val_bar, 0, a.timeout_ns)) {
      // The bulk copy did not land in time: report it and keep this tile's
      // unverified payloads out of the output (its look-back still runs, so
      // later tiles are released).  The copy writes this CTA's shared memory,
      // so it gets a further bounded period to finish before the CTA moves on.
      atomicCAS(a.error, kErrNone, kErrLookback);
      s.skip_stores = 1;
      mbar_wait_bounded(io.val_bar, 0, kCopyDrainNs);
    }
    // The payloads are staged in the buffer they were loaded into: read
    // every thread's payloads before any is overwritten.
    const bool vin = VK == kValU32 || io.vals_in;
    uint32_t v[ITEMS];
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int p = wpos + i * kWarp;
      v[i] = !vin ? static_cast<uint32_t>(tile_begin + p)
                  : (((FULL || p < valid) && in_bounds(p < TILE, a.error, 4)) ? io.vals[p] : 0u);
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < ITEMS; ++i)
      if (in_bounds(half(packed[i >> 1], i) < TILE, a.error, 5))
        io.vals[half(packed[i >> 1], i)] = v[i];
  }
  LSDRS_PHASE(3);  // staging (thread 0's share)

  // ---- 6. decoupled look-back (thread d, digit d) ------------------------
  // Sums the counts of the row's earlier tiles up to the first inclusive
  // prefix and publishes this tile's inclusive prefix.  (PRE: the tile's
  // output offsets were computed before the pass from per-tile digit counts,
  // so there is nothing to wait for.)  Output positions are below 2^32.
  if (PRE && tid < R) {
    s.g_off[tid] = a.offsets[(row * a.tiles_per_row + t) * R + tid] - start;
  } else if (tid < R) {
    SW excl = 0;
    if (t > 0) {
      excl = look_back<R, WIN>(status_row + tid, t, a.error, a.timeout_ns, trips, polls);
      if (FULL) st_relaxed(status_tile + tid, LW::kFlagP | (excl + my_count));
    }
    s.g_off[tid] = a.bases[row * a.bases_row_stride + tid] + static_cast<uint32_t>(excl) - start;
  }
  LSDRS_PHASE(4);  // thread 0's look-back
#if LSDRS_STATS
  if (trips) atomicAdd(a.error + kStatsWord, trips);
  if (polls) atomicAdd(a.error + kStatsWord + 1, polls);
#endif
  __syncthreads();
  LSDRS_PHASE(5);  // wait for the slowest digit's look-back
  if (s.skip_stores) return;  // (uniform: read after the barrier)

  // ---- 7. contiguous per-digit runs out ---------------------------------
  const PassBufs<DYN> pb{DYN ? s.code : a.code, a};
  T* kout = static_cast<T*>(pb.keys_out()) + row_base;
  uint32_t* vout32 = static_cast<uint32_t*>(pb.template vals_out<VK>()) + row_base;
  int64_t* vout64 = static_cast<int64_t*>(pb.template vals_out<VK>()) + row_base;
  const bool wide = VK == kValIdx && pb.last();
  const bool last_run = pb.last();  // (kEnc) write T^-1 of the carried keys
  if (kPack && pb.last()) {
    // the packed words leave as the row's values and their int64 columns
    uint16_t* v16 = static_cast<uint16_t*>(pb.keys_out()) + row_base;
#pragma unroll
    for (int i = 0; i < ITEMS; ++i) {
      const int j = i * THREADS + tid;
      if (FULL || j < valid) {
        const T k = io.stage_keys[j];
        const uint32_t d = pass_digit<DK, BYTE>(k, a);
        if (!in_bounds(d < R, a.error, 6)) continue;
        const uint32_t g = s.g_off[d] + static_cast<uint32_t>(j);
        if (!in_bounds(g < a.cols, a.error, 7)) continue;
        v16[g] = KeyF16Packed::bits(k, a.xf);
        vout64[g] = static_cast<int64_t>(k & 0xFFFFu);
      }
    }
    return;
  }
#pragma unroll
  for (int i = 0; i < ITEMS; ++i) {
    const int j = i * THREADS + tid;
    if (FULL || j < valid) {
      const T k = io.stage_keys[j];
      uint32_t v = 0;
      if constexpr (kVals) v = io.vals[j];
      const uint32_t d = pass_digit<DK, BYTE>(k, a);
      if (!in_bounds(d < R, a.error, 6)) continue;
      const uint32_t g = s.g_off[d] + static_cast<uint32_t>(j);
      if (!in_bounds(g < a.cols, a.error, 7)) continue;
      T kw = k;
      if constexpr (kEnc) kw = last_run ? static_cast<T>(KeyOp::decode(k, a.xf)) : k;
      out_store(kout + g, kw);
      if constexpr (kVals) {
        if (wide)
          out_store(vout64 + g, static_cast<int64_t>(static_cast<int32_t>(v)));
        else
          out_store(vout32 + g, v);
      }
    }
  }
  LSDRS_PHASE(6);  // write-out
}

// Shared memory of one tile.
template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS>
struct SweepSmem {
  using T = typename KeyOp::T;
  static constexpr int kTile = THREADS * ITEMS;
  static constexpr bool kVals = VK == kValU32 || VK == kValIdx;
  alignas(128) T stage[kTile];                    // keys in tile-sorted order
  alignas(128) uint32_t vals[kVals ? kTile : 4];  // payloads in, then their stage
  TileScratch<THREADS / kWarp, (1 << BITS)> scratch;
  uint64_t bar;  // the tile's bulk copies (keys, payloads) complete on it
  uint32_t tile_id;
  uint32_t abort;
};

// One CTA, one tile, taken from the tile counter: ids below
// rows * full_per_row are the full tiles of every row, in row-major order;
// id rows * full_per_row + r is row r's partial last tile, if rows have one.
// DYN: the schedule (which passes run, between which buffers) comes from
// K-SCAN through the tile counter; otherwise it is the host's static one in
// the kernel arguments (every pass runs).
template <bool DYN, bool PRE, class KeyOp, int BITS, int VK, int THREADS, int ITEMS, int WIN,
          bool BYTE, bool WIDE>
__device__ __forceinline__ void onesweep_body(const SweepArgs& a) {
  using S = SweepSmem<KeyOp, BITS, VK, THREADS, ITEMS>;
  using SW = std::conditional_t<WIDE, uint64_t, uint32_t>;  // look-back word
  using T = typename KeyOp::T;
  constexpr int R = 1 << BITS;
  constexpr int W = THREADS / kWarp;
  constexpr int TILE = S::kTile;
  static_assert(R <= THREADS, "one thread per digit");
  static_assert(TILE < 65536, "ranks and staging slots are packed in 16 bits");

  extern __shared__ __align__(128) unsigned char smem_raw[];
  S& s = *reinterpret_cast<S*>(smem_raw);
  const int tid = threadIdx.x;
  grid_dependency_sync();

  // the tile id and this pass's schedule code in one word
  if (tid == 0) {
    const uint32_t v = atomicAdd(a.tile_counter, 1u);
    s.tile_id = v & kTileMask;
    if (DYN) s.scratch.code = v >> kCodeShift;
    s.abort = ld_relaxed(a.error) != kErrNone;
    s.scratch.skip_stores = 0;
    // the bulk copies' barriers, initialised before the block-wide barrier
    // below so that every thread that waits on one sees it initialised
    if (LSDRS_VALS_TMA || LSDRS_KEYS_TMA) mbar_init(&s.bar, 1);
  }
  static_assert((W * R) % 4 == 0, "counters are zeroed 16 bytes at a time");
  for (int i = tid; i < W * R / 4; i += THREADS)
    reinterpret_cast<uint4*>(&s.scratch.warp_cnt[0][0])[i] = make_uint4(0u, 0u, 0u, 0u);
  __syncthreads();

  const uint32_t fpr = static_cast<uint32_t>(a.full_per_row);
  const uint32_t n_full = static_cast<uint32_t>(a.rows) * fpr;
  const bool full = s.tile_id < n_full;
  int64_t row, t, tile_begin;
  if (!full) {
    row = s.tile_id - n_full;
    t = a.full_per_row;
    tile_begin = t * TILE;
  } else {
    // tile ids are below 2^24, so 32-bit arithmetic suffices
    const uint32_t id = s.tile_id;
    const uint32_t r32 = id / fpr;
    row = r32;
    t = id - r32 * fpr;
    tile_begin = t * TILE;
  }
  const int valid = full ? TILE : static_cast<int>(a.cols - tile_begin);
  const int64_t off = row * a.cols + tile_begin;
  if (DYN && (s.scratch.code & kCodeSkip)) return;  // an identity pass: not run
  const PassBufs<DYN> pb{DYN ? s.scratch.code : a.code, a};
  // look-back words are indexed by full tile, row-major: row r's tile t at
  // r * full_per_row + t; partial tiles publish none
  SW* status_row = static_cast<SW*>(pb.status()) + (row * a.full_per_row) * R;
  TileIo<KeyOp> io;
  io.key_src = static_cast<const T*>(pb.keys_in()) + off;
  if (VK == kValPack16 && pb.first())  // 16-bit keys: offset in 16-bit units
    io.key_src = reinterpret_cast<const T*>(static_cast<const uint16_t*>(pb.keys_in()) + off);
  io.stage_keys = s.stage;
  io.vals = s.vals;
  io.val_bar = nullptr;
  io.key_bar = nullptr;
  io.vals_in = false;
  if (s.abort) {  // an earlier tile failed: release successors and stop
    if (full && !PRE && tid < R) st_relaxed(status_row + t * R + tid, LookbackWord<SW>::kFlagP);
  } else {
    // Bulk copies into shared memory, for a full tile from 16-byte aligned
    // sources: the keys into the stage buffer (free until the keys are in
    // registers) and the payloads into their buffer, both completing on one
    // barrier.  The keys are read right away, so the CTA waits for the
    // copies before ranking; payloads alone are waited for at the staging
    // step.  Sources that do not qualify are loaded by the threads: keys by
    // each thread for itself, payloads by the CTA into their buffer (the
    // tile's first block-wide barrier makes them visible).
    const uint32_t kbytes = TILE * ((VK == kValPack16 && pb.first()) ? 2u : sizeof(T));
    if ((VK == kValNone ? LSDRS_L2_PREFETCH >= 1 : VK == kValU32 && LSDRS_L2_PREFETCH >= 2) &&
        a.prefetch_tiles != 0 && a.rows == 1) {
      // a flat sort: the tile handed out about one resident-grid later
      const uint32_t nt = s.tile_id + a.prefetch_tiles;
      if (nt < n_full) {
        const char* kb = static_cast<const char*>(pb.keys_in()) +
                         static_cast<uint64_t>(nt) * TILE * sizeof(T);
        const uint32_t klines = TILE * static_cast<uint32_t>(sizeof(T)) / 128u;
        for (uint32_t l = tid; l < klines; l += THREADS) prefetch_l2(kb + 128u * l);
      }
    }
    const bool keys_tma =
        LSDRS_KEYS_TMA && full && (reinterpret_cast<uintptr_t>(io.key_src) & 15) == 0;
    const uint32_t* vsrc = nullptr;
    bool vals_tma = false;
    if ((VK == kValU32 || VK == kValIdx) && pb.template vals_in<VK>() != nullptr) {
      vsrc = static_cast<const uint32_t*>(pb.template vals_in<VK>()) + off;
      io.vals_in = true;
      vals_tma = LSDRS_VALS_TMA && full && (reinterpret_cast<uintptr_t>(vsrc) & 15) == 0;
    }
    if (tid == 0 && (keys_tma || vals_tma)) {
      const uint32_t vbytes = TILE * static_cast<uint32_t>(sizeof(uint32_t));
      mbar_arrive_expect_tx(&s.bar, (keys_tma ? kbytes : 0u) + (vals_tma ? vbytes : 0u));
      if (keys_tma) bulk_copy_g2s(s.stage, io.key_src, kbytes, &s.bar);
      if (vals_tma) bulk_copy_g2s(s.vals, vsrc, vbytes, &s.bar);
    }
    if (vals_tma) io.val_bar = &s.bar;
    if (vsrc != nullptr && !vals_tma)
      for (int i = tid; i < valid; i += THREADS) s.vals[i] = ld_stream(vsrc + i);
    if (keys_tma) {
      io.key_bar = &s.bar;
      if (!mbar_wait_bounded(&s.bar, 0, a.timeout_ns)) {
        // The copy did not land in time: report it, keep this tile's stores
        // out of the output (its look-back still runs), and give the copy a
        // further bounded period to finish before the buffers are reused.
        atomicCAS(a.error, kErrNone, kErrLookback);
        s.scratch.skip_stores = 1;
        mbar_wait_bounded(&s.bar, 0, kCopyDrainNs);
      }
    }
    if (!full) {
      sweep_tile<false, DYN, PRE, KeyOp, BITS, VK, THREADS, ITEMS, WIN, BYTE>(
          a, s.scratch, io, status_row, row, t, tile_begin, valid);
    } else {
      sweep_tile<true, DYN, PRE, KeyOp, BITS, VK, THREADS, ITEMS, WIN, BYTE>(
          a, s.scratch, io, status_row, row, t, tile_begin, valid);
    }
  }
  SW* zero = static_cast<SW*>(PassBufs<DYN>{DYN ? s.scratch.code : a.code, a}.status_zero());
  if (full && !PRE && zero != nullptr && tid < R)
    zero[static_cast<int64_t>(s.tile_id) * R + tid] = 0;
}

template <bool DYN, bool PRE, class KeyOp, int BITS, int VK, int THREADS, int ITEMS, int MINB,
          int WIN, bool BYTE, bool WIDE>
__global__ void __launch_bounds__(THREADS, MINB) onesweep_kernel(SweepArgs a) {
  onesweep_body<DYN, PRE, KeyOp, BITS, VK, THREADS, ITEMS, WIN, BYTE, WIDE>(a);
}

template <class K>
cudaError_t launch_with_smem(K kern, unsigned grid, int threads, size_t smem, cudaStream_t s,
                             const SweepArgs& a) {
  if (smem > 48 * 1024) {
    cudaError_t e =
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  return launch_kernel(kern, grid, threads, smem, s, a);
}

// One pass: every full tile, then each row's partial tile, in one launch.
// Returns the number of kernels launched in *launched.
// PRE: offsets precomputed by the tile-count kernels (row-wise sorts only).
// WIDE: 64-bit look-back words (flat sorts of 2^30 keys or more).
template <class KeyOp, int BITS, int VK, int THREADS, int ITEMS, int MINB, int WIN,
          bool PRE = false, bool WIDE = false>
cudaError_t launch_sweep_t(const SweepArgs& args, int* launched, cudaStream_t s) {
  using S = SweepSmem<KeyOp, BITS, VK, THREADS, ITEMS>;
  constexpr int TILE = S::kTile;
  const SweepArgs& a = args;
  *launched = 0;
  const int64_t full = a.rows * a.full_per_row;
  const bool partial = a.rows > 0 && a.cols % TILE != 0;
  const int64_t grid = full + (partial ? a.rows : 0);
  if (grid <= 0) return cudaSuccess;
  // whole-byte digits (every 8-bit pass but a narrower last one) of keys of
  // at most 32 bits take the byte-permute instantiation (for 64-bit keys
  // it measured slower than shift and mask: 13.02 vs 12.34 ms per 2^28
  // key-value sort)
  constexpr bool B8 = LSDRS_BYTE_DIGITS && BITS == 8 && sizeof(typename KeyOp::T) <= 4;
  const bool byte = B8 && a.shift % 8 == 0 && a.mask == 0xFFu;
  const unsigned g = static_cast<unsigned>(grid);
  cudaError_t e;
  if (byte)
    e = a.dynamic
            ? launch_with_smem(onesweep_kernel<true, PRE, KeyOp, BITS, VK, THREADS, ITEMS, MINB,
                                               WIN, B8, WIDE>, g, THREADS, sizeof(S), s, a)
            : launch_with_smem(onesweep_kernel<false, PRE, KeyOp, BITS, VK, THREADS, ITEMS, MINB,
                                               WIN, B8, WIDE>, g, THREADS, sizeof(S), s, a);
  else
    e = a.dynamic
            ? launch_with_smem(onesweep_kernel<true, PRE, KeyOp, BITS, VK, THREADS, ITEMS, MINB,
                                               WIN, false, WIDE>, g, THREADS, sizeof(S), s, a)
            : launch_with_smem(onesweep_kernel<false, PRE, KeyOp, BITS, VK, THREADS, ITEMS, MINB,
                                               WIN, false, WIDE>, g, THREADS, sizeof(S), s, a);
  if (e != cudaSuccess) return e;
  *launched = 1;
  return cudaSuccess;
}

template <class KeyOp, int VK, int THREADS, int ITEMS, int MINB, int WIN, bool WIDE = false>
cudaError_t launch_sweep_bits(int bits, const SweepArgs& a, int* launched, cudaStream_t s) {
  switch (bits) {
    case 1: return launch_sweep_t<KeyOp, 1, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 2: return launch_sweep_t<KeyOp, 2, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 3: return launch_sweep_t<KeyOp, 3, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 4: return launch_sweep_t<KeyOp, 4, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 5: return launch_sweep_t<KeyOp, 5, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 6: return launch_sweep_t<KeyOp, 6, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 7: return launch_sweep_t<KeyOp, 7, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    case 8: return launch_sweep_t<KeyOp, 8, VK, THREADS, ITEMS, MINB, WIN, false, WIDE>(a, launched, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace lsdrs
