/*
 * lsdrs -- least-significant-digit radix sort for NVIDIA GB300 (sm_103a).
 *
 * The method (CUDA Handbook ch. 16 "Radix Sort", opening section and
 * Listings 16-8/16-9; DSA CUDA from First Principles ch. 13, sections
 * 13.1-13.3): keys are sorted one b-bit digit at a time, least significant
 * digit first.  Each pass histograms the digit, turns the counts into bucket
 * bases with an exclusive scan, and scatters every key stably to
 * base[digit] + (number of earlier keys with the same digit).  Passes
 * ping-pong between two buffers.
 *
 * On the GPU one sort is: an upfront kernel that reads the keys once and
 * counts the digits of every pass; a scan kernel that turns those counts
 * into bases; then one "onesweep" scatter kernel per pass, in which tiles
 * rank their keys in shared memory, learn the counts of earlier tiles by a
 * decoupled look-back, and write each digit's keys as one contiguous run.
 * A sort whose rows (the whole input, for a flat sort) hold at most 8,192
 * keys, with 4- or 8-bit digits, runs in one kernel instead: one CTA per row
 * does every pass in shared memory (see RS_OPT_NO_SMALL_SORT).
 *
 * Conventions shared by every call:
 *  - Pointers marked (device) are device memory of the current device; the
 *    caller owns all of them, including `temp`.  The library allocates
 *    nothing on the sort path.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream).  Every sort call is asynchronous: it validates on the host,
 *    enqueues its kernels on `stream` and returns; it never synchronises.
 *  - Inputs are never written (sorting is out of place; "100 Days of GPU"
 *    day 35, Pitfalls: never re-sort your own output).  keys_out may equal
 *    keys_in (and vals_out vals_in) for an in-place sort; any other overlap
 *    is rejected.
 *  - Sorting is stable and ascending on bits [begin_bit, end_bit) of the
 *    key; bits outside that range do not take part in the order but are
 *    carried in the output keys.  The number of passes is
 *    ceil((end_bit - begin_bit) / digit_bits); the last digit may be
 *    narrower.
 *  - Host-side argument errors return RS_ERR_INVALID or
 *    RS_ERR_TEMP_TOO_SMALL before anything is enqueued.  A failed launch
 *    returns RS_ERR_CUDA.  Errors raised on the device (a look-back wait
 *    that exceeded its time limit) are recorded in `temp` and returned by
 *    radix_sort_device_status().
 *  - Modes (pass skipping, precomputed tile offsets, the one-kernel path for
 *    short rows, the wait limit) are options of the call that wants them
 *    (rs_options); the library keeps no mode state between calls, so calls
 *    from different threads or streams never change each other's schedule.
 */
#ifndef LSDRS_H
#define LSDRS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum rs_status {
  RS_OK = 0,
  RS_ERR_INVALID = 1,          /* bad argument, found before any launch */
  RS_ERR_TEMP_TOO_SMALL = 2,   /* temp_bytes below the size query's answer */
  RS_ERR_CUDA = 3,             /* a CUDA runtime call or launch failed */
  RS_ERR_LOOKBACK_TIMEOUT = 4  /* device: a look-back wait ran out of time */
} rs_status;

typedef enum rs_float_kind { RS_F16 = 0, RS_BF16 = 1 } rs_float_kind;

/* Key types of the typed global sorts. */
typedef enum rs_key_type {
  RS_KEY_U32 = 0, RS_KEY_I32 = 1, RS_KEY_F32 = 2,   /* 4-byte keys */
  RS_KEY_U64 = 3, RS_KEY_I64 = 4, RS_KEY_F64 = 5    /* 8-byte keys */
} rs_key_type;

/* Largest number of keys in one flat sort: output positions are 32-bit.
 * The look-back words of a sort hold a flag pair and a count in 32 bits (a
 * 30-bit count) below 2^30 keys, and in 64 bits (a 62-bit count) for a flat
 * sort of 2^30 keys or more; the scratch size accounts for it. */
#define RS_MAX_KEYS ((size_t)0xFFFFFFFFu)
/* Largest row of a row-wise sort (FlagTree PR #1084, "radix_sort"
 * signature: n < 2^30). */
#define RS_MAX_ROW_KEYS ((size_t)((1u << 30) - 1u))

/* Options of one sort call.  A NULL rs_options* means all defaults; a
 * zero-initialised struct is the same.
 *   flags  RS_OPT_* bits (unknown bits: RS_ERR_INVALID)
 *     RS_OPT_PASS_SKIPPING  a pass in which every key (every key of every
 *            row, for a row-wise sort) has the same digit is the identity
 *            permutation and is not run; decided on the device from the
 *            upfront histograms, so nothing waits, and the output is the
 *            same.  Off by default: a sort of keys that vary in every digit
 *            pays about 1% for the device-side schedule.
 *     RS_OPT_TILE_OFFSETS   row-wise sorts only: before each pass a kernel
 *            counts the digits of every tile and a per-row scan turns the
 *            counts into offsets, so the scatter never waits on another tile
 *            (FlagTree PR #1084, section 2, "precompute each tile"); it reads
 *            the keys once more per pass.  Pass skipping does not apply.
 *     RS_OPT_NO_SMALL_SORT  sorts whose rows hold at most 8,192 keys take the
 *            multi-kernel path like longer rows instead of the one-kernel
 *            path (which runs every pass: it never skips).
 *   lookback_timeout_ns  limit on one look-back or copy wait inside the
 *            scatter kernels; 0 = the default, 2 s; at most 60 s.  A wait
 *            that runs past it records RS_ERR_LOOKBACK_TIMEOUT (read it with
 *            radix_sort_device_status) and releases every later tile.
 * The results never depend on the options. */
typedef struct rs_options {
  unsigned flags;
  uint64_t lookback_timeout_ns;
} rs_options;
#define RS_OPT_PASS_SKIPPING 0x1u
#define RS_OPT_TILE_OFFSETS 0x2u
#define RS_OPT_NO_SMALL_SORT 0x4u

/* Size in bytes of the scratch buffer a flat sort needs (keys only or
 * key-value; the same size serves any options).
 *   n           number of keys (0 <= n <= RS_MAX_KEYS)
 *   key_bytes   4 (u32) or 8 (u64)
 *   value_bytes 0 (keys only) or 4 (u32 payload)
 *   begin_bit, end_bit, digit_bits  as for the sort calls
 * Writes the size to *bytes.  Host only; enqueues nothing. */
rs_status radix_sort_keys_temp_bytes(size_t n, int key_bytes, int value_bytes,
                                     int begin_bit, int end_bit, int digit_bits,
                                     size_t* bytes);

/* Keys-only LSD radix sort of n unsigned 32-bit keys.
 * (CUDA Handbook ch. 16, Listing 16-9 "RadixSort": one counting-sort pass per
 * digit, ping-ponging between two buffers.)
 *   keys_in   (device) n keys, read only
 *   keys_out  (device) n keys, the sorted result
 *   n         0 <= n <= RS_MAX_KEYS; n == 0 enqueues nothing
 *   begin_bit 0 <= begin_bit < end_bit <= 32
 *   digit_bits 1..8 (2^digit_bits buckets per pass)
 *   temp, temp_bytes (device) scratch of at least radix_sort_keys_temp_bytes()
 *   stream    cudaStream_t as void*
 * Every option at its default (see radix_sort_keys_typed for options). */
rs_status radix_sort_keys_u32(const uint32_t* keys_in, uint32_t* keys_out, size_t n,
                              int begin_bit, int end_bit, int digit_bits,
                              void* temp, size_t temp_bytes, void* stream);

/* As radix_sort_keys_u32 for unsigned 64-bit keys; end_bit <= 64. */
rs_status radix_sort_keys_u64(const uint64_t* keys_in, uint64_t* keys_out, size_t n,
                              int begin_bit, int end_bit, int digit_bits,
                              void* temp, size_t temp_bytes, void* stream);

/* Key-value sort: a u32 payload rides with every key move, so equal keys
 * keep their payloads in input order ("100 Days of GPU", day 35, Exercise:
 * carry a second array through the sort).
 *   vals_in   (device) n payloads, read only
 *   vals_out  (device) n payloads, permuted like the keys
 * Other arguments as radix_sort_keys_u32. */
rs_status radix_sort_pairs_u32(const uint32_t* keys_in, uint32_t* keys_out,
                               const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                               int begin_bit, int end_bit, int digit_bits,
                               void* temp, size_t temp_bytes, void* stream);

/* As radix_sort_pairs_u32 with unsigned 64-bit keys. */
rs_status radix_sort_pairs_u64(const uint64_t* keys_in, uint64_t* keys_out,
                               const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                               int begin_bit, int end_bit, int digit_bits,
                               void* temp, size_t temp_bytes, void* stream);

/* Typed keys-only sort: stable sort of signed (two's complement), IEEE
 * float or unsigned keys, ascending or descending.  A radix sort orders bit
 * patterns, which is the wanted order only for unsigned keys ("100 Days of
 * GPU", day 35, Pitfalls: sort signed and float keys through a bijection on
 * the way in).  Keys are ordered by T(k) = k XOR (top bit of k ? neg : pos):
 * signed keys flip the sign bit; float keys set the sign bit of non-negative
 * patterns and complement negative ones; descending complements T.  So
 * -0.0 sorts before +0.0, a NaN with the sign bit clear after +inf and one
 * with it set before -inf (the order of the bit patterns under T), and
 * equal keys keep input order in both directions.  T is applied on the fly;
 * the keys written out are the input bits.
 *   type       an rs_key_type; 4-byte types take 4-byte keys, 8-byte 8-byte
 *   descending 0 or 1
 *   begin_bit, end_bit  the bits of T(k) sorted (all of them: 0 and 8*size)
 *   temp       scratch of radix_sort_keys_temp_bytes() for the key size
 *   opts       (host) options of this call, or NULL for the defaults
 * Other arguments and errors as radix_sort_keys_u32; an unknown type or a
 * descending flag other than 0/1 is RS_ERR_INVALID.  RS_KEY_U32/RS_KEY_U64
 * ascending is the unsigned sort with options. */
rs_status radix_sort_keys_typed(rs_key_type type, int descending, const void* keys_in,
                                void* keys_out, size_t n, int begin_bit, int end_bit,
                                int digit_bits, void* temp, size_t temp_bytes,
                                const rs_options* opts, void* stream);

/* Typed key-value sort: radix_sort_keys_typed with a u32 payload, as
 * radix_sort_pairs_u32. */
rs_status radix_sort_pairs_typed(rs_key_type type, int descending, const void* keys_in,
                                 void* keys_out, const uint32_t* vals_in, uint32_t* vals_out,
                                 size_t n, int begin_bit, int end_bit, int digit_bits,
                                 void* temp, size_t temp_bytes, const rs_options* opts,
                                 void* stream);

/* Scratch size of a row-wise sort of a (rows, cols) 16-bit array. */
rs_status radix_segmented_sort_temp_bytes(int64_t rows, int64_t cols, size_t* bytes);

/* Row-wise stable sort of 16-bit floats along the last dimension, returning
 * the sorted values and their int64 column indices (FlagTree PR #1084: a
 * radix `sort` of fp16/bf16 rows with a descending flag folded into an
 * order-preserving key, two 8-bit passes, compact indices inside and int64
 * on the way out).  Between the passes a row of at most 65,536 columns
 * carries each key and its column in one 32-bit word (key << 16 | column);
 * longer rows, and the pass-skipping and precomputed-offset modes, carry an
 * int32 index array beside 16-bit keys.  The results are the same.
 *   in        (device) rows*cols 16-bit patterns, row-major, contiguous
 *   vals_out  (device) rows*cols patterns: each row sorted
 *   idx_out   (device) rows*cols int64: idx_out[r][j] is the column of in[r]
 *             that landed at position j
 *   rows >= 0, 0 <= cols <= RS_MAX_ROW_KEYS (cols <= RS_MAX_KEYS when
 *             rows == 1); rows*cols == 0 enqueues nothing
 *   kind      RS_F16 or RS_BF16 (both orders come from the sign bit, so the
 *             result does not depend on it; it is validated and recorded)
 *   descending 0 = ascending, 1 = descending.  Ascending order is the order
 *             of the bijection T(u) = sign ? ~u : u | 0x8000: -NaN < -inf <
 *             negatives < -0 < +0 < positives < +inf < +NaN; descending is
 *             the order of ~T(u).  Equal patterns keep input order in both.
 *   temp, temp_bytes (device) scratch of radix_segmented_sort_temp_bytes()
 * Every option at its default. */
rs_status radix_segmented_sort_f16(const uint16_t* in, uint16_t* vals_out, int64_t* idx_out,
                                   int64_t rows, int64_t cols, rs_float_kind kind,
                                   int descending, void* temp, size_t temp_bytes,
                                   void* stream);

/* radix_segmented_sort_f16 with the options of this call (NULL: defaults). */
rs_status radix_segmented_sort_f16_ex(const uint16_t* in, uint16_t* vals_out, int64_t* idx_out,
                                      int64_t rows, int64_t cols, rs_float_kind kind,
                                      int descending, void* temp, size_t temp_bytes,
                                      const rs_options* opts, void* stream);

/* Upfront all-pass digit histograms and their exclusive scans, the first two
 * stages of a sort, exposed on their own (FlagTree PR #1084, section 2:
 * per-pass histograms of shape (passes, 2^b) from one read of the keys;
 * DSA CUDA from First Principles section 13.1: bases are the exclusive
 * prefix sums of the counts).
 *   keys      (device) n keys of key_bytes (4 or 8) bytes
 *   hist_out  (device) passes * 2^digit_bits u32 counts, pass-major
 *   bases_out (device) the same shape: exclusive scan of each pass's counts
 *   temp      (device) scratch of radix_sort_keys_temp_bytes(n, key_bytes, 0, ...) */
rs_status radix_sort_histograms(const void* keys, int key_bytes, size_t n,
                                int begin_bit, int end_bit, int digit_bits,
                                uint32_t* hist_out, uint32_t* bases_out,
                                void* temp, size_t temp_bytes, void* stream);

/* Synchronises `stream` and returns the device-side status of the last sort
 * that used `temp` (RS_OK or RS_ERR_LOOKBACK_TIMEOUT), or RS_ERR_CUDA. */
rs_status radix_sort_device_status(const void* temp, void* stream);

/* Passes run by the last sort enqueued with this scratch buffer (all of
 * them unless RS_OPT_PASS_SKIPPING was given).  Synchronises `stream` and reads the
 * count.
 *   temp    (device) the scratch buffer of that sort
 *   passes  (host) receives the count (0 .. passes of the bit range) */
rs_status radix_sort_passes_run(const void* temp, int* passes, void* stream);

/* 1 when this library is the bounds-checked build (compiled with
 * LSDRS_CHECKED=1: every shared and global index of the scatter, histogram
 * and one-kernel sorts is tested before the access, and a failed test is
 * recorded in the scratch header instead of performed), else 0.  A
 * verification aid standing in for memory checkers; no counterpart on the
 * pages. */
int rs_checked_build(void);

/* Bounds-checked builds: synchronises `stream`, writes the number of failed
 * index tests recorded in `temp` since the last call (*count) and the site
 * code of the first (*first_site, 0 if none), then clears both.  Clear them
 * once before the first sort on a new scratch buffer.  Other builds record
 * nothing, so after a clear the count stays 0.
 *   temp  (device) scratch of a sort (at least 1 KiB) */
rs_status radix_sort_checked_violations(void* temp, void* stream, uint32_t* count,
                                        uint32_t* first_site);

/* Human-readable name of a status code (static storage). */
const char* rs_status_string(rs_status status);

/* Failure-detection check: runs the scatter kernels' bounded look-back wait
 * on a status word that nothing ever sets, with the given limit
 * (0 < timeout_ns <= 60 s).  Writes the status the wait produced
 * (RS_ERR_LOOKBACK_TIMEOUT when it expired) to *result after synchronising
 * `stream`.  word: (device) two u32 scratch words (the status word and an
 * error word), overwritten. */
rs_status rs_lookback_timeout_probe(uint32_t* word, uint64_t timeout_ns, void* stream,
                                    rs_status* result);

/* Bandwidth probe: copies `bytes` from src to dst with 16-byte vector loads
 * and stores on every SM (the "copy, no sort" row of "100 Days of GPU",
 * day 35, Results).  Both pointers (device), 16-byte aligned, bytes % 16 == 0. */
rs_status rs_copy_probe(void* dst, const void* src, size_t bytes, void* stream);

/* Per-kernel timing for measurement.  While enabled, every kernel the
 * library enqueues is bracketed by two CUDA events on its stream.
 * rs_profile_read synchronises on the last event and writes up to `max`
 * records (kernel id, milliseconds, keys processed), oldest first, then
 * clears the log; it returns the number written.  Kernel ids: 0 upfront
 * histogram, 1 scan, 2 onesweep pass, 3 copy probe. */
typedef struct rs_kernel_time {
  int kernel;
  float ms;
  uint64_t units;
} rs_kernel_time;
rs_status rs_profile_enable(int enable);
int rs_profile_read(rs_kernel_time* out, int max);

/* Number of kernels the library enqueued since the last call (a launch
 * count for measurement); resets the counter. */
uint64_t rs_launch_count_reset(void);

/* Key-value sort for callers that cannot allocate device memory where they
 * sort (the pages have no counterpart of this entry point): callers whose
 * device memory belongs to a pool they may not grow, or plugins and
 * callbacks handed only the buffers they work on, with no allocator of their
 * own.  Same result and arguments as radix_sort_pairs_u32 without
 * temp/temp_bytes, with every option at its default: the scratch is a fixed
 * 4 MiB array inside the library's device code, which every GPU that loads
 * the library holds until the process exits.  No call allocates or frees
 * anything.
 *   n         0 <= n <= 262,144 (2^18); larger n returns RS_ERR_INVALID
 *             before anything is enqueued
 * The first call on a device looks up that device's address of the array
 * (make that first call, or a call of radix_sort_pairs_u32_noalloc_status,
 * before any stream capture on the device).  The address is kept for the
 * life of the process: a process that resets a device (cudaDeviceReset) must
 * not call these two entry points on it afterwards.  Every call on a device
 * shares the one array and it keeps the last call's contents; each call
 * clears what must start at zero.  Calls whose work overlaps on the GPU (for
 * example on two streams) race and give wrong results; calls on one stream
 * are safe. */
rs_status radix_sort_pairs_u32_noalloc(const uint32_t* keys_in, uint32_t* keys_out,
                                       const uint32_t* vals_in, uint32_t* vals_out, size_t n,
                                       int begin_bit, int end_bit, int digit_bits,
                                       void* stream);

/* Synchronises `stream` and returns the device-side status of the last
 * radix_sort_pairs_u32_noalloc enqueued on the current device (RS_OK or
 * RS_ERR_LOOKBACK_TIMEOUT), or RS_ERR_CUDA: the radix_sort_device_status of
 * that entry point, whose scratch the caller cannot name.  Allocates
 * nothing. */
rs_status radix_sort_pairs_u32_noalloc_status(void* stream);

/* Verification of the status path above (no sort): runs the look-back's
 * bounded wait on a word of the no-allocation array that nothing sets, with
 * the given limit (1 ns .. 60 s), so that it records RS_ERR_LOOKBACK_TIMEOUT
 * in the array's device-side status word, exactly where a timed-out sort of
 * radix_sort_pairs_u32_noalloc records it; the next such sort clears it.
 * Synchronises `stream`; writes the probe's own reading of the word to
 * *result.  Allocates nothing. */
rs_status rs_noalloc_timeout_probe(uint64_t timeout_ns, void* stream, rs_status* result);

#ifdef __cplusplus
}
#endif

#endif /* LSDRS_H */
