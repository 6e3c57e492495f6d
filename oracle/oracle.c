/*
 * ORACLE -- test infrastructure, not product code.
 *
 * A plain, slow, single-threaded CPU statement of what LSD radix sort
 * computes.  Only the test suite, the smoke check and the CPU-baseline leg
 * of the benchmark may load this file's library; the CUDA path shares no
 * code, header, table or helper with it.
 *
 * Every sort here is built from the three loops of one counting-sort pass
 * (CUDA Handbook ch. 16 "Radix Sort", Listing 16-8):
 *   1. histogram  : counts[d] += 1 for the digit d of every key;
 *   2. scan       : counts -> exclusive prefix sums (the digit's base offset;
 *                   DSA CUDA from First Principles ch. 13, section 13.1,
 *                   "COMMON TRAP": exclusive, not inclusive);
 *   3. scatter    : walk the input in order, place each key at its digit's
 *                   running offset and advance it (section 13.2: the forward
 *                   walk is what makes the pass stable).
 * The driver applies one pass per digit, least significant digit first,
 * ping-ponging between two buffers (Listing 16-9; section 13.3).
 *
 * The three loops are written once, over an array of precomputed digits, so
 * that the base-10 worked example of section 13.1/13.2/13.3 runs through the
 * very same code as the bit-field sorts.
 *
 * Readings of the pages taken here (each also listed in the design notes):
 *  - Listing 16-9 advances the digit window by one bit; the text sorts one
 *    digit at a time, so the window advances by the digit width b.
 *  - The pass count comes from the requested bit range [begin_bit, end_bit):
 *    ceil((end_bit - begin_bit) / b) passes; the last digit may be narrower.
 *  - Bits outside [begin_bit, end_bit) take no part in the ordering but are
 *    carried in the output keys.
 *  - 16-bit floats (fp16 and bf16 share the layout sign|exponent|mantissa)
 *    are sorted through the bijection T(u) = (u & 0x8000) ? ~u : u | 0x8000,
 *    whose unsigned order is the float order (100 Days of GPU, day 35,
 *    "Pitfalls": a bijection on the way in); descending order sorts ~T(u)
 *    ascending, so ties keep input order in both directions.
 *  - Typed 32/64-bit keys follow the same plain reading of that passage:
 *    two's-complement keys flip the sign bit; IEEE floats complement
 *    negative patterns and set the sign bit of non-negative ones (the
 *    16-bit rule at full width); descending complements the result.  -0.0
 *    and +0.0, and NaNs of either sign, are ordered by their patterns under
 *    that map (the page gives no other rule).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_OK 0
#define OR_ERR_INVALID 1
#define OR_ERR_NOMEM 2

/* ---- the three loops of one counting-sort pass, over a digit array ---- */

/* 1. Histogram (Listing 16-8 step 1; section 13.1 count[]). */
void or_histogram(const uint32_t *digit, size_t n, uint32_t radix,
                  uint64_t *counts) {
  for (uint32_t d = 0; d < radix; d++) counts[d] = 0;
  for (size_t i = 0; i < n; i++) counts[digit[i]] += 1;
}

/* 2. Exclusive scan: offsets[d] = sum of counts[e] for e < d
 *    (Listing 16-8 step 2; section 13.1 offset[]). */
void or_exclusive_scan(const uint64_t *counts, uint32_t radix,
                       uint64_t *offsets) {
  uint64_t sum = 0;
  for (uint32_t d = 0; d < radix; d++) {
    uint64_t c = counts[d];
    offsets[d] = sum;
    sum += c;
  }
}

/* 3. Stable destinations: walk the input in order; element i goes to its
 *    digit's running offset, which then advances (Listing 16-8 step 3;
 *    section 13.2 "pos[d]++" walk).  Returns OR_ERR_NOMEM, with dest left
 *    unwritten, when its working array cannot be allocated. */
int or_stable_destinations(const uint32_t *digit, size_t n, uint32_t radix,
                           const uint64_t *offsets, uint64_t *dest) {
  uint64_t *pos = (uint64_t *)malloc(sizeof(uint64_t) * radix);
  if (!pos) return OR_ERR_NOMEM;
  for (uint32_t d = 0; d < radix; d++) pos[d] = offsets[d];
  for (size_t i = 0; i < n; i++) {
    uint32_t d = digit[i];
    dest[i] = pos[d];
    pos[d] += 1;
  }
  free(pos);
  return OR_OK;
}

/* One whole pass on a digit array: dest[i] is where element i lands. */
int or_counting_pass(const uint32_t *digit, size_t n, uint32_t radix,
                     uint64_t *counts, uint64_t *offsets, uint64_t *dest) {
  if (radix == 0) return OR_ERR_INVALID;
  for (size_t i = 0; i < n; i++)
    if (digit[i] >= radix) return OR_ERR_INVALID;
  or_histogram(digit, n, radix, counts);
  or_exclusive_scan(counts, radix, offsets);
  return or_stable_destinations(digit, n, radix, offsets, dest);
}

/* ---- bit-field LSD sorts (Listing 16-9 driver with the readings above) ---- */

static int check_range(int key_bits, int begin_bit, int end_bit, int b) {
  if (begin_bit < 0 || end_bit > key_bits || begin_bit >= end_bit) return 0;
  if (b < 1 || b > 16) return 0;
  return 1;
}

/* Number of passes for bits [begin_bit, end_bit) at digit width b. */
int or_num_passes(int begin_bit, int end_bit, int b) {
  if (b < 1 || end_bit <= begin_bit) return 0;
  return (end_bit - begin_bit + b - 1) / b;
}

/* Digit width of pass p: b, except a narrower last digit. */
static int pass_width(int begin_bit, int end_bit, int b, int p) {
  int shift = begin_bit + p * b;
  int w = end_bit - shift;
  return w < b ? w : b;
}

/* The sort for one key width.  Keys are widened to 64 bits only inside the
 * digit extraction; moves copy the caller's element type. */
#define OR_DEFINE_SORT(NAME, KEY_T, KEY_BITS)                                  \
  int NAME(const KEY_T *keys_in, KEY_T *keys_out, const uint32_t *vals_in,     \
           uint32_t *vals_out, size_t n, int begin_bit, int end_bit, int b) {  \
    if (!check_range(KEY_BITS, begin_bit, end_bit, b)) return OR_ERR_INVALID;  \
    if (n == 0) return OR_OK;                                                  \
    int passes = or_num_passes(begin_bit, end_bit, b);                         \
    uint32_t radix = 1u << b;                                                  \
    KEY_T *kbuf[2];                                                            \
    uint32_t *vbuf[2] = {0, 0};                                                \
    kbuf[0] = (KEY_T *)malloc(sizeof(KEY_T) * n);                              \
    kbuf[1] = (KEY_T *)malloc(sizeof(KEY_T) * n);                              \
    if (vals_in) {                                                             \
      vbuf[0] = (uint32_t *)malloc(sizeof(uint32_t) * n);                      \
      vbuf[1] = (uint32_t *)malloc(sizeof(uint32_t) * n);                      \
    }                                                                          \
    uint32_t *digit = (uint32_t *)malloc(sizeof(uint32_t) * n);                \
    uint64_t *dest = (uint64_t *)malloc(sizeof(uint64_t) * n);                 \
    uint64_t *counts = (uint64_t *)malloc(sizeof(uint64_t) * radix);           \
    uint64_t *offsets = (uint64_t *)malloc(sizeof(uint64_t) * radix);          \
    int rc = OR_OK;                                                            \
    if (!kbuf[0] || !kbuf[1] || !digit || !dest || !counts || !offsets ||      \
        (vals_in && (!vbuf[0] || !vbuf[1]))) {                                 \
      rc = OR_ERR_NOMEM;                                                       \
      goto done;                                                               \
    }                                                                          \
    memcpy(kbuf[0], keys_in, sizeof(KEY_T) * n);                               \
    if (vals_in) memcpy(vbuf[0], vals_in, sizeof(uint32_t) * n);               \
    int cur = 0; /* buffer holding the current order */                        \
    for (int p = 0; p < passes; p++) {                                         \
      int shift = begin_bit + p * b;                                           \
      int w = pass_width(begin_bit, end_bit, b, p);                            \
      uint64_t mask = (w >= 64) ? ~0ull : ((1ull << w) - 1ull);                \
      const KEY_T *src = kbuf[cur];                                            \
      KEY_T *dst = kbuf[1 - cur];                                              \
      for (size_t i = 0; i < n; i++)                                           \
        digit[i] = (uint32_t)((((uint64_t)src[i]) >> shift) & mask);           \
      rc = or_counting_pass(digit, n, radix, counts, offsets, dest);           \
      if (rc != OR_OK) goto done;                                              \
      for (size_t i = 0; i < n; i++) dst[dest[i]] = src[i];                    \
      if (vals_in) {                                                           \
        const uint32_t *vs = vbuf[cur];                                        \
        uint32_t *vd = vbuf[1 - cur];                                          \
        for (size_t i = 0; i < n; i++) vd[dest[i]] = vs[i];                    \
      }                                                                        \
      cur = 1 - cur; /* ping-pong, Listing 16-9 */                             \
    }                                                                          \
    memcpy(keys_out, kbuf[cur], sizeof(KEY_T) * n);                            \
    if (vals_in && vals_out) memcpy(vals_out, vbuf[cur], sizeof(uint32_t) * n);\
  done:                                                                        \
    free(kbuf[0]); free(kbuf[1]); free(vbuf[0]); free(vbuf[1]);                \
    free(digit); free(dest); free(counts); free(offsets);                      \
    return rc;                                                                 \
  }

OR_DEFINE_SORT(or_sort_u32, uint32_t, 32)
OR_DEFINE_SORT(or_sort_u64, uint64_t, 64)

/* Digit histograms of every pass from the unsorted keys:
 * hist[p * 2^b + d] = #{i : digit_p(key_i) == d}.  A pass only reorders the
 * keys, so the histogram of pass p's digit is the same before and after the
 * earlier passes; this is what an upfront all-pass histogram computes. */
#define OR_DEFINE_PASS_HIST(NAME, KEY_T, KEY_BITS)                             \
  int NAME(const KEY_T *keys, size_t n, int begin_bit, int end_bit, int b,     \
           uint64_t *hist) {                                                   \
    if (!check_range(KEY_BITS, begin_bit, end_bit, b)) return OR_ERR_INVALID;  \
    int passes = or_num_passes(begin_bit, end_bit, b);                         \
    uint32_t radix = 1u << b;                                                  \
    uint32_t *digit = (uint32_t *)malloc(sizeof(uint32_t) * (n ? n : 1));      \
    if (!digit) return OR_ERR_NOMEM;                                           \
    for (int p = 0; p < passes; p++) {                                         \
      int shift = begin_bit + p * b;                                           \
      int w = pass_width(begin_bit, end_bit, b, p);                            \
      uint64_t mask = (w >= 64) ? ~0ull : ((1ull << w) - 1ull);                \
      for (size_t i = 0; i < n; i++)                                           \
        digit[i] = (uint32_t)((((uint64_t)keys[i]) >> shift) & mask);          \
      or_histogram(digit, n, radix, hist + (size_t)p * radix);                 \
    }                                                                          \
    free(digit);                                                               \
    return OR_OK;                                                              \
  }

OR_DEFINE_PASS_HIST(or_pass_histograms_u32, uint32_t, 32)
OR_DEFINE_PASS_HIST(or_pass_histograms_u64, uint64_t, 64)

/* ---- 16-bit floats: order-preserving bijection and row-wise sort ---- */

/* T(u): negative patterns (sign set) are complemented so that larger
 * magnitudes come first; non-negative patterns get the sign bit set so that
 * they follow every negative one.  Descending complements the result. */
uint16_t or_order_key16(uint16_t u, int descending) {
  uint16_t t = (u & 0x8000u) ? (uint16_t)(~u) : (uint16_t)(u | 0x8000u);
  return descending ? (uint16_t)(~t) : t;
}

/* Row-wise sort of a row-major (rows, cols) array of 16-bit float patterns
 * (fp16 or bf16: the bijection only reads the sign bit).  Each row is an
 * independent LSD sort of T(x) with 8-bit digits (two passes), carrying the
 * original bit pattern and the int64 column index (the FlagTree PR #1084
 * sort returns values and int64 indices along the last dimension). */
int or_segmented_sort16(const uint16_t *in, uint16_t *vals_out,
                        int64_t *idx_out, int64_t rows, int64_t cols,
                        int descending) {
  if (rows < 0 || cols < 0) return OR_ERR_INVALID;
  if (rows == 0 || cols == 0) return OR_OK;
  size_t n = (size_t)cols;
  const uint32_t radix = 256;
  uint16_t *kb[2], *vb[2];
  int64_t *ib[2];
  kb[0] = (uint16_t *)malloc(2 * n); kb[1] = (uint16_t *)malloc(2 * n);
  vb[0] = (uint16_t *)malloc(2 * n); vb[1] = (uint16_t *)malloc(2 * n);
  ib[0] = (int64_t *)malloc(8 * n);  ib[1] = (int64_t *)malloc(8 * n);
  uint32_t *digit = (uint32_t *)malloc(4 * n);
  uint64_t *dest = (uint64_t *)malloc(8 * n);
  uint64_t counts[256], offsets[256];
  int rc = OR_OK;
  if (!kb[0] || !kb[1] || !vb[0] || !vb[1] || !ib[0] || !ib[1] || !digit ||
      !dest) {
    rc = OR_ERR_NOMEM;
    goto done;
  }
  for (int64_t r = 0; r < rows; r++) {
    const uint16_t *row = in + (size_t)r * n;
    for (size_t i = 0; i < n; i++) {
      kb[0][i] = or_order_key16(row[i], descending);
      vb[0][i] = row[i];
      ib[0][i] = (int64_t)i;
    }
    int cur = 0;
    for (int p = 0; p < 2; p++) {
      int shift = 8 * p;
      for (size_t i = 0; i < n; i++) digit[i] = (kb[cur][i] >> shift) & 0xFFu;
      rc = or_counting_pass(digit, n, radix, counts, offsets, dest);
      if (rc != OR_OK) goto done;
      for (size_t i = 0; i < n; i++) {
        kb[1 - cur][dest[i]] = kb[cur][i];
        vb[1 - cur][dest[i]] = vb[cur][i];
        ib[1 - cur][dest[i]] = ib[cur][i];
      }
      cur = 1 - cur;
    }
    memcpy(vals_out + (size_t)r * n, vb[cur], 2 * n);
    memcpy(idx_out + (size_t)r * n, ib[cur], 8 * n);
  }
done:
  free(kb[0]); free(kb[1]); free(vb[0]); free(vb[1]);
  free(ib[0]); free(ib[1]); free(digit); free(dest);
  return rc;
}

/* Per-row digit histograms of both 8-bit passes of T(x):
 * hist[(r * 2 + p) * 256 + d]. */
int or_segmented_histograms16(const uint16_t *in, int64_t rows, int64_t cols,
                              int descending, uint64_t *hist) {
  if (rows < 0 || cols < 0) return OR_ERR_INVALID;
  size_t n = (size_t)cols;
  uint32_t *digit = (uint32_t *)malloc(4 * (n ? n : 1));
  if (!digit) return OR_ERR_NOMEM;
  for (int64_t r = 0; r < rows; r++) {
    const uint16_t *row = in + (size_t)r * n;
    for (int p = 0; p < 2; p++) {
      for (size_t i = 0; i < n; i++)
        digit[i] = (or_order_key16(row[i], descending) >> (8 * p)) & 0xFFu;
      or_histogram(digit, n, 256, hist + ((size_t)r * 2 + p) * 256);
    }
  }
  free(digit);
  return OR_OK;
}

/* ---- typed 32/64-bit keys: bijection to unsigned order, then the sort ---- */

enum { OR_UNSIGNED = 0, OR_SIGNED = 1, OR_FLOAT = 2 };

/* T(k) for a key of `type`: unsigned keys are their own order; signed keys
 * flip the sign bit (two's complement order -> unsigned order); floats
 * complement negative patterns (larger magnitudes first) and set the sign
 * bit of the others.  Descending complements T. */
uint32_t or_order_key32(uint32_t k, int type, int descending) {
  const uint32_t sign = 0x80000000u;
  uint32_t t = k;
  if (type == OR_SIGNED) t = k ^ sign;
  if (type == OR_FLOAT) t = (k & sign) ? ~k : (k | sign);
  return descending ? ~t : t;
}

uint64_t or_order_key64(uint64_t k, int type, int descending) {
  const uint64_t sign = 0x8000000000000000ull;
  uint64_t t = k;
  if (type == OR_SIGNED) t = k ^ sign;
  if (type == OR_FLOAT) t = (k & sign) ? ~k : (k | sign);
  return descending ? ~t : t;
}

/* Stable sort of typed keys on bits [begin_bit, end_bit) of T(k): sort T(k)
 * with each key's input position as payload, then gather the original keys
 * (and payloads) in that order. */
#define OR_DEFINE_TYPED(NAME, KEY_T, ORDER, SORT)                              \
  int NAME(const KEY_T *keys_in, KEY_T *keys_out, const uint32_t *vals_in,     \
           uint32_t *vals_out, size_t n, int type, int descending,             \
           int begin_bit, int end_bit, int b) {                                \
    if (type < OR_UNSIGNED || type > OR_FLOAT) return OR_ERR_INVALID;          \
    if (descending != 0 && descending != 1) return OR_ERR_INVALID;             \
    if (n == 0) return SORT(keys_in, keys_out, NULL, NULL, 0, begin_bit,       \
                            end_bit, b);                                       \
    KEY_T *t = (KEY_T *)malloc(sizeof(KEY_T) * n);                             \
    KEY_T *ts = (KEY_T *)malloc(sizeof(KEY_T) * n);                            \
    uint32_t *pos = (uint32_t *)malloc(4 * n);                                 \
    uint32_t *order = (uint32_t *)malloc(4 * n);                               \
    int rc = OR_ERR_NOMEM;                                                     \
    if (t && ts && pos && order) {                                             \
      for (size_t i = 0; i < n; i++) {                                         \
        t[i] = ORDER(keys_in[i], type, descending);                            \
        pos[i] = (uint32_t)i;                                                  \
      }                                                                        \
      rc = SORT(t, ts, pos, order, n, begin_bit, end_bit, b);                  \
      if (rc == OR_OK) {                                                       \
        for (size_t i = 0; i < n; i++) {                                       \
          keys_out[i] = keys_in[order[i]];                                     \
          if (vals_in) vals_out[i] = vals_in[order[i]];                        \
        }                                                                      \
      }                                                                        \
    }                                                                          \
    free(t); free(ts); free(pos); free(order);                                 \
    return rc;                                                                 \
  }

OR_DEFINE_TYPED(or_sort_typed32, uint32_t, or_order_key32, or_sort_u32)
OR_DEFINE_TYPED(or_sort_typed64, uint64_t, or_order_key64, or_sort_u64)
