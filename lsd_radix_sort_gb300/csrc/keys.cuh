// Key encodings: how a stored key becomes the unsigned integer whose b-bit
// digits are sorted.
//
// A radix sort orders bit patterns, which is the wanted order only for
// unsigned integers ("100 Days of GPU", day 35, Pitfalls: negatives come
// after positives and negative floats come out backwards; the fix is a
// bijection on the way in).  The bijection used here is
//     T(k) = k XOR (top bit of k set ? neg : pos)
// with two constants per key type (width w, sign bit s = 1 << (w-1)):
//     unsigned        pos = neg = 0
//     two's-complement pos = neg = s          (flip the sign bit)
//     IEEE float      pos = s, neg = all ones (non-negative: set the sign
//                                              bit; negative: complement)
// and descending order complements T (pos and neg complemented), so that
// equal patterns still keep input order.  fp16 and bf16 share the float
// layout (FlagTree PR #1084 folds the descending flag into the key
// conversion of every load).  encode() gives T(k) whole.  The scatter
// passes of signed, float or descending 32/64-bit keys apply T once, when
// the first pass run loads a key, carry T(k) through the ping-pong buffers
// and invert it when the last pass run writes the key out ("100 Days of
// GPU", day 35: a bijection on the way in, its inverse on the way out):
// `Stored` names the encoding whose digits those passes take from T(k), and
// decode() is the inverse.  Every other key type is carried as stored
// (`Stored` is the type itself) and T is applied at each digit extraction.
// The upfront histogram always reads the caller's keys and applies T.
#pragma once
#include <cstdint>

#include "kernels.h"

namespace lsdrs {

// digit_byte(k, sel, hi, xf): the digit when it is one whole byte of T(k)
// (8-bit digits starting at a multiple of 8): byte (sel & 3) of the high
// (hi) or low 32-bit word of T(k), by one byte permute; sel is
// 0x4440 | byte index, so the upper three bytes of the result are zero.

// Unsigned 32-bit keys in ascending order: T is the identity.
struct KeyU32 {
  using T = uint32_t;
  using Stored = KeyU32;
  static constexpr int kBits = 32;
  __device__ __forceinline__ static uint32_t encode(T k, const KeyXform&) { return k; }
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   const KeyXform&) {
    return (k >> shift) & mask;
  }
  __device__ __forceinline__ static uint32_t digit_byte(T k, uint32_t sel, bool,
                                                        const KeyXform&) {
    return __byte_perm(k, 0u, sel);
  }
};

// Any other 32-bit key: signed or float, or descending.
struct KeyX32 {
  using T = uint32_t;
  using Stored = KeyU32;  // the scatter passes carry T(k)
  static constexpr int kBits = 32;
  __device__ __forceinline__ static uint32_t encode(T k, const KeyXform& x) {
    return k ^ (static_cast<int32_t>(k) < 0 ? static_cast<uint32_t>(x.neg)
                                            : static_cast<uint32_t>(x.pos));
  }
  // The inverse of T: pos and neg have the same top bit for every key type
  // and direction, so the top bit of T(k) ^ pos is the top bit of k.
  __device__ __forceinline__ static uint32_t decode(uint32_t t, const KeyXform& x) {
    return t ^ (static_cast<int32_t>(t ^ static_cast<uint32_t>(x.pos)) < 0
                    ? static_cast<uint32_t>(x.neg)
                    : static_cast<uint32_t>(x.pos));
  }
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   const KeyXform& x) {
    const uint32_t t = k ^ (static_cast<int32_t>(k) < 0 ? static_cast<uint32_t>(x.neg)
                                                        : static_cast<uint32_t>(x.pos));
    return (t >> shift) & mask;
  }
  __device__ __forceinline__ static uint32_t digit_byte(T k, uint32_t sel, bool,
                                                        const KeyXform& x) {
    return __byte_perm(encode(k, x), 0u, sel);
  }
};

struct KeyU64 {
  using T = uint64_t;
  using Stored = KeyU64;
  static constexpr int kBits = 64;
  __device__ __forceinline__ static uint64_t encode(T k, const KeyXform&) { return k; }
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   const KeyXform&) {
    return static_cast<uint32_t>(k >> shift) & mask;
  }
  __device__ __forceinline__ static uint32_t digit_byte(T k, uint32_t sel, bool hi,
                                                        const KeyXform&) {
    return __byte_perm(hi ? static_cast<uint32_t>(k >> 32) : static_cast<uint32_t>(k), 0u, sel);
  }
};

struct KeyX64 {
  using T = uint64_t;
  using Stored = KeyU64;  // the scatter passes carry T(k)
  static constexpr int kBits = 64;
  __device__ __forceinline__ static uint64_t encode(T k, const KeyXform& x) {
    return k ^ (static_cast<int64_t>(k) < 0 ? x.neg : x.pos);
  }
  // The inverse of T (see KeyX32::decode).
  __device__ __forceinline__ static uint64_t decode(uint64_t t, const KeyXform& x) {
    return t ^ (static_cast<int64_t>(t ^ x.pos) < 0 ? x.neg : x.pos);
  }
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   const KeyXform& x) {
    const uint64_t t = k ^ (static_cast<int64_t>(k) < 0 ? x.neg : x.pos);
    return static_cast<uint32_t>(t >> shift) & mask;
  }
  __device__ __forceinline__ static uint32_t digit_byte(T k, uint32_t sel, bool hi,
                                                        const KeyXform& x) {
    const uint64_t t = encode(k, x);
    return __byte_perm(hi ? static_cast<uint32_t>(t >> 32) : static_cast<uint32_t>(t), 0u, sel);
  }
};

// 16-bit float keys (fp16 / bf16 bit patterns).
struct KeyF16Bits {
  using T = uint16_t;
  using Stored = KeyF16Bits;
  static constexpr int kBits = 16;
  // T(k) in the low 16 bits (the bits above are not part of the key)
  __device__ __forceinline__ static uint32_t encode(T k, const KeyXform& x) {
    const uint32_t u = k;
    return u ^ ((u & 0x8000u) ? static_cast<uint32_t>(x.neg) : static_cast<uint32_t>(x.pos));
  }
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   const KeyXform& x) {
    const uint32_t u = k;
    const uint32_t t = u ^ ((u & 0x8000u) ? static_cast<uint32_t>(x.neg)
                                          : static_cast<uint32_t>(x.pos));
    return (t >> shift) & mask;
  }
  __device__ __forceinline__ static uint32_t digit_byte(T k, uint32_t sel, bool,
                                                        const KeyXform& x) {
    return __byte_perm(encode(k, x), 0u, sel);
  }
};

// A 16-bit float key packed with its 16-bit column index into one word,
// (T(bits) << 16) | column: the form a row of at most 65,536 columns takes
// between the two passes of a row-wise sort, so that each pass moves and
// stages one 32-bit word per key.  The order-preserving transform is applied
// once, when the word is made (pack), and undone once, when the last pass
// writes the value out (bits): a digit is then one byte permute.
struct KeyF16Packed {
  using T = uint32_t;
  using Stored = KeyF16Packed;
  static constexpr int kBits = 16;
  __device__ __forceinline__ static uint32_t pack(uint16_t bits, uint32_t col,
                                                  const KeyXform& x) {
    return (KeyF16Bits::encode(bits, x) << 16) | col;
  }
  // The 16-bit pattern of the word's key: T is u ^ pos for u >= 0 and
  // u ^ neg for u < 0, and the sign bit of T(u) ^ pos is set exactly for the
  // latter, so the key's sign is read back from T.
  __device__ __forceinline__ static uint16_t bits(T w, const KeyXform& x) {
    const uint32_t t = w >> 16;
    const uint32_t pos = static_cast<uint32_t>(x.pos), neg = static_cast<uint32_t>(x.neg);
    return static_cast<uint16_t>(t ^ (((t ^ pos) & 0x8000u) ? neg : pos));
  }
  __device__ __forceinline__ static uint32_t encode(T w, const KeyXform&) { return w >> 16; }
  __device__ __forceinline__ static uint32_t digit(T w, int shift, uint32_t mask,
                                                   const KeyXform&) {
    return (w >> (16 + shift)) & mask;
  }
  // sel selects byte b (0 or 1) of T: bytes 2 and 3 of the word
  __device__ __forceinline__ static uint32_t digit_byte(T w, uint32_t sel, bool,
                                                        const KeyXform&) {
    return __byte_perm(w, 0u, sel + 2u);
  }
};

}  // namespace lsdrs
