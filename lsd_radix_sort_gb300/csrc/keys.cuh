// Key encodings: how a stored key becomes the unsigned integer whose b-bit
// digits are sorted.
//
// Unsigned integers are their own sort key.  16-bit floats (fp16 and bf16
// share the layout sign|exponent|mantissa) use an order-preserving bijection:
// a negative pattern is complemented (larger magnitude first), a
// non-negative one gets its sign bit set (after every negative).  Descending
// order complements that key, so equal patterns still keep input order.
// ("100 Days of GPU", day 35, Pitfalls: sort floats through a bijection on
// the way in; FlagTree PR #1084 folds the descending flag into the key
// conversion of every load.)  The stored bits are carried unchanged, so no
// inverse transform is needed on the way out.
#pragma once
#include <cstdint>

namespace lsdrs {

struct KeyU32 {
  using T = uint32_t;
  static constexpr int kBits = 32;
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   uint32_t /*flip*/) {
    return (k >> shift) & mask;
  }
};

struct KeyU64 {
  using T = uint64_t;
  static constexpr int kBits = 64;
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   uint32_t /*flip*/) {
    return static_cast<uint32_t>(k >> shift) & mask;
  }
};

// 16-bit float patterns; flip = 0xFFFF for descending, 0 for ascending.
struct KeyF16Bits {
  using T = uint16_t;
  static constexpr int kBits = 16;
  __device__ __forceinline__ static uint32_t order_key(T u, uint32_t flip) {
    uint32_t x = u;
    uint32_t t = (x & 0x8000u) ? (~x & 0xFFFFu) : (x | 0x8000u);
    return t ^ flip;
  }
  __device__ __forceinline__ static uint32_t digit(T k, int shift, uint32_t mask,
                                                   uint32_t flip) {
    return (order_key(k, flip) >> shift) & mask;
  }
};

}  // namespace lsdrs
