// Onesweep instantiations for unsigned 64-bit keys with 64-bit look-back words: flat sorts
// of 2^30 keys or more (keys only and u32 pairs), with the tile shapes of the
// 32-bit-word kernels.
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_u64_wide(ValKind v, int bits, const SweepArgs& a, int* launched,
                                  cudaStream_t s) {
  if (v == kValNone)
    return launch_sweep_bits<KeyU64, kValNone, kShapeU64Keys.threads, kShapeU64Keys.items, kShapeU64Keys.min_blocks,
                             kShapeU64Keys.window, true>(bits, a, launched, s);
  if (v == kValU32)
    return launch_sweep_bits<KeyU64, kValU32, kShapeU64Pairs.threads, kShapeU64Pairs.items, kShapeU64Pairs.min_blocks,
                             kShapeU64Pairs.window, true>(bits, a, launched, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
