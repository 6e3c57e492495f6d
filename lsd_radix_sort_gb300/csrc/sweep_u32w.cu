// Onesweep instantiations for unsigned 32-bit keys with 64-bit look-back words: flat sorts
// of 2^30 keys or more (keys only and u32 pairs), with the tile shapes of the
// 32-bit-word kernels.
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_u32_wide(ValKind v, int bits, const SweepArgs& a, int* launched,
                                  cudaStream_t s) {
  if (v == kValNone)
    return launch_sweep_bits<KeyU32, kValNone, kShapeU32Keys.threads, kShapeU32Keys.items, kShapeU32Keys.min_blocks,
                             kShapeU32Keys.window, true>(bits, a, launched, s);
  if (v == kValU32)
    return launch_sweep_bits<KeyU32, kValU32, kShapeU32Pairs.threads, kShapeU32Pairs.items, kShapeU32Pairs.min_blocks,
                             kShapeU32Pairs.window, true>(bits, a, launched, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
