// Onesweep instantiations for unsigned 32-bit keys (keys only, u32 pairs).
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_u32(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s) {
  if (mid_tiles(kKeyU32, v, a.rows, a.cols)) return launch_sweep_u32_mid(v, bits, a, launched, s);
  if (v == kValNone)
    return launch_sweep_bits<KeyU32, kValNone, kShapeU32Keys.threads, kShapeU32Keys.items, kShapeU32Keys.min_blocks, kShapeU32Keys.window>(bits, a, launched, s);
  if (v == kValU32)
    return launch_sweep_bits<KeyU32, kValU32, kShapeU32Pairs.threads, kShapeU32Pairs.items, kShapeU32Pairs.min_blocks, kShapeU32Pairs.window>(bits, a, launched, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
