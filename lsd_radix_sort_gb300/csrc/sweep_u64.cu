// Onesweep instantiations for unsigned 64-bit keys (keys only, u32 pairs).
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_u64(ValKind v, int bits, const SweepArgs& a, int* launched,
                             cudaStream_t s) {
  if (v == kValNone)
    return launch_sweep_bits<KeyU64, kValNone, kShapeU64Keys.threads, kShapeU64Keys.items, kShapeU64Keys.min_blocks, kShapeU64Keys.window>(bits, a, launched, s);
  if (v == kValU32)
    return launch_sweep_bits<KeyU64, kValU32, kShapeU64Pairs.threads, kShapeU64Pairs.items, kShapeU64Pairs.min_blocks, kShapeU64Pairs.window>(bits, a, launched, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
