// Onesweep instantiations for flat sorts of at most kMidMaxKeys unsigned
// 32-bit keys (keys only, u32 pairs): the smaller tiles of the mid-size shapes.
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_u32_mid(ValKind v, int bits, const SweepArgs& a, int* launched,
                                 cudaStream_t s) {
  if (v == kValNone)
    return launch_sweep_bits<KeyU32, kValNone, kShapeU32KeysMid.threads, kShapeU32KeysMid.items,
                             kShapeU32KeysMid.min_blocks, kShapeU32KeysMid.window>(bits, a,
                                                                                  launched, s);
  if (v == kValU32)
    return launch_sweep_bits<KeyU32, kValU32, kShapeU32PairsMid.threads,
                             kShapeU32PairsMid.items, kShapeU32PairsMid.min_blocks,
                             kShapeU32PairsMid.window>(bits, a, launched, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
