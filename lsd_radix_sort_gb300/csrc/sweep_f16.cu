// Onesweep instantiation for 16-bit float rows: 8-bit digits of the
// order-preserving key, column-index payload.
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_f16(const SweepArgs& a, int* launched, cudaStream_t s) {
  constexpr SweepShape S = kShapeF16Idx;
  if (a.offsets != nullptr)
    return launch_sweep_t<KeyF16Bits, 8, kValIdx, S.threads, S.items, S.min_blocks, S.window,
                          true>(a, launched, s);
  return launch_sweep_t<KeyF16Bits, 8, kValIdx, S.threads, S.items, S.min_blocks, S.window>(
      a, launched, s);
}

}  // namespace lsdrs
