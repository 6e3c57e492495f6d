// Onesweep instantiation for 16-bit float rows: 8-bit digits of the
// order-preserving key, column-index payload.
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_f16(const SweepArgs& a, int* launched, cudaStream_t s) {
  return launch_sweep_t<KeyF16Bits, 8, kValIdx, kShapeF16Idx.threads, kShapeF16Idx.items, kShapeF16Idx.min_blocks, kShapeF16Idx.window>(a, launched, s);
}

}  // namespace lsdrs
