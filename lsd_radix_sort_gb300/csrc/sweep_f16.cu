// Onesweep instantiations for 16-bit float rows: 8-bit digits of the
// order-preserving key, with the column index as a payload array, or (rows
// of at most 65,536 columns) packed with the key into one 32-bit word.
#include "onesweep.cuh"

namespace lsdrs {

cudaError_t launch_sweep_f16(const SweepArgs& a, int* launched, cudaStream_t s) {
  if (a.packed) {  // rows of at most 65,536 columns: key and column in one word
    constexpr SweepShape P = kShapeF16Packed;
    return launch_sweep_t<KeyF16Packed, 8, kValPack16, P.threads, P.items, P.min_blocks,
                          P.window>(a, launched, s);
  }
  constexpr SweepShape S = kShapeF16Idx;
  if (a.offsets != nullptr)
    return launch_sweep_t<KeyF16Bits, 8, kValIdx, S.threads, S.items, S.min_blocks, S.window,
                          true>(a, launched, s);
  return launch_sweep_t<KeyF16Bits, 8, kValIdx, S.threads, S.items, S.min_blocks, S.window>(
      a, launched, s);
}

}  // namespace lsdrs
