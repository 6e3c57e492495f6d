// K-HIST for transformed 32- and 64-bit keys (signed, float, descending).
#include "hist.cuh"

namespace lsdrs {

cudaError_t launch_hist_x(KeyKind k, int bits, const HistArgs& a, int grid, cudaStream_t s) {
  if (k == kKeyX32) return launch_hist_k<KeyX32>(bits, a, grid, s);
  if (k == kKeyX64) return launch_hist_k<KeyX64>(bits, a, grid, s);
  return cudaErrorInvalidValue;
}

}  // namespace lsdrs
