// K-HIST for unsigned and 16-bit float keys (the templates are in
// hist.cuh; signed, float and descending 32/64-bit keys are instantiated in
// hist_x.cu), and K-SCAN: per-pass exclusive scans of the counts into bucket
// bases (DSA CUDA from First Principles, section 13.1: the base of digit d
// is the exclusive prefix sum of the counts of the digits below it).
#include "hist.cuh"

namespace lsdrs {

namespace {

// One CTA per (row, pass): add the slots of the row's chunks, then an
// exclusive scan over the digits.  Q threads share each digit's sum (Q
// independent partial sums in flight) when the row has many chunks.
template <int Q>
__global__ void __launch_bounds__(kScanThreads * Q) digit_scan_kernel(ScanArgs a) {
  __shared__ uint32_t part[Q][kScanThreads];
  __shared__ uint32_t warp_sums[kScanThreads / kWarp];
  grid_dependency_sync();
  const int tid = threadIdx.x;
  const int d = tid % kScanThreads;  // digit (when < radix)
  const int q = tid / kScanThreads;  // share of the chunks
  const int64_t row = blockIdx.x / a.passes;
  const int p = blockIdx.x % a.passes;
  const int nb = a.passes * a.radix;

  uint32_t total = 0;
  if (d < a.radix) {
    const uint32_t* s = a.slots + row * a.chunks_per_row * static_cast<int64_t>(nb) +
                        p * a.radix + d;
    int c = q;
    for (; c + 3 * Q < a.chunks_per_row; c += 4 * Q) {
      const uint32_t s0 = s[static_cast<int64_t>(c) * nb];
      const uint32_t s1 = s[static_cast<int64_t>(c + Q) * nb];
      const uint32_t s2 = s[static_cast<int64_t>(c + 2 * Q) * nb];
      const uint32_t s3 = s[static_cast<int64_t>(c + 3 * Q) * nb];
      total += (s0 + s1) + (s2 + s3);
    }
    for (; c < a.chunks_per_row; c += Q) total += s[static_cast<int64_t>(c) * nb];
  }
  if (Q > 1) {
    part[q][d] = total;
    __syncthreads();
    if (q != 0) return;
    total = 0;
#pragma unroll
    for (int k = 0; k < Q; ++k) total += part[k][d];
  }
  // block-wide exclusive scan of the totals over the first kScanThreads threads
  const int lane = d & 31, warp = d >> 5;
  uint32_t incl = total;
#pragma unroll
  for (int o = 1; o < kWarp; o <<= 1) {
    uint32_t y = __shfl_up_sync(kFull, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == kWarp - 1) warp_sums[warp] = incl;
  asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads));
  if (warp == 0) {
    uint32_t w = lane < kScanThreads / kWarp ? warp_sums[lane] : 0;
    uint32_t wi = w;
#pragma unroll
    for (int o = 1; o < kWarp; o <<= 1) {
      uint32_t y = __shfl_up_sync(kFull, wi, o);
      if (lane >= o) wi += y;
    }
    if (lane < kScanThreads / kWarp) warp_sums[lane] = wi - w;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads));
  const uint32_t excl = incl - total + warp_sums[warp];
  if (d < a.radix) {
    const int64_t o = (row * a.passes + p) * a.radix + d;
    a.bases[o] = excl;
    if (a.hist_out) a.hist_out[o] = total;
    if (a.bases_out) a.bases_out[o] = excl;
  }

  // Without pass skipping every pass runs.
  if (!a.dynamic) {
    if (blockIdx.x == 0 && d == 0) a.header[kHdrPassesRun] = a.passes;
    return;
  }
  // Pass p of this row is the identity when one digit holds every key of the
  // row; record the passes where some row is not.  The last CTA to finish
  // turns the flags into the schedule.
  __shared__ int one_digit;
  __shared__ bool last_cta;
  if (d == 0) one_digit = 0;
  asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads));
  if (d < a.radix && static_cast<int64_t>(total) == a.cols) one_digit = 1;
  asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads));
  if (d == 0) {
    uint32_t* hdr = a.header;
    if (!one_digit) atomicOr(hdr + kHdrNontrivial + p, 1u);
    __threadfence();
    const uint32_t done = atomicAdd(hdr + kHdrScanDone, 1u);
    last_cta = done == gridDim.x - 1;
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads));
  if (!last_cta) return;
  __shared__ uint32_t nontrivial[kMaxPasses];
  if (d < a.passes) {
    __threadfence();
    nontrivial[d] = ld_relaxed(a.header + kHdrNontrivial + d);
  }
  asm volatile("bar.sync 1, %0;" ::"n"(kScanThreads));
  if (d == 0) {
    uint32_t m = 0;
    for (int q = 0; q < a.passes; ++q) m += nontrivial[q] != 0;
    uint32_t k = 0, prev = kBufIn;
    for (int q = 0; q < a.passes; ++q) {
      uint32_t code = kCodeSkip;
      if (nontrivial[q] != 0) {
        code = pass_code(k, m, prev, a.in_place != 0);
        prev = (code & kCodeDst) >> 2;
        ++k;
      }
      a.header[kHdrTileCounter + q] = code << kCodeShift;
    }
    a.header[kHdrPassesRun] = m;
  }
}

}  // namespace

cudaError_t launch_hist(KeyKind k, int bits, const HistArgs& a, int grid, cudaStream_t s) {
  switch (k) {
    case kKeyU32: return launch_hist_k<KeyU32>(bits, a, grid, s);
    case kKeyU64: return launch_hist_k<KeyU64>(bits, a, grid, s);
    case kKeyF16:
      if (bits != 8) return cudaErrorInvalidValue;
      return launch_hist_t<KeyF16Bits, 8>(a, grid, s);
    case kKeyX32:
    case kKeyX64:
      return launch_hist_x(k, bits, a, grid, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_scan(const ScanArgs& a, cudaStream_t s) {
  const int64_t grid = a.rows * a.passes;
  if (a.chunks_per_row >= 16)
    return launch_kernel(digit_scan_kernel<4>, static_cast<unsigned>(grid), kScanThreads * 4, 0,
                         s, a);
  return launch_kernel(digit_scan_kernel<1>, static_cast<unsigned>(grid), kScanThreads, 0, s, a);
}

}  // namespace lsdrs
