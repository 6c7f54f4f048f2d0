// Exact top-k machinery shared by the top-k kernels: the scratch layout and
// the radix threshold search.
//
// Completion counters: the filter phase counts finished chunks per row with
// one atomicAdd each; the CTA that sees the last count selects the row and
// resets the counter and the row's histogram to zero. Nothing waits on
// another CTA, so no launch order or co-residency is assumed.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kBins1 = 2048;   // level-1 digit: key bits 21..31
constexpr int kChunk = 4096;   // scores per histogram / filter work item
constexpr int kChunkThreads = 256;

// Device view of the top-k scratch (see TopkLayout in internal.h).
struct TopkWs {
  unsigned* ghist;     // [R, 2048] level-1 histograms (zero between calls)
  unsigned* ghist2;    // [R, 2048] level-2 histograms of the bin-b1 keys (zero between calls)
  unsigned* done2;     // [R] completion counters of the filter phase (zero between calls)
  unsigned* counts;    // [R, nch] kept-list length of each chunk
  uint2* list;         // [R, Tmax] (key, token) with key >> 21 >= b1, per chunk in token order
  int nch;             // chunks per row = ceil(Tmax / kChunk)
};

inline TopkWs topk_ws_view(const TopkLayout& L) {
  TopkWs w;
  w.ghist = static_cast<unsigned*>(L.ghist);
  w.ghist2 = static_cast<unsigned*>(L.ghist2);
  w.done2 = static_cast<unsigned*>(L.done2);
  w.counts = static_cast<unsigned*>(L.counts);
  w.list = static_cast<uint2*>(L.list);
  w.nch = L.nch;
  return w;
}

// Shared-memory slot of histogram bin b: the low 5 bits (the bank) are XOR-
// folded with the higher bits, a bijection per 32-bin block, so digit
// patterns that vary only in high bits (e.g. integer-valued scores, whose low
// mantissa bits are all zero) still spread over all banks.
__device__ __forceinline__ int hslot(int b) { return (b & ~31) | ((b ^ (b >> 5) ^ (b >> 10)) & 31); }

// Adds 1 to bin `bin` of a shared histogram (slot hslot(bin)) when `pred`.
// Shared atomics to one address are combined by the hardware; bank conflicts
// between different addresses are what serialises them, and hslot spreads
// those.
__device__ __forceinline__ void warp_hist_add(unsigned* h, unsigned bin, bool pred) {
  if (pred) atomicAdd(h + hslot(static_cast<int>(bin)), 1u);
}

// Scanning a histogram from its highest bin down, finds the bin where the
// running count first reaches `need` (1 <= need <= total). Writes out[0] =
// bin, out[1] = count in the bins above it (0, 0 if no bin qualifies).
// nbins must be a multiple of blockDim.x. GLOBAL: the histogram is in global
// memory written by other CTAs' atomics, read through L2 (bin b at index b);
// otherwise it is a shared histogram filled by warp_hist_add (bin b at hslot(b)).
template <bool GLOBAL>
__device__ __forceinline__ void find_threshold_bin(const unsigned* hist, int nbins, unsigned need, unsigned* sh_scan,
                                   unsigned* out) {
  const int per = nbins / blockDim.x;
  const int hi = nbins - per * threadIdx.x;
  if (threadIdx.x == 0) {
    out[0] = 0;
    out[1] = 0;
  }
  unsigned c = 0;
  for (int i = 1; i <= per; ++i) c += GLOBAL ? __ldcg(hist + hi - i) : hist[hslot(hi - i)];
  unsigned total;
  const unsigned before = block_excl_scan(c, sh_scan, &total);
  if (before < need && before + c >= need) {
    unsigned run = before;
    for (int i = 1; i <= per; ++i) {
      const unsigned h = GLOBAL ? __ldcg(hist + hi - i) : hist[hslot(hi - i)];
      if (run + h >= need) {
        out[0] = hi - i;
        out[1] = run;
        break;
      }
      run += h;
    }
  }
  __syncthreads();
}

// Rows that need a selection at all: 0 < K_eff < T.
__device__ __forceinline__ bool needs_selection(int k, int T) { return k > 0 && k < T; }

}  // namespace ds
