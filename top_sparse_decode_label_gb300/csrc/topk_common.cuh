// Exact top-k machinery shared by the fused scoring kernel and the top-k
// kernels: the scratch layout, the radix threshold search and the level-1
// epilogue that turns a row's 2048-bin histogram of the top 11 key bits into
// (threshold bin b1, number of keys above it).
//
// Completion counters: a multi-CTA phase counts finished CTAs per row (or per
// request and head block) with one atomicAdd each; the CTA that sees the last
// count does the per-row follow-up and resets the counter to zero. Nothing
// waits on another CTA, so no launch order or co-residency is assumed.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace ds {

constexpr int kBins1 = 2048;   // level-1 digit: key bits 21..31
constexpr int kChunk = 4096;   // scores per filter CTA
constexpr int kChunkThreads = 256;

// Device view of the top-k scratch (see TopkLayout in internal.h).
struct TopkWs {
  unsigned* ghist;     // [R, 2048] level-1 histograms (zero between calls)
  unsigned* done1;     // [R] completion counters of the histogram phase (zero between calls)
  unsigned* done2;     // [R] completion counters of the filter phase (zero between calls)
  uint2* row_state;    // [R] (b1, count above b1)
  unsigned* counts;    // [R, nch] kept-list length of each chunk
  uint2* list;         // [R, Tmax] (key, token) with key >> 21 >= b1, per chunk in token order
  int nch;             // chunks per row = ceil(Tmax / kChunk)
};

inline TopkWs topk_ws_view(const TopkLayout& L) {
  TopkWs w;
  w.ghist = static_cast<unsigned*>(L.ghist);
  w.done1 = static_cast<unsigned*>(L.done1);
  w.done2 = static_cast<unsigned*>(L.done2);
  w.row_state = static_cast<uint2*>(L.row_state);
  w.counts = static_cast<unsigned*>(L.counts);
  w.list = static_cast<uint2*>(L.list);
  w.nch = L.nch;
  return w;
}

// Scanning a histogram from its highest bin down, finds the bin where the
// running count first reaches `need` (1 <= need <= total). Writes out[0] =
// bin, out[1] = count in the bins above it (0, 0 if no bin qualifies).
// nbins must be a multiple of blockDim.x. GLOBAL: the histogram is in global
// memory written by other CTAs' atomics, read through L2.
template <bool GLOBAL>
__device__ void find_threshold_bin(const unsigned* hist, int nbins, unsigned need, unsigned* sh_scan,
                                   unsigned* out) {
  const int per = nbins / blockDim.x;
  const int hi = nbins - per * threadIdx.x;
  if (threadIdx.x == 0) {
    out[0] = 0;
    out[1] = 0;
  }
  unsigned c = 0;
  for (int i = 1; i <= per; ++i) c += GLOBAL ? __ldcg(hist + hi - i) : hist[hi - i];
  unsigned total;
  const unsigned before = block_excl_scan(c, sh_scan, &total);
  if (before < need && before + c >= need) {
    unsigned run = before;
    for (int i = 1; i <= per; ++i) {
      const unsigned h = GLOBAL ? __ldcg(hist + hi - i) : hist[hi - i];
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

// Level-1 epilogue of one row, run by every thread of the CTA that finished
// the row's histogram last: records (b1, above) and clears the histogram.
__device__ __forceinline__ void level1_threshold(const TopkWs& w, int row, int keff, unsigned* sh_scan,
                                                 unsigned* sh_res) {
  unsigned* h = w.ghist + static_cast<size_t>(row) * kBins1;
  find_threshold_bin<true>(h, kBins1, static_cast<unsigned>(keff), sh_scan, sh_res);
  if (threadIdx.x == 0) w.row_state[row] = make_uint2(sh_res[0], sh_res[1]);
  for (int i = threadIdx.x; i < kBins1; i += blockDim.x) __stcg(h + i, 0u);
  __syncthreads();
}

// Level-1 epilogue of one row run by a single warp: lane l holds bins
// [2048 - 64(l+1), 2048 - 64 l) in registers (one round of loads), a warp
// prefix over lanes from the top finds the lane holding the K_eff-th key,
// which scans its bins. Records (b1, above) and clears the histogram.
__device__ __forceinline__ void level1_threshold_warp(const TopkWs& w, int row, int keff) {
  const int lane = threadIdx.x & 31;
  unsigned* h = w.ghist + static_cast<size_t>(row) * kBins1 + (kBins1 - 64 * (lane + 1));
  uint4 v[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __ldcg(reinterpret_cast<const uint4*>(h) + i);
  unsigned c = 0;
#pragma unroll
  for (int i = 0; i < 16; ++i) c += v[i].x + v[i].y + v[i].z + v[i].w;
  const unsigned inc = warp_incl_scan(c);
  const unsigned before = inc - c;
  const unsigned need = static_cast<unsigned>(keff);
  if (before < need && inc >= need) {
    unsigned run = before;
    unsigned bin = 0, above = 0;
    bool found = false;
#pragma unroll
    for (int i = 15; i >= 0; --i) {
      const unsigned e[4] = {v[i].w, v[i].z, v[i].y, v[i].x};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (!found && run + e[q] >= need) {
          found = true;
          bin = kBins1 - 64 * (lane + 1) + 4 * i + (3 - q);
          above = run;
        }
        run += e[q];
      }
    }
    w.row_state[row] = make_uint2(bin, above);
  }
#pragma unroll
  for (int i = 0; i < 16; ++i) __stcg(reinterpret_cast<uint4*>(h) + i, make_uint4(0u, 0u, 0u, 0u));
}

// Rows that need a selection at all: 0 < K_eff < T.
__device__ __forceinline__ bool needs_selection(int k, int T) { return k > 0 && k < T; }

}  // namespace ds
