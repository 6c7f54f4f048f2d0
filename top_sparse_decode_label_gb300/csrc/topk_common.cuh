// Radix digits and shared-memory histograms of the exact top-k.
#pragma once

#include "common.cuh"

namespace ds {

constexpr int kBins1 = 2048;   // digits 1 and 2: key bits 21..31 and 10..20
constexpr int kBins3 = 1024;   // digit 3: key bits 0..9

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

// Rows that need a selection at all: 0 < K_eff < T.
__device__ __forceinline__ bool needs_selection(int k, int T) { return k > 0 && k < T; }

}  // namespace ds
