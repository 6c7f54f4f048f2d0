// Stage 2: exact top-k per (request, KV head) row with lowest-token-index
// tie-breaking, output ascending by token index.
//
// sglang PR #43527 "QSA cache sharding", "Distributed QSA execution": local
// candidates are merged into an exact Top-K using deterministic global
// token-ID tie-breaking. "Support double sparsity" (PR #1459): keep the
// heavy-token count of tokens per head.
//
// Scores are mapped to order-preserving 32-bit keys (-0.0 == +0.0, NaN
// lowest). Let K_eff = min(k, T). Three launches, all multi-CTA except the last:
//   hist    : 2048-bin histogram of key >> 21 per row (shared-memory
//             histogram per 4096-score chunk, flushed with global atomics).
//   filter  : every CTA finds the bin b1 holding the K_eff-th largest key from
//             the row histogram, then streams its chunk: keys in bins above b1
//             are certainly kept ("sure" list), keys in b1 are candidates.
//   select  : one CTA per row refines the threshold key among the candidates
//             with two more radix digits (11 + 10 bits), giving the exact
//             K_eff-th key `thr` and how many tokens with key == thr to keep.
//             Kept tokens are marked in a shared-memory bitmap over token
//             positions; the first r ties in token order are found with a
//             popcount prefix over the bitmap, and a second popcount prefix
//             writes the kept tokens ascending. Rows longer than the bitmap
//             window are processed window by window.
// The score buffer is read twice (hist, filter); everything else touches only
// the candidates, typically a few thousand per row.
#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kBins1 = 2048;          // top 11 bits
constexpr int kChunk = 4096;          // scores per hist/filter CTA
constexpr int kChunkThreads = 256;
constexpr int kSelThreads = 1024;
constexpr int kWindow = 1 << 20;      // tokens per bitmap window (128 KB of shared memory)

struct Layout {
  unsigned* hist;    // [R, 2048]
  unsigned* state;   // [R, 4]: sure count, candidate count
  int32_t* sure;     // [R, k]
  uint32_t* ckey;    // [R, Tmax]
  int32_t* ctok;     // [R, Tmax]
  size_t bytes;
  size_t clear_bytes;  // hist + state, zeroed per call
};

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

Layout make_layout(void* base, int R, int Tmax, int k) {
  Layout L;
  char* p = static_cast<char*>(base);
  size_t off = 0;
  L.hist = reinterpret_cast<unsigned*>(p + off);
  off += static_cast<size_t>(R) * kBins1 * 4;
  L.state = reinterpret_cast<unsigned*>(p + off);
  off += static_cast<size_t>(R) * 16;
  L.clear_bytes = off;
  off = align256(off);
  L.sure = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (k > 0 ? k : 1) * 4);
  L.ckey = reinterpret_cast<uint32_t*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (Tmax > 0 ? Tmax : 1) * 4);
  L.ctok = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (Tmax > 0 ? Tmax : 1) * 4);
  L.bytes = off;
  return L;
}

struct TopkParams {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* idx;
  unsigned* err;
  int Hkv, Tmax, lim, k;
  Layout L;
};

__device__ __forceinline__ int row_len(const TopkParams& p, int b, bool flag) {
  int T = p.seq_lens[b];
  if (T < 0 || T > p.lim) {
    if (flag) flag_error(p.err, 1u);
    T = T < 0 ? 0 : p.lim;
  }
  return T;
}

// Scanning `hist` from its highest bin down, finds the bin where the running
// count first reaches `need` (1 <= need <= total). Writes out[0] = bin,
// out[1] = count in the bins above it. nbins must be a multiple of blockDim.x.
__device__ void find_threshold_bin(const unsigned* hist, int nbins, unsigned need, unsigned* sh_scan,
                                   unsigned* out) {
  const int per = nbins / blockDim.x;
  const int hi = nbins - per * threadIdx.x;
  if (threadIdx.x == 0) {  // defined result even if `need` were out of range
    out[0] = 0;
    out[1] = 0;
  }
  unsigned c = 0;
  for (int i = 1; i <= per; ++i) c += hist[hi - i];
  unsigned total;
  const unsigned before = block_excl_scan(c, sh_scan, &total);
  if (before < need && before + c >= need) {
    unsigned run = before;
    for (int i = 1; i <= per; ++i) {
      const unsigned h = hist[hi - i];
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

__device__ __forceinline__ unsigned warp_append(bool pred, unsigned* counter) {
  const int lane = threadIdx.x & 31;
  const unsigned mask = __ballot_sync(kFull, pred);
  unsigned base = 0;
  const int leader = mask ? __ffs(mask) - 1 : 0;
  if (mask && lane == leader) base = atomicAdd(counter, __popc(mask));
  base = __shfl_sync(kFull, base, leader);
  return base + __popc(mask & ((1u << lane) - 1u));
}

__global__ void __launch_bounds__(kChunkThreads) topk_hist_kernel(const TopkParams p) {
  __shared__ unsigned h[kBins1];
  const int row = blockIdx.y;
  const int b = row / p.Hkv;
  const int T = row_len(p, b, blockIdx.x == 0 && threadIdx.x == 0 && row % p.Hkv == 0);
  const int keff = min(p.k, T);
  const int c0 = blockIdx.x * kChunk;
  if (keff == 0 || keff == T || c0 >= T) return;
  for (int i = threadIdx.x; i < kBins1; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const float* s = p.scores + static_cast<long long>(row) * p.Tmax;
  const int c1 = min(T, c0 + kChunk);
  for (int t = c0 + threadIdx.x; t < c1; t += blockDim.x) atomicAdd(&h[order_key(s[t]) >> 21], 1u);
  __syncthreads();
  unsigned* g = p.L.hist + static_cast<size_t>(row) * kBins1;
  for (int i = threadIdx.x; i < kBins1; i += blockDim.x)
    if (h[i]) atomicAdd(&g[i], h[i]);
}

__global__ void __launch_bounds__(kChunkThreads) topk_filter_kernel(const TopkParams p) {
  __shared__ unsigned sh_scan[33];
  __shared__ unsigned sh_res[2];
  const int row = blockIdx.y;
  const int b = row / p.Hkv;
  const int T = row_len(p, b, false);
  const int keff = min(p.k, T);
  const int c0 = blockIdx.x * kChunk;
  if (keff == 0 || keff == T || c0 >= T) return;
  find_threshold_bin(p.L.hist + static_cast<size_t>(row) * kBins1, kBins1, keff, sh_scan, sh_res);
  const unsigned b1 = sh_res[0];
  const float* s = p.scores + static_cast<long long>(row) * p.Tmax;
  unsigned* st = p.L.state + static_cast<size_t>(row) * 4;
  int32_t* sure = p.L.sure + static_cast<size_t>(row) * p.k;
  uint32_t* ckey = p.L.ckey + static_cast<size_t>(row) * p.Tmax;
  int32_t* ctok = p.L.ctok + static_cast<size_t>(row) * p.Tmax;
  const int c1 = min(T, c0 + kChunk);
  // Uniform trip count so whole warps take part in the appends.
  for (int base = c0; base < c1; base += blockDim.x) {
    const int t = base + threadIdx.x;
    uint32_t key = 0;
    if (t < c1) key = order_key(s[t]);
    const unsigned bin = key >> 21;
    const bool is_sure = t < c1 && bin > b1;
    const bool is_cand = t < c1 && bin == b1;
    const unsigned ps = warp_append(is_sure, &st[0]);
    const unsigned pc = warp_append(is_cand, &st[1]);
    if (is_sure) sure[ps] = t;
    if (is_cand) {
      ckey[pc] = key;
      ctok[pc] = t;
    }
  }
}

__global__ void __launch_bounds__(kSelThreads) topk_select_kernel(const TopkParams p, int win_words) {
  extern __shared__ unsigned bitmap[];
  __shared__ unsigned sh_scan[33];
  __shared__ unsigned sh_hist[kBins1];
  __shared__ unsigned sh_res[2];
  const int row = blockIdx.x;
  const int b = row / p.Hkv;
  const int T = row_len(p, b, false);
  const int keff = min(p.k, T);
  int32_t* out = p.idx + static_cast<size_t>(row) * p.k;
  const int tid = threadIdx.x;

  if (keff == 0 || keff == T) {
    for (int i = tid; i < p.k; i += blockDim.x) out[i] = (i < keff) ? i : -1;
    return;
  }
  // Level 1: the bin of the top 11 bits (same histogram the filter used).
  find_threshold_bin(p.L.hist + static_cast<size_t>(row) * kBins1, kBins1, keff, sh_scan, sh_res);
  const unsigned b1 = sh_res[0];
  const unsigned need = keff - sh_res[1];
  const unsigned* st = p.L.state + static_cast<size_t>(row) * 4;
  const int nsure = st[0];
  const int ncand = st[1];
  const uint32_t* ckey = p.L.ckey + static_cast<size_t>(row) * p.Tmax;
  const int32_t* ctok = p.L.ctok + static_cast<size_t>(row) * p.Tmax;
  const int32_t* sure = p.L.sure + static_cast<size_t>(row) * p.k;

  // Level 2: bits 10..20 among the candidates.
  for (int i = tid; i < kBins1; i += blockDim.x) sh_hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < ncand; i += blockDim.x) atomicAdd(&sh_hist[(ckey[i] >> 10) & 2047u], 1u);
  __syncthreads();
  find_threshold_bin(sh_hist, kBins1, need, sh_scan, sh_res);
  const unsigned d2 = sh_res[0];
  const unsigned need2 = need - sh_res[1];
  // Level 3: bits 0..9 among the candidates that match so far.
  for (int i = tid; i < 1024; i += blockDim.x) sh_hist[i] = 0;
  __syncthreads();
  for (int i = tid; i < ncand; i += blockDim.x) {
    const uint32_t key = ckey[i];
    if (((key >> 10) & 2047u) == d2) atomicAdd(&sh_hist[key & 1023u], 1u);
  }
  __syncthreads();
  find_threshold_bin(sh_hist, 1024, need2, sh_scan, sh_res);
  const unsigned d3 = sh_res[0];
  const unsigned r_eq = need2 - sh_res[1];          // ties to keep, in token order
  const unsigned eq_total = sh_hist[d3];
  const uint32_t thr = (b1 << 21) | (d2 << 10) | d3;
  __syncthreads();

  const bool prune = eq_total > r_eq;
  unsigned eq_before = 0;   // ties kept in earlier windows
  unsigned out_off = 0;
  const int win = win_words * 32;
  for (int w0 = 0; w0 < T; w0 += win) {
    const int wl = min(win, T - w0);
    const int nwords = (wl + 31) >> 5;
    const int per = (nwords + blockDim.x - 1) / blockDim.x;
    const int wb = tid * per;
    const int we = min(nwords, wb + per);
    for (int i = tid; i < nwords; i += blockDim.x) bitmap[i] = 0;
    __syncthreads();
    // Ties at the threshold key.
    for (int i = tid; i < ncand; i += blockDim.x) {
      const int t = ctok[i] - w0;
      if (ckey[i] == thr && t >= 0 && t < wl) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    if (prune) {
      unsigned c = 0;
      for (int i = wb; i < we; ++i) c += __popc(bitmap[i]);
      unsigned total;
      unsigned before = block_excl_scan(c, sh_scan, &total) + eq_before;
      for (int i = wb; i < we; ++i) {
        unsigned w = bitmap[i];
        unsigned keepw = 0;
        while (w) {
          const unsigned bit = w & (0u - w);
          if (before < r_eq) keepw |= bit;
          ++before;
          w ^= bit;
        }
        bitmap[i] = keepw;
      }
      eq_before += total;
      __syncthreads();
    }
    // Everything strictly above the threshold.
    for (int i = tid; i < ncand; i += blockDim.x) {
      const int t = ctok[i] - w0;
      if (ckey[i] > thr && t >= 0 && t < wl) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    }
    for (int i = tid; i < nsure; i += blockDim.x) {
      const int t = sure[i] - w0;
      if (t >= 0 && t < wl) atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    }
    __syncthreads();
    // Ascending compaction.
    unsigned c = 0;
    for (int i = wb; i < we; ++i) c += __popc(bitmap[i]);
    unsigned total;
    unsigned pos = out_off + block_excl_scan(c, sh_scan, &total);
    for (int i = wb; i < we; ++i) {
      unsigned w = bitmap[i];
      while (w) {
        const int bit = __ffs(w) - 1;
        if (pos < static_cast<unsigned>(p.k)) out[pos] = w0 + i * 32 + bit;
        ++pos;
        w &= w - 1;
      }
    }
    out_off += total;
    __syncthreads();
  }
  for (int i = keff + tid; i < p.k; i += blockDim.x) out[i] = -1;
}

}  // namespace

size_t topk_workspace_bytes(int B, int Hkv, int Tmax, int k) {
  return make_layout(nullptr, B * Hkv, Tmax, k).bytes;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  const int R = a.B * a.Hkv;
  if (R == 0 || a.k == 0) {
    return cudaSuccess;
  }
  TopkParams p;
  p.scores = a.scores;
  p.seq_lens = a.seq_lens;
  p.idx = a.idx;
  p.err = a.err;
  p.Hkv = a.Hkv;
  p.Tmax = a.Tmax;
  p.lim = a.maxp_tokens < a.Tmax ? a.maxp_tokens : a.Tmax;
  p.k = a.k;
  p.L = make_layout(a.ws, R, a.Tmax, a.k);
  cudaError_t e = cudaMemsetAsync(p.L.hist, 0, p.L.clear_bytes, stream);
  if (e != cudaSuccess) return e;
  if (a.Tmax > 0) {
    dim3 grid((a.Tmax + kChunk - 1) / kChunk, R);
    topk_hist_kernel<<<grid, kChunkThreads, 0, stream>>>(p);
    topk_filter_kernel<<<grid, kChunkThreads, 0, stream>>>(p);
  }
  int tw = a.Tmax < kWindow ? a.Tmax : kWindow;
  int win_words = (tw + 31) / 32;
  if (win_words < 1) win_words = 1;
  const size_t smem = static_cast<size_t>(win_words) * 4;
  e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  topk_select_kernel<<<R, kSelThreads, smem, stream>>>(p, win_words);
  return cudaGetLastError();
}

}  // namespace ds
