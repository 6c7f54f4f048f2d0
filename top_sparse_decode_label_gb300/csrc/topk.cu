// Stage 2: exact top-k per (request, KV head) row with lowest-token-index
// tie-breaking, output ascending by token index.
//
// sglang PR #43527 "QSA cache sharding", "Distributed QSA execution": local
// candidates are merged into an exact Top-K using deterministic global
// token-ID tie-breaking. "Support double sparsity" (PR #1459): keep the
// heavy-token count of tokens per head.
//
// Scores map to order-preserving 32-bit keys (-0.0 == +0.0, NaN lowest).
// With K_eff = min(k, T), rows with 0 < K_eff < T go through three radix
// digits (11 + 11 + 10 bits) in two launches:
//   histogram: one CTA per 4096-score chunk of a row builds a 2048-bin
//     histogram of key >> 21 in shared memory and adds its nonzero bins into
//     the row's global histogram (a few dozen atomics per CTA).
//   filter + select (persistent CTAs over (row, chunk) work items): a CTA
//     finds, from the row's histogram, the bin b1 holding the K_eff-th largest
//     key, then keeps every (key, token) of its chunk with key >> 21 >= b1, in
//     token order, in the chunk's slot of the row's list (one block-wide
//     prefix sum). The CTA that completes the row's last chunk selects: it
//     gathers the row's list (typically K_eff plus a few thousand entries)
//     into shared memory, refines the threshold key over the entries whose
//     top bits equal b1 (two more digits), giving the exact K_eff-th key `thr`
//     and the number r of ties to keep, and writes the kept tokens -- key >
//     thr, or key == thr and tie rank < r -- ascending with two block-wide
//     prefix sums. It then clears the row's histogram and counter.
// Completion is detected with per-row counters (the last CTA continues);
// nothing waits on another CTA. Both kernels use programmatic dependent
// launch and wait for the previous kernel before touching its outputs.
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ds {

namespace {

constexpr int kElems = kChunk / kChunkThreads;   // 16 scores per thread
constexpr int kMaxChunks = 4096;                 // rows of up to 16M tokens
constexpr int kListCap = 8192;                   // kept entries selected from shared memory (64 KB)

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct TopkParams {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* idx;
  unsigned* err;
  int Hkv, Tmax, lim, k, R;
  TopkWs w;
};

// Keys of scores [t0, t0 + kElems) of a row (only t < c1 is meaningful); four
// 16-byte loads in flight when aligned, else scalar loads.
__device__ __forceinline__ void load_keys(const float* s, int t0, int c1, uint32_t (&keys)[kElems]) {
  if (((reinterpret_cast<uintptr_t>(s) & 15u) == 0) && (t0 + kElems <= c1)) {
    float4 v[kElems / 4];
#pragma unroll
    for (int i = 0; i < kElems / 4; ++i) v[i] = *reinterpret_cast<const float4*>(s + t0 + 4 * i);
#pragma unroll
    for (int i = 0; i < kElems / 4; ++i) {
      keys[4 * i] = order_key(v[i].x);
      keys[4 * i + 1] = order_key(v[i].y);
      keys[4 * i + 2] = order_key(v[i].z);
      keys[4 * i + 3] = order_key(v[i].w);
    }
  } else {
#pragma unroll
    for (int i = 0; i < kElems; ++i) keys[i] = (t0 + i < c1) ? order_key(s[t0 + i]) : 0u;
  }
}

__device__ __forceinline__ int row_len(const TopkParams& p, int b, bool flag) {
  int T = p.seq_lens[b];
  if (T < 0 || T > p.lim) {
    if (flag) flag_error(p.err, 1u);
    T = T < 0 ? 0 : p.lim;
  }
  return T;
}

// Level-1 histograms of the rows that need a selection.
__global__ void __launch_bounds__(kChunkThreads) topk_hist_kernel(const TopkParams p) {
  __shared__ unsigned h[kBins1];
  grid_dependency_wait();
  const int row = blockIdx.y;
  const int b = row / p.Hkv;
  const int T = row_len(p, b, blockIdx.x == 0 && threadIdx.x == 0 && row % p.Hkv == 0);
  if (!needs_selection(p.k, T)) return;
  const int c0 = blockIdx.x * kChunk;
  if (c0 >= T) return;
  for (int i = threadIdx.x; i < kBins1; i += blockDim.x) h[i] = 0;
  __syncthreads();
  const float* s = p.scores + static_cast<long long>(row) * p.Tmax;
  const int c1 = min(T, c0 + kChunk);
  const int t0 = c0 + threadIdx.x * kElems;
  uint32_t keys[kElems];
  load_keys(s, t0, c1, keys);
#pragma unroll
  for (int i = 0; i < kElems; ++i) warp_hist_add(h, keys[i] >> 21, t0 + i < c1);
  __syncthreads();
  unsigned* g = p.w.ghist + static_cast<size_t>(row) * kBins1;
  for (int i = threadIdx.x; i < kBins1; i += blockDim.x) {
    const unsigned v = h[hslot(i)];
    if (v) atomicAdd(&g[i], v);
  }
}

// Walks entries [e, ...) of a row's list (chunk slots concatenated).
struct ListWalker {
  const uint2* base;   // row's list
  const unsigned* pref;  // shared: chunk prefix, nch + 1 entries
  int ci, off;
  __device__ void seek(int e, int nch) {
    int lo = 0, hi = nch - 1;  // largest ci with pref[ci] <= e
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (pref[mid] <= static_cast<unsigned>(e)) lo = mid; else hi = mid - 1;
    }
    ci = lo;
    off = e - static_cast<int>(pref[ci]);
  }
  __device__ uint2 next() {
    while (static_cast<unsigned>(off) >= pref[ci + 1] - pref[ci]) {
      ++ci;
      off = 0;
    }
    const uint2 v = __ldcg(base + static_cast<size_t>(ci) * kChunk + off);
    ++off;
    return v;
  }
};

// Select phase of one row, run by the CTA that completed the row's filter.
// `lst` holds the kept entries of the row in token order when M <= cap
// (copied to shared memory); otherwise they are walked in global memory.
__device__ __forceinline__ void select_row(const TopkParams& p, int row, int T, int nch, unsigned b1, unsigned above1,
                           uint2* sm_list, int cap, unsigned* sh_pref, unsigned* sh_hist, unsigned* sh_scan,
                           unsigned* sh_res) {
  const int tid = threadIdx.x;
  const int keff = min(p.k, T);
  int32_t* out = p.idx + static_cast<size_t>(row) * p.k;
  const unsigned* counts = p.w.counts + static_cast<size_t>(row) * p.w.nch;
  const uint2* base = p.w.list + static_cast<size_t>(row) * p.Tmax;

  // Chunk prefix of the list lengths.
  const int cpt = (nch + kChunkThreads - 1) / kChunkThreads;
  {
    unsigned mine = 0;
    for (int i = tid * cpt; i < min(nch, (tid + 1) * cpt); ++i) mine += __ldcg(counts + i);
    unsigned tot;
    unsigned run = block_excl_scan(mine, sh_scan, &tot);
    for (int i = tid * cpt; i < min(nch, (tid + 1) * cpt); ++i) {
      sh_pref[i] = run;
      run += __ldcg(counts + i);
    }
    if (tid == 0) sh_pref[nch] = tot;
  }
  __syncthreads();
  const int M = static_cast<int>(sh_pref[nch]);
  const bool in_smem = M <= cap;
  if (in_smem) {
    // Gather the list into shared memory: warp w copies chunks w, w+8, ...,
    // eight independent loads in flight per lane.
    const int lane = tid & 31, warp = tid >> 5;
    for (int ci = warp; ci < nch; ci += kChunkThreads / 32) {
      const int n = static_cast<int>(sh_pref[ci + 1] - sh_pref[ci]);
      const uint2* src = base + static_cast<size_t>(ci) * kChunk;
      uint2* dst = sm_list + sh_pref[ci];
      for (int j0 = lane; j0 < n; j0 += 8 * 32) {
        uint2 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (j0 + i * 32 < n) v[i] = __ldcg(src + j0 + i * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          if (j0 + i * 32 < n) dst[j0 + i * 32] = v[i];
      }
    }
    __syncthreads();
  }
  auto key_at = [&](int e, ListWalker& wk) -> uint2 { return in_smem ? sm_list[e] : wk.next(); };
  const unsigned need = static_cast<unsigned>(keff) - above1;

  // Level 2: bits 10..20 of the bin-b1 keys, histogram built by the filter CTAs.
  unsigned* gh2 = p.w.ghist2 + static_cast<size_t>(row) * kBins1;
  find_threshold_bin<true>(gh2, kBins1, need, sh_scan, sh_res);
  for (int i = tid; i < kBins1; i += blockDim.x) __stcg(gh2 + i, 0u);
  const unsigned d2 = sh_res[0];
  const unsigned need2 = need - sh_res[1];
  // Level 3: bits 0..9 of the entries that match so far.
  const uint32_t hi22 = (b1 << 11) | d2;
  for (int i = tid; i < 1024; i += blockDim.x) sh_hist[i] = 0;
  __syncthreads();
  if (in_smem) {
    for (int e0 = 0; e0 < M; e0 += 4 * kChunkThreads) {
      uint32_t key[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int e = e0 + i * kChunkThreads + tid;
        key[i] = e < M ? sm_list[e].x : 0u;
      }
#pragma unroll
      for (int i = 0; i < 4; ++i)
        warp_hist_add(sh_hist, key[i] & 1023u, e0 + i * kChunkThreads + tid < M && (key[i] >> 10) == hi22);
    }
  } else {
    const int lane = tid & 31, warp = tid >> 5;
    for (int ci = warp; ci < nch; ci += kChunkThreads / 32) {
      const int n = static_cast<int>(sh_pref[ci + 1] - sh_pref[ci]);
      for (int j0 = 0; j0 < n; j0 += 32) {
        const int j = j0 + lane;
        const uint32_t key = j < n ? __ldcg(base + static_cast<size_t>(ci) * kChunk + j).x : 0u;
        warp_hist_add(sh_hist, key & 1023u, j < n && (key >> 10) == hi22);
      }
    }
  }
  __syncthreads();
  find_threshold_bin<false>(sh_hist, 1024, need2, sh_scan, sh_res);
  const unsigned d3 = sh_res[0];
  const unsigned r_eq = need2 - sh_res[1];
  const unsigned eq_total = sh_hist[hslot(static_cast<int>(d3))];
  const uint32_t thr = (hi22 << 10) | d3;
  __syncthreads();

  // Ordered output: thread segments in token order, prefix sums across threads.
  const int seg = (M + kChunkThreads - 1) / kChunkThreads;
  const int e0 = min(M, tid * seg);
  const int e1 = min(M, e0 + seg);
  ListWalker wk{base, sh_pref, 0, 0};
  unsigned eq_base = 0;
  if (eq_total > r_eq) {
    unsigned eqc = 0;
    if (!in_smem && e0 < e1) wk.seek(e0, nch);
    for (int e = e0; e < e1; ++e) eqc += (key_at(e, wk).x == thr);
    unsigned tot;
    eq_base = block_excl_scan(eqc, sh_scan, &tot);
  }
  unsigned selc = 0;
  {
    if (!in_smem && e0 < e1) wk.seek(e0, nch);
    unsigned eq = eq_base;
    for (int e = e0; e < e1; ++e) {
      const uint32_t key = key_at(e, wk).x;
      if (key > thr) {
        ++selc;
      } else if (key == thr) {
        selc += (eq < r_eq);
        ++eq;
      }
    }
  }
  unsigned tot_sel;
  unsigned opos = block_excl_scan(selc, sh_scan, &tot_sel);
  {
    if (!in_smem && e0 < e1) wk.seek(e0, nch);
    unsigned eq = eq_base;
    for (int e = e0; e < e1; ++e) {
      const uint2 v = key_at(e, wk);
      bool keep = v.x > thr;
      if (v.x == thr) {
        keep = eq < r_eq;
        ++eq;
      }
      if (keep) {
        if (opos < static_cast<unsigned>(p.k)) out[opos] = static_cast<int32_t>(v.y);
        ++opos;
      }
    }
  }
  for (int i = keff + tid; i < p.k; i += blockDim.x) out[i] = -1;
  // Every chunk of the row has read the histogram: clear it for the next call.
  unsigned* gh = p.w.ghist + static_cast<size_t>(row) * kBins1;
  for (int i = tid; i < kBins1; i += blockDim.x) __stcg(gh + i, 0u);
  __syncthreads();
}

// Persistent filter: CTAs walk (row, chunk) work items; the CTA that completes
// a row's last chunk selects the row.
__global__ void __launch_bounds__(kChunkThreads) topk_filter_select_kernel(const TopkParams p, int cap) {
  extern __shared__ __align__(16) unsigned char dsmem[];
  uint2* sm_list = reinterpret_cast<uint2*>(dsmem);                         // [cap]
  unsigned* sh_pref = reinterpret_cast<unsigned*>(dsmem + static_cast<size_t>(cap) * 8);  // [nch + 1]
  __shared__ unsigned sh_scan[33];
  __shared__ unsigned sh_res[2];
  __shared__ int sh_last;
  __shared__ unsigned sh_hist[kBins1];
  const int tid = threadIdx.x;
  const int nitems = p.R * p.w.nch;
  const int w0 = static_cast<int>(static_cast<long long>(blockIdx.x) * nitems / gridDim.x);
  const int w1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * nitems / gridDim.x);
  grid_dependency_wait();
  int cur_row = -1;
  unsigned b1 = 0, above1 = 0;
  for (int item = w0; item < w1; ++item) {
    const int row = item / p.w.nch;
    const int c = item - row * p.w.nch;
    const int b = row / p.Hkv;
    const int T = row_len(p, b, false);
    const int keff = min(p.k, T);
    if (!needs_selection(p.k, T)) {
      if (c == 0) {
        int32_t* out = p.idx + static_cast<size_t>(row) * p.k;
        for (int i = tid; i < p.k; i += blockDim.x) out[i] = (i < keff) ? i : -1;
      }
      continue;
    }
    const int nch = (T + kChunk - 1) / kChunk;
    if (c >= nch) continue;
    if (row != cur_row) {
      // Level 1: the bin holding the K_eff-th largest key, from the row's histogram.
      find_threshold_bin<true>(p.w.ghist + static_cast<size_t>(row) * kBins1, kBins1, static_cast<unsigned>(keff),
                               sh_scan, sh_res);
      b1 = sh_res[0];
      above1 = sh_res[1];
      cur_row = row;
    }

    // ---- filter: keep key >> 21 >= b1 of this chunk, in token order
    const int c0 = c * kChunk;
    const int c1 = min(T, c0 + kChunk);
    const float* s = p.scores + static_cast<long long>(row) * p.Tmax;
    const int t0 = c0 + tid * kElems;
    uint32_t keys[kElems];
    unsigned flags = 0, cnt = 0;
    load_keys(s, t0, c1, keys);
    for (int i = tid; i < kBins1; i += blockDim.x) sh_hist[i] = 0;
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kElems; ++i) {
      if (t0 + i < c1 && (keys[i] >> 21) >= b1) {
        flags |= 1u << i;
        ++cnt;
      }
      warp_hist_add(sh_hist, (keys[i] >> 10) & 2047u, t0 + i < c1 && (keys[i] >> 21) == b1);
    }
    unsigned total;
    unsigned pos = block_excl_scan(cnt, sh_scan, &total);
    uint2* lst = p.w.list + static_cast<size_t>(row) * p.Tmax + c0;
#pragma unroll
    for (int i = 0; i < kElems; ++i)
      if ((flags >> i) & 1u) lst[pos++] = make_uint2(keys[i], static_cast<unsigned>(t0 + i));
    if (tid == 0) p.w.counts[static_cast<size_t>(row) * p.w.nch + c] = total;
    {
      unsigned* gh2 = p.w.ghist2 + static_cast<size_t>(row) * kBins1;
      for (int i = tid; i < kBins1; i += blockDim.x) {
        const unsigned v = sh_hist[hslot(i)];
        if (v) atomicAdd(gh2 + i, v);
      }
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) sh_last = (atomicAdd(p.w.done2 + row, 1u) + 1 == static_cast<unsigned>(nch));
    __syncthreads();
    if (!sh_last) continue;
    __threadfence();
    select_row(p, row, T, nch, b1, above1, sm_list, cap, sh_pref, sh_hist, sh_scan, sh_res);
    if (tid == 0) atomicExch(p.w.done2 + row, 0u);
  }
}

cudaError_t allow_select_smem(int bytes) {
  static int done[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && done[dev] >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(topk_filter_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = bytes;
  return e;
}

}  // namespace

TopkLayout topk_layout(void* base, int R, int Tmax) {
  TopkLayout L;
  char* p = static_cast<char*>(base);
  const int T1 = Tmax > 0 ? Tmax : 1;
  L.nch = (T1 + kChunk - 1) / kChunk;
  size_t off = 0;
  L.ghist = p + off;
  off += static_cast<size_t>(R) * kBins1 * 4;
  L.ghist2 = p + off;
  off += static_cast<size_t>(R) * kBins1 * 4;
  L.done2 = p + off;
  off += static_cast<size_t>(R) * 4;
  L.zero_bytes = off;
  off = align256(off);
  L.counts = p + off;
  off = align256(off + static_cast<size_t>(R) * L.nch * 4);
  L.list = p + off;
  off = align256(off + static_cast<size_t>(R) * T1 * 8);
  L.bytes = off;
  return L;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  const int R = a.B * a.Hkv;
  if (R == 0 || a.k == 0) return cudaSuccess;
  const int T1 = a.Tmax > 0 ? a.Tmax : 1;
  if ((T1 + kChunk - 1) / kChunk > kMaxChunks) return cudaErrorNotSupported;
  TopkParams p{};
  p.scores = a.scores;
  p.seq_lens = a.seq_lens;
  p.idx = a.idx;
  p.err = a.err;
  p.Hkv = a.Hkv;
  p.Tmax = a.Tmax;
  p.lim = a.maxp_tokens < a.Tmax ? a.maxp_tokens : a.Tmax;
  p.k = a.k;
  p.w = topk_ws_view(a.L);
  p.R = R;
  cudaError_t e;
  if (!a.zeroed) {
    e = cudaMemsetAsync(a.L.ghist, 0, a.L.zero_bytes, stream);
    if (e != cudaSuccess) return e;
  }
  if (a.Tmax > 0) {
    e = launch_pdl(topk_hist_kernel, dim3(a.L.nch, R), dim3(kChunkThreads), 0, stream, p);
    if (e != cudaSuccess) return e;
  }
  // Shared memory: the selected row's kept list (up to kListCap entries) and the chunk prefix.
  const int smem = kListCap * 8 + (a.L.nch + 1) * 4;
  e = allow_select_smem(smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, topk_filter_select_kernel, kChunkThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  long long blocks = static_cast<long long>(sm_count()) * per_sm;
  const long long items = static_cast<long long>(R) * a.L.nch;
  if (items < blocks) blocks = items;
  e = launch_pdl(topk_filter_select_kernel, dim3(static_cast<unsigned>(blocks)), dim3(kChunkThreads), smem, stream,
                 p, static_cast<int>(kListCap));
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
