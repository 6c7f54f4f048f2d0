// Exact top-k computed the way the QSA cache-sharding page distributes it,
// emulated on one GPU: sglang PR #43527 "QSA cache sharding", "QSA cache
// placement" (each cache page has one owner shard; page-interleaved: logical
// page p of a request belongs to shard p mod S) and "Distributed QSA
// execution" (each shard produces local candidates, merged into an exact
// global Top-K with deterministic global token-ID tie-breaking).
//
// Kernels, on the caller's stream:
//  1. shard_gather_kernel: row (b, g) of the scores becomes S shard rows,
//     shard j holding the scores of its pages in token order, and the shard
//     rows' lengths.
//  2. the cluster top-k on the R*S shard rows: each shard's local top-k
//     (positions in shard order, ascending).
//  3. mark_kernel: the local picks, mapped back to global token indices, are
//     set in a per-row bitmap of the row's tokens.
//  4. assemble_kernel: one CTA per row walks the bitmap in token order and
//     writes the candidates' scores and tokens, so that candidate position
//     order is global token order; it clears the bitmap as it goes.
//  5. the cluster top-k on the candidate rows: the merge. Equal scores go to
//     the lower candidate position, i.e. the lower global token index.
//  6. map_kernel: candidate positions back to token indices (ascending, -1
//     padded), the output of ds_topk_select.
#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kThreads = 256;

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

// Tokens of shard j (of S) among the first T tokens of a request (pages of 64).
__host__ __device__ __forceinline__ int shard_tokens(int T, int S, int j) {
  const int pages = (T + kPage - 1) / kPage;
  if (j >= pages) return 0;
  const int owned = (pages - 1 - j) / S + 1;   // pages j, j + S, ... below `pages`
  int n = owned * kPage;
  const int last = pages - 1;
  if (last % S == j && T % kPage) n -= kPage - T % kPage;
  return n;
}

// Global token of shard-local position l in shard j.
__device__ __forceinline__ int global_token(int l, int S, int j) {
  return ((l / kPage) * S + j) * kPage + (l & (kPage - 1));
}

__global__ void __launch_bounds__(kThreads) shard_gather_kernel(const float* scores, const int32_t* seq_lens,
                                                                int Hkv, int Tmax, int lim, int S, int Ls,
                                                                float* shard_scores, int32_t* shard_len,
                                                                unsigned* err) {
  const int rs = blockIdx.y;            // (row, shard)
  const int row = rs / S, j = rs - row * S;
  const int b = row / Hkv;
  int T = seq_lens[b];
  if (T < 0 || T > lim) {
    if (threadIdx.x == 0 && blockIdx.x == 0 && j == 0 && row % Hkv == 0) flag_error(err, 1u);
    T = T < 0 ? 0 : lim;
  }
  const int n = shard_tokens(T, S, j);
  if (blockIdx.x == 0 && threadIdx.x == 0) shard_len[rs] = n;
  const float* src = scores + static_cast<long long>(row) * Tmax;
  float* dst = shard_scores + static_cast<long long>(rs) * Ls;
  for (int l = blockIdx.x * kThreads + threadIdx.x; l < n; l += gridDim.x * kThreads)
    dst[l] = __ldcg(src + global_token(l, S, j));
}

__global__ void __launch_bounds__(kThreads) mark_kernel(const int32_t* local_idx, int k, int S, int words,
                                                        unsigned* bitmap) {
  const int rs = blockIdx.y;
  const int row = rs / S, j = rs - row * S;
  const int32_t* li = local_idx + static_cast<long long>(rs) * k;
  unsigned* bm = bitmap + static_cast<long long>(row) * words;
  for (int i = blockIdx.x * kThreads + threadIdx.x; i < k; i += gridDim.x * kThreads) {
    const int l = li[i];
    if (l < 0) continue;
    const int t = global_token(l, S, j);
    atomicOr(bm + (t >> 5), 1u << (t & 31));
  }
}

// One CTA per row: candidates in token order from the bitmap (then cleared).
__global__ void __launch_bounds__(kThreads) assemble_kernel(const float* scores, int Tmax, int words, int cap,
                                                            unsigned* bitmap, float* cand_scores,
                                                            int32_t* cand_tokens, int32_t* cand_len) {
  __shared__ unsigned scan[33];
  const int row = blockIdx.x;
  const int tid = threadIdx.x;
  unsigned* bm = bitmap + static_cast<long long>(row) * words;
  const float* s = scores + static_cast<long long>(row) * Tmax;
  float* cs = cand_scores + static_cast<long long>(row) * cap;
  int32_t* ct = cand_tokens + static_cast<long long>(row) * cap;
  // Contiguous word ranges per thread keep the output in token order.
  const int per = (words + kThreads - 1) / kThreads;
  const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
  unsigned n = 0;
  for (int w = w0; w < w1; ++w) n += __popc(bm[w]);
  unsigned tot;
  unsigned pos = block_excl_scan(n, scan, &tot);
  for (int w = w0; w < w1; ++w) {
    unsigned m = bm[w];
    if (!m) continue;
    bm[w] = 0u;
    while (m) {
      const int bit = __ffs(m) - 1;
      m &= m - 1;
      const int t = w * 32 + bit;
      if (pos < static_cast<unsigned>(cap)) {
        ct[pos] = t;
        cs[pos] = __ldcg(s + t);
      }
      ++pos;
    }
  }
  if (tid == 0) cand_len[row] = static_cast<int>(min(tot, static_cast<unsigned>(cap)));
}

__global__ void __launch_bounds__(kThreads) map_kernel(const int32_t* pos_idx, const int32_t* cand_tokens, int k,
                                                       int cap, int R, int32_t* idx) {
  const long long n = static_cast<long long>(R) * k;
  for (long long i = static_cast<long long>(blockIdx.x) * kThreads + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * kThreads) {
    const int row = static_cast<int>(i / k);
    const int p = pos_idx[i];
    idx[i] = p >= 0 ? cand_tokens[static_cast<long long>(row) * cap + p] : -1;
  }
}

struct ShardedLayout {
  float* shard_scores;    // [R*S, Ls]
  int32_t* shard_len;     // [R*S]
  int32_t* local_idx;     // [R*S, k]
  TopkLayout topk1;
  unsigned* bitmap;       // [R, words]
  float* cand_scores;     // [R, cap]
  int32_t* cand_tokens;   // [R, cap]
  int32_t* cand_len;      // [R]
  int32_t* pos_idx;       // [R, k]
  TopkLayout topk2;
  size_t bitmap_bytes;
  size_t bytes;
  int Ls, words, cap;
};

ShardedLayout sharded_layout(void* base, int R, int Tmax, int k, int S) {
  ShardedLayout L{};
  const int T1 = Tmax > 0 ? Tmax : 1;
  const int pages = (T1 + kPage - 1) / kPage;
  L.Ls = ((pages + S - 1) / S) * kPage;
  L.words = (T1 + 31) / 32;
  const long long capl = static_cast<long long>(S) * (k > 0 ? k : 1);
  L.cap = static_cast<int>(capl < T1 ? capl : T1);
  char* p = static_cast<char*>(base);
  size_t off = 0;
  auto take = [&](size_t bytes) {
    char* q = p ? p + off : nullptr;
    off = align256(off + bytes);
    return q;
  };
  const size_t RS = static_cast<size_t>(R) * S;
  L.bitmap = reinterpret_cast<unsigned*>(take(static_cast<size_t>(R) * L.words * 4));
  L.bitmap_bytes = align256(static_cast<size_t>(R) * L.words * 4);
  L.shard_scores = reinterpret_cast<float*>(take(RS * L.Ls * 4));
  L.shard_len = reinterpret_cast<int32_t*>(take(RS * 4));
  L.local_idx = reinterpret_cast<int32_t*>(take(RS * (k > 0 ? k : 1) * 4));
  const TopkLayout t1 = topk_layout(nullptr, static_cast<int>(RS), L.Ls);
  char* t1p = take(t1.bytes);
  L.topk1 = topk_layout(t1p, static_cast<int>(RS), L.Ls);
  L.cand_scores = reinterpret_cast<float*>(take(static_cast<size_t>(R) * L.cap * 4));
  L.cand_tokens = reinterpret_cast<int32_t*>(take(static_cast<size_t>(R) * L.cap * 4));
  L.cand_len = reinterpret_cast<int32_t*>(take(static_cast<size_t>(R) * 4));
  L.pos_idx = reinterpret_cast<int32_t*>(take(static_cast<size_t>(R) * (k > 0 ? k : 1) * 4));
  const TopkLayout t2 = topk_layout(nullptr, R, L.cap);
  char* t2p = take(t2.bytes);
  L.topk2 = topk_layout(t2p, R, L.cap);
  L.bytes = off;
  return L;
}

}  // namespace

size_t topk_sharded_workspace_bytes(int R, int Tmax, int k, int S) {
  return sharded_layout(nullptr, R, Tmax, k, S).bytes;
}

cudaError_t launch_topk_sharded(const float* scores, const int32_t* seq_lens, int B, int Hkv, int Tmax, int lim,
                                int k, int S, int32_t* idx, void* ws, unsigned* err, cudaStream_t stream) {
  const int R = B * Hkv;
  if (R == 0 || k == 0) return cudaSuccess;
  if (static_cast<long long>(R) * S > 65535) return cudaErrorNotSupported;
  const ShardedLayout L = sharded_layout(ws, R, Tmax, k, S);
  cudaError_t e = cudaMemsetAsync(L.bitmap, 0, L.bitmap_bytes, stream);
  if (e != cudaSuccess) return e;
  // 1. shard rows
  {
    const int chunks = (L.Ls + kThreads * 8 - 1) / (kThreads * 8);
    shard_gather_kernel<<<dim3(chunks, R * S), kThreads, 0, stream>>>(scores, seq_lens, Hkv, Tmax, lim, S, L.Ls,
                                                                      L.shard_scores, L.shard_len, err);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 2. local top-k of every shard row (rows as requests of one head)
  {
    TopkArgs a{L.shard_scores, L.shard_len, L.local_idx, err, R * S, 1, L.Ls, L.Ls, k, L.topk1};
    if ((e = launch_topk(a, stream)) != cudaSuccess) return e;
  }
  // 3-4. candidates of each row in global token order
  {
    const int chunks = (k + kThreads - 1) / kThreads;
    mark_kernel<<<dim3(chunks, R * S), kThreads, 0, stream>>>(L.local_idx, k, S, L.words, L.bitmap);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    assemble_kernel<<<R, kThreads, 0, stream>>>(scores, Tmax, L.words, L.cap, L.bitmap, L.cand_scores,
                                                L.cand_tokens, L.cand_len);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // 5. the exact merge: top-k of the candidate rows
  {
    TopkArgs a{L.cand_scores, L.cand_len, L.pos_idx, err, R, 1, L.cap, L.cap, k, L.topk2};
    if ((e = launch_topk(a, stream)) != cudaSuccess) return e;
  }
  // 6. candidate positions -> token indices
  {
    const long long n = static_cast<long long>(R) * k;
    const int blocks = static_cast<int>((n + kThreads - 1) / kThreads < 4096 ? (n + kThreads - 1) / kThreads : 4096);
    map_kernel<<<blocks, kThreads, 0, stream>>>(L.pos_idx, L.cand_tokens, k, L.cap, R, idx);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace ds
