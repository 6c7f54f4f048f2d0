// Block-compressed QSA selection: the compressed index cache and the
// block-level selection that precedes the sparse attention.
//
// sglang PR #43527 "QSA cache sharding", "Summary": the sequence-dependent
// QSA state has a raw K/V history and a compressed cache; its review thread
// has the global merge choose "512 of 1024 blocks". The pages do not say how
// a block's key is formed from its tokens. Readings taken here:
//   - a block is one 64-token KV page of a request (block j covers logical
//     tokens [64j, 64j + 64) below the sequence length);
//   - its compressed key is the per-channel mean of its tokens' index keys:
//     their sum in double in token order, divided by the number of tokens
//     present, rounded to the nearest bf16 (ties to even), stored at the
//     page's physical id;
//   - a block is scored like a token, with its compressed key; the top-k
//     blocks of each (request, KV head) are kept with the exact top-k rule
//     (ties to the lower block index), and the attention runs over every
//     token of the kept blocks below the sequence length.
//
// Kernels (each on the caller's stream, programmatic dependent launch):
//   block_compress_kernel  one warp per (request, logical page)
//   block_score_kernel     one thread per (request, block), every KV head
//   block_expand_kernel    kept blocks -> ascending token indices, -1 padded
// The block top-k is the cluster top-k of the token path on rows of block
// scores.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

// Nearest bf16 to a double, ties to even, in one rounding: round to odd into
// float (keep the truncated value and make its last bit sticky when anything
// was dropped), then CUDA's float -> bf16 rounding to nearest even. Float has
// 24 significant bits against bf16's 8, and the same exponent range, so the
// odd intermediate cannot create a false tie.
__device__ __forceinline__ uint16_t bf16_from_double(double x) {
  float f = __double2float_rz(x);
  if (static_cast<double>(f) != x) f = __uint_as_float(__float_as_uint(f) | 1u);
  return __bfloat16_as_ushort(__float2bfloat16_rn(f));
}

// grid (max_pages, B), 32 threads: warp (j, b) writes the key of logical page j
// of request b (only the last page of each request when last_only).
__global__ void __launch_bounds__(32) block_compress_kernel(const uint16_t* keys, const int32_t* page_table,
                                                            const int32_t* seq_lens, int C, int maxp, int num_pages,
                                                            int last_only, uint16_t* block_keys, unsigned* err) {
  const int j = blockIdx.x, b = blockIdx.y, lane = threadIdx.x;
  grid_dependency_wait();
  grid_launch_dependents();
  int T = seq_lens[b];
  if (T < 0 || T > maxp * kPage) {
    if (lane == 0 && j == 0) flag_error(err, 1u);
    return;
  }
  const int nb = (T + kPage - 1) / kPage;
  if (j >= nb || (last_only && j != nb - 1)) return;
  const int pid = page_table[static_cast<long long>(b) * maxp + j];
  if (pid < 0 || pid >= num_pages) {
    if (lane == 0) flag_error(err, 2u);
    return;
  }
  const int t0 = j * kPage, n = min(T, t0 + kPage) - t0;
  // Lane l holds channels 2l and 2l + 1 (one 32-bit word of each key row).
  const int c = 2 * lane;
  if (c >= C) return;
  const uint32_t* rows = reinterpret_cast<const uint32_t*>(keys + static_cast<long long>(pid) * kPage * C) + lane;
  // Rows in batches of 16 loads in flight; the sums stay in token order.
  double s0 = 0.0, s1 = 0.0;
  for (int t0b = 0; t0b < n; t0b += 16) {
    uint32_t w[16];
#pragma unroll
    for (int u = 0; u < 16; ++u) w[u] = t0b + u < n ? __ldg(rows + static_cast<long long>(t0b + u) * (C / 2)) : 0u;
#pragma unroll
    for (int u = 0; u < 16; ++u) {
      if (t0b + u < n) {
        s0 += static_cast<double>(bf16_lo(w[u]));
        s1 += static_cast<double>(bf16_hi(w[u]));
      }
    }
  }
  const uint32_t lo = bf16_from_double(__ddiv_rn(s0, static_cast<double>(n)));
  const uint32_t hi = bf16_from_double(__ddiv_rn(s1, static_cast<double>(n)));
  reinterpret_cast<uint32_t*>(block_keys + static_cast<long long>(pid) * C)[lane] = lo | (hi << 16);
}

// grid (ceil(maxp / 128), B), 128 threads (lim: the largest valid sequence
// length): thread (x, b) scores block
// j = 128 x + threadIdx.x of request b for every KV head g,
//   s[b, g, j] = sum_c (sum_{h in g} qp[b, h, c]) * K_blk[pid(b, j), c],
// and CTA (0, b) writes the request's block count.
template <int C>
__global__ void __launch_bounds__(128) block_score_kernel(const uint16_t* qp, const uint16_t* block_keys,
                                                          const int32_t* page_table, const int32_t* seq_lens, int Hq,
                                                          int Hkv, int maxp, int num_pages, int lim, float* scores,
                                                          int32_t* nblocks, unsigned* err) {
  extern __shared__ float qg[];   // [Hkv][C] group queries
  const int b = blockIdx.y;
  const int G = Hq / Hkv;
  grid_dependency_wait();   // the queries and keys may come from the previous kernel
  grid_launch_dependents();
  for (int i = threadIdx.x; i < Hkv * C; i += blockDim.x) {
    const int g = i / C, c = i - g * C;
    float q = 0.f;
    for (int h = g * G; h < (g + 1) * G; ++h) q += bf16_lo(__ldg(qp + (static_cast<long long>(b) * Hq + h) * C + c));
    qg[i] = q;
  }
  __syncthreads();
  int T = seq_lens[b];
  if (T < 0 || T > lim) {
    if (blockIdx.x == 0 && threadIdx.x == 0) flag_error(err, 1u);
    T = T < 0 ? 0 : lim;
  }
  const int nb = (T + kPage - 1) / kPage;
  if (blockIdx.x == 0 && threadIdx.x == 0) nblocks[b] = nb;
  const int j = blockIdx.x * blockDim.x + threadIdx.x;
  if (j >= nb) return;
  const int pid = page_table[static_cast<long long>(b) * maxp + j];
  float* out = scores + static_cast<long long>(b) * Hkv * maxp + j;
  if (pid < 0 || pid >= num_pages) {
    flag_error(err, 2u);
    for (int g = 0; g < Hkv; ++g) out[static_cast<long long>(g) * maxp] = -INFINITY;
    return;
  }
  uint32_t kw[C / 2];
  const uint4* kr = reinterpret_cast<const uint4*>(block_keys + static_cast<long long>(pid) * C);
#pragma unroll
  for (int v = 0; v < C / 8; ++v) {
    const uint4 x = __ldg(kr + v);
    kw[4 * v] = x.x;
    kw[4 * v + 1] = x.y;
    kw[4 * v + 2] = x.z;
    kw[4 * v + 3] = x.w;
  }
  for (int g = 0; g < Hkv; ++g) {
    const float* q = qg + g * C;
    float s = 0.f;
#pragma unroll
    for (int w = 0; w < C / 2; ++w) {
      s = fmaf(q[2 * w], bf16_lo(kw[w]), s);
      s = fmaf(q[2 * w + 1], bf16_hi(kw[w]), s);
    }
    out[static_cast<long long>(g) * maxp] = s;
  }
}

// grid (B * Hkv), 256 threads: position i of row (b, g) is token
// 64 * blocks[i / 64] + i % 64 when that block was kept and the token lies
// below the sequence length, else -1. Kept blocks ascend and only the last
// block of a request can be partial, so the valid positions form a prefix.
__global__ void __launch_bounds__(256) block_expand_kernel(const int32_t* blocks, const int32_t* seq_lens, int Hkv,
                                                           int kb, int lim, int32_t* idx) {
  const int row = blockIdx.x;
  grid_dependency_wait();
  grid_launch_dependents();
  int T = seq_lens[row / Hkv];
  T = T < 0 ? 0 : (T > lim ? lim : T);
  const int32_t* blk = blocks + static_cast<long long>(row) * kb;
  int32_t* out = idx + static_cast<long long>(row) * kb * kPage;
  for (int i = threadIdx.x; i < kb * kPage; i += blockDim.x) {
    const int bj = blk[i / kPage];
    const int t = bj * kPage + (i % kPage);
    out[i] = (bj >= 0 && t < T) ? t : -1;
  }
}

}  // namespace

cudaError_t launch_block_compress(const void* keys, const int32_t* page_table, const int32_t* seq_lens, int B,
                                  int C, int maxp, int num_pages, int last_only, void* block_keys, unsigned* err,
                                  cudaStream_t stream) {
  if (B == 0 || maxp == 0) return cudaSuccess;
  if (B > 65535 || (C != 16 && C != 32 && C != 64)) return cudaErrorNotSupported;
  return launch_pdl(block_compress_kernel, dim3(static_cast<unsigned>(maxp), static_cast<unsigned>(B)), dim3(32), 0,
                    stream, static_cast<const uint16_t*>(keys), page_table, seq_lens, C, maxp, num_pages, last_only,
                    static_cast<uint16_t*>(block_keys), err);
}

cudaError_t launch_block_score(const void* qp, const void* block_keys, const int32_t* page_table,
                               const int32_t* seq_lens, int B, int Hq, int Hkv, int C, int maxp, int num_pages,
                               int lim, float* scores, int32_t* nblocks, unsigned* err, cudaStream_t stream) {
  if (B == 0) return cudaSuccess;
  if (B > 65535 || Hkv <= 0 || Hq % Hkv) return cudaErrorNotSupported;
  const size_t smem = static_cast<size_t>(Hkv) * C * 4;
  if (smem > 48 * 1024) return cudaErrorNotSupported;
  const dim3 grid(static_cast<unsigned>((maxp + 127) / 128 > 0 ? (maxp + 127) / 128 : 1), static_cast<unsigned>(B));
  const uint16_t* q = static_cast<const uint16_t*>(qp);
  const uint16_t* k = static_cast<const uint16_t*>(block_keys);
  switch (C) {
    case 16:
      return launch_pdl(block_score_kernel<16>, grid, dim3(128), smem, stream, q, k, page_table, seq_lens, Hq, Hkv,
                        maxp, num_pages, lim, scores, nblocks, err);
    case 32:
      return launch_pdl(block_score_kernel<32>, grid, dim3(128), smem, stream, q, k, page_table, seq_lens, Hq, Hkv,
                        maxp, num_pages, lim, scores, nblocks, err);
    case 64:
      return launch_pdl(block_score_kernel<64>, grid, dim3(128), smem, stream, q, k, page_table, seq_lens, Hq, Hkv,
                        maxp, num_pages, lim, scores, nblocks, err);
  }
  return cudaErrorNotSupported;
}

cudaError_t launch_block_expand(const int32_t* blocks, const int32_t* seq_lens, int B, int Hkv, int kb, int lim,
                                int32_t* idx, cudaStream_t stream) {
  if (B == 0 || kb == 0) return cudaSuccess;
  return launch_pdl(block_expand_kernel, dim3(static_cast<unsigned>(B * Hkv)), dim3(256), 0, stream, blocks, seq_lens,
                    Hkv, kb, lim, idx);
}

}  // namespace ds
