// Stage 4: log-sum-exp merge of split-KV partials.
//
// sglang PR #43527 "QSA cache sharding", "Distributed QSA execution":
// owner-side partial outputs are merged with FP32 log-sum-exp normalisation.
//   lse = ln sum_j exp(lse_j),  out = sum_j exp(lse_j - lse) * o_j
// One warp per output row; each lane owns 4 consecutive dims (float4 loads of
// every partial). Chunks with lse_j = -inf weigh nothing; a row whose chunks
// are all empty gets out = 0 and lse = -inf.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kMergeWarps = 8;

__global__ void __launch_bounds__(kMergeWarps * 32)
lse_merge_kernel(int S, int rows, int D, const float* __restrict__ o_part, const float* __restrict__ lse_part,
                 __nv_bfloat16* __restrict__ out, float* __restrict__ lse_out) {
  grid_dependency_wait();
  const int lane = threadIdx.x & 31;
  const long long r = static_cast<long long>(blockIdx.x) * kMergeWarps + (threadIdx.x >> 5);
  if (r >= rows) return;
  float M = -INFINITY;
  for (int s = lane; s < S; s += 32) M = fmaxf(M, lse_part[static_cast<long long>(s) * rows + r]);
#pragma unroll
  for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, o));
  float L = 0.f;
  if (M != -INFINITY)
    for (int s = lane; s < S; s += 32) L += expf(lse_part[static_cast<long long>(s) * rows + r] - M);
#pragma unroll
  for (int o = 16; o; o >>= 1) L += __shfl_xor_sync(kFull, L, o);
  const float lse = (M == -INFINITY) ? -INFINITY : M + logf(L);
  for (int d4 = lane; d4 < D / 4; d4 += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -INFINITY) {
      // Eight splits per step, loads issued before use so they overlap.
      for (int s0 = 0; s0 < S; s0 += 8) {
        float ls[8];
        float4 v[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          ls[i] = -INFINITY;
          if (s0 + i < S) {
            ls[i] = lse_part[static_cast<long long>(s0 + i) * rows + r];
            v[i] = *reinterpret_cast<const float4*>(o_part + (static_cast<long long>(s0 + i) * rows + r) * D + d4 * 4);
          }
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (ls[i] == -INFINITY) continue;
          const float w = expf(ls[i] - lse);
          acc.x = fmaf(w, v[i].x, acc.x);
          acc.y = fmaf(w, v[i].y, acc.y);
          acc.z = fmaf(w, v[i].z, acc.z);
          acc.w = fmaf(w, v[i].w, acc.w);
        }
      }
    }
    __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
    __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
    __nv_bfloat162* dst = reinterpret_cast<__nv_bfloat162*>(out + r * D + d4 * 4);
    dst[0] = lo;
    dst[1] = hi;
  }
  if (lane == 0 && lse_out) lse_out[r] = lse;
}

}  // namespace

cudaError_t launch_lse_merge(int S, int rows, int D, const float* o_part, const float* lse_part, void* out,
                             float* lse, cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const unsigned blocks = static_cast<unsigned>((rows + kMergeWarps - 1) / kMergeWarps);
  cudaError_t e = launch_pdl(lse_merge_kernel, dim3(blocks), dim3(kMergeWarps * 32), 0, stream, S, rows, D, o_part,
                             lse_part, static_cast<__nv_bfloat16*>(out), lse);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
