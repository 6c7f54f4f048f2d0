// The step before the path: append each request's new token to the caches.
//
// "Support double sparsity" (sglang PR #1459), review thread: the label cache
// of a token is the per-head gather of its K at the heavy channels (a
// torch.gather over [tokens, heads, channels]). "QSA HiSparse - SGLang
// plugin", "Supported versions": FP8 E4M3 KV cache with page size 64. sglang
// PR #39721: the indexer's raw index keys are stored per token.
//
// For request b, the token at logical position t = positions[b] goes to slot
// page_table[b][t / 64] * 64 + t % 64: its K and V rows (bf16 copied; e4m3 as
// the fp32 quotient by the page's scale rounded to nearest even and
// saturated to +-448) and its label row -- K[g, channels[g, c]] per KV head,
// or the given index key. One CTA of 128 threads per (request, KV head). A negative position skips the request; a position
// past the page table, a page id outside the pool or a channel outside
// [0, 128) is skipped and flagged in the device error word.
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

struct AppendParams {
  const uint16_t* k_new;     // bf16 [B, Hkv, 128]
  const uint16_t* v_new;
  void* kc;                  // [slots, Hkv, 128] bf16 or e4m3
  void* vc;
  const float* ks;           // [num_pages] (e4m3)
  const float* vs;
  const int32_t* page_table; // [B, maxp]
  const int32_t* positions;  // [B]
  const int32_t* channels;   // [Hkv, C] or null
  const uint16_t* index_key; // [B, C] or null
  uint16_t* label;           // [slots, HL, C] or null
  unsigned* err;
  int Hkv, maxp, num_pages, fp8, HL, C, D;
};

constexpr int kAppendThreads = 128;

__global__ void __launch_bounds__(kAppendThreads) cache_append_kernel(const AppendParams p) {
  const int b = blockIdx.x;
  const int g = blockIdx.y;
  const int tid = threadIdx.x;
  const int t = __ldg(p.positions + b);
  if (t < 0) return;
  if (t >= p.maxp * kPage) {
    if (tid == 0 && g == 0) flag_error(p.err, 1u);
    return;
  }
  const int pid = __ldg(p.page_table + static_cast<long long>(b) * p.maxp + (t >> 6));
  if (pid < 0 || pid >= p.num_pages) {
    if (tid == 0 && g == 0) flag_error(p.err, 2u);
    return;
  }
  const long long slot = static_cast<long long>(pid) * kPage + (t & (kPage - 1));
  for (int d = tid; d < p.D; d += kAppendThreads) {
    const long long src = (static_cast<long long>(b) * p.Hkv + g) * p.D + d;
    const long long dst = (slot * p.Hkv + g) * p.D + d;
    const uint16_t kb = __ldg(p.k_new + src), vb = __ldg(p.v_new + src);
    if (p.fp8) {
      const float kq = __fdiv_rn(__uint_as_float(static_cast<uint32_t>(kb) << 16), __ldg(p.ks + pid));
      const float vq = __fdiv_rn(__uint_as_float(static_cast<uint32_t>(vb) << 16), __ldg(p.vs + pid));
      static_cast<uint8_t*>(p.kc)[dst] = __nv_cvt_float_to_fp8(kq, __NV_SATFINITE, __NV_E4M3);
      static_cast<uint8_t*>(p.vc)[dst] = __nv_cvt_float_to_fp8(vq, __NV_SATFINITE, __NV_E4M3);
    } else {
      static_cast<uint16_t*>(p.kc)[dst] = kb;
      static_cast<uint16_t*>(p.vc)[dst] = vb;
    }
  }
  // Label row of this KV head (a shared index key: written by head 0's CTA).
  if (!p.label || g >= p.HL) return;
  for (int c = tid; c < p.C; c += kAppendThreads) {
    uint16_t v;
    if (p.channels) {
      const int ch = __ldg(p.channels + g * p.C + c);
      if (ch < 0 || ch >= p.D) {
        flag_error(p.err, 16u);
        continue;
      }
      v = __ldg(p.k_new + (static_cast<long long>(b) * p.Hkv + g) * p.D + ch);
    } else {
      v = __ldg(p.index_key + static_cast<long long>(b) * p.C + c);
    }
    p.label[(slot * p.HL + g) * p.C + c] = v;
  }
}

}  // namespace

cudaError_t launch_cache_append(const AppendArgs& a, cudaStream_t stream) {
  if (a.B == 0) return cudaSuccess;
  AppendParams p{};
  p.k_new = static_cast<const uint16_t*>(a.k_new);
  p.v_new = static_cast<const uint16_t*>(a.v_new);
  p.kc = a.k_cache;
  p.vc = a.v_cache;
  p.ks = a.k_scale;
  p.vs = a.v_scale;
  p.page_table = a.page_table;
  p.positions = a.positions;
  p.channels = a.channels;
  p.index_key = static_cast<const uint16_t*>(a.index_key);
  p.label = static_cast<uint16_t*>(a.label);
  p.err = a.err;
  p.Hkv = a.Hkv;
  p.maxp = a.maxp;
  p.num_pages = a.num_pages;
  p.fp8 = a.fp8;
  p.HL = a.HL;
  p.C = a.C;
  p.D = a.D;
  if (a.Hkv > 65535) return cudaErrorNotSupported;
  cache_append_kernel<<<dim3(a.B, a.Hkv), kAppendThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ds
