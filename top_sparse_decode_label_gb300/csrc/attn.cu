// Stage 3: sparse GQA decode attention over the selected tokens, gathered
// from a paged bf16 or FP8-E4M3 KV cache.
//
// "Support double sparsity" (sglang PR #1459): attention over the heavy
// tokens only. sglang PR #39721: sparse_gqa over the indexer's selection.
// "QSA HiSparse - SGLang plugin", "Supported versions": FP8 E4M3 KV cache with
// page size 64 (here with one fp32 scale per physical page for K and for V).
// sglang PR #43527, "Distributed QSA execution": owner-side partial outputs,
// merged later by log-sum-exp.
//
// One CTA per (request b, KV head g, split j); 4 warps. Each warp takes tiles
// of 32 selected positions: lane l resolves the slot of position l (index ->
// page table -> slot), then the warp walks the tile in sub-tiles of J tokens.
// A K or V row (D = 128) is read by the whole warp in one coalesced
// instruction (8 B bf16 or 4 B e4m3 per lane: dims 4l..4l+3). The G query
// heads of the group are in registers (4 dims per lane, pre-scaled by
// sm_scale * log2 e), so a lane forms J x G partial dot products; a transposed
// butterfly leaves one finished logit per lane. Online softmax keeps per-head
// running max and sum; P.V accumulates into 4 dims x G heads per lane. At the
// end the warps' states are combined in shared memory (the same log-sum-exp
// merge as stage 4) and the CTA writes either the final bf16 output (one
// split) or fp32 partials.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kWarps = 4;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  const uint16_t* q;
  const uint8_t* kc;
  const uint8_t* vc;
  const float* ks;
  const float* vs;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* idx;
  float* o_part;
  float* lse_part;
  __nv_bfloat16* out;
  float* lse;
  unsigned* err;
  int B, Hq, Hkv, maxp, num_pages, lim, k, S, split_mode, n_known;
  float qscale;  // sm_scale * log2(e)
};

template <int G, bool FP8>
__global__ void __launch_bounds__(kWarps * 32) sparse_attn_kernel(const AttnParams p) {
  constexpr int J = (G >= 4) ? 32 / G : 8;   // tokens per sub-tile
  constexpr int V = J * G;                   // logits per sub-tile (<= 32)
  constexpr int SH = (V >= 32) ? 0 : (V == 16 ? 1 : (V == 8 ? 2 : 3));  // lane -> value shift
  constexpr int NSUB = 32 / J;
  constexpr int ROWB = FP8 ? kHeadDim : kHeadDim * 2;  // bytes per K/V row

  __shared__ float sm_m[kWarps][G];
  __shared__ float sm_l[kWarps][G];
  __shared__ float sm_o[kWarps][G][kHeadDim];
  __shared__ unsigned sh_cnt[kWarps];

  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int j = blockIdx.x % p.S;
  const int bg = blockIdx.x / p.S;
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;
  const int32_t* row = p.idx + static_cast<long long>(bg) * p.k;

  int T = p.seq_lens[b];
  if (T < 0 || T > p.lim) T = T < 0 ? 0 : p.lim;  // flagged by the scoring / top-k stages

  // Number of valid (leading, non-negative) entries of the index row: known
  // from the length when the row comes from the top-k stage, else counted.
  int n;
  if (p.n_known) {
    n = min(p.k, T);
  } else {
    unsigned cnt = 0;
    for (int i = threadIdx.x; i < p.k; i += blockDim.x) cnt += row[i] >= 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if (lane == 0) sh_cnt[warp] = cnt;
    __syncthreads();
    n = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) n += sh_cnt[w];
  }

  int p0, p1;
  if (p.split_mode == 0) {
    p0 = static_cast<int>(static_cast<long long>(j) * n / p.S);
    p1 = static_cast<int>(static_cast<long long>(j + 1) * n / p.S);
  } else {
    p0 = 0;
    p1 = n;
  }

  // Query heads g*G .. g*G+G-1, dims 4*lane .. 4*lane+3, scaled to log2 units.
  float qf[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint2 w = *reinterpret_cast<const uint2*>(p.q + (static_cast<long long>(b) * p.Hq + g * G + h) * kHeadDim + lane * 4);
    qf[h][0] = bf16_lo(w.x) * p.qscale;
    qf[h][1] = bf16_hi(w.x) * p.qscale;
    qf[h][2] = bf16_lo(w.y) * p.qscale;
    qf[h][3] = bf16_hi(w.y) * p.qscale;
  }
  float m[G], o[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    m[h] = -INFINITY;
#pragma unroll
    for (int i = 0; i < 4; ++i) o[h][i] = 0.f;
  }
  float lsum = 0.f;  // running sum of the (token, head) value this lane holds
  const int my_v = lane >> SH;
  const int my_h = my_v % G;
  const int my_j = my_v / G;

  for (int tb = p0 + warp * 32; tb < p1; tb += kWarps * 32) {
    const int pos = tb + lane;
    bool valid = pos < p1;
    int t = valid ? row[pos] : -1;
    valid = valid && t >= 0;
    if (valid && t >= T) {
      flag_error(p.err, 4u);
      valid = false;
    }
    if (valid && p.split_mode == 1 && (t / kPage) % p.S != j) valid = false;
    int pid = 0;
    if (valid) {
      pid = p.page_table[static_cast<long long>(b) * p.maxp + t / kPage];
      if (pid < 0 || pid >= p.num_pages) {
        flag_error(p.err, 2u);
        valid = false;
        pid = 0;
      }
    }
    const long long rowoff = ((static_cast<long long>(pid) * kPage + (t & (kPage - 1))) * p.Hkv + g) * ROWB;
    float kscale = 1.f, vscale = 1.f;
    if (FP8 && valid) {
      kscale = p.ks[pid];
      vscale = p.vs[pid];
    }
    const unsigned vmask = __ballot_sync(kFull, valid);
    if (!vmask) continue;

#pragma unroll 2
    for (int sub = 0; sub < NSUB; ++sub) {
      const unsigned smask = (vmask >> (sub * J)) & ((J == 32) ? kFull : ((1u << J) - 1u));
      if (!smask) continue;
      // Gather J K rows and J V rows, one coalesced warp instruction each.
      uint2 kx[J], vx[J];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        const long long ro = __shfl_sync(kFull, rowoff, sub * J + jj);
        if ((smask >> jj) & 1u) {
          if (FP8) {
            kx[jj].x = ld_nc_na_4(p.kc + ro + lane * 4);
            vx[jj].x = ld_nc_na_4(p.vc + ro + lane * 4);
          } else {
            kx[jj] = ld_nc_na_8(p.kc + ro + lane * 8);
            vx[jj] = ld_nc_na_8(p.vc + ro + lane * 8);
          }
        } else {
          kx[jj] = make_uint2(0u, 0u);
          vx[jj] = make_uint2(0u, 0u);
        }
      }
      float part[V];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        float k0, k1, k2, k3;
        if (FP8) {
          const float2 a = e4m3x2_to_float2(kx[jj].x);
          const float2 c = e4m3x2_to_float2(kx[jj].x >> 16);
          k0 = a.x; k1 = a.y; k2 = c.x; k3 = c.y;
        } else {
          k0 = bf16_lo(kx[jj].x); k1 = bf16_hi(kx[jj].x); k2 = bf16_lo(kx[jj].y); k3 = bf16_hi(kx[jj].y);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          float a = qf[h][0] * k0;
          a = fmaf(qf[h][1], k1, a);
          a = fmaf(qf[h][2], k2, a);
          a = fmaf(qf[h][3], k3, a);
          part[jj * G + h] = a;
        }
      }
      transposed_reduce<32, V>(part);
      // This lane now holds the logit of (token my_j, head my_h) of the sub-tile.
      const int src = sub * J + my_j;
      const bool tv = (smask >> my_j) & 1u;
      const float ksrc = FP8 ? __shfl_sync(kFull, kscale, src) : 1.f;
      float z = tv ? part[0] * ksrc : -INFINITY;
      // Sub-tile max per head: reduce over lanes of other tokens.
      float zm = z;
#pragma unroll
      for (int off = (1 << SH) * G; off < 32; off <<= 1) zm = fmaxf(zm, __shfl_xor_sync(kFull, zm, off));
      float mnew[G], corr[G];
#pragma unroll
      for (int h = 0; h < G; ++h) {
        const float tm = __shfl_sync(kFull, zm, h << SH);
        mnew[h] = fmaxf(m[h], tm);
        corr[h] = (mnew[h] == -INFINITY) ? 1.f : exp2f(m[h] - mnew[h]);
        m[h] = mnew[h];
      }
      float my_m = mnew[0], my_corr = corr[0];
#pragma unroll
      for (int h = 1; h < G; ++h) {
        my_m = (my_h == h) ? mnew[h] : my_m;
        my_corr = (my_h == h) ? corr[h] : my_corr;
      }
      const float pw = (z == -INFINITY) ? 0.f : exp2f(z - my_m);
      lsum = lsum * my_corr + pw;
      const float pv = FP8 ? pw * __shfl_sync(kFull, vscale, src) : pw;
#pragma unroll
      for (int h = 0; h < G; ++h)
#pragma unroll
        for (int i = 0; i < 4; ++i) o[h][i] *= corr[h];
#pragma unroll
      for (int jj = 0; jj < J; ++jj) {
        float v0, v1, v2, v3;
        if (FP8) {
          const float2 a = e4m3x2_to_float2(vx[jj].x);
          const float2 c = e4m3x2_to_float2(vx[jj].x >> 16);
          v0 = a.x; v1 = a.y; v2 = c.x; v3 = c.y;
        } else {
          v0 = bf16_lo(vx[jj].x); v1 = bf16_hi(vx[jj].x); v2 = bf16_lo(vx[jj].y); v3 = bf16_hi(vx[jj].y);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
          const float pj = __shfl_sync(kFull, pv, (jj * G + h) << SH);
          o[h][0] = fmaf(pj, v0, o[h][0]);
          o[h][1] = fmaf(pj, v1, o[h][1]);
          o[h][2] = fmaf(pj, v2, o[h][2]);
          o[h][3] = fmaf(pj, v3, o[h][3]);
        }
      }
    }
  }

  // Per-head sums of this warp: add the lanes of the other tokens.
#pragma unroll
  for (int off = (1 << SH) * G; off < 32; off <<= 1) lsum += __shfl_xor_sync(kFull, lsum, off);
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const float lh = __shfl_sync(kFull, lsum, h << SH);
    if (lane == 0) {
      sm_m[warp][h] = m[h];
      sm_l[warp][h] = lh;
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) sm_o[warp][h][lane * 4 + i] = o[h][i];
  }
  __syncthreads();

  // Combine the warps: the log-sum-exp merge of kWarps partial states.
  for (int e = threadIdx.x; e < G * kHeadDim; e += blockDim.x) {
    const int h = e / kHeadDim;
    const int d = e % kHeadDim;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, sm_m[w][h]);
    float L = 0.f, acc = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < kWarps; ++w) {
        const float c = (sm_m[w][h] == -INFINITY) ? 0.f : exp2f(sm_m[w][h] - M);
        L += c * sm_l[w][h];
        acc += c * sm_o[w][h][d];
      }
    }
    const float val = (L > 0.f) ? acc / L : 0.f;
    const float lse = (L > 0.f) ? (M + log2f(L)) * kLn2 : -INFINITY;
    const long long qrow = static_cast<long long>(b) * p.Hq + g * G + h;
    if (p.S == 1) {
      p.out[qrow * kHeadDim + d] = __float2bfloat16_rn(val);
      if (d == 0 && p.lse) p.lse[qrow] = lse;
    } else {
      const long long prow = static_cast<long long>(j) * p.B * p.Hq + qrow;
      p.o_part[prow * kHeadDim + d] = val;
      if (d == 0) p.lse_part[prow] = lse;
    }
  }
}

using KernelFn = void (*)(const AttnParams);

template <bool FP8>
KernelFn pick(int G) {
  switch (G) {
    case 1: return sparse_attn_kernel<1, FP8>;
    case 2: return sparse_attn_kernel<2, FP8>;
    case 4: return sparse_attn_kernel<4, FP8>;
    case 8: return sparse_attn_kernel<8, FP8>;
  }
  return nullptr;
}

}  // namespace

bool sparse_attn_supported(int G) { return pick<false>(G) != nullptr; }

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  KernelFn fn = a.fp8 ? pick<true>(G) : pick<false>(G);
  if (!fn) return cudaErrorNotSupported;
  const long long blocks = static_cast<long long>(a.B) * a.Hkv * a.S;
  if (blocks == 0) return cudaSuccess;
  AttnParams p;
  p.q = static_cast<const uint16_t*>(a.q);
  p.kc = static_cast<const uint8_t*>(a.k_cache);
  p.vc = static_cast<const uint8_t*>(a.v_cache);
  p.ks = a.k_scale;
  p.vs = a.v_scale;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.idx = a.idx;
  p.o_part = a.o_part;
  p.lse_part = a.lse_part;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.err = a.err;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.maxp = a.maxp;
  p.num_pages = a.num_pages;
  p.lim = a.maxp * kPage < a.Tmax ? a.maxp * kPage : a.Tmax;
  p.k = a.k;
  p.S = a.S;
  p.split_mode = a.split_mode;
  p.qscale = a.sm_scale * kLog2e;
  p.n_known = a.n_from_seq_len;
  fn<<<static_cast<unsigned>(blocks), kWarps * 32, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ds
