// Stage 1: proxy scoring of every cached token.
//
// "Support double sparsity" (sglang PR #1459): the query's heavy channels are
// dotted with a label cache that holds, per token and KV head, the same heavy
// channels of K. sglang PR #39721 / #43527: the QSA indexer scans per-token
// index keys and scores them against an index query. Both are
//   s[b, g, t] = sum_{h in group g} sum_c qp[b, h, c] * L[slot(b, t), gL, c]
// with gL = g (per-head label cache, HL = Hkv) or gL = 0 (shared key, HL = 1).
// Because the sum over the group's query heads commutes with the channel sum,
// each lane first adds its group's proxy queries (fp32) and then needs one dot
// product per (token, group).
//
// HBM-bound scan. Each warp instruction reads 512 contiguous bytes of one
// page's label block (16 B per lane, L1 bypassed): C/8 lanes cover one C-wide
// row, so an instruction covers 256/C rows. Rows are ordered (token, head) in
// memory; the warp walks a page either several tokens per instruction (when a
// token's block is shorter than 512 B) or a fixed block of heads of one token
// per instruction (per-head label with many heads). Every lane therefore keeps
// the same (head, channel chunk) for a whole page and holds its slice of the
// summed query in registers. After U instructions the U x NGR partial dot
// products of a lane group are combined by a transposed butterfly.
#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

struct ScoreParams {
  const uint16_t* qp;
  const uint16_t* label;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float* scores;
  unsigned* err;
  int Hq, Hkv, HL, maxp, num_pages, Tmax, nhb;
  long long tasks;  // B * nhb * maxp warp tasks, page fastest
};

// C: proxy width; NGR: groups fed by one label row (1 for a per-head label,
// Hkv for a shared index key); TPI: tokens covered by one warp instruction.
template <int C, int NGR, int TPI>
__global__ void __launch_bounds__(256) index_score_kernel(const ScoreParams p) {
  constexpr int LPR = C / 8;            // lanes per row
  constexpr int RPI = 32 / LPR;         // rows per instruction
  constexpr int HPB = RPI / TPI;        // label heads per instruction
  constexpr int IPP = kPage / TPI;      // instructions per page
  constexpr int U = IPP < 8 ? IPP : 8;  // instructions per batch
  constexpr int V = U * NGR;            // partial sums per lane per batch
  constexpr int PER = V / LPR;          // full sums per lane after the reduction
  static_assert(V >= LPR && V % LPR == 0, "reduction shape");

  const int lane = threadIdx.x & 31;
  const int chunk = lane % LPR;
  const int rin = lane / LPR;
  const int tok_off = rin / HPB;
  const int hin = rin % HPB;
  const int G = p.Hq / p.Hkv;
  const long long wpb = blockDim.x >> 5;
  const long long gw = blockIdx.x * wpb + (threadIdx.x >> 5);
  const long long nw = gridDim.x * wpb;
  const long long t_begin = gw * p.tasks / nw;
  const long long t_end = (gw + 1) * p.tasks / nw;

  long long cur = -1;
  int b = 0, T = 0, hl = 0;
  float q[NGR][8];

  for (long long task = t_begin; task < t_end; ++task) {
    const long long bh = task / p.maxp;
    const int page = static_cast<int>(task - bh * p.maxp);
    if (bh != cur) {
      cur = bh;
      b = static_cast<int>(bh / p.nhb);
      const int hb = static_cast<int>(bh % p.nhb);
      hl = hb * HPB + hin;
      int Tb = p.seq_lens[b];
      const int lim = min(p.Tmax, p.maxp * kPage);
      if (Tb < 0 || Tb > lim) {
        if (lane == 0 && hb == 0 && page == 0) flag_error(p.err, 1u);
        Tb = Tb < 0 ? 0 : lim;
      }
      T = Tb;
      // Summed proxy query of this lane's groups, channels chunk*8 .. chunk*8+7.
#pragma unroll
      for (int n = 0; n < NGR; ++n) {
        const int g = (NGR == 1) ? hl : n;
#pragma unroll
        for (int i = 0; i < 8; ++i) q[n][i] = 0.f;
        for (int h = g * G; h < (g + 1) * G; ++h) {
          const uint4 w = *reinterpret_cast<const uint4*>(p.qp + (static_cast<long long>(b) * p.Hq + h) * C + chunk * 8);
          q[n][0] += bf16_lo(w.x); q[n][1] += bf16_hi(w.x);
          q[n][2] += bf16_lo(w.y); q[n][3] += bf16_hi(w.y);
          q[n][4] += bf16_lo(w.z); q[n][5] += bf16_hi(w.z);
          q[n][6] += bf16_lo(w.w); q[n][7] += bf16_hi(w.w);
        }
      }
    }
    const int tok0 = page * kPage;
    if (tok0 >= T) continue;  // past the request's length: page-table entry is never read
    const int pid = p.page_table[static_cast<long long>(b) * p.maxp + page];
    const bool ok = pid >= 0 && pid < p.num_pages;
    if (!ok && lane == 0) flag_error(p.err, 2u);
    const long long slot0 = static_cast<long long>(ok ? pid : 0) * kPage;

#pragma unroll 1
    for (int ib = 0; ib < IPP; ib += U) {
      uint4 x[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int toff = (ib + u) * TPI + tok_off;
        if (ok && tok0 + toff < T) {
          const long long e = ((slot0 + toff) * p.HL + hl) * C + chunk * 8;
          x[u] = ld_nc_na_16(p.label + e);
        } else {
          x[u] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      float acc[V];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const float f0 = bf16_lo(x[u].x), f1 = bf16_hi(x[u].x), f2 = bf16_lo(x[u].y), f3 = bf16_hi(x[u].y);
        const float f4 = bf16_lo(x[u].z), f5 = bf16_hi(x[u].z), f6 = bf16_lo(x[u].w), f7 = bf16_hi(x[u].w);
#pragma unroll
        for (int n = 0; n < NGR; ++n) {
          float a = q[n][0] * f0;
          a = fmaf(q[n][1], f1, a); a = fmaf(q[n][2], f2, a); a = fmaf(q[n][3], f3, a);
          a = fmaf(q[n][4], f4, a); a = fmaf(q[n][5], f5, a); a = fmaf(q[n][6], f6, a);
          a = fmaf(q[n][7], f7, a);
          acc[u * NGR + n] = a;
        }
      }
      transposed_reduce<LPR, V>(acc);
#pragma unroll
      for (int k = 0; k < PER; ++k) {
        const int v = chunk * PER + k;
        const int u = v / NGR;
        const int n = v % NGR;
        const int t = tok0 + (ib + u) * TPI + tok_off;
        const int g = (NGR == 1) ? hl : n;
        if (t < T)
          p.scores[(static_cast<long long>(b) * p.Hkv + g) * p.Tmax + t] = ok ? acc[k] : __int_as_float(0x7fc00000);
      }
    }
  }
}

using KernelFn = void (*)(const ScoreParams);

template <int C, int NGR>
KernelFn pick_tpi(int tpi) {
  constexpr int RPI = 256 / C;
  switch (tpi) {
    case 1: return index_score_kernel<C, NGR, 1>;
    case 2: if constexpr (RPI >= 2) return index_score_kernel<C, NGR, 2>; break;
    case 4: if constexpr (RPI >= 4) return index_score_kernel<C, NGR, 4>; break;
    case 8: if constexpr (RPI >= 8) return index_score_kernel<C, NGR, 8>; break;
    case 16: if constexpr (RPI >= 16) return index_score_kernel<C, NGR, 16>; break;
  }
  return nullptr;
}

template <int C>
KernelFn pick(int HL, int Hkv) {
  constexpr int RPI = 256 / C;
  if (HL == 1) {
    // Shared key (or a single KV head): one row per token, feeds every group.
    switch (Hkv) {
      case 1: return index_score_kernel<C, 1, RPI>;
      case 2: return index_score_kernel<C, 2, RPI>;
      case 4: return index_score_kernel<C, 4, RPI>;
      case 8: return index_score_kernel<C, 8, RPI>;
    }
    return nullptr;
  }
  if (HL != Hkv) return nullptr;
  // Per-head label: tokens per instruction = RPI / HL when HL divides RPI, else 1.
  if (HL < RPI) {
    if (RPI % HL) return nullptr;
    return pick_tpi<C, 1>(RPI / HL);
  }
  if (HL % RPI) return nullptr;
  return pick_tpi<C, 1>(1);
}

KernelFn select_kernel(int C, int HL, int Hkv) {
  switch (C) {
    case 16: return pick<16>(HL, Hkv);
    case 32: return pick<32>(HL, Hkv);
    case 64: return pick<64>(HL, Hkv);
  }
  return nullptr;
}

}  // namespace

bool index_score_supported(int C, int HL, int Hkv, int G) {
  (void)G;
  return select_kernel(C, HL, Hkv) != nullptr;
}

cudaError_t launch_index_score(const ScoreArgs& a, cudaStream_t stream) {
  KernelFn fn = select_kernel(a.C, a.HL, a.Hkv);
  if (!fn) return cudaErrorNotSupported;
  if (a.B == 0) return cudaSuccess;
  const int rpi = 256 / a.C;
  const int nhb = (a.HL > rpi) ? a.HL / rpi : 1;
  ScoreParams p;
  p.qp = static_cast<const uint16_t*>(a.qp);
  p.label = static_cast<const uint16_t*>(a.label);
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.scores = a.scores;
  p.err = a.err;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.HL = a.HL;
  p.maxp = a.maxp;
  p.num_pages = a.num_pages;
  p.Tmax = a.Tmax;
  p.nhb = nhb;
  p.tasks = static_cast<long long>(a.B) * nhb * a.maxp;
  constexpr int kThreads = 256;
  int per_sm = 0;
  cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kThreads, 0);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  long long want = (p.tasks + (kThreads / 32) - 1) / (kThreads / 32);
  long long blocks = static_cast<long long>(sm_count()) * per_sm;
  if (want < blocks) blocks = want;
  fn<<<static_cast<unsigned>(blocks), kThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ds
