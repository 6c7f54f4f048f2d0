// Stage 1: proxy scoring of every cached token, optionally fused with the
// first radix pass of the exact top-k.
//
// "Support double sparsity" (sglang PR #1459): the query's heavy channels are
// dotted with a label cache that holds, per token and KV head, the same heavy
// channels of K. sglang PR #39721 / #43527: the QSA indexer scans per-token
// index keys and scores them against an index query. Both are
//   s[b, g, t] = sum_{h in group g} sum_c qp[b, h, c] * L[slot(b, t), gL, c]
// with gL = g (per-head label cache, HL = Hkv) or gL = 0 (shared key, HL = 1).
// The sum over the group's query heads commutes with the channel sum, so each
// lane first adds its group's proxy queries (fp32) and then needs one dot
// product per (token, group).
//
// HBM-bound scan. The label cache is cut into 16 KB units: consecutive tokens
// of one request, either whole token rows (HL*C*2 bytes <= 512) or one
// 512-byte block of heads of each token (per-head label with many heads). A
// persistent grid gives each CTA a contiguous range of units; the CTA streams
// them through a ring of cp.async stages (16-byte copies, L1 bypassed, L2
// zero-fill past the request's length), so 64-128 KB per SM are
// in flight without holding registers. Each of the 8 warps then reads 4
// consecutive 512-byte pieces of a unit from shared memory: C/8 lanes hold one
// C-wide row, every lane keeps the same (head, channel chunk) for the whole
// unit, its slice of the summed query sits in registers, and the partial dot
// products of a lane group are combined by a transposed butterfly.
//
// With a top-k to follow, the kernel also builds each row's histogram of the
// top 11 bits of the order-preserving score key in shared memory (two 16-bit
// counters per word), adds it into the row's global histogram when the CTA
// leaves a (request, head block), and the CTA that finishes a (request, head
// block) last turns the histograms into the level-1 threshold bins.
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ds {

namespace {

constexpr int kScoreThreads = 256;
constexpr int kUnitBytes = 16384;               // 32 warp instructions of 512 B
constexpr int kWarps = kScoreThreads / 32;

struct ScoreParams {
  const uint16_t* qp;
  const uint8_t* label;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float* scores;
  unsigned* err;
  int Hq, Hkv, HL, maxp, num_pages, Tmax, nhb, k;
  int units;        // B * nhb * upb (< 2^31, checked on the host)
  int upb;          // units per (request, head block)
  int nst;          // cp.async ring stages
  int hist;         // build level-1 top-k histograms
  TopkWs tw;
};

__device__ __forceinline__ int clamp_len(const ScoreParams& p, int b) {
  const int lim = min(p.Tmax, p.maxp * kPage);
  const int T = __ldg(p.seq_lens + b);
  return T < 0 ? 0 : (T > lim ? lim : T);
}

// Index of the CTA whose unit range holds unit i (ranges [c*U/n, (c+1)*U/n)).
__device__ __forceinline__ int cta_of(long long i, long long units, long long n) {
  return static_cast<int>(((i + 1) * n + units - 1) / units - 1);
}

// C: proxy width; NGR: groups fed by one label row (1 for a per-head label,
// Hkv for a shared index key); TPI: tokens covered by one 512-byte piece.
template <int C, int NGR, int TPI>
__global__ void __launch_bounds__(kScoreThreads) index_score_kernel(const ScoreParams p) {
  constexpr int LPR = C / 8;                    // lanes per C-wide row
  constexpr int RPI = 32 / LPR;                 // rows per 512-byte piece
  constexpr int HPB = RPI / TPI;                // label heads per piece
  constexpr int BR = 512 / TPI;                 // bytes of one token's block
  constexpr int TPU = kUnitBytes / BR;          // tokens per unit
  constexpr int U = kUnitBytes / 512 / kWarps;  // pieces per warp per unit (4)
  constexpr int V = U * NGR;                    // partial sums per lane
  constexpr int PER = V >= LPR ? V / LPR : 1;   // finished sums per lane
  constexpr int RB = (NGR == 1) ? HPB : NGR;    // histogram rows of a (request, head block)
  constexpr int CPT = kUnitBytes / 16 / kScoreThreads;

  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* ring = smem;
  unsigned* hist = reinterpret_cast<unsigned*>(smem + static_cast<size_t>(p.nst) * kUnitBytes);
  __shared__ int sh_last;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int chunk = lane % LPR;
  const int rin = lane / LPR;
  const int tok_off = rin / HPB;
  const int hin = rin % HPB;
  const int G = p.Hq / p.Hkv;
  const int u0 = static_cast<int>(static_cast<long long>(blockIdx.x) * p.units / gridDim.x);
  const int u1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * p.units / gridDim.x);

  if (p.hist)
    for (int i = tid; i < RB * 1024; i += kScoreThreads) hist[i] = 0;

  // Copies unit (bh, ui) into ring stage `stage`.
  auto issue = [&](int bh, int ui, int stage) {
    const int b = (p.nhb == 1) ? bh : bh / p.nhb;
    const int hb = bh - b * p.nhb;
    const int T = clamp_len(p, b);
    const int* pt = p.page_table + b * p.maxp;
    const long long head0 = static_cast<long long>(hb) * HPB * (C * 2);
    unsigned char* dst = ring + stage * kUnitBytes;
#pragma unroll
    for (int c = 0; c < CPT; ++c) {
      const int ch = c * kScoreThreads + tid;
      const int t = ui * TPU + ch / (BR / 16);
      const int byte = (ch % (BR / 16)) * 16;
      bool ok = t < T;
      const uint8_t* src = p.label;
      if (ok) {
        const int pid = __ldg(pt + (t >> 6));
        ok = pid >= 0 && pid < p.num_pages;
        if (ok) {
          const int slot = pid * kPage + (t & (kPage - 1));
          src = p.label + static_cast<long long>(slot) * (p.HL * C * 2) + head0 + byte;
        }
      }
      cp_async16(dst + ch * 16, src, ok);
    }
  };

  int cur = -1;
  int flushed_at = 0;  // unit of the last histogram flush (16-bit counters must not overflow)
  int b = 0, hb = 0, T = 0, hl = 0;
  bool sel = false;
  float q[NGR][8];

  // Adds the CTA's shared histogram of (b, hb) into the global one and clears it.
  auto flush_hist = [&]() {
      for (int i = tid; i < RB * 1024; i += kScoreThreads) {
        const unsigned v = hist[i];
        if (v) {
          const int r = i >> 10;
          const int w = i & 1023;
          const int g = (NGR == 1) ? hb * HPB + r : r;
          unsigned* gh = p.tw.ghist + (static_cast<size_t>(b) * p.Hkv + g) * kBins1 + 2 * w;
          if (v & 0xffffu) atomicAdd(gh, v & 0xffffu);
          if (v >> 16) atomicAdd(gh + 1, v >> 16);
          hist[i] = 0;
        }
      }
  };
  // Leaving (b, hb): flush, count this CTA done for (b, hb), and let the
  // last CTA compute the level-1 thresholds of its rows.
  auto finish = [&]() {
    __syncthreads();
    if (sel) {
      flush_hist();
      __threadfence();
      __syncthreads();
      if (tid == 0) {
        const long long s = static_cast<long long>(cur) * p.upb;
        const int expected = cta_of(s + p.upb - 1, p.units, gridDim.x) - cta_of(s, p.units, gridDim.x) + 1;
        const unsigned prev = atomicAdd(p.tw.done1 + cur, 1u);
        sh_last = (prev + 1 == static_cast<unsigned>(expected));
      }
      __syncthreads();
      if (sh_last) {
        __threadfence();
        for (int r = warp; r < RB; r += kWarps) {
          const int g = (NGR == 1) ? hb * HPB + r : r;
          level1_threshold_warp(p.tw, b * p.Hkv + g, p.k);
        }
        if (tid == 0) atomicExch(p.tw.done1 + cur, 0u);
      }
    }
  };

  // Compute cursor (bh, ui) and issue cursor, advanced without divisions.
  int c_bh = u0 / p.upb;
  int c_ui = u0 - c_bh * p.upb;
  int i_bh = c_bh, i_ui = c_ui;
  for (int s = 0; s < p.nst; ++s) {
    if (u0 + s < u1) {
      issue(i_bh, i_ui, s);
      if (++i_ui == p.upb) { i_ui = 0; ++i_bh; }
    }
    cp_async_commit();
  }

  int stage = 0;
  for (int u = u0; u < u1; ++u) {
    cp_async_wait_dyn(p.nst - 1);
    __syncthreads();
    const int bh = c_bh;
    if (bh != cur) {
      if (cur >= 0 && p.hist) finish();
      cur = bh;
      flushed_at = u;
      b = (p.nhb == 1) ? bh : bh / p.nhb;
      hb = bh - b * p.nhb;
      hl = hb * HPB + hin;
      T = clamp_len(p, b);
      sel = p.hist && needs_selection(p.k, T);
      if (tid == 0 && hb == 0 && c_ui == 0) {
        const int raw = __ldg(p.seq_lens + b);
        if (raw < 0 || raw > min(p.Tmax, p.maxp * kPage)) flag_error(p.err, 1u);
      }
#pragma unroll
      for (int n = 0; n < NGR; ++n) {
        const int g = (NGR == 1) ? hl : n;
#pragma unroll
        for (int i = 0; i < 8; ++i) q[n][i] = 0.f;
        for (int h = g * G; h < (g + 1) * G; ++h) {
          const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.qp + (static_cast<long long>(b) * p.Hq + h) * C + chunk * 8));
          q[n][0] += bf16_lo(w.x); q[n][1] += bf16_hi(w.x);
          q[n][2] += bf16_lo(w.y); q[n][3] += bf16_hi(w.y);
          q[n][4] += bf16_lo(w.z); q[n][5] += bf16_hi(w.z);
          q[n][6] += bf16_lo(w.w); q[n][7] += bf16_hi(w.w);
        }
      }
    }
    if (sel && (u - flushed_at) * TPU > 60000) {
      flush_hist();
      __syncthreads();
      flushed_at = u;
    }

    // ---- dot products of this unit
    const int tbase = c_ui * TPU;
    if (tbase < T) {
      const unsigned char* src = ring + stage * kUnitBytes + (warp * U) * 512 + lane * 16;
      float acc[V];
#pragma unroll
      for (int uu = 0; uu < U; ++uu) {
        const uint4 x = *reinterpret_cast<const uint4*>(src + uu * 512);
        const float f0 = bf16_lo(x.x), f1 = bf16_hi(x.x), f2 = bf16_lo(x.y), f3 = bf16_hi(x.y);
        const float f4 = bf16_lo(x.z), f5 = bf16_hi(x.z), f6 = bf16_lo(x.w), f7 = bf16_hi(x.w);
#pragma unroll
        for (int n = 0; n < NGR; ++n) {
          float a = q[n][0] * f0;
          a = fmaf(q[n][1], f1, a); a = fmaf(q[n][2], f2, a); a = fmaf(q[n][3], f3, a);
          a = fmaf(q[n][4], f4, a); a = fmaf(q[n][5], f5, a); a = fmaf(q[n][6], f6, a);
          a = fmaf(q[n][7], f7, a);
          acc[uu * NGR + n] = a;
        }
      }
      transposed_reduce<LPR, V>(acc);
#pragma unroll
      for (int kk = 0; kk < PER; ++kk) {
        const int v = (V >= LPR) ? chunk * PER + kk : (chunk * V) / LPR;
        const bool writer = (V >= LPR) || ((chunk * V) % LPR == 0);
        const int uu = v / NGR;
        const int n = v % NGR;
        const int t = tbase + (warp * U + uu) * TPI + tok_off;
        const int g = (NGR == 1) ? hl : n;
        if (writer && t < T) {
          float sc = acc[kk];
          const int pid = __ldg(p.page_table + b * p.maxp + (t >> 6));
          if (pid < 0 || pid >= p.num_pages) {
            sc = __int_as_float(0x7fc00000);
            flag_error(p.err, 2u);
          }
          p.scores[(static_cast<long long>(b) * p.Hkv + g) * p.Tmax + t] = sc;
          if (sel) {
            const unsigned bin = order_key(sc) >> 21;
            const int r = (NGR == 1) ? hin : n;
            atomicAdd(hist + r * 1024 + (bin >> 1), 1u << ((bin & 1u) << 4));
          }
        }
      }
    }
    __syncthreads();
    if (u + p.nst < u1) {
      issue(i_bh, i_ui, stage);
      if (++i_ui == p.upb) { i_ui = 0; ++i_bh; }
    }
    cp_async_commit();
    if (++c_ui == p.upb) { c_ui = 0; ++c_bh; }
    if (++stage == p.nst) stage = 0;
  }
  if (cur >= 0 && p.hist) finish();
  cp_async_wait<0>();
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
KernelFn pick(int HL, int Hkv, int* tpi_out) {
  constexpr int RPI = 256 / C;
  if (HL == 1) {
    // Shared key (or a single KV head): one row per token, feeds every group.
    *tpi_out = RPI;
    switch (Hkv) {
      case 1: return index_score_kernel<C, 1, RPI>;
      case 2: return index_score_kernel<C, 2, RPI>;
      case 4: return index_score_kernel<C, 4, RPI>;
      case 8: return index_score_kernel<C, 8, RPI>;
    }
    return nullptr;
  }
  if (HL != Hkv) return nullptr;
  // Per-head label: tokens per piece = RPI / HL when HL divides RPI, else 1.
  if (HL < RPI) {
    if (RPI % HL) return nullptr;
    *tpi_out = RPI / HL;
    return pick_tpi<C, 1>(RPI / HL);
  }
  if (HL % RPI) return nullptr;
  *tpi_out = 1;
  return pick_tpi<C, 1>(1);
}

KernelFn select_kernel(int C, int HL, int Hkv, int* tpi) {
  switch (C) {
    case 16: return pick<16>(HL, Hkv, tpi);
    case 32: return pick<32>(HL, Hkv, tpi);
    case 64: return pick<64>(HL, Hkv, tpi);
  }
  return nullptr;
}

// Sets the dynamic shared memory limit of a kernel once per (kernel, size) per device.
cudaError_t allow_smem(KernelFn fn, int bytes) {
  struct Entry { KernelFn fn; int dev; int bytes; };
  static Entry done[256];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < n; ++i)
    if (done[i].fn == fn && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < 256) done[n++] = Entry{fn, dev, bytes};
  return e;
}

}  // namespace

bool index_score_supported(int C, int HL, int Hkv, int G) {
  (void)G;
  int tpi = 0;
  return select_kernel(C, HL, Hkv, &tpi) != nullptr;
}

cudaError_t launch_index_score(const ScoreArgs& a, cudaStream_t stream) {
  int tpi = 0;
  KernelFn fn = select_kernel(a.C, a.HL, a.Hkv, &tpi);
  if (!fn) return cudaErrorNotSupported;
  if (a.B == 0 || a.Tmax == 0) return cudaSuccess;
  const int rpi = 256 / a.C;
  const int hpb = rpi / tpi;
  const int nhb = (a.HL > rpi) ? a.HL / rpi : 1;
  const int tpu = kUnitBytes / (512 / tpi);
  const int rb = (a.HL == 1) ? a.Hkv : hpb;
  ScoreParams p{};
  p.qp = static_cast<const uint16_t*>(a.qp);
  p.label = static_cast<const uint8_t*>(a.label);
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
  p.k = a.k;
  const long long upb = (static_cast<long long>(a.maxp) * kPage + tpu - 1) / tpu;
  const long long units = static_cast<long long>(a.B) * nhb * upb;
  if (units >= (1LL << 31) || static_cast<long long>(a.B) * a.maxp >= (1LL << 31)) return cudaErrorNotSupported;
  p.upb = static_cast<int>(upb);
  p.units = static_cast<int>(units);
  p.hist = a.topk != nullptr;
  if (p.hist) p.tw = topk_ws_view(*a.topk);
  const int hist_bytes = p.hist ? rb * 4096 : 0;
  // Two CTAs per SM when the histogram is small, else one with a deeper ring.
  int nst = (104 * 1024 - hist_bytes) / kUnitBytes;
  if (nst < 4) nst = (220 * 1024 - hist_bytes) / kUnitBytes;
  if (nst > 8) nst = 8;
  if (nst < 2) return cudaErrorNotSupported;
  p.nst = nst;
  const int smem = nst * kUnitBytes + hist_bytes;
  cudaError_t e = allow_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kScoreThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  long long blocks = static_cast<long long>(sm_count()) * per_sm;
  if (p.units < blocks) blocks = p.units;
  fn<<<static_cast<unsigned>(blocks), kScoreThreads, smem, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace ds
