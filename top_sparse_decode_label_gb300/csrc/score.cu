// Stage 1: proxy scoring of every cached token.
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
// HBM-bound scan. The label rows are read once, with an evict-first L2
// policy; the scores are written with an evict-last one, so that the top-k
// after the scan reads them from L2. The label cache is cut into 16 KB units
// of whole token rows (HL*C*2 bytes each) of one request; only units that
// hold tokens of a sequence count. A persistent grid splits them evenly: CTA
// c takes a contiguous range of them in request order (a shared counter with
// dynamic claims was measured slower: its returning atomics queue at one L2
// address). In each CTA a producer warp loads the page ids of a chunk's pages
// together, a chunk before they are needed, and streams the units into a
// ring of shared-memory stages with bulk copies -- one per page span -- that
// complete on the stage's mbarrier; eight consumer warps wait on it, read it
// into registers, release it through a second mbarrier and then compute, so
// copies run ahead by the ring depth with no CTA-wide barrier per unit; each
// stage carries its unit's request and index, and a stage marked -1 ends the
// consumers.
//
// CUDA-core consumers: each warp reads 4 consecutive 512-byte pieces of a
// unit; C/8 lanes hold one C-wide row (one head of one token), every lane
// keeps the same (head block, channel chunk) for the whole unit, its slices of
// the summed queries sit in registers, packed fp32 FMAs form the partial dot
// products, and a transposed butterfly combines them across the row's lanes.
//
// Tensor-core consumers (shared 64-wide index keys): the producer copies
// whole 64-token pages with tiled tensor copies that swizzle 16-byte chunks
// by row, each consumer warp forms the scores of 16 tokens for every group
// with ldmatrix and mma.sync (bf16 in, fp32 accumulate) against the group
// queries held in registers. These warps also write the largest score of
// each 16-token block per group (three shuffles over the fragment rows), from
// which the top-k bounds its threshold without reading every score. Every
// mbarrier wait is bounded: on timeout it sets DS_DEVERR_TIMEOUT and carries
// on.

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kScoreThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kUnitBytes = 16384;                     // 32 pieces of 512 B
constexpr int kMaxStages = 12;
constexpr uint32_t kWaitLimit = 1u << 22;             // bounded mbarrier polls
constexpr int kChunkUnits = 4;                        // units whose page ids are loaded together

struct ScoreParams {
  CUtensorMap tmap;   // tensor-core path: the key cache as [slots, 64] bf16 rows, 64 x 64 boxes, 128-byte swizzle
  const uint16_t* qp;
  const uint8_t* label;
  const int32_t* page_table;
  const int32_t* seq_lens;
  float* scores;
  unsigned* err;
  int B, Hq, Hkv, HL, maxp, num_pages, Tmax;
  int nst;          // ring stages
  float* bmax;      // tensor-core path: [B, Hkv, nbr] maxima of 16-token blocks, or null
  int nbr;          // blocks per row of bmax: ceil(Tmax / 16)
};

__device__ __forceinline__ int clamp_len(const ScoreParams& p, int b) {
  const int lim = min(p.Tmax, p.maxp * kPage);
  const int T = __ldg(p.seq_lens + b);
  return T < 0 ? 0 : (T > lim ? lim : T);
}

// C: proxy width; NGR: groups fed by one label row (1 for a per-head label,
// Hkv for a shared index key); TPI: tokens covered by one 512-byte piece.
template <int C, int NGR, int TPI, int PPT, bool MMA>
__global__ void __launch_bounds__(kScoreThreads, (NGR >= 8 && !MMA) ? 1 : 2)
    index_score_kernel(const __grid_constant__ ScoreParams p) {
  static_assert(!MMA || (C == 64 && TPI == 4 && PPT == 1), "tensor-core path: shared 64-wide keys");
  static_assert(PPT == 1 || (TPI == 1 && NGR == 1), "several pieces per token only for a per-head label");
  constexpr int LPR = C / 8;                             // lanes per C-wide row
  constexpr int RPI = 32 / LPR;                          // rows per 512-byte piece
  constexpr int HPB = RPI / TPI;                         // label heads per piece
  constexpr int BR = 512 * PPT / TPI;                    // bytes of one token's label row
  constexpr int TPU = kUnitBytes / BR;                   // tokens per unit
  constexpr int U = kUnitBytes / 512 / kConsumerWarps;   // pieces per consumer warp per unit (4)
  constexpr int V = U * NGR;                             // partial sums per lane
  constexpr int PER = V >= LPR ? V / LPR : 1;            // finished sums per lane
  constexpr int NQ = NGR > 1 ? NGR : (PPT < U ? PPT : U);  // query register sets per lane

  extern __shared__ __align__(128) unsigned char smem[];
  // Ring of stages. The tensor-core path aligns it to 1024 bytes for the
  // 128-byte swizzle of its tensor copies (its launch adds 1 KB for that).
  unsigned char* ring = MMA ? smem + ((1024u - (smem_u32(smem) & 1023u)) & 1023u) : smem;
  __shared__ __align__(8) uint64_t full_bar[kMaxStages];
  __shared__ __align__(8) uint64_t empty_bar[kMaxStages];
  __shared__ int stage_unit[kMaxStages];   // unit held by each ring stage, -1: no more units
  __shared__ int stage_req[kMaxStages];    // and its request (the producer's quotient, for the consumers)

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;

  if (tid == 0) {
    for (int s = 0; s < p.nst; ++s) {
      mbar_init(&full_bar[s], 1);
      mbar_init(&empty_bar[s], kConsumerWarps);
    }
    mbar_fence_init();
  }
  __syncthreads();
  grid_dependency_wait();
  grid_launch_dependents();

  // The label rows stream through once and go first from L2; the scores and
  // block maxima stay there for the top-k, which reads them next.
  const uint64_t stream_pol = l2_evict_first();
  const uint64_t keep_pol = l2_evict_last();
  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer warp
    // The work is the valid units of all requests in request order (a
    // request of T tokens has ceil(T / TPU) of them) and this CTA takes an
    // equal contiguous share: no global counter, no units past a sequence.
    // The units come in chunks of kChunkUnits; the page ids of a chunk's
    // pages are loaded together, one lane per page, a chunk before the chunk
    // is copied, so no global round trip sits on the per-unit path.
    constexpr int PPU = TPU >= kPage ? TPU / kPage : 1;   // pages per unit
    static_assert(PPU * kChunkUnits <= 32, "one lane per page of a chunk");
    // upre[b]: valid units of the requests before b (upre[B]: all of them);
    // ulen[b]: request b's length, clamped.
    int* upre = reinterpret_cast<int*>(smem + p.nst * kUnitBytes + (MMA ? 1024 : 0));
    int* ulen = upre + p.B + 1;
    int carry = 0;
    for (int b0 = 0; b0 < p.B; b0 += 32) {
      const int rb = b0 + lane;
      const int T = rb < p.B ? clamp_len(p, rb) : 0;
      const int nv = (T + TPU - 1) / TPU;
      const int inc = static_cast<int>(warp_incl_scan(static_cast<unsigned>(nv)));
      if (rb < p.B) {
        upre[rb] = carry + inc - nv;
        ulen[rb] = T;
      }
      carry += __shfl_sync(kFull, inc, 31);
    }
    if (lane == 0) upre[p.B] = carry;
    __syncwarp();
    const int v0 = static_cast<int>(static_cast<long long>(blockIdx.x) * carry / gridDim.x);
    const int v1 = static_cast<int>(static_cast<long long>(blockIdx.x + 1) * carry / gridDim.x);
    // Lane l's unit of chunk [a, e) is a + l / PPU: its request rb (the last
    // one with upre[rb] <= unit), its index rui in the request and the id of
    // its page l % PPU (-1 past the sequence or the chunk).
    auto load_chunk = [&](int a, int e, int& rb, int& rui) -> int {
      const int v = a + lane / PPU;
      int pid = -1;
      rb = 0;
      rui = 0;
      if (v < e) {
        int lo = 0, hi = p.B - 1;
        while (lo < hi) {
          const int mid = (lo + hi + 1) >> 1;
          if (upre[mid] <= v) lo = mid;
          else hi = mid - 1;
        }
        rb = lo;
        rui = v - upre[lo];
        const int pg = ((rui * TPU) >> 6) + lane % PPU;
        if (pg * kPage < ulen[lo]) pid = __ldg(p.page_table + static_cast<long long>(lo) * p.maxp + pg);
      }
      return pid;
    };
    int cu = v0, ce = min(v1, v0 + kChunkUnits);
    int cb, cui, nb, nui;
    int cpid = load_chunk(cu, ce, cb, cui);
    int na = ce, ne = min(v1, na + kChunkUnits);
    int npid = load_chunk(na, ne, nb, nui);
    int ca = cu;          // first unit of the current chunk
    int s = 0;
    uint32_t fill = 0;  // how many times stage s has been filled before
    for (;;) {
      if (cu >= ce && na < ne) {
        // Next chunk: its page ids were loaded a chunk ago; start loading the
        // one after it.
        cu = na;
        ce = ne;
        ca = cu;
        cpid = npid;
        cb = nb;
        cui = nui;
        na = ce;
        ne = min(v1, na + kChunkUnits);
        npid = load_chunk(na, ne, nb, nui);
      }
      const int unit = cu < ce ? cu++ : -1;
      if (fill > 0 && !mbar_wait(&empty_bar[s], (fill - 1) & 1u, kWaitLimit) && lane == 0)
        flag_error(p.err, 8u);
      if (unit < 0) {
        // No more units: a stage marked -1 (plain arrive, no bytes) stops the consumers.
        if (lane == 0) {
          stage_unit[s] = -1;
          mbar_arrive(&full_bar[s]);
        }
        break;
      }
      const int lane0 = (unit - ca) * PPU;   // lane of this unit's first page id
      const int b = __shfl_sync(kFull, cb, lane0);
      const int ui = __shfl_sync(kFull, cui, lane0);
      const int T = ulen[b];
      const int t0 = ui * TPU;
      const int t1 = min(T, t0 + TPU);
      const int pbase = lane0;
      unsigned char* dst = ring + s * kUnitBytes;
      uint32_t nbytes = 0;
      const uint8_t* src = p.label;
      int dst_off = 0;
      if constexpr (MMA) {
        // Tensor copies: one 64-token page (64 x 64 bf16, 8 KB) per lane,
        // swizzled into the stage for conflict-free ldmatrix reads.
        const int pid = __shfl_sync(kFull, cpid, (pbase + lane) & 31);
        const int pg = (t0 >> 6) + lane;
        if (lane < PPU && pg * kPage < t1) {
          if (pid >= 0 && pid < p.num_pages) {
            nbytes = 8192u;
            dst_off = lane * 8192;
          } else {
            flag_error(p.err, 2u);
          }
        }
        uint32_t total = nbytes;
#pragma unroll
        for (int o = 16; o; o >>= 1) total += __shfl_xor_sync(kFull, total, o);
        if (lane == 0) {
          stage_unit[s] = ui;
          stage_req[s] = b;
          mbar_arrive_expect_tx(&full_bar[s], total);
        }
        __syncwarp();
        if (nbytes) tensor_g2s_2d_hint(dst + dst_off, &p.tmap, 0, pid * kPage, &full_bar[s], stream_pol);
        if (++s == p.nst) {
          s = 0;
          ++fill;
        }
        continue;
      } else {
        // Whole token rows: one contiguous span per page of the unit.
        const int pid = __shfl_sync(kFull, cpid, (pbase + lane) & 31);
        const int pg = (t0 >> 6) + lane;
        const int ts = max(t0, pg * kPage);
        const int te = min(t1, pg * kPage + kPage);
        if (lane < PPU && ts < te) {
          if (pid >= 0 && pid < p.num_pages) {
            nbytes = static_cast<uint32_t>(te - ts) * BR;
            src = p.label + static_cast<long long>(pid * kPage + (ts & (kPage - 1))) * BR;
            dst_off = (ts - t0) * BR;
          } else {
            flag_error(p.err, 2u);
          }
        }
      }
      uint32_t total = nbytes;
#pragma unroll
      for (int o = 16; o; o >>= 1) total += __shfl_xor_sync(kFull, total, o);
      if (lane == 0) {
        stage_unit[s] = ui;
        stage_req[s] = b;
        mbar_arrive_expect_tx(&full_bar[s], total);
      }
      __syncwarp();
      if (nbytes) bulk_g2s_hint(dst + dst_off, src, nbytes, &full_bar[s], stream_pol);
      if (++s == p.nst) {
        s = 0;
        ++fill;
      }
    }
  } else {
    // ------------------------------------------------------------ consumer warps
    if constexpr (MMA) {
      // Tensor cores: warp w takes tokens [16w, 16w + 16) of each 128-token
      // unit and forms D[16 tokens x 8] = K_tile[16 x 64] . B[64 x 8] with
      // mma.sync m16n8k16 (bf16 in, fp32 accumulate). Column 2g of B holds
      // the group-g query summed over its heads, rounded to bf16 (hi);
      // column 2g + 1 the bf16 rounding of the remainder (lo), so hi + lo
      // carries the fp32 sum to about 2^-16 relative and integer-valued sums
      // exactly; the score of group g is D[., 2g] + D[., 2g + 1].
      constexpr int NT = (2 * NGR + 7) / 8;   // n8 tiles
      const int gr = lane >> 2, qc = lane & 3;
      const int G = p.Hq / p.Hkv;
      uint32_t qb[NT][4][2];
      int cur = -1, b = 0, T = 0;
      int s = 0;
      uint32_t fill = 0;
      for (;;) {
        const bool ok = mbar_wait(&full_bar[s], fill & 1u, kWaitLimit);
        if (!ok && lane == 0) flag_error(p.err, 8u);
        const int unit = ok ? stage_unit[s] : -1;   // a wait that ran out stops this warp
        if (unit < 0) break;
        const int ub = stage_req[s];
        const int ui = unit;
        if (ub != cur) {
          cur = ub;
          b = ub;
          T = clamp_len(p, b);
          if (tid == 0 && ui == 0) {
            const int raw = __ldg(p.seq_lens + b);
            if (raw < 0 || raw > min(p.Tmax, p.maxp * kPage)) flag_error(p.err, 1u);
          }
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int n = nt * 8 + gr;   // this lane's B column
            const int g = n >> 1;
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) {
              float qs[4] = {0.f, 0.f, 0.f, 0.f};   // channels 16ks + 2qc, +1, +8, +9
              if (g < NGR) {
                for (int h = g * G; h < (g + 1) * G; ++h) {
                  const uint16_t* qrow = p.qp + (static_cast<long long>(b) * p.Hq + h) * C + 16 * ks + 2 * qc;
                  const uint32_t w0 = __ldg(reinterpret_cast<const uint32_t*>(qrow));
                  const uint32_t w1 = __ldg(reinterpret_cast<const uint32_t*>(qrow + 8));
                  qs[0] += bf16_lo(w0);
                  qs[1] += bf16_hi(w0);
                  qs[2] += bf16_lo(w1);
                  qs[3] += bf16_hi(w1);
                }
              }
              uint16_t part[4];
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const __nv_bfloat16 hi = __float2bfloat16_rn(qs[i]);
                const __nv_bfloat16 v = (n & 1) ? __float2bfloat16_rn(qs[i] - __bfloat162float(hi)) : hi;
                part[i] = __bfloat16_as_ushort(v);
              }
              qb[nt][ks][0] = static_cast<uint32_t>(part[0]) | (static_cast<uint32_t>(part[1]) << 16);
              qb[nt][ks][1] = static_cast<uint32_t>(part[2]) | (static_cast<uint32_t>(part[3]) << 16);
            }
          }
        }
        const int tw = ui * TPU + 16 * warp;   // this warp's first token
        bool released = false;
        if (ok && tw < T) {
          const int row0 = (16 * warp) & (kPage - 1);
          const uint32_t tile = smem_u32(ring + s * kUnitBytes + ((16 * warp) >> 6) * 8192);
          const int r = row0 + (lane & 15);
          float acc[NT][4];
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
#pragma unroll
            for (int i = 0; i < 4; ++i) acc[nt][i] = 0.f;
#pragma unroll
          for (int ks = 0; ks < 4; ++ks) {
            const int chunk = 2 * ks + (lane >> 4);
            uint32_t a0, a1, a2, a3;
            ldsm_x4(tile + r * 128 + ((chunk ^ (r & 7)) << 4), a0, a1, a2, a3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt) mma_bf16(acc[nt], a0, a1, a2, a3, qb[nt][ks][0], qb[nt][ks][1]);
          }
          // The stage has been read into registers: hand it back to the
          // producer before the scores are written.
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
          released = true;
          const int t_lo = tw + gr, t_hi = tw + gr + 8;
          const bool full = tw + 16 <= T;   // the warp's 16 tokens all lie inside the sequence
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            const int g = nt * 4 + qc;
            const float s_lo = acc[nt][0] + acc[nt][1];
            const float s_hi = acc[nt][2] + acc[nt][3];
            if (g < NGR) {
              float* srow = p.scores + (static_cast<long long>(b) * p.Hkv + g) * p.Tmax;
              if (full || t_lo < T) st_hint(srow + t_lo, s_lo, keep_pol);
              if (full || t_hi < T) st_hint(srow + t_hi, s_hi, keep_pol);
            }
            if (p.bmax) {
              // The largest of the warp's 16 scores of group g (lanes with
              // this qc, rows gr and gr + 8): the very values stored above,
              // combined with fmaxf, which passes over NaN and positions
              // past the sequence (NaN here) as the top-k's keys rank NaN
              // lowest.
              const float nan = __int_as_float(0x7fffffff);
              float m = full ? fmaxf(s_lo, s_hi) : fmaxf(t_lo < T ? s_lo : nan, t_hi < T ? s_hi : nan);
              m = fmaxf(m, __shfl_xor_sync(kFull, m, 4));
              m = fmaxf(m, __shfl_xor_sync(kFull, m, 8));
              m = fmaxf(m, __shfl_xor_sync(kFull, m, 16));
              if (gr == 0 && g < NGR)
                st_hint(p.bmax + (static_cast<long long>(b) * p.Hkv + g) * p.nbr + (tw >> 4), m, keep_pol);
            }
          }
        }
        if (!released) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty_bar[s]);
        }
        if (++s == p.nst) {
          s = 0;
          ++fill;
        }
      }
    } else {
    const int chunk = lane % LPR;
    const int rin = lane / LPR;
    const int tok_off = rin / HPB;
    const int hin = rin % HPB;
    const int G = p.Hq / p.Hkv;
    int cur = -1;
    int b = 0, T = 0;
    float2 q[NQ][4];
    // Label head of query set n (per-head label): piece warp * U + n of a unit
    // holds head block (warp * U + n) % PPT of its token.
    auto head_of = [&](int n) { return ((warp * U + n) % PPT) * HPB + hin; };

    int s = 0;
    uint32_t fill = 0;
    for (;;) {
      const bool ok = mbar_wait(&full_bar[s], fill & 1u, kWaitLimit);
      if (!ok && lane == 0) flag_error(p.err, 8u);
      const int unit = ok ? stage_unit[s] : -1;   // a wait that ran out stops this warp
      if (unit < 0) break;
      const int ub = stage_req[s];
      const int ui = unit;
      if (ub != cur) {
        cur = ub;
        b = ub;
        T = clamp_len(p, b);
        if (tid == 0 && ui == 0) {
          const int raw = __ldg(p.seq_lens + b);
          if (raw < 0 || raw > min(p.Tmax, p.maxp * kPage)) flag_error(p.err, 1u);
        }
#pragma unroll
        for (int n = 0; n < NQ; ++n) {
          const int g = (NGR == 1) ? head_of(n) : n;
          float qs[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
          for (int h = g * G; h < (g + 1) * G; ++h) {
            const uint4 w = __ldg(reinterpret_cast<const uint4*>(p.qp + (static_cast<long long>(b) * p.Hq + h) * C + chunk * 8));
            qs[0] += bf16_lo(w.x); qs[1] += bf16_hi(w.x);
            qs[2] += bf16_lo(w.y); qs[3] += bf16_hi(w.y);
            qs[4] += bf16_lo(w.z); qs[5] += bf16_hi(w.z);
            qs[6] += bf16_lo(w.w); qs[7] += bf16_hi(w.w);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i) q[n][i] = make_float2(qs[2 * i], qs[2 * i + 1]);
        }
      }

      const int tbase = ui * TPU;
      bool released = false;
      if (ok && tbase < T) {
        const unsigned char* src = ring + s * kUnitBytes + (warp * U) * 512 + lane * 16;
        float acc[V];
#pragma unroll
        for (int uu = 0; uu < U; ++uu) {
          const uint4 x = *reinterpret_cast<const uint4*>(src + uu * 512);
          const float2 x0 = make_float2(bf16_lo(x.x), bf16_hi(x.x));
          const float2 x1 = make_float2(bf16_lo(x.y), bf16_hi(x.y));
          const float2 x2 = make_float2(bf16_lo(x.z), bf16_hi(x.z));
          const float2 x3 = make_float2(bf16_lo(x.w), bf16_hi(x.w));
#pragma unroll
          for (int n = 0; n < NGR; ++n) {
            const int qi = NGR > 1 ? n : uu % NQ;
            float2 a = make_float2(q[qi][0].x * x0.x, q[qi][0].y * x0.y);
            a = __ffma2_rn(q[qi][1], x1, a);
            a = __ffma2_rn(q[qi][2], x2, a);
            a = __ffma2_rn(q[qi][3], x3, a);
            acc[uu * NGR + n] = a.x + a.y;
          }
        }
        // The stage has been read into registers: hand it back to the
        // producer before the sums are combined and written.
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
        released = true;
        transposed_reduce<LPR, V>(acc);
#pragma unroll
        for (int kk = 0; kk < PER; ++kk) {
          const int v = (V >= LPR) ? chunk * PER + kk : (chunk * V) / LPR;
          const bool writer = (V >= LPR) || ((chunk * V) % LPR == 0);
          const int uu = v / NGR;
          const int n = v % NGR;
          const int t = tbase + ((warp * U + uu) / PPT) * TPI + tok_off;
          const int g = (NGR == 1) ? head_of(uu) : n;
          if (writer && t < T) st_hint(p.scores + (static_cast<long long>(b) * p.Hkv + g) * p.Tmax + t, acc[kk], keep_pol);
        }
      }
      if (!released) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty_bar[s]);
      }
      if (++s == p.nst) {
        s = 0;
        ++fill;
      }
    }
    }
  }
}

using KernelFn = void (*)(const ScoreParams);

template <int C, int NGR>
KernelFn pick_tpi(int tpi) {
  constexpr int RPI = 256 / C;
  switch (tpi) {
    case 1: return index_score_kernel<C, NGR, 1, 1, false>;
    case 2: if constexpr (RPI >= 2) return index_score_kernel<C, NGR, 2, 1, false>; break;
    case 4: if constexpr (RPI >= 4) return index_score_kernel<C, NGR, 4, 1, false>; break;
    case 8: if constexpr (RPI >= 8) return index_score_kernel<C, NGR, 8, 1, false>; break;
    case 16: if constexpr (RPI >= 16) return index_score_kernel<C, NGR, 16, 1, false>; break;
  }
  return nullptr;
}

template <int C>
KernelFn pick(int HL, int Hkv, int* tpi_out, bool* mma) {
  constexpr int RPI = 256 / C;
  *mma = false;
  if (HL == 1) {
    // Shared key (or a single KV head): one row per token, feeds every group.
    // 64-wide keys: the tensor-core path.
    *tpi_out = RPI;
    if constexpr (C == 64) {
      *mma = true;
      switch (Hkv) {
        case 1: return index_score_kernel<C, 1, RPI, 1, true>;
        case 2: return index_score_kernel<C, 2, RPI, 1, true>;
        case 4: return index_score_kernel<C, 4, RPI, 1, true>;
        case 8: return index_score_kernel<C, 8, RPI, 1, true>;
      }
      return nullptr;
    }
    switch (Hkv) {
      case 1: return index_score_kernel<C, 1, RPI, 1, false>;
      case 2: return index_score_kernel<C, 2, RPI, 1, false>;
      case 4: return index_score_kernel<C, 4, RPI, 1, false>;
      case 8: return index_score_kernel<C, 8, RPI, 1, false>;
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
  // Rows of several 512-byte pieces: PPT pieces (head blocks) per token.
  if (HL % RPI) return nullptr;
  *tpi_out = 1;
  switch (HL / RPI) {
    case 1: return index_score_kernel<C, 1, 1, 1, false>;
    case 2: return index_score_kernel<C, 1, 1, 2, false>;
    case 4: return index_score_kernel<C, 1, 1, 4, false>;
    case 8: return index_score_kernel<C, 1, 1, 8, false>;
  }
  return nullptr;
}

KernelFn select_kernel(int C, int HL, int Hkv, int* tpi, bool* mma) {
  switch (C) {
    case 16: return pick<16>(HL, Hkv, tpi, mma);
    case 32: return pick<32>(HL, Hkv, tpi, mma);
    case 64: return pick<64>(HL, Hkv, tpi, mma);
  }
  return nullptr;
}

// Tensor map of a shared 64-wide bf16 key cache: rows = slots, 64 x 64 boxes
// (one page), 128-byte swizzle. The encoder is the driver's, fetched once.
cudaError_t key_tensor_map(CUtensorMap* map, const void* keys, long long slots) {
  using Encode = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
  static Encode encode = nullptr;
  if (!encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess || !fn)
      return cudaErrorNotSupported;
    encode = reinterpret_cast<Encode>(fn);
  }
  const cuuint64_t dims[2] = {64, static_cast<cuuint64_t>(slots)};
  const cuuint64_t strides[1] = {128};
  const cuuint32_t box[2] = {64, 64};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = encode(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(keys), dims, strides, box,
                            estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
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

bool index_score_block_maxima(int C, int HL, int Hkv) {
  int tpi = 0;
  bool mma = false;
  return select_kernel(C, HL, Hkv, &tpi, &mma) != nullptr && mma;
}

bool index_score_supported(int C, int HL, int Hkv, int G) {
  (void)G;
  int tpi = 0;
  bool mma = false;
  return select_kernel(C, HL, Hkv, &tpi, &mma) != nullptr;
}

cudaError_t launch_index_score(const ScoreArgs& a, cudaStream_t stream) {
  int tpi = 0;
  bool mma = false;
  KernelFn fn = select_kernel(a.C, a.HL, a.Hkv, &tpi, &mma);
  if (!fn) return cudaErrorNotSupported;
  if (a.B == 0 || a.Tmax == 0) return cudaSuccess;
  const int tpu = kUnitBytes / (a.HL * a.C * 2);   // whole token rows per unit
  ScoreParams p{};
  p.qp = static_cast<const uint16_t*>(a.qp);
  p.label = static_cast<const uint8_t*>(a.label);
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.scores = a.scores;
  p.err = a.err;
  p.B = a.B;
  p.Hq = a.Hq;
  p.Hkv = a.Hkv;
  p.HL = a.HL;
  p.maxp = a.maxp;
  p.num_pages = a.num_pages;
  p.Tmax = a.Tmax;
  // Units of all requests at their longest: their count must fit an int.
  const long long upb = (static_cast<long long>(a.maxp) * kPage + tpu - 1) / tpu;
  const long long units = static_cast<long long>(a.B) * upb;
  if (units >= (1LL << 31) || static_cast<long long>(a.B) * a.maxp >= (1LL << 31)) return cudaErrorNotSupported;
  if (mma) {
    const cudaError_t te = key_tensor_map(&p.tmap, a.label, static_cast<long long>(a.num_pages) * kPage);
    if (te != cudaSuccess) return te;
    p.bmax = a.bmax;
    p.nbr = (a.Tmax + kMaxBlock - 1) / kMaxBlock;
  }
  // Two CTAs per SM, each with a ring of 7 x 16 KB stages (6 on the
  // tensor-core path, which aligns the ring to 1024 bytes), and the
  // producer's per-request unit prefix and lengths after it.
  p.nst = mma ? 6 : 7;
  const int smem = p.nst * kUnitBytes + (mma ? 1024 : 0) + 8 * (a.B + 1);
  cudaError_t e = allow_smem(fn, smem);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kScoreThreads, smem);
  if (e != cudaSuccess) return e;
  if (per_sm < 1) per_sm = 1;
  long long blocks = static_cast<long long>(sm_count()) * per_sm;
  if (units < blocks) blocks = units;
  e = launch_pdl(fn, dim3(static_cast<unsigned>(blocks)), dim3(kScoreThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
