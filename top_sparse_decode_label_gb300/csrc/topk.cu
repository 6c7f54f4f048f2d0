// Stage 2: exact top-k per (request, KV head) row with lowest-token-index
// tie-breaking, output ascending by token index.
//
// sglang PR #43527 "QSA cache sharding", "Distributed QSA execution": local
// candidates are merged into an exact Top-K using deterministic global
// token-ID tie-breaking. "Support double sparsity" (PR #1459): keep the
// heavy-token count of tokens per head.
//
// Scores map to order-preserving 32-bit keys (-0.0 == +0.0, NaN lowest).
// With K_eff = min(k, T), a row with 0 < K_eff < T is selected by one
// thread-block cluster of CS CTAs (CS a power of two, up to 16), CTA q owning
// the contiguous token slice q of the row. The threshold key -- the K_eff-th
// largest -- is found digit by digit (11 + 11 + 10 bits): each CTA builds the
// histogram of its slice's digits in shared memory and adds its nonzero bins
// into the bins' owner CTA (bins are split evenly over the cluster) with
// distributed-shared-memory atomics; after a cluster barrier every CTA reads
// the row's totals from the owners and finds the digit where the running
// count from the top reaches the remaining need. After digit 1 each CTA
// compacts the (key, token) pairs of its slice whose first digit is at least
// the threshold's into a token-ordered list (shared memory, or the workspace
// when it overflows); digits 2 and 3 and the output work on that list. With
// `thr` the threshold key and r the number of keys equal to it that must be
// kept, a CTA keeps its keys > thr and its equal keys whose rank in the row's
// token order is below r; the counts of the CTAs before it give its output
// offset. No global atomics, no completion counters, nothing to clear.
//
// Rows with slices of two passes or more and K_eff <= T/128 first try a
// filtered pass (a kernel variant with one CTA per SM, launched when
// full-length rows qualify): a filter key that all CTAs of the cluster share
// lets only the keys at or above it into the candidate lists and their
// digit-1 histogram. The filter key comes from the scan's 16-token block
// maxima when there are any (the first-digit bin where the row's block maxima
// reach K_eff, an exact lower bound; only blocks whose maximum reaches it are
// read), otherwise from a sample of the keys (the key where the sample, counted from
// the top, reaches the kept fraction plus three standard deviations; the
// cluster takes its CTAs' smallest). Either way every key at or above the
// filter is a candidate, so a digit-1 crossing in the candidates' totals is
// the true one and the lists hold every key that can be kept; when there is
// none (too few keys passed) or a list overflows, the cluster clears its
// histograms and takes the two passes above.
#include "common.cuh"
#include "internal.h"
#include "topk_common.cuh"

namespace ds {

namespace {

constexpr int kThreads = 512;
constexpr int kPer = 16;                      // scores per thread per pass
constexpr int kBatch = kThreads * kPer;       // scores per CTA pass
constexpr int kListCap = 4096;                // kept (key, token) pairs in shared memory
constexpr int kMaxCluster = 16;
constexpr int kPtCap = 1040;                  // page-table entries of a slice kept in shared memory
constexpr int kWarps = kThreads / 32;
constexpr int kPerF = 32;                     // scores per lane per step of the filtered pass
constexpr int kStep = 32 * kPerF;             // keys of one warp step of the filtered pass
constexpr int kWarpCap = kListCap / kWarps;   // (key, token) pairs one warp keeps in the filtered pass
constexpr int kBmPer = 8;                     // block maxima per thread (block-maxima filter)
constexpr int kBmCap = kThreads * kBmPer;     // 16-token blocks of a CTA slice that takes the block-maxima filter
constexpr int kGatherRounds = 4;              // rounds of kThreads / 4 candidate blocks read in one round trip

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct TopkParams {
  const float* scores;
  const int32_t* seq_lens;
  int32_t* idx;
  unsigned* err;
  uint2* list;     // [R, Tmax] overflow lists
  int Hkv, Tmax, lim, k;
  // Chained call only (slots == nullptr otherwise): the physical slot of each
  // kept token and, for an FP8 cache (sscale non-null), its page's K and V
  // scales, so that the attention resolves both with one load.
  const int32_t* page_table;
  int32_t* slots;  // [R, k]
  const float* ks;
  const float* vs;
  float2* sscale;  // [R, k]
  int maxp, num_pages;
  int pre_wait;    // inputs may be read before the previous kernel completes
  const float* bmax;   // [R, nbr] maxima of the rows' 16-token blocks, or null
  int nbr;
};

struct __align__(16) Smem {
  unsigned h1[kBins1];   // this CTA's digit histograms, bin b at hslot(b)
  unsigned h2[kBins1];
  unsigned h3[kBins3];
  unsigned t1[kBins1];   // row totals of the bins this CTA owns, bin b at b
  unsigned t2[kBins1];
  unsigned t3[kBins3];
  unsigned long long scan[33];
  unsigned cnt[2];       // this CTA's keys above the threshold, equal to it
  unsigned res[4];
  unsigned lmax;         // filtered pass: the highest filter bin of the cluster (rank 0's copy)
  unsigned lmin;         // sampled filter: the smallest filter key of the cluster (rank 0's copy)
  unsigned wcnt[kThreads / 32];   // filtered pass: candidates of each warp's token range
  unsigned woff[kThreads / 32];
  int pt[kPtCap];        // page-table entries of this CTA's slice (chained call)
  float2 psc[kPtCap];    // and, for an FP8 cache, the (K, V) scales of those pages
  uint2 list[kListCap];
};
constexpr int kZeroWords = 4 * kBins1 + 2 * kBins3;   // h1 .. t3

// Shared memory the filtered variant adds after Smem: the block-maxima filter.
struct __align__(16) FiltX {
  unsigned hm[kBins1];              // first-digit histogram of this CTA's block maxima, bin b at hslot(b)
  unsigned tm[kBins1];              // row totals of the maxima bins this CTA owns, bin b at b
  unsigned short cblk[kBmCap];      // the slice's candidate blocks, in token order
};

// The smallest score whose key is `key` (a multiple of 2^21). For the keys of
// bins 1..3 that float is a NaN bit pattern, while every score but NaN has a
// key in bin 3 or above (-inf's key is 0x007fffff): those bins, like bin 0,
// take every key.
__device__ __forceinline__ float key_floor(uint32_t key) {
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7fffffffu) : ~key);
}

// Keys of one thread's share of a tile of NT threads x N scores starting at
// token `base` of a row: group i (4 consecutive scores) of thread r is tokens
// base + 4 (i NT + r) .. + 3, so each 16-byte load instruction of a warp reads
// 512 contiguous bytes (only tokens < c1 are meaningful; scalar loads where a
// row is not 16-byte aligned or at its end).
// The scores stay raw in registers until the tile is processed, so the loads
// of the next tile are in flight while the current one is.
template <int G, int NT>
__device__ __forceinline__ void load_tile(const float* s, int base, int r, int c1, float4 (&v)[G]) {
  const bool al = (reinterpret_cast<uintptr_t>(s + base) & 15u) == 0;
#pragma unroll
  for (int i = 0; i < G; ++i) {
    const int t = base + 4 * (i * NT + r);
    if (al && t + 4 <= c1) {
      v[i] = __ldcg(reinterpret_cast<const float4*>(s + t));
    } else {
      v[i].x = t < c1 ? __ldcg(s + t) : 0.f;
      v[i].y = t + 1 < c1 ? __ldcg(s + t + 1) : 0.f;
      v[i].z = t + 2 < c1 ? __ldcg(s + t + 2) : 0.f;
      v[i].w = t + 3 < c1 ? __ldcg(s + t + 3) : 0.f;
    }
  }
}
template <int G>
__device__ __forceinline__ void tile_keys(const float4 (&v)[G], uint32_t (&keys)[4 * G]) {
#pragma unroll
  for (int i = 0; i < G; ++i) {
    keys[4 * i] = order_key(v[i].x);
    keys[4 * i + 1] = order_key(v[i].y);
    keys[4 * i + 2] = order_key(v[i].z);
    keys[4 * i + 3] = order_key(v[i].w);
  }
}
// Token of key q of thread r in that tile.
template <int NT>
__device__ __forceinline__ int tile_token(int base, int r, int q) {
  return base + 4 * ((q >> 2) * NT + r) + (q & 3);
}

// Rows that try the filtered pass: CTA slices of two passes or more, and at
// most 1/128 of the row kept (with more kept, the two passes of the other
// variant, two CTAs per SM, were measured faster on GB300).
__host__ __device__ __forceinline__ bool filtered_row(int slice, long long keff, int T) {
  return slice >= 2 * kBatch && keff * 128 <= T;
}
// Filtered rows that bound the threshold with the scan's block maxima:
// slices of at most kBmCap blocks.
__host__ __device__ __forceinline__ bool block_maxima_row(int slice) { return slice <= kMaxBlock * kBmCap; }

// Adds this CTA's histogram h (nbins bins, slots hslot) into the owners'
// totals t: bin b belongs to cluster rank b / (nbins / cs).
template <int NB>
__device__ __forceinline__ void push_bins(const unsigned* h, unsigned* t, unsigned cs) {
  constexpr int per = NB / kThreads;
  const int own_shift = __ffs(NB / static_cast<int>(cs)) - 1;
#pragma unroll
  for (int j = 0; j < per; ++j) {
    const int b = threadIdx.x * per + j;
    const unsigned v = h[hslot(b)];
    if (v) cluster_red_add(cluster_map(smem_u32(t + b), static_cast<unsigned>(b >> own_shift)), v);
  }
}

// Reads the row totals of bins hi-1 .. hi-PER (hi = NB - PER * tid) from
// their owner: c[j] = total of bin hi-1-j.
template <int NB, int PER>
__device__ __forceinline__ void read_totals(const unsigned* t, unsigned cs, unsigned (&c)[PER]) {
  const int hi = NB - PER * static_cast<int>(threadIdx.x);
  const int own_shift = __ffs(NB / static_cast<int>(cs)) - 1;
  const uint32_t a = cluster_map(smem_u32(t + hi - PER), static_cast<unsigned>((hi - PER) >> own_shift));
  if constexpr (PER == 4) {
    const uint4 v = cluster_ld4(a);
    c[0] = v.w;
    c[1] = v.z;
    c[2] = v.y;
    c[3] = v.x;
  } else {
    static_assert(PER == 2, "two or four bins per thread");
    const uint2 v = cluster_ld2(a);
    c[0] = v.y;
    c[1] = v.x;
  }
}

// Bins hi-1 .. hi-PER per thread (thread 0 the highest): finds the bin where
// the count from the top first reaches `need` (1 <= need <= total) and writes
// res[0] = bin, res[1] = count in the bins above it.
template <int NB, int PER>
__device__ __forceinline__ void find_crossing(const unsigned (&c)[PER], unsigned need, Smem& S) {
  const int hi = NB - PER * static_cast<int>(threadIdx.x);
  unsigned sum = 0;
#pragma unroll
  for (int j = 0; j < PER; ++j) sum += c[j];
  unsigned tot;
  unsigned run = block_excl_scan(sum, reinterpret_cast<unsigned*>(S.scan), &tot);
  if (run < need && run + sum >= need) {
#pragma unroll
    for (int j = 0; j < PER; ++j) {
      if (run + c[j] >= need) {
        S.res[0] = static_cast<unsigned>(hi - 1 - j);
        S.res[1] = run;
        break;
      }
      run += c[j];
    }
  }
  __syncthreads();
}

__device__ __forceinline__ int row_len(const TopkParams& p, int b, bool flag) {
  int T = p.seq_lens[b];
  if (T < 0 || T > p.lim) {
    if (flag) flag_error(p.err, 1u);
    T = T < 0 ? 0 : p.lim;
  }
  return T;
}

// Writes kept token t at output position pos; in the chained call also its
// physical slot and, for an FP8 cache, its page's (K, V) scales.
__device__ __forceinline__ void emit(const TopkParams& p, const Smem& S, int row, int b, int pg0, int npg, int pos,
                                     int t) {
  const size_t o = static_cast<size_t>(row) * p.k + pos;
  p.idx[o] = t;
  if (!p.slots) return;
  const int pg = t >> 6;
  const bool cached = npg <= kPtCap && pg - pg0 < npg;
  const int pid = cached ? S.pt[pg - pg0] : __ldg(p.page_table + static_cast<long long>(b) * p.maxp + pg);
  int slot = -1;
  float2 sc = make_float2(1.f, 1.f);
  if (pid < 0 || pid >= p.num_pages) {
    flag_error(p.err, 2u);
  } else {
    slot = pid * kPage + (t & (kPage - 1));
    if (p.sscale) sc = cached ? S.psc[pg - pg0] : make_float2(__ldg(p.ks + pid), __ldg(p.vs + pid));
  }
  p.slots[o] = slot;
  if (p.sscale) p.sscale[o] = sc;
}

// FILT: the variant that tries the filtered pass first (one CTA per SM, so
// that its deeper loads keep their registers); the other one runs two CTAs
// per SM. KPER: keys per thread per pass of the two passes (16, or 20 so that
// slices of up to 10,240 keys take one pass and the second pass reuses the
// keys still in registers).
template <bool FILT, int KPER = kPer>
__global__ void __launch_bounds__(kThreads, FILT ? 1 : 2) topk_cluster_kernel(const TopkParams p) {
  constexpr int PASS = kThreads * KPER;            // keys per CTA pass
  constexpr int FB = KPER / 4 <= 4 ? 16 : 12;      // bits per group count in the packed scan
  extern __shared__ __align__(16) unsigned char dsm[];
  Smem& S = *reinterpret_cast<Smem*>(dsm);
  const int tid = threadIdx.x;
  const unsigned cs = cluster_nctarank();
  const unsigned q = cluster_ctarank();
  const int row = static_cast<int>(blockIdx.x / cs);
  {
    uint4* z = reinterpret_cast<uint4*>(S.h1);
    for (int i = tid; i < kZeroWords / 4; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
    if (FILT) {
      uint4* zx = reinterpret_cast<uint4*>(dsm + sizeof(Smem));   // FiltX::hm and ::tm
      for (int i = tid; i < 2 * kBins1 / 4; i += kThreads) zx[i] = make_uint4(0u, 0u, 0u, 0u);
    }
    if (tid == 0) {
      S.lmax = 0u;
      S.lmin = 0xffffffffu;
      S.res[0] = 0u;
    }
  }
  const int b = row / p.Hkv;
  const int g = row - b * p.Hkv;
  int T = 0, s0 = 0, s1 = 0, pg0 = 0, npg = 0;
  // This CTA's token slice and, in the chained call, its page-table entries.
  auto setup = [&]() {
    T = row_len(p, b, q == 0 && tid == 0 && g == 0);
    const int SL = ((T + static_cast<int>(cs) - 1) / static_cast<int>(cs) + 15) & ~15;
    s0 = min(T, static_cast<int>(q) * SL);
    s1 = min(T, s0 + SL);
    if (p.slots && s1 > s0) {
      pg0 = s0 >> 6;
      npg = ((s1 - 1) >> 6) - pg0 + 1;
      if (npg <= kPtCap) {
        for (int i = tid; i < npg; i += kThreads) {
          const int pid = __ldg(p.page_table + static_cast<long long>(b) * p.maxp + pg0 + i);
          S.pt[i] = pid;
          if (p.sscale)
            S.psc[i] = (pid >= 0 && pid < p.num_pages) ? make_float2(__ldg(p.ks + pid), __ldg(p.vs + pid))
                                                       : make_float2(1.f, 1.f);
        }
      }
    }
  };
  if (p.pre_wait) setup();
  grid_dependency_wait();
  grid_launch_dependents();
  if (!p.pre_wait) setup();
  __syncthreads();
  int32_t* out = p.idx + static_cast<size_t>(row) * p.k;
  const int keff = min(p.k, T);
  if (!needs_selection(p.k, T)) {
    // The whole cluster takes this branch (same row): no shared memory is
    // exchanged, so CTAs leave independently. Every token is kept.
    for (int t = s0 + tid; t < min(s1, p.k); t += kThreads) emit(p, S, row, b, pg0, npg, t, t);
    for (int i = keff + static_cast<int>(q) * kThreads + tid; i < p.k; i += static_cast<int>(cs) * kThreads) {
      out[i] = -1;
      if (p.slots) p.slots[static_cast<size_t>(row) * p.k + i] = -1;
    }
    return;
  }
  cluster_arrive();   // this CTA's totals are zero: owners may receive adds

  const float* s = p.scores + static_cast<long long>(row) * p.Tmax;
  unsigned b1 = 0, above1 = 0, M = 0;
  uint2* lst = S.list;
  bool filtered = false;
  // Filtered rows (see the top of the file): a shared filter key lets only
  // the keys at or above it into the candidate lists; when too few pass, or a
  // list overflows, every CTA of the cluster falls back to the two passes
  // below.
  const int SLr = ((T + static_cast<int>(cs) - 1) / static_cast<int>(cs) + 15) & ~15;
  if (FILT && filtered_row(SLr, keff, T)) {
    const int warp = tid >> 5, lane = tid & 31;
    const int len = s1 - s0;
    // With the scan's block maxima (block_maxima_row), the filter bin is
    // exact instead of sampled: the first-digit bin where the
    // row's block maxima, counted from the top, reach K_eff. Each of those
    // blocks holds its maximum, so at least K_eff keys lie in that bin or
    // above and so does the threshold; only blocks whose maximum reaches the
    // bin can hold a kept key, and only they are read.
    const bool bm_path = p.bmax != nullptr && block_maxima_row(SLr);
    uint2* sub = S.list + warp * kWarpCap;   // sample path: this warp's candidates, in token order
    unsigned n = 0;    // sample path: this warp's candidates so far (only the first kWarpCap are kept)
    unsigned mc = 0;   // block-maxima path: the CTA's candidates (only the first kListCap are kept)
    unsigned lbin = 0;
    if (bm_path) {
      FiltX& X = *reinterpret_cast<FiltX*>(dsm + sizeof(Smem));
      const int nbk = (len + kMaxBlock - 1) / kMaxBlock;   // s0 is a multiple of 16
      const float* bm = p.bmax + static_cast<long long>(row) * p.nbr + s0 / kMaxBlock;
      uint32_t mk[kBmPer];
      {
        // Thread t's kBmPer maxima, as two 16-byte loads where they are whole
        // and aligned (a quarter of the sectors the scalar loads request).
        float mf[kBmPer];
        const int blk0 = tid * kBmPer;
        if ((reinterpret_cast<uintptr_t>(bm + blk0) & 15u) == 0 && blk0 + kBmPer <= nbk) {
#pragma unroll
          for (int i = 0; i < kBmPer / 4; ++i) {
            const float4 f = __ldcg(reinterpret_cast<const float4*>(bm + blk0) + i);
            mf[4 * i] = f.x;
            mf[4 * i + 1] = f.y;
            mf[4 * i + 2] = f.z;
            mf[4 * i + 3] = f.w;
          }
        } else {
#pragma unroll
          for (int i = 0; i < kBmPer; ++i) mf[i] = blk0 + i < nbk ? __ldcg(bm + blk0 + i) : 0.f;
        }
#pragma unroll
        for (int i = 0; i < kBmPer; ++i) {
          const int blk = blk0 + i;
          mk[i] = blk < nbk ? order_key(mf[i]) : 0u;
          warp_hist_add(X.hm, mk[i] >> 21, blk < nbk);
        }
      }
      __syncthreads();
      cluster_wait();
      push_bins<kBins1>(X.hm, X.tm, cs);
      cluster_sync();
      {
        unsigned c[4];
        read_totals<kBins1, 4>(X.tm, cs, c);
        find_crossing<kBins1, 4>(c, static_cast<unsigned>(keff), S);   // the row has at least 8 K_eff blocks
      }
      lbin = S.res[0];
      cluster_arrive();   // no more reads of the maxima totals; paired with the wait before the next push
      // The candidate blocks (maximum in the bin or above), in token order.
      const uint32_t lb = lbin << 21;
      unsigned cnt = 0;
#pragma unroll
      for (int i = 0; i < kBmPer; ++i) cnt += (tid * kBmPer + i < nbk && mk[i] >= lb) ? 1u : 0u;
      unsigned nc;
      unsigned pos = block_excl_scan(cnt, reinterpret_cast<unsigned*>(S.scan), &nc);
#pragma unroll
      for (int i = 0; i < kBmPer; ++i)
        if (tid * kBmPer + i < nbk && mk[i] >= lb) X.cblk[pos++] = static_cast<unsigned short>(tid * kBmPer + i);
      __syncthreads();
      // Their keys in the bin or above, appended in token order.
      const float flb = key_floor(lb);
      const bool take_all = lbin < 4u;
      const bool al = (reinterpret_cast<uintptr_t>(s) & 15u) == 0;
      // Batches of kGatherRounds x kThreads / 4 candidate blocks. In round u
      // thread t reads the 16-byte quarter t % 4 of block
      // cb + u kThreads / 4 + t / 4, so each warp load covers 8 whole blocks
      // (whole 32-byte sectors); all rounds' loads are issued before any is
      // used, and one block scan of per-round counts (16 bits each) orders
      // the batch: token order is round, then thread order.
      constexpr int BPR = kThreads / 4;   // blocks per round
      for (int cb = 0; cb < static_cast<int>(nc); cb += kGatherRounds * BPR) {
        float4 v[kGatherRounds];
        int tb[kGatherRounds];
#pragma unroll
        for (int u = 0; u < kGatherRounds; ++u) {
          const int ci = cb + u * BPR + (tid >> 2);
          tb[u] = ci < static_cast<int>(nc) ? s0 + kMaxBlock * static_cast<int>(X.cblk[ci]) + 4 * (tid & 3) : s1;
          if (al && tb[u] + 4 <= s1) {
            v[u] = __ldcg(reinterpret_cast<const float4*>(s + tb[u]));
          } else {
            v[u].x = tb[u] < s1 ? __ldcg(s + tb[u]) : 0.f;
            v[u].y = tb[u] + 1 < s1 ? __ldcg(s + tb[u] + 1) : 0.f;
            v[u].z = tb[u] + 2 < s1 ? __ldcg(s + tb[u] + 2) : 0.f;
            v[u].w = tb[u] + 3 < s1 ? __ldcg(s + tb[u] + 3) : 0.f;
          }
        }
        unsigned m[kGatherRounds];
        unsigned long long packed = 0;
#pragma unroll
        for (int u = 0; u < kGatherRounds; ++u) {
          const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
          m[u] = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((take_all || x[j] >= flb) && tb[u] + j < s1) m[u] |= 1u << j;
          packed += static_cast<unsigned long long>(__popc(m[u])) << (16 * u);
        }
        unsigned long long tot;
        const unsigned long long ex = block_excl_scan64(packed, S.scan, &tot);
        unsigned base = mc;
#pragma unroll
        for (int u = 0; u < kGatherRounds; ++u) {
          unsigned q = base + static_cast<unsigned>((ex >> (16 * u)) & 65535u);
          const float x[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if ((m[u] >> j) & 1u) {
              if (q < static_cast<unsigned>(kListCap))
                S.list[q] = make_uint2(order_key(x[j]), static_cast<unsigned>(tb[u] + j));
              ++q;
            }
          }
          base += static_cast<unsigned>((tot >> (16 * u)) & 65535u);
        }
        mc = base;
      }
      __syncthreads();
      // Digit-1 histogram of the candidates (an overflowing list is not used).
      for (unsigned e = static_cast<unsigned>(tid); e < min(mc, static_cast<unsigned>(kListCap)); e += kThreads)
        warp_hist_add(S.h1, S.list[e].x >> 21, true);
    } else {
      // Warp w owns the contiguous token range [w0, w1) of the slice, in tiles
      // of kStep keys (kPerF per lane), so each warp appends its candidates in
      // token order without block-wide barriers.
      const int SW = ((len + kWarps - 1) / kWarps + kStep - 1) / kStep * kStep;
      const int w0 = min(s1, s0 + warp * SW), w1 = min(s1, w0 + SW);
      const int nst = (w1 - w0 + kStep - 1) / kStep;
      // The tiles stay raw floats: order_key is monotone, so key >= lb is
      // compared as score >= the float of key lb, and only candidates are
      // converted.
      float4 raw[kPerF / 4];
      float cur[kPerF];
      auto tile_floats = [&]() {
#pragma unroll
        for (int i = 0; i < kPerF / 4; ++i) {
          cur[4 * i] = raw[i].x;
          cur[4 * i + 1] = raw[i].y;
          cur[4 * i + 2] = raw[i].z;
          cur[4 * i + 3] = raw[i].w;
        }
      };
      if (nst > 0) load_tile<kPerF / 4, 32>(s, w0, lane, w1, raw);
      tile_floats();
      // Sample: two keys of each lane's first tile (up to 1024 per CTA,
      // spread over the warps' token ranges). The CTA's filter key is where
      // the sampled keys, counted from the top, reach the row's kept
      // fraction of the sample plus three standard deviations plus two --
      // found on the sample digit by digit (11 bits, then 11 more inside that
      // bin) -- and the cluster filters with the smallest of its CTAs' keys.
      // A sample whose kept share rounds to all of it gives key 0: no filter.
      uint32_t lb = 0;
      {
        FiltX& X = *reinterpret_cast<FiltX*>(dsm + sizeof(Smem));
        constexpr int kSamp[2] = {0, kPerF / 2};
        uint32_t sk[2];
        bool sv[2];
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          sv[j] = nst > 0 && tile_token<32>(w0, lane, kSamp[j]) < w1;
          sk[j] = order_key(cur[kSamp[j]]);
          warp_hist_add(S.h2, sk[j] >> 21, sv[j]);
        }
        if (tid == 0) S.res[0] = 0xffffffffu;
        unsigned ns;
        block_excl_scan(static_cast<unsigned>(sv[0]) + static_cast<unsigned>(sv[1]),
                        reinterpret_cast<unsigned*>(S.scan), &ns);
        const float mu = static_cast<float>(keff) / static_cast<float>(T) * static_cast<float>(ns);
        const unsigned m = static_cast<unsigned>(ceilf(mu + 3.f * sqrtf(mu) + 2.f));
        const int hi = kBins1 - 4 * tid;
        unsigned c[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) c[j] = S.h2[hslot(hi - 1 - j)];
        if (m < ns) find_crossing<kBins1, 4>(c, m, S);
        const unsigned bs = S.res[0], above = S.res[1];
#pragma unroll
        for (int j = 0; j < 4; ++j) S.h2[hslot(hi - 1 - j)] = 0u;   // digit 2 starts from zero
        if (bs != 0xffffffffu) {
#pragma unroll
          for (int j = 0; j < 2; ++j) warp_hist_add(X.hm, (sk[j] >> 10) & 2047u, sv[j] && (sk[j] >> 21) == bs);
          __syncthreads();
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            c[j] = X.hm[hslot(hi - 1 - j)];
            X.hm[hslot(hi - 1 - j)] = 0u;
          }
          find_crossing<kBins1, 4>(c, m - above, S);   // the bin holds the m-th sample
          lb = (bs << 21) | (S.res[0] << 10);
        }
      }
      cluster_wait();   // every CTA has set up its shared memory
      cluster_red_min(cluster_map(smem_u32(&S.lmin), 0u), lb);
      cluster_sync();
      lb = cluster_ld(cluster_map(smem_u32(&S.lmin), 0u));
      cluster_arrive();   // no more reads of rank 0's filter key; paired with the wait before the next push
      lbin = lb >> 21;
      // Keys below -inf's are NaN patterns: such a filter takes every key.
      const float flb = key_floor(lb);
      const bool take_all = lb < (4u << 21);
      // ---- the filtered pass: the candidate list of the keys >= lb, then their digit-1 histogram
      for (int st = 0; st < (lb != 0 ? nst : 0); ++st) {
        const int tb = w0 + st * kStep;
        if (st > 0) tile_floats();
        if (st + 1 < nst) load_tile<kPerF / 4, 32>(s, tb + kStep, lane, w1, raw);
        // Group g of the tile (4 keys per lane) is 128 contiguous tokens, lane
        // by lane: a warp ballot per key index gives every lane the number of
        // candidates before its own, and groups without any are skipped.
        const bool full = tb + kStep <= w1;
#pragma unroll
        for (int g = 0; g < kPerF / 4; ++g) {
          bool tk[4];
          unsigned bal[4], any = 0;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            tk[j] = (take_all || cur[4 * g + j] >= flb) && (full || tile_token<32>(tb, lane, 4 * g + j) < w1);
            bal[j] = __ballot_sync(kFull, tk[j]);
            any |= bal[j];
          }
          if (any) {
            const unsigned lt = (1u << lane) - 1u;
            unsigned q = n, tot = 0;
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              q += __popc(bal[j] & lt);
              tot += __popc(bal[j]);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              if (tk[j]) {
                if (q < static_cast<unsigned>(kWarpCap))
                  sub[q] = make_uint2(order_key(cur[4 * g + j]),
                                      static_cast<unsigned>(tile_token<32>(tb, lane, 4 * g + j)));
                ++q;
              }
            }
            n += tot;
          }
        }
      }
      // Digit-1 histogram of the candidates (an overflowing list is not used).
      for (unsigned e = static_cast<unsigned>(lane); e < min(n, static_cast<unsigned>(kWarpCap)); e += 32)
        atomicAdd(S.h1 + hslot(static_cast<int>(sub[e].x >> 21)), 1u);
      if (lane == 0) S.wcnt[warp] = n;
    }
    __syncthreads();
    cluster_wait();
    push_bins<kBins1>(S.h1, S.t1, cs);
    if (tid == 0) {
      // This CTA's filter bin into rank 0's maximum; a list that overflowed
      // posts one past the last bin, which fails the check.
      bool over = mc > static_cast<unsigned>(kListCap);
      if (!bm_path)
        for (int w = 0; w < kWarps; ++w) over |= S.wcnt[w] > static_cast<unsigned>(kWarpCap);
      cluster_red_max(cluster_map(smem_u32(&S.lmax), 0u), over ? static_cast<unsigned>(kBins1) : lbin);
      S.res[0] = 0xffffffffu;   // no crossing yet
    }
    cluster_sync();
    const unsigned lmax = cluster_ld(cluster_map(smem_u32(&S.lmax), 0u));
    {
      unsigned c[4];
      read_totals<kBins1, 4>(S.t1, cs, c);
      find_crossing<kBins1, 4>(c, static_cast<unsigned>(keff), S);
    }
    b1 = S.res[0];
    above1 = S.res[1];
    // Every CTA counted every key of the bins >= its own filter bin, so the
    // totals are exact from lmax up; a crossing there is the true one, and
    // every list holds all keys of its slice whose first digit reaches it.
    filtered = b1 != 0xffffffffu && b1 >= lmax;
    if (filtered && bm_path) {
      // One token-ordered list already; its entries below b1 fail every
      // later test (digit 2 and 3 match on the higher digits, the output
      // compares with the threshold), so it is used as it is.
      M = mc;
      for (int e = tid; e < static_cast<int>(M); e += kThreads) {
        const uint32_t key = S.list[e].x;
        warp_hist_add(S.h2, (key >> 10) & 2047u, (key >> 21) == b1);
      }
    } else if (filtered) {
      // The warps' lists, concatenated in warp (= token) order, keeping only
      // the entries whose first digit reaches b1 (the filter bin may lie
      // below it). In place, through registers: a warp's destination may
      // cover another warp's entries, so every entry is read before any is
      // written.
      const unsigned lt = (1u << lane) - 1u;
      uint2 v[kWarpCap / 32];
      unsigned pos[kWarpCap / 32];
      unsigned kept = 0, keepbits = 0;
#pragma unroll
      for (int j = 0; j < kWarpCap / 32; ++j) {
        const unsigned e = static_cast<unsigned>(j * 32 + lane);
        v[j] = e < n ? sub[e] : make_uint2(0u, 0u);
        const bool kp = e < n && (v[j].x >> 21) >= b1;
        const unsigned bal = __ballot_sync(kFull, kp);
        pos[j] = kept + __popc(bal & lt);
        kept += __popc(bal);
        keepbits |= static_cast<unsigned>(kp) << j;
      }
      if (lane == 0) S.wcnt[warp] = kept;
      __syncthreads();
      if (warp == 0) {
        const unsigned c = lane < kWarps ? S.wcnt[lane] : 0u;
        const unsigned inc = warp_incl_scan(c);
        if (lane < kWarps) S.woff[lane] = inc - c;
        if (lane == 31) S.res[2] = inc;
      }
      __syncthreads();
      M = S.res[2];
      const unsigned o = S.woff[warp];
#pragma unroll
      for (int j = 0; j < kWarpCap / 32; ++j)
        if ((keepbits >> j) & 1u) S.list[o + pos[j]] = v[j];
      __syncthreads();
      // digit 2 (bits 10..20) of the candidates whose first digit is b1
      for (int e = tid; e < static_cast<int>(M); e += kThreads) {
        const uint32_t key = S.list[e].x;
        warp_hist_add(S.h2, (key >> 10) & 2047u, (key >> 21) == b1);
      }
    } else {
      // Back to the two passes: clear the digit-1 histogram and, once every
      // CTA has read its totals, the owners' totals.
      uint4* z = reinterpret_cast<uint4*>(S.h1);
      for (int i = tid; i < kBins1 / 4; i += kThreads) z[i] = make_uint4(0u, 0u, 0u, 0u);
      cluster_sync();
      uint4* zt = reinterpret_cast<uint4*>(S.t1);
      for (int i = tid; i < kBins1 / 4; i += kThreads) zt[i] = make_uint4(0u, 0u, 0u, 0u);
      __syncthreads();
      cluster_arrive();
    }
  }

  if (!filtered) {
    // ---- digit 1 (key bits 21..31) over the slice
    const int nb = (s1 - s0 + PASS - 1) / PASS;
    // Passes over the slice with the next pass's loads in flight.
    float4 raw[KPER / 4];
    uint32_t cur[KPER];
    if (nb > 0) load_tile<KPER / 4, kThreads>(s, s0, tid, s1, raw);
    for (int bt = 0; bt < nb; ++bt) {
      const int tb = s0 + bt * PASS;
      tile_keys(raw, cur);
      if (bt + 1 < nb) load_tile<KPER / 4, kThreads>(s, tb + PASS, tid, s1, raw);
#pragma unroll
      for (int i = 0; i < KPER; ++i) warp_hist_add(S.h1, cur[i] >> 21, tile_token<kThreads>(tb, tid, i) < s1);
    }
    __syncthreads();
    cluster_wait();
    push_bins<kBins1>(S.h1, S.t1, cs);
    cluster_sync();
    {
      // Row totals and this CTA's own counts scanned together (lo | own << 32).
      unsigned c[4], l[4];
      read_totals<kBins1, 4>(S.t1, cs, c);
      const int hi = kBins1 - 4 * tid;
      unsigned sc = 0, sl = 0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        l[j] = S.h1[hslot(hi - 1 - j)];
        sc += c[j];
        sl += l[j];
      }
      const unsigned long long v = static_cast<unsigned long long>(sc) | (static_cast<unsigned long long>(sl) << 32);
      const unsigned long long before = block_excl_scan64(v, S.scan, nullptr);
      unsigned run = static_cast<unsigned>(before), lrun = static_cast<unsigned>(before >> 32);
      const unsigned need = static_cast<unsigned>(keff);
      if (run < need && run + sc >= need) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if (run + c[j] >= need) {
            S.res[0] = static_cast<unsigned>(hi - 1 - j);
            S.res[1] = run;
            S.res[2] = lrun + l[j];   // this CTA's keys with digit 1 >= the threshold's
            break;
          }
          run += c[j];
          lrun += l[j];
        }
      }
      __syncthreads();
      b1 = S.res[0];
      above1 = S.res[1];
      M = S.res[2];
    }

    // ---- compaction of the candidates (digit 1 >= b1), token order; digit 2
    // (bits 10..20) histogram of the keys whose digit 1 equals b1
    lst = (M <= static_cast<unsigned>(kListCap)) ? S.list : p.list + static_cast<size_t>(row) * p.Tmax + s0;
    unsigned base = 0;
    // (with one pass, raw still holds it)
    if (nb > 1) load_tile<KPER / 4, kThreads>(s, s0, tid, s1, raw);
    for (int bt = 0; bt < nb; ++bt) {
      const int tb = s0 + bt * PASS;
      tile_keys(raw, cur);
      if (bt + 1 < nb) load_tile<KPER / 4, kThreads>(s, tb + PASS, tid, s1, raw);
      // Candidates per group of 4 (group g = 2048 contiguous tokens of the
      // pass), packed FB bits per group: one block scan orders them.
      unsigned flags = 0;
      unsigned long long packed = 0;
#pragma unroll
      for (int i = 0; i < KPER; ++i) {
        const bool valid = tile_token<kThreads>(tb, tid, i) < s1;
        const unsigned d1 = cur[i] >> 21;
        if (valid && d1 >= b1) {
          flags |= 1u << i;
          packed += 1ull << (FB * (i >> 2));
        }
        warp_hist_add(S.h2, (cur[i] >> 10) & 2047u, valid && d1 == b1);
      }
      unsigned long long tot;
      const unsigned long long ex = block_excl_scan64(packed, S.scan, &tot);
      unsigned gbase = base;
#pragma unroll
      for (int g = 0; g < KPER / 4; ++g) {
        unsigned pos = gbase + static_cast<unsigned>((ex >> (FB * g)) & ((1u << FB) - 1u));
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = 4 * g + j;
          if ((flags >> i) & 1u) lst[pos++] = make_uint2(cur[i], static_cast<unsigned>(tile_token<kThreads>(tb, tid, i)));
        }
        gbase += static_cast<unsigned>((tot >> (FB * g)) & ((1u << FB) - 1u));
      }
      base = gbase;
    }
  }
  const unsigned need1 = static_cast<unsigned>(keff) - above1;
  __syncthreads();
  push_bins<kBins1>(S.h2, S.t2, cs);
  cluster_sync();
  unsigned d2, need2;
  {
    unsigned c[4];
    read_totals<kBins1, 4>(S.t2, cs, c);
    find_crossing<kBins1, 4>(c, need1, S);
    d2 = S.res[0];
    need2 = need1 - S.res[1];
  }

  // ---- digit 3 (bits 0..9) of the candidates whose top 22 bits match
  const uint32_t hi22 = (b1 << 11) | d2;
  for (int e = tid; e < static_cast<int>(M); e += kThreads) {
    const uint32_t key = lst[e].x;
    warp_hist_add(S.h3, key & 1023u, (key >> 10) == hi22);
  }
  __syncthreads();
  push_bins<kBins3>(S.h3, S.t3, cs);
  cluster_sync();
  uint32_t thr;
  unsigned r_eq;
  {
    unsigned c[2];
    read_totals<kBins3, 2>(S.t3, cs, c);
    find_crossing<kBins3, 2>(c, need2, S);
    thr = (hi22 << 10) | S.res[0];
    r_eq = need2 - S.res[1];   // keys equal to thr that are kept, lowest tokens first
  }

  // ---- output: per-thread contiguous list segments in token order
  const int seg = (static_cast<int>(M) + kThreads - 1) / kThreads;
  const int e0 = min(static_cast<int>(M), tid * seg);
  const int e1 = min(static_cast<int>(M), e0 + seg);
  unsigned gt = 0, eq = 0;
  for (int e = e0; e < e1; ++e) {
    const uint32_t key = lst[e].x;
    gt += key > thr;
    eq += key == thr;
  }
  unsigned long long tot;
  const unsigned long long ex =
      block_excl_scan64(static_cast<unsigned long long>(gt) | (static_cast<unsigned long long>(eq) << 32), S.scan,
                        &tot);
  if (tid == 0) {
    S.cnt[0] = static_cast<unsigned>(tot);
    S.cnt[1] = static_cast<unsigned>(tot >> 32);
  }
  cluster_sync();
  if (tid < 32) {
    unsigned g = 0, e = 0;
    if (static_cast<unsigned>(tid) < q) {
      const uint2 v = cluster_ld2(cluster_map(smem_u32(S.cnt), static_cast<unsigned>(tid)));
      g = v.x;
      e = v.y;
    }
    g = __reduce_add_sync(kFull, g);
    e = __reduce_add_sync(kFull, e);
    if (tid == 0) {
      S.res[2] = g;
      S.res[3] = e;
    }
  }
  __syncthreads();
  cluster_arrive();   // no more reads of other CTAs' shared memory
  const unsigned gt_before = S.res[2], eq_before = S.res[3];
  const unsigned admit = r_eq > eq_before ? r_eq - eq_before : 0u;   // ties this CTA may keep
  unsigned eqr = static_cast<unsigned>(ex >> 32);
  unsigned pos = gt_before + min(r_eq, eq_before) + static_cast<unsigned>(ex) + min(admit, eqr);
  for (int e = e0; e < e1; ++e) {
    const uint2 v = lst[e];
    bool keep = v.x > thr;
    if (v.x == thr) {
      keep = eqr < admit;
      ++eqr;
    }
    if (keep) {
      if (pos < static_cast<unsigned>(p.k)) emit(p, S, row, b, pg0, npg, static_cast<int>(pos), static_cast<int>(v.y));
      ++pos;
    }
  }
  for (int i = keff + static_cast<int>(q) * kThreads + tid; i < p.k; i += static_cast<int>(cs) * kThreads) {
    out[i] = -1;
    if (p.slots) p.slots[static_cast<size_t>(row) * p.k + i] = -1;
  }
  cluster_wait();   // keep this CTA's shared memory until every CTA is done with it
}

// Clusters of `cs` CTAs of variant FILT the current device keeps resident at
// once (cached per device; 0 if unknown). Also sets the kernel's attributes.
template <bool FILT, int KPER = kPer>
int resident_clusters(int cs, int smem) {
  static int cache[64][5] = {};
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  if (!attr_done[dev]) {
    if (cudaFuncSetAttribute(topk_cluster_kernel<FILT, KPER>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) !=
        cudaSuccess)
      return 0;
    if (cudaFuncSetAttribute(topk_cluster_kernel<FILT, KPER>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
        cudaSuccess)
      cudaGetLastError();
    attr_done[dev] = true;
  }
  const int ci = cs == 1 ? 0 : cs == 2 ? 1 : cs == 4 ? 2 : cs == 8 ? 3 : 4;
  int& c = cache[dev][ci];
  if (c) return c > 0 ? c : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<FILT, KPER>, &cfg) != cudaSuccess || n < 0) n = 0;
  cudaGetLastError();
  c = n > 0 ? n : -1;
  return n;
}

}  // namespace

TopkLayout topk_layout(void* base, int R, int Tmax) {
  TopkLayout L;
  const int T1 = Tmax > 0 ? Tmax : 1;
  L.list = base;
  L.bytes = align256(static_cast<size_t>(R) * T1 * 8);
  return L;
}

cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream) {
  const int R = a.B * a.Hkv;
  if (R == 0 || a.k == 0) return cudaSuccess;
  TopkParams p{};
  p.scores = a.scores;
  p.seq_lens = a.seq_lens;
  p.idx = a.idx;
  p.err = a.err;
  p.list = static_cast<uint2*>(a.L.list);
  p.Hkv = a.Hkv;
  p.Tmax = a.Tmax;
  p.lim = a.maxp_tokens < a.Tmax ? a.maxp_tokens : a.Tmax;
  p.k = a.k;
  p.page_table = a.page_table;
  p.slots = a.slots;
  p.ks = a.k_scale;
  p.vs = a.v_scale;
  p.sscale = a.sscale;
  p.maxp = a.maxp;
  p.num_pages = a.num_pages;
  p.pre_wait = a.pre_wait;
  p.bmax = a.bmax;
  p.nbr = (a.Tmax + kMaxBlock - 1) / kMaxBlock;
  const int smem = static_cast<int>(sizeof(Smem));
  const int smem_f = static_cast<int>(sizeof(Smem) + sizeof(FiltX));   // the filtered variant
  // Cluster size: one pass of kBatch scores per CTA where possible, but no
  // more clusters than the device keeps resident at once (a second wave would
  // double the latency-bound selection). The occupancy query assumes an empty
  // GPU: the scan before this kernel has finished when its CTAs start work,
  // and the attention after it is only scheduled once all of them run.
  auto cluster_size = [&](auto resident) {
    int cs = 1;
    while (cs < kMaxCluster && static_cast<long long>(cs) * kBatch < a.Tmax) {
      const int n = resident(cs * 2);
      if (n <= 0 || R > n) break;
      cs *= 2;
    }
    return cs;
  };
  // The filtered variant when full-length rows would take the filtered pass
  // with its cluster size; otherwise the two-CTA-per-SM variant.
  bool filt = false;
  int cs = 1;
  const long long keff_max = a.k < a.Tmax ? a.k : a.Tmax;
  if (filtered_row(2 * kBatch, keff_max, a.Tmax) && resident_clusters<true>(1, smem_f) > 0) {
    cs = cluster_size([&](int c) { return resident_clusters<true>(c, smem_f); });
    filt = filtered_row(((a.Tmax + cs - 1) / cs + 15) & ~15, keff_max, a.Tmax);
  }
  bool wide = false;   // the two-pass variant with 20 keys per thread per pass
  if (!filt) {
    if (resident_clusters<false>(1, smem) <= 0) return cudaErrorNotSupported;
    cs = cluster_size([&](int c) { return resident_clusters<false>(c, smem); });
    // Full-length slices of one pass at 20 keys per thread but two at 16:
    // the wider pass, whose second pass reuses the keys in registers.
    const int slice = ((a.Tmax + cs - 1) / cs + 15) & ~15;
    wide = slice > kBatch && slice <= kThreads * 20 && resident_clusters<false, 20>(cs, smem) >= R;
  }
  if (static_cast<long long>(R) * cs > 0x7fffffffLL) return cudaErrorNotSupported;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(R * cs));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = filt ? smem_f : smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  cudaError_t e = filt   ? cudaLaunchKernelEx(&cfg, topk_cluster_kernel<true>, p)
                  : wide ? cudaLaunchKernelEx(&cfg, topk_cluster_kernel<false, 20>, p)
                         : cudaLaunchKernelEx(&cfg, topk_cluster_kernel<false>, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
