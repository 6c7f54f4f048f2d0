// Stage 3: sparse GQA decode attention over the selected tokens, gathered
// from a paged bf16 or FP8-E4M3 KV cache, with the log-sum-exp merge of the
// split partials.
//
// "Support double sparsity" (sglang PR #1459): attention over the heavy
// tokens only. sglang PR #39721: sparse_gqa over the indexer's selection.
// "QSA HiSparse - SGLang plugin", "Supported versions": FP8 E4M3 KV cache with
// page size 64 (here with one fp32 scale per physical page for K and for V).
// sglang PR #43527, "Distributed QSA execution": owner-side partial outputs
// merged with FP32 log-sum-exp normalisation.
//
// One CTA per (request b, KV head g, split j), 4 warps. The CTA resolves the
// physical slot (index -> page table -> slot) of every selected token of its
// chunk into shared memory, in order, with one prefix sum. Each warp then
// takes every fourth 16-token tile and gathers its K and V rows into its own
// ring of shared-memory stages with 16-byte cp.async copies (rows XOR-swizzled
// by 16-byte chunk so that ldmatrix reads are conflict-free), waiting only on
// its own copies. Per tile the warp computes, on the tensor cores
// (mma.sync m16n8k16, fp32 accumulators):
//   S^T[16 tokens x 8 heads] = K_tile[16 x 128] . Q^T[128 x 8]
//   O^T[128 dims x 8 heads] += V_tile^T[128 x 16] . P^T[16 x 8]
// with the group's G <= 8 query heads as the N = 8 columns, an online softmax
// on the S^T fragments (exp2 domain), and P^T moved into the B-operand layout
// with movmatrix. bf16 caches feed bf16 MMAs directly; e4m3 rows are loaded
// as byte pairs and converted to f16 in registers (the dimension order inside
// each 16-wide step is permuted identically in K and in Q, and the V rows'
// dimension order is undone when writing the output), the query is scaled by
// a power of two into f16 range, and the per-page K scale multiplies the
// logits and the V scale the probabilities. The warps' states are combined in
// shared memory. One split writes bf16 out; several write fp32 partials, or,
// when the splits of a (b, g) run as one thread-block cluster, merge through
// distributed shared memory with no global round trip.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTok = 16;      // tokens per warp tile
constexpr int kSeg = 512;     // selected positions resolved at a time
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
  const int32_t* slots;   // non-null: physical slot per selected position (-1 = skip); idx unused
  const float2* sscale;   // with slots and FP8: (K, V) page scales per selected position
  float* o_part;
  float* lse_part;
  __nv_bfloat16* out;
  float* lse;
  unsigned* err;
  int B, Hq, Hkv, maxp, num_pages, lim, k, S, split_mode, n_known;
  int cluster_merge;   // the S splits of a (b, g) are one cluster: merge in shared memory
  int pre_wait;        // q may be read before waiting on the previous kernel
  float qscale;        // sm_scale * log2(e)
};

// Stores 4 consecutive bf16 outputs (x, y, z, w) * scale as two bf16 pairs
// (the output row offset is a multiple of 4 elements; rows are 4-byte aligned).
__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* dst, float4 v, float scale) {
  __nv_bfloat162* d2 = reinterpret_cast<__nv_bfloat162*>(dst);
  d2[0] = __floats2bfloat162_rn(v.x * scale, v.y * scale);
  d2[1] = __floats2bfloat162_rn(v.z * scale, v.w * scale);
}

template <bool FP8, int D>
struct Cfg {
  static constexpr int ROWB = FP8 ? D : D * 2;   // bytes per K or V row
  // Ring stages per warp. At D = 256 half as many (a 64 KB ring, three CTAs
  // per SM), so that twice the splits stay resident in one wave.
  static constexpr int NST = D == 128 ? (FP8 ? 4 : 2) : (FP8 ? 2 : 1);
  static constexpr int STAGE = 2 * kTok * ROWB;                 // K tile then V tile
  static constexpr int RING = kWarps * NST * STAGE;
  static constexpr int SMEM = RING + kSeg * 4 + (FP8 ? kSeg * 8 : 0);
};

template <int G, bool FP8, int D>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(const AttnParams p) {
  using C = Cfg<FP8, D>;
  constexpr int KS = D / 16;              // 16-wide steps over the head dimension
  constexpr int ROWB = C::ROWB;
  constexpr int NST = C::NST;
  constexpr int CPR = ROWB / 16;          // 16-byte chunks per row
  constexpr int RPI = 32 / CPR;           // rows a warp copies per instruction
  constexpr int NI = kTok / RPI;          // copy instructions per lane per K (or V) tile

  extern __shared__ __align__(128) unsigned char smem[];
  unsigned char* ring = smem;
  int* sl = reinterpret_cast<int*>(smem + C::RING);                 // [kSeg] slots
  float2* sc = reinterpret_cast<float2*>(sl + kSeg);                // [kSeg] (k scale, v scale)
  __shared__ float wm[kWarps][8], wl[kWarps][8];
  __shared__ float cw[kWarps][8];          // each warp's weight per head in the combine
  __shared__ float cm[8], cl[8];
  __shared__ float mw[16][8], mm[8], ml[8];   // each split's normalised weight per head in the merge
  __shared__ unsigned long long sh_scan[33];
  __shared__ unsigned sh_cnt[kWarps];

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int pr = lane >> 2;   // fragment row group
  const int qc = lane & 3;    // fragment column pair
  const int j = blockIdx.x % p.S;
  const int bg = blockIdx.x / p.S;
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;

  // ---- query B fragments: head pr of the group (0 past G), 8 k-steps.
  uint32_t qb[KS][2];
  float qs = p.qscale;
  auto load_q = [&]() {
    float qv[KS][4];
    const bool hv = pr < G;
    const uint16_t* qrow = p.q + (static_cast<long long>(b) * p.Hq + g * G + (hv ? pr : 0)) * D;
#pragma unroll
    for (int kk = 0; kk < KS; ++kk) {
      // bf16: dims 16kk + 2qc (+1) and +8; e4m3 order: dims 16kk + 4qc .. 4qc + 3
      const int d0 = FP8 ? 16 * kk + 4 * qc : 16 * kk + 2 * qc;
      const int d1 = FP8 ? d0 + 2 : d0 + 8;
      const uint32_t w0 = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d0)) : 0u;
      const uint32_t w1 = hv ? __ldg(reinterpret_cast<const uint32_t*>(qrow + d1)) : 0u;
      if (!FP8) {
        qb[kk][0] = w0;
        qb[kk][1] = w1;
      } else {
        qv[kk][0] = bf16_lo(w0);
        qv[kk][1] = bf16_hi(w0);
        qv[kk][2] = bf16_lo(w1);
        qv[kk][3] = bf16_hi(w1);
      }
    }
    if (FP8) {
      // Scale the query by 2^sh so that its largest magnitude lies in
      // [2^13, 2^14): f16 keeps every bf16 mantissa there without overflow.
      float mx = 0.f;
#pragma unroll
      for (int kk = 0; kk < KS; ++kk)
#pragma unroll
        for (int i = 0; i < 4; ++i) mx = fmaxf(mx, fabsf(qv[kk][i]));
#pragma unroll
      for (int o = 16; o; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, o));
      int sh = 0;
      if (mx > 0.f && mx < INFINITY) sh = 13 - (static_cast<int>((__float_as_uint(mx) >> 23) & 0xff) - 127);
      sh = max(-100, min(100, sh));
      const float up = __uint_as_float(static_cast<uint32_t>(127 + sh) << 23);   // 2^sh, exact
      qs = p.qscale * __uint_as_float(static_cast<uint32_t>(127 - sh) << 23);
#pragma unroll
      for (int kk = 0; kk < KS; ++kk) {
        qb[kk][0] = pack_f16(qv[kk][0] * up, qv[kk][1] * up);
        qb[kk][1] = pack_f16(qv[kk][2] * up, qv[kk][3] * up);
      }
    }
  };
  if (p.pre_wait) load_q();
  grid_dependency_wait();
  grid_launch_dependents();
  if (!p.pre_wait) load_q();

  int T = p.seq_lens[b];
  if (T < 0 || T > p.lim) T = T < 0 ? 0 : p.lim;  // flagged by the scoring / top-k stages
  const int32_t* row = p.idx + static_cast<long long>(bg) * p.k;

  int n;
  if (p.n_known) {
    n = min(p.k, T);
  } else {
    unsigned cnt = 0;
    for (int i = tid; i < p.k; i += kThreads) cnt += row[i] >= 0;
#pragma unroll
    for (int o = 16; o; o >>= 1) cnt += __shfl_xor_sync(kFull, cnt, o);
    if (lane == 0) sh_cnt[warp] = cnt;
    __syncthreads();
    n = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) n += sh_cnt[w];
  }
  int p0 = 0, p1 = n;
  if (p.split_mode == 0) {
    p0 = static_cast<int>(static_cast<long long>(j) * n / p.S);
    p1 = static_cast<int>(static_cast<long long>(j + 1) * n / p.S);
  }

  float m0 = -INFINITY, m1 = -INFINITY;   // running max of heads 2qc, 2qc+1 (log2 units)
  float l0 = 0.f, l1 = 0.f;                // this lane's share of the running sums
  float acc[KS][4];
#pragma unroll
  for (int mt = 0; mt < KS; ++mt)
#pragma unroll
    for (int i = 0; i < 4; ++i) acc[mt][i] = 0.f;

  const long long head_off = static_cast<long long>(g) * ROWB;
  const long long slot_stride = static_cast<long long>(p.Hkv) * ROWB;
  unsigned char* wring = ring + warp * NST * C::STAGE;
  const uint32_t wring_s = smem_u32(wring);

  for (int sb = p0; sb < p1; sb += kSeg) {
    const int se = min(p1, sb + kSeg);
    // ---- resolve the slots of this segment, in order: in round i thread t
    // takes position sb + i kThreads + t (coalesced loads), and one scan of
    // the rounds' counts (16 bits each) orders them, round by round.
    constexpr int PPT = kSeg / kThreads;
    static_assert(PPT <= 4, "four 16-bit round counts in the scan");
    int slot_v[PPT];
    float2 sc_v[PPT];
    unsigned long long packed = 0;
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
      const int pos = sb + i * kThreads + tid;
      slot_v[i] = -1;
      sc_v[i] = make_float2(1.f, 1.f);
      if (pos < se && p.slots) {
        const int sv = __ldcg(p.slots + static_cast<long long>(bg) * p.k + pos);
        // Loaded with the slot, not after it: one round trip for both.
        const float2 given = (FP8 && p.sscale) ? __ldcg(p.sscale + static_cast<long long>(bg) * p.k + pos)
                                               : make_float2(1.f, 1.f);
        if (sv >= 0) {
          slot_v[i] = sv;
          if (FP8) sc_v[i] = p.sscale ? given : make_float2(__ldg(p.ks + sv / kPage), __ldg(p.vs + sv / kPage));
          packed += 1ull << (16 * i);
        }
      } else if (pos < se) {
        const int t = row[pos];
        bool ok = t >= 0;
        if (ok && t >= T) {
          flag_error(p.err, 4u);
          ok = false;
        }
        if (ok && p.split_mode == 1 && (t / kPage) % p.S != j) ok = false;
        if (ok) {
          const int pid = __ldg(p.page_table + static_cast<long long>(b) * p.maxp + t / kPage);
          if (pid < 0 || pid >= p.num_pages) {
            flag_error(p.err, 2u);
          } else {
            slot_v[i] = pid * kPage + (t & (kPage - 1));
            if (FP8) sc_v[i] = make_float2(__ldg(p.ks + pid), __ldg(p.vs + pid));
            packed += 1ull << (16 * i);
          }
        }
      }
    }
    unsigned long long tot;
    const unsigned long long ex = block_excl_scan64(packed, sh_scan, &tot);
    unsigned nseg_u = 0;
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
      if (slot_v[i] >= 0) {
        const unsigned wpos = nseg_u + static_cast<unsigned>((ex >> (16 * i)) & 65535u);
        sl[wpos] = slot_v[i];
        if (FP8) sc[wpos] = sc_v[i];
      }
      nseg_u += static_cast<unsigned>((tot >> (16 * i)) & 65535u);
    }
    __syncthreads();
    const int nseg = static_cast<int>(nseg_u);
    const int ntile = (nseg + kTok - 1) / kTok;
    const int nt_w = ntile > warp ? (ntile - warp + kWarps - 1) / kWarps : 0;   // this warp's tiles

    // Copies of tile `tile` into stage `st` of this warp's ring: chunk c of
    // row r lands at chunk position c ^ (r & 7).
    auto issue = [&](int tile, int st) {
      unsigned char* dst = wring + st * C::STAGE;
      const int c = lane % CPR;
#pragma unroll
      for (int i = 0; i < NI; ++i) {
        const int r = lane / CPR + RPI * i;
        const int e = tile * kTok + r;
        const bool ok = e < nseg;
        const long long off = ok ? static_cast<long long>(sl[e]) * slot_stride + head_off + c * 16 : 0;
        const int so = r * ROWB + ((c ^ (r & 7)) << 4);
        cp_async16(dst + so, p.kc + off, ok);
        cp_async16(dst + kTok * ROWB + so, p.vc + off, ok);
      }
    };

#pragma unroll
    for (int s = 0; s < NST; ++s) {
      if (s < nt_w) issue(warp + kWarps * s, s);
      cp_async_commit();
    }
    for (int it = 0; it < nt_w; ++it) {
      const int st = it % NST;
      const int tile = warp + kWarps * it;
      cp_async_wait<NST - 1>();
      __syncwarp();
      const uint32_t kb = wring_s + st * C::STAGE;
      const uint32_t vb = kb + kTok * ROWB;

      // ---- S^T = K . Q^T
      float sa[4] = {0.f, 0.f, 0.f, 0.f};
      if (!FP8) {
        const int r = lane & 15;
        const uint32_t rb = kb + r * ROWB;
        const int x = (lane >> 4) ^ (r & 7);
#pragma unroll
        for (int kk = 0; kk < KS; ++kk) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(rb + (((2 * kk) ^ x) << 4), a0, a1, a2, a3);
          mma_bf16(sa, a0, a1, a2, a3, qb[kk][0], qb[kk][1]);
        }
      } else {
        const int mi = lane >> 3;
        const int r = (lane & 7) + 8 * (mi & 1);
        const uint32_t rb = kb + r * ROWB;
        const int x = (mi >> 1) ^ (lane & 7);
#pragma unroll
        for (int cc = 0; cc < KS / 2; ++cc) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(rb + (((2 * cc) ^ x) << 4), r0, r1, r2, r3);
          mma_f16(sa, e4m3x2_to_f16x2(r0), e4m3x2_to_f16x2(r1), e4m3x2_to_f16x2(r0 >> 16),
                  e4m3x2_to_f16x2(r1 >> 16), qb[2 * cc][0], qb[2 * cc][1]);
          mma_f16(sa, e4m3x2_to_f16x2(r2), e4m3x2_to_f16x2(r3), e4m3x2_to_f16x2(r2 >> 16),
                  e4m3x2_to_f16x2(r3 >> 16), qb[2 * cc + 1][0], qb[2 * cc + 1][1]);
        }
      }

      // ---- online softmax on tokens pr (lo) and pr + 8 (hi), heads 2qc, 2qc + 1
      const int e_lo = tile * kTok + pr;
      const int e_hi = e_lo + 8;
      float kl = qs, kh = qs, vl = 1.f, vh = 1.f;
      if (FP8) {
        if (e_lo < nseg) {
          const float2 t = sc[e_lo];
          kl *= t.x;
          vl = t.y;
        }
        if (e_hi < nseg) {
          const float2 t = sc[e_hi];
          kh *= t.x;
          vh = t.y;
        }
      }
      const float s0 = e_lo < nseg ? sa[0] * kl : -INFINITY;
      const float s1 = e_lo < nseg ? sa[1] * kl : -INFINITY;
      const float s2 = e_hi < nseg ? sa[2] * kh : -INFINITY;
      const float s3 = e_hi < nseg ? sa[3] * kh : -INFINITY;
      float t0 = fmaxf(s0, s2), t1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        t0 = fmaxf(t0, __shfl_xor_sync(kFull, t0, o));
        t1 = fmaxf(t1, __shfl_xor_sync(kFull, t1, o));
      }
      const float n0 = fmaxf(m0, t0), n1 = fmaxf(m1, t1);   // finite: the tile has a valid token
      const float c0 = exp2f(m0 - n0), c1 = exp2f(m1 - n1);
      m0 = n0;
      m1 = n1;
      const float e0 = exp2f(s0 - n0), e1 = exp2f(s1 - n1), e2 = exp2f(s2 - n0), e3 = exp2f(s3 - n1);
      l0 = l0 * c0 + e0 + e2;
      l1 = l1 * c1 + e1 + e3;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        acc[mt][0] *= c0;
        acc[mt][1] *= c1;
        acc[mt][2] *= c0;
        acc[mt][3] *= c1;
      }
      uint32_t pb0, pb1;
      if (!FP8) {
        pb0 = movm_t(pack_bf16(e0, e1));
        pb1 = movm_t(pack_bf16(e2, e3));
      } else {
        pb0 = movm_t(pack_f16(e0 * vl, e1 * vl));
        pb1 = movm_t(pack_f16(e2 * vh, e3 * vh));
      }

      // ---- O^T += V^T . P^T
      {
        const int mi = lane >> 3;
        if (!FP8) {
          // matrices: (tokens 0-7, chunk 2mt), (tokens 0-7, chunk 2mt+1),
          //           (tokens 8-15, chunk 2mt), (tokens 8-15, chunk 2mt+1)
          const uint32_t rb = vb + ((lane & 7) + 8 * (mi >> 1)) * ROWB;
          const int x = (mi & 1) ^ (lane & 7);
#pragma unroll
          for (int mt = 0; mt < KS; ++mt) {
            uint32_t a0, a1, a2, a3;
            ldsm_x4_t(rb + (((2 * mt) ^ x) << 4), a0, a1, a2, a3);
            mma_bf16(acc[mt], a0, a1, a2, a3, pb0, pb1);
          }
        } else {
          // matrices: (tokens 0-7, chunk 2cc), (tokens 8-15, chunk 2cc),
          //           (tokens 0-7, chunk 2cc+1), (tokens 8-15, chunk 2cc+1)
          const int r8 = (lane & 7) + 8 * (mi & 1);
          const uint32_t rb8 = vb + r8 * ROWB;
          const int x = (mi >> 1) ^ (lane & 7);
#pragma unroll
          for (int cc = 0; cc < KS / 2; ++cc) {
            uint32_t r0, r1, r2, r3;
            ldsm_x4_t(rb8 + (((2 * cc) ^ x) << 4), r0, r1, r2, r3);
            // (token 2qc, dims 2pr, 2pr+1), (token 2qc+1, ...) -> per-dim token pairs
            const uint32_t u0 = __byte_perm(r0, 0, 0x3120), u1 = __byte_perm(r1, 0, 0x3120);
            const uint32_t u2 = __byte_perm(r2, 0, 0x3120), u3 = __byte_perm(r3, 0, 0x3120);
            mma_f16(acc[2 * cc], e4m3x2_to_f16x2(u0), e4m3x2_to_f16x2(u0 >> 16), e4m3x2_to_f16x2(u1),
                    e4m3x2_to_f16x2(u1 >> 16), pb0, pb1);
            mma_f16(acc[2 * cc + 1], e4m3x2_to_f16x2(u2), e4m3x2_to_f16x2(u2 >> 16), e4m3x2_to_f16x2(u3),
                    e4m3x2_to_f16x2(u3 >> 16), pb0, pb1);
          }
        }
      }
      __syncwarp();
      if (it + NST < nt_w) issue(warp + kWarps * (it + NST), st);
      cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();
  }

  // ---- this warp's state -> shared memory (the ring is free now)
#pragma unroll
  for (int o = 4; o < 32; o <<= 1) {
    l0 += __shfl_xor_sync(kFull, l0, o);
    l1 += __shfl_xor_sync(kFull, l1, o);
  }
  float* wo = reinterpret_cast<float*>(ring);   // [kWarps][G][D]
  const int h0 = 2 * qc, h1 = 2 * qc + 1;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    // bf16: rows pr / pr + 8 are dims 16mt + pr / + 8; e4m3: dims 16mt + 2pr / + 1
    const int da = FP8 ? 16 * mt + 2 * pr : 16 * mt + pr;
    const int db = FP8 ? da + 1 : da + 8;
    if (h0 < G) {
      wo[(warp * G + h0) * D + da] = acc[mt][0];
      wo[(warp * G + h0) * D + db] = acc[mt][2];
    }
    if (h1 < G) {
      wo[(warp * G + h1) * D + da] = acc[mt][1];
      wo[(warp * G + h1) * D + db] = acc[mt][3];
    }
  }
  if (pr == 0) {
    if (h0 < G) {
      wm[warp][h0] = m0;
      wl[warp][h0] = l0;
    }
    if (h1 < G) {
      wm[warp][h1] = m1;
      wl[warp][h1] = l1;
    }
  }
  __syncthreads();

  // ---- combine the warps: state (M, L, O unnormalised) per (head, dim); each
  // warp's weight per head is computed once, and the outputs go 4 dims at a time
  float* co = wo + kWarps * G * D;   // [G][D]
  if (tid < G) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) M = fmaxf(M, wm[w][tid]);
    float L = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = (M == -INFINITY || wm[w][tid] == -INFINITY) ? 0.f : exp2f(wm[w][tid] - M);
      cw[w][tid] = wt;
      L += wt * wl[w][tid];
    }
    cm[tid] = M;
    cl[tid] = L;
  }
  __syncthreads();
  for (int e = 4 * tid; e < G * D; e += 4 * kThreads) {
    const int h = e / D;
    const int d = e % D;
    float4 acc_o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      const float wt = cw[w][h];
      const float4 v = *reinterpret_cast<const float4*>(wo + (w * G + h) * D + d);
      acc_o.x += wt * v.x;
      acc_o.y += wt * v.y;
      acc_o.z += wt * v.z;
      acc_o.w += wt * v.w;
    }
    const float M = cm[h];
    const float L = cl[h];
    const long long qrow = static_cast<long long>(b) * p.Hq + g * G + h;
    if (p.cluster_merge) {
      *reinterpret_cast<float4*>(co + e) = acc_o;
    } else if (p.S == 1) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      store_bf16x4(p.out + qrow * D + d, acc_o, inv);
      if (d == 0 && p.lse) p.lse[qrow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    } else {
      const long long prow = static_cast<long long>(j) * p.B * p.Hq + qrow;
      const float inv = L > 0.f ? 1.f / L : 0.f;
      float* op = p.o_part + prow * D + d;
      op[0] = acc_o.x * inv;
      op[1] = acc_o.y * inv;
      op[2] = acc_o.z * inv;
      op[3] = acc_o.w * inv;
      if (d == 0) p.lse_part[prow] = L > 0.f ? (M + log2f(L)) * kLn2 : -INFINITY;
    }
  }
  if (!p.cluster_merge) return;

  // ---- merge the cluster's S splits. Every CTA reads each split's (M, L) per
  // head once and turns them into normalised weights; CTA j then finishes
  // elements [e0, e1) of G x D, 4 at a time, from every split's partial.
  cluster_sync();
  if (tid < G) {
    float Ms[16], Ls[16];
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < p.S) {
        Ms[s] = __uint_as_float(cluster_ld(cluster_map(smem_u32(cm + tid), s)));
        Ls[s] = __uint_as_float(cluster_ld(cluster_map(smem_u32(cl + tid), s)));
        M = fmaxf(M, Ms[s]);
      }
    }
    float L = 0.f;
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < p.S && M != -INFINITY && Ms[s] != -INFINITY) L += exp2f(Ms[s] - M) * Ls[s];
#pragma unroll
    for (int s = 0; s < 16; ++s)
      if (s < p.S) mw[s][tid] = (L > 0.f && Ms[s] != -INFINITY) ? exp2f(Ms[s] - M) / L : 0.f;
    mm[tid] = M;
    ml[tid] = L;
  }
  __syncthreads();
  const int E = G * D;
  const int e0 = j * E / p.S, e1 = (j + 1) * E / p.S;   // multiples of 4 (E and S powers of two, E / S >= 8)
  for (int e = e0 + 4 * tid; e < e1; e += 4 * kThreads) {
    const int h = e / D;
    const int d = e % D;
    float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < 16; ++s) {
      if (s < p.S) {
        const uint4 u = cluster_ld4(cluster_map(smem_u32(co + e), s));
        const float wt = mw[s][h];
        o.x += wt * __uint_as_float(u.x);
        o.y += wt * __uint_as_float(u.y);
        o.z += wt * __uint_as_float(u.z);
        o.w += wt * __uint_as_float(u.w);
      }
    }
    const long long qrow = static_cast<long long>(b) * p.Hq + g * G + h;
    store_bf16x4(p.out + qrow * D + d, o, 1.f);
    const float L = ml[h];
    if (d == 0 && p.lse) p.lse[qrow] = L > 0.f ? (mm[h] + log2f(L)) * kLn2 : -INFINITY;
  }
  cluster_sync();   // keep this CTA's shared memory until every CTA has read it
}

using KernelFn = void (*)(const AttnParams);

template <bool FP8, int D>
KernelFn pick_g(int G) {
  switch (G) {
    case 1: return sparse_attn_kernel<1, FP8, D>;
    case 2: return sparse_attn_kernel<2, FP8, D>;
    case 4: return sparse_attn_kernel<4, FP8, D>;
    case 8: return sparse_attn_kernel<8, FP8, D>;
  }
  return nullptr;
}

KernelFn pick(int G, int fp8, int D) {
  if (D == 128) return fp8 ? pick_g<true, 128>(G) : pick_g<false, 128>(G);
  if (D == 256) return fp8 ? pick_g<true, 256>(G) : pick_g<false, 256>(G);
  return nullptr;
}

int smem_bytes(int fp8, int D) {
  if (D == 256) return fp8 ? Cfg<true, 256>::SMEM : Cfg<false, 256>::SMEM;
  return fp8 ? Cfg<true, 128>::SMEM : Cfg<false, 128>::SMEM;
}

cudaError_t prepare(KernelFn fn, int bytes) {
  struct Entry { KernelFn fn; int dev; };
  static Entry done[64];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < n; ++i)
    if (done[i].fn == fn && done[i].dev == dev) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
  if (e != cudaSuccess) {
    cudaGetLastError();   // clusters stay at the portable size
  }
  if (n < 64) done[n++] = Entry{fn, dev};
  return cudaSuccess;
}

}  // namespace

bool sparse_attn_supported(int G, int D) { return pick(G, 0, D) != nullptr; }

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  KernelFn fn = pick(G, a.fp8, a.D);
  if (!fn) return cudaErrorNotSupported;
  const long long blocks = static_cast<long long>(a.B) * a.Hkv * a.S;
  if (blocks == 0) return cudaSuccess;
  // The merge hands each CTA G * D / S outputs, 4 at a time: S a power of two up to 16.
  if (a.cluster_merge && (a.S > 16 || (a.S & (a.S - 1)) || a.split_mode != 0)) return cudaErrorInvalidValue;
  AttnParams p{};
  p.q = static_cast<const uint16_t*>(a.q);
  p.kc = static_cast<const uint8_t*>(a.k_cache);
  p.vc = static_cast<const uint8_t*>(a.v_cache);
  p.ks = a.k_scale;
  p.vs = a.v_scale;
  p.page_table = a.page_table;
  p.seq_lens = a.seq_lens;
  p.idx = a.idx;
  p.slots = a.slots;
  p.sscale = a.sscale;
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
  p.cluster_merge = a.cluster_merge;
  p.pre_wait = a.pre_wait;
  const int smem = smem_bytes(a.fp8, a.D);
  cudaError_t e = prepare(fn, smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = a.cluster_merge ? a.S : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, fn, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

int sparse_attn_resident_clusters(int G, int fp8, int S, int D) {
  static int cache[2][2][9][5][64] = {};
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || G < 1 || G > 8) {
    cudaGetLastError();
    return 0;
  }
  const int si = S == 1 ? 0 : S == 2 ? 1 : S == 4 ? 2 : S == 8 ? 3 : S == 16 ? 4 : -1;
  if (si < 0) return 0;
  if (D != 128 && D != 256) return 0;
  int& c = cache[D == 256 ? 1 : 0][fp8 ? 1 : 0][G][si][dev];
  if (c) return c > 0 ? c : 0;
  KernelFn fn = pick(G, fp8, D);
  if (!fn) return 0;
  const int smem = smem_bytes(fp8, D);
  if (prepare(fn, smem) != cudaSuccess) return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = S;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, fn, &cfg) != cudaSuccess || n < 0) n = 0;
  cudaGetLastError();
  c = n > 0 ? n : -1;
  return n;
}

}  // namespace ds
