// Stage 3: sparse GQA decode attention over the selected tokens, gathered
// from a paged bf16 or FP8-E4M3 KV cache, with the log-sum-exp merge of the
// split partials optionally fused into the last CTA of each (request, KV head).
//
// "Support double sparsity" (sglang PR #1459): attention over the heavy
// tokens only. sglang PR #39721: sparse_gqa over the indexer's selection.
// "QSA HiSparse - SGLang plugin", "Supported versions": FP8 E4M3 KV cache with
// page size 64 (here with one fp32 scale per physical page for K and for V).
// sglang PR #43527, "Distributed QSA execution": owner-side partial outputs
// merged with FP32 log-sum-exp normalisation.
//
// One CTA per (request b, KV head g, split j), 4 warps. The CTA first
// resolves the physical slot (index -> page table -> slot) of every selected
// token of its chunk into shared memory, in order, with one prefix sum. The
// K and V rows of those slots are then gathered in tiles of 32 tokens
// through a ring of cp.async stages (16-byte copies; a bf16 row is 256 B,
// an e4m3 row 128 B), so the gather keeps many rows in flight per SM. Each
// warp takes 8 tokens of a tile: one K or V row is read by the whole warp in
// one conflict-free shared-memory instruction (dims 4l..4l+3 in lane l); the
// G query heads of the group are in registers (pre-scaled by sm_scale*log2 e),
// a transposed butterfly turns the J x G partial dot products into one logit
// per lane, and online softmax accumulates P.V into 4 dims x G heads per lane.
// The warps' states are combined in shared memory; the CTA writes the final
// bf16 output (one split) or fp32 partials, and with a fused merge the CTA
// that finishes a (b, g) last merges all splits.
#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace ds {

namespace {

constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTile = 32;     // tokens per gather stage
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
  float* o_part;
  float* lse_part;
  __nv_bfloat16* out;
  float* lse;
  unsigned* err;
  unsigned* merge_done;
  int B, Hq, Hkv, maxp, num_pages, lim, k, S, split_mode, n_known, nst;
  float qscale;  // sm_scale * log2(e)
};

template <int G, bool FP8>
__global__ void __launch_bounds__(kThreads) sparse_attn_kernel(const AttnParams p) {
  constexpr int J = (G >= 4) ? 32 / G : 8;   // tokens per sub-tile
  constexpr int V = J * G;                   // logits per sub-tile (<= 32)
  constexpr int SH = (V >= 32) ? 0 : (V == 16 ? 1 : (V == 8 ? 2 : 3));  // lane -> value shift
  constexpr int ROWB = FP8 ? kHeadDim : kHeadDim * 2;  // bytes per K/V row
  constexpr int CPR = ROWB / 16;                        // 16-byte copies per row
  constexpr int STAGE = 2 * kTile * ROWB;               // K tile then V tile
  constexpr int CPT = 2 * kTile * CPR / kThreads;       // copies per thread per stage
  constexpr int WTOK = kTile / kWarps;                  // tokens per warp per tile (8)

  extern __shared__ __align__(16) unsigned char smem[];
  unsigned char* ring = smem;
  int* sl = reinterpret_cast<int*>(smem + static_cast<size_t>(p.nst) * STAGE);   // [kSeg] slots
  float2* sc = reinterpret_cast<float2*>(sl + kSeg);                             // [kSeg] (kscale, vscale)
  __shared__ float sm_m[kWarps][G];
  __shared__ float sm_l[kWarps][G];
  __shared__ float sm_o[kWarps][G][kHeadDim];
  __shared__ unsigned sh_scan[33];
  __shared__ unsigned sh_cnt[kWarps];
  __shared__ int sh_last;

  const int tid = threadIdx.x;
  const int lane = tid & 31;
  const int warp = tid >> 5;
  const int j = blockIdx.x % p.S;
  const int bg = blockIdx.x / p.S;
  const int g = bg % p.Hkv;
  const int b = bg / p.Hkv;
  const int32_t* row = p.idx + static_cast<long long>(bg) * p.k;
  grid_dependency_wait();

  int T = p.seq_lens[b];
  if (T < 0 || T > p.lim) T = T < 0 ? 0 : p.lim;  // flagged by the scoring / top-k stages

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

  // Query heads g*G .. g*G+G-1, dims 4*lane .. 4*lane+3, scaled to log2 units.
  float qf[G][4];
#pragma unroll
  for (int h = 0; h < G; ++h) {
    const uint2 w = __ldg(reinterpret_cast<const uint2*>(p.q + (static_cast<long long>(b) * p.Hq + g * G + h) * kHeadDim + lane * 4));
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

  const long long head_off = static_cast<long long>(g) * ROWB;
  const long long slot_stride = static_cast<long long>(p.Hkv) * ROWB;

  for (int sb = p0; sb < p1; sb += kSeg) {
    const int se = min(p1, sb + kSeg);
    // ---- resolve the slots of this segment, in order
    constexpr int PPT = kSeg / kThreads;
    int slot_v[PPT];
    float2 sc_v[PPT];
    unsigned cnt = 0;
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
      const int pos = sb + tid * PPT + i;
      slot_v[i] = -1;
      sc_v[i] = make_float2(1.f, 1.f);
      if (pos < se) {
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
            ++cnt;
          }
        }
      }
    }
    unsigned nseg;
    unsigned wpos = block_excl_scan(cnt, sh_scan, &nseg);
#pragma unroll
    for (int i = 0; i < PPT; ++i) {
      if (slot_v[i] >= 0) {
        sl[wpos] = slot_v[i];
        if (FP8) sc[wpos] = sc_v[i];
        ++wpos;
      }
    }
    __syncthreads();
    const int ntile = (static_cast<int>(nseg) + kTile - 1) / kTile;

    auto issue = [&](int tile, int stage) {
      unsigned char* dst = ring + stage * STAGE;
#pragma unroll
      for (int c = 0; c < CPT; ++c) {
        const int id = c * kThreads + tid;          // 0 .. 2*kTile*CPR-1
        const int kv = id / (kTile * CPR);          // 0: K, 1: V
        const int r = (id / CPR) % kTile;
        const int part = id % CPR;
        const int e = tile * kTile + r;
        const bool ok = e < static_cast<int>(nseg);
        const uint8_t* base = kv ? p.vc : p.kc;
        const uint8_t* src = ok ? base + sl[e] * slot_stride + head_off + part * 16 : base;
        cp_async16(dst + id * 16, src, ok);
      }
    };

    for (int s = 0; s < p.nst; ++s) {
      if (s < ntile) issue(s, s);
      cp_async_commit();
    }
    for (int tile = 0; tile < ntile; ++tile) {
      const int stage = tile % p.nst;
      cp_async_wait_dyn(p.nst - 1);
      __syncthreads();
      const unsigned char* kt = ring + stage * STAGE;
      const unsigned char* vt = kt + kTile * ROWB;
      const int tok_base = tile * kTile + warp * WTOK;   // entry index of this warp's first token
#pragma unroll
      for (int sub = 0; sub < WTOK / J; ++sub) {
        const int r0 = warp * WTOK + sub * J;           // row within the tile
        const int e0 = tok_base + sub * J;              // entry index
        const int nvalid = min(J, static_cast<int>(nseg) - e0);
        if (nvalid <= 0) break;
        float part[V];
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          float k0, k1, k2, k3;
          if (FP8) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(kt + (r0 + jj) * ROWB + lane * 4);
            const float2 a = e4m3x2_to_float2(w);
            const float2 c = e4m3x2_to_float2(w >> 16);
            k0 = a.x; k1 = a.y; k2 = c.x; k3 = c.y;
          } else {
            const uint2 w = *reinterpret_cast<const uint2*>(kt + (r0 + jj) * ROWB + lane * 8);
            k0 = bf16_lo(w.x); k1 = bf16_hi(w.x); k2 = bf16_lo(w.y); k3 = bf16_hi(w.y);
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
        const bool tv = my_j < nvalid;
        float2 scl = make_float2(1.f, 1.f);
        if (FP8 && tv) scl = sc[e0 + my_j];
        const float z = tv ? part[0] * scl.x : -INFINITY;
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
        const float pv = FP8 ? pw * scl.y : pw;
#pragma unroll
        for (int h = 0; h < G; ++h)
#pragma unroll
          for (int i = 0; i < 4; ++i) o[h][i] *= corr[h];
#pragma unroll
        for (int jj = 0; jj < J; ++jj) {
          float v0, v1, v2, v3;
          if (FP8) {
            const uint32_t w = *reinterpret_cast<const uint32_t*>(vt + (r0 + jj) * ROWB + lane * 4);
            const float2 a = e4m3x2_to_float2(w);
            const float2 c = e4m3x2_to_float2(w >> 16);
            v0 = a.x; v1 = a.y; v2 = c.x; v3 = c.y;
          } else {
            const uint2 w = *reinterpret_cast<const uint2*>(vt + (r0 + jj) * ROWB + lane * 8);
            v0 = bf16_lo(w.x); v1 = bf16_hi(w.x); v2 = bf16_lo(w.y); v3 = bf16_hi(w.y);
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
      __syncthreads();
      if (tile + p.nst < ntile) issue(tile + p.nst, stage);
      cp_async_commit();
    }
    cp_async_wait<0>();
    __syncthreads();
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
  for (int e = tid; e < G * kHeadDim; e += kThreads) {
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
  if (p.S == 1 || !p.merge_done) return;

  // ---- fused merge: the CTA that finishes (b, g) last merges its S splits.
  __threadfence();
  __syncthreads();
  if (tid == 0) sh_last = (atomicAdd(p.merge_done + bg, 1u) + 1 == static_cast<unsigned>(p.S));
  __syncthreads();
  if (!sh_last) return;
  __threadfence();
  const long long rows = static_cast<long long>(p.B) * p.Hq;
  const long long qrow0 = static_cast<long long>(b) * p.Hq + g * G;
  // All split lse values of the group's heads in one round of loads, then the
  // merge weights exp(lse_s - lse) in shared memory (reusing the ring).
  float* sw = reinterpret_cast<float*>(ring);          // [S][G] weights
  float* slse = sw + p.S * G;                          // [G] merged lse
  for (int i = tid; i < p.S * G; i += kThreads) sw[i] = __ldcg(p.lse_part + (i / G) * rows + qrow0 + (i % G));
  __syncthreads();
  if (tid < G) {
    float M = -INFINITY;
    for (int s = 0; s < p.S; ++s) M = fmaxf(M, sw[s * G + tid]);
    float L = 0.f;
    if (M != -INFINITY)
      for (int s = 0; s < p.S; ++s) L += expf(sw[s * G + tid] - M);
    const float lse = (M == -INFINITY) ? -INFINITY : M + logf(L);
    slse[tid] = lse;
    for (int s = 0; s < p.S; ++s) {
      const float ls = sw[s * G + tid];
      sw[s * G + tid] = (ls == -INFINITY) ? 0.f : expf(ls - lse);
    }
  }
  __syncthreads();
  for (int e = tid; e < G * kHeadDim; e += kThreads) {
    const int h = e / kHeadDim;
    const int d = e % kHeadDim;
    float acc = 0.f;
    for (int s0 = 0; s0 < p.S; s0 += 8) {
      float v[8];
#pragma unroll
      for (int i = 0; i < 8; ++i)
        v[i] = (s0 + i < p.S) ? __ldcg(p.o_part + ((s0 + i) * rows + qrow0 + h) * kHeadDim + d) : 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (s0 + i < p.S) acc = fmaf(sw[(s0 + i) * G + h], v[i], acc);
    }
    p.out[(qrow0 + h) * kHeadDim + d] = __float2bfloat16_rn(acc);
    if (d == 0 && p.lse) p.lse[qrow0 + h] = slse[h];
  }
  if (tid == 0) atomicExch(p.merge_done + bg, 0u);
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

cudaError_t allow_smem(KernelFn fn, int bytes) {
  struct Entry { KernelFn fn; int dev; int bytes; };
  static Entry done[64];
  static int n = 0;
  int dev = 0;
  cudaGetDevice(&dev);
  for (int i = 0; i < n; ++i)
    if (done[i].fn == fn && done[i].dev == dev && done[i].bytes >= bytes) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess && n < 64) done[n++] = Entry{fn, dev, bytes};
  return e;
}

}  // namespace

bool sparse_attn_supported(int G) { return pick<false>(G) != nullptr; }

cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream) {
  const int G = a.Hq / a.Hkv;
  KernelFn fn = a.fp8 ? pick<true>(G) : pick<false>(G);
  if (!fn) return cudaErrorNotSupported;
  const long long blocks = static_cast<long long>(a.B) * a.Hkv * a.S;
  if (blocks == 0) return cudaSuccess;
  AttnParams p{};
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
  p.merge_done = a.merge_done;
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
  const int rowb = a.fp8 ? kHeadDim : kHeadDim * 2;
  const int stage = 2 * kTile * rowb;
  p.nst = a.fp8 ? 6 : 4;
  const int smem = p.nst * stage + kSeg * (a.fp8 ? 4 + 8 : 4);
  cudaError_t e = allow_smem(fn, smem);
  if (e != cudaSuccess) return e;
  e = launch_pdl(fn, dim3(static_cast<unsigned>(blocks)), dim3(kThreads), smem, stream, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace ds
