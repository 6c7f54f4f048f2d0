// Host-side launchers shared between the C ABI (api.cu) and the kernel files.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

namespace ds {

constexpr int kHeadDimMax = 256;  // head dimensions: 128 and 256
constexpr int kPageSupported = 64;
constexpr long long kDecodeTargetCtas = 456;  // attention CTAs the chained call aims for (3 per SM)

// Streaming multiprocessors of the current device (cached per device).
int sm_count();

// Scratch of the exact top-k for R rows of up to Tmax scores: a (key, token)
// list per row, used only by rows whose candidates overflow shared memory.
// Needs no initialisation.
struct TopkLayout {
  void* list;        // uint2 [R, Tmax]
  size_t bytes;
};
TopkLayout topk_layout(void* base, int R, int Tmax);

struct ScoreArgs {
  const void* qp;          // bf16 [B, Hq, C]
  const void* label;       // bf16 [slots, HL, C]
  const int32_t* page_table;
  const int32_t* seq_lens;
  float* scores;           // [B, Hkv, Tmax]
  unsigned* err;
  int B, Hq, Hkv, HL, C, maxp, num_pages, Tmax;
  float* bmax;             // [B, Hkv, ceil(Tmax / 16)] largest score of each 16-token block, or null
                           // (written only by kernels for which index_score_block_maxima is true)
};
// Returns a cudaError_t; cudaErrorNotSupported for shapes without a kernel.
cudaError_t launch_index_score(const ScoreArgs& a, cudaStream_t stream);
bool index_score_supported(int C, int HL, int Hkv, int G);
// Whether the scan for this shape also writes the 16-token block maxima.
bool index_score_block_maxima(int C, int HL, int Hkv);
constexpr int kMaxBlock = 16;   // tokens per block of the block maxima

struct TopkArgs {
  const float* scores;     // [B, Hkv, Tmax]
  const int32_t* seq_lens;
  int32_t* idx;            // [B, Hkv, k]
  unsigned* err;
  int B, Hkv, Tmax, maxp_tokens, k;
  TopkLayout L;
  // Chained call only (slots == nullptr otherwise): physical slots of the kept
  // tokens ([B, Hkv, k], -1 past K_eff) and, with an FP8 cache (sscale
  // non-null), the (K, V) scales of their pages.
  int32_t* slots;
  const int32_t* page_table;
  const float* k_scale;
  const float* v_scale;
  float2* sscale;          // [B, Hkv, k]
  int maxp, num_pages;
  int pre_wait;            // inputs may be read before the previous kernel completes
  // Largest score of each 16-token block of each row ([B, Hkv, ceil(Tmax / 16)],
  // exactly the maxima of `scores`), or null. Long rows with a small k use
  // them to read only the blocks that can hold a kept token.
  const float* bmax;
};
cudaError_t launch_topk(const TopkArgs& a, cudaStream_t stream);

// Top-k by S page-interleaved shards and an exact merge (ds_topk_select_sharded).
size_t topk_sharded_workspace_bytes(int R, int Tmax, int k, int S);
cudaError_t launch_topk_sharded(const float* scores, const int32_t* seq_lens, int B, int Hkv, int Tmax, int lim,
                                int k, int S, int32_t* idx, void* ws, unsigned* err, cudaStream_t stream);

struct AttnArgs {
  const void* q;           // bf16 [B, Hq, D]
  const void* k_cache;     // [slots, Hkv, D]
  const void* v_cache;
  const float* k_scale;    // [num_pages] (fp8)
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  const int32_t* idx;      // [B, Hkv, k]
  float* o_part;           // [S, B, Hq, D] (S > 1)
  float* lse_part;         // [S, B, Hq]
  void* out;               // bf16 [B, Hq, D] (S == 1, or S > 1 with a fused merge)
  float* lse;              // [B, Hq] (may be null)
  unsigned* err;
  int B, Hq, Hkv, maxp, num_pages, Tmax, k, S, split_mode, fp8;
  float sm_scale;
  const int32_t* slots;    // non-null: physical slots per selected position ([B, Hkv, k], -1 = skip), idx unused
  const float2* sscale;    // with slots and an FP8 cache: the (K, V) page scales per selected position
  int n_from_seq_len;      // 1: each idx row holds exactly min(k, seq_len) valid entries (top-k output)
  int cluster_merge;       // 1: the S (<= 16) splits of a (b, g) run as one cluster and merge into out
  int pre_wait;            // 1: q may be read before the previous kernel of the stream completes
  int D;                   // head dimension: 128 or 256
};
cudaError_t launch_sparse_attn(const AttnArgs& a, cudaStream_t stream);
bool sparse_attn_supported(int G, int D);
// Clusters of S attention CTAs the current device keeps resident at once (0
// when it cannot be determined).
int sparse_attn_resident_clusters(int G, int fp8, int S, int D);

struct AppendArgs {
  const void* k_new;       // bf16 [B, Hkv, 128]
  const void* v_new;
  void* k_cache;           // [slots, Hkv, 128] bf16 or e4m3
  void* v_cache;
  const float* k_scale;    // [num_pages], e4m3 only
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* positions;
  const int32_t* channels; // [Hkv, C]: per-head label gathered from K; null: index_key copied
  const void* index_key;   // bf16 [B, C]
  void* label;             // bf16 [slots, HL, C] or null
  unsigned* err;
  int B, Hkv, maxp, num_pages, fp8, HL, C, D;
};
cudaError_t launch_cache_append(const AppendArgs& a, cudaStream_t stream);

cudaError_t launch_lse_merge(int S, int rows, int D, const float* o_part, const float* lse_part,
                             void* out, float* lse, cudaStream_t stream);

// Block-compressed selection: compressed keys, block scores, kept blocks -> tokens.
cudaError_t launch_block_compress(const void* keys, const int32_t* page_table, const int32_t* seq_lens, int B,
                                  int C, int maxp, int num_pages, int last_only, void* block_keys, unsigned* err,
                                  cudaStream_t stream);
cudaError_t launch_block_score(const void* qp, const void* block_keys, const int32_t* page_table,
                               const int32_t* seq_lens, int B, int Hq, int Hkv, int C, int maxp, int num_pages,
                               int lim, float* scores, int32_t* nblocks, unsigned* err, cudaStream_t stream);
cudaError_t launch_block_expand(const int32_t* blocks, const int32_t* seq_lens, int B, int Hkv, int kb, int lim,
                                int32_t* idx, cudaStream_t stream);

}  // namespace ds

namespace ds {

// Launches `kernel` on `stream` with programmatic dependent launch enabled, so
// its CTAs may start while the previous kernel of the stream drains; the
// kernel must call grid_dependency_wait() before using earlier results.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

}  // namespace ds
