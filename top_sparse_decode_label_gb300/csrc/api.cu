// C ABI of libdssparse: argument validation, workspace layout and the chained
// decode step. Every entry point validates on the host and then only enqueues
// work on the caller's stream; nothing here allocates or synchronises, except
// ds_device_errors which is documented to synchronise.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <cstdint>

#include "ds_sparse.h"
#include "internal.h"

// Sticky device error word (DS_DEVERR_* bits), one per device.
static __device__ unsigned g_ds_device_errors;

namespace ds {

namespace {

constexpr int kMaxDevices = 64;
constexpr int kMaxShards = 64;   // virtual shards of ds_topk_select_sharded

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  return dev;
}

// Device address of the error word on the current device (looked up once per
// device; concurrent first lookups store the same address).
unsigned* error_word() {
  static std::atomic<unsigned*> ptrs[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return nullptr;
  unsigned* w = ptrs[dev].load(std::memory_order_acquire);
  if (!w) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_ds_device_errors) != cudaSuccess) return nullptr;
    w = static_cast<unsigned*>(p);
    ptrs[dev].store(w, std::memory_order_release);
  }
  return w;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

ds_status from_cuda(cudaError_t e) {
  if (e == cudaSuccess) return DS_OK;
  if (e == cudaErrorNotSupported) return DS_ERR_UNSUPPORTED;
  return DS_ERR_CUDA;
}

ds_status check_shape(const ds_shape* s) {
  if (!s) return DS_ERR_INVALID_ARG;
  if (s->batch < 0 || s->num_q_heads <= 0 || s->num_kv_heads <= 0 || s->max_pages_per_req <= 0 ||
      s->num_pages <= 0 || s->max_seq_len < 0 || s->head_dim <= 0 || s->page_size <= 0)
    return DS_ERR_INVALID_ARG;
  if (s->num_q_heads % s->num_kv_heads) return DS_ERR_INVALID_ARG;
  const int G = s->num_q_heads / s->num_kv_heads;
  if (G != 1 && G != 2 && G != 4 && G != 8) return DS_ERR_UNSUPPORTED;
  if ((s->head_dim != 128 && s->head_dim != kHeadDimMax) || s->page_size != kPageSupported) return DS_ERR_UNSUPPORTED;
  // Slot and element offsets are 64-bit; page ids and token indices are int32.
  if (static_cast<long long>(s->num_pages) * s->page_size > 0x7fffffffLL) return DS_ERR_UNSUPPORTED;
  return DS_OK;
}

}  // namespace

int sm_count() {
  static int counts[kMaxDevices] = {};
  const int dev = current_device();
  if (dev < 0) return 1;
  if (!counts[dev]) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
    counts[dev] = n;
  }
  return counts[dev];
}

// Internal split count of the chained call: the largest power of two up to
// 16 (the splits of a (request, KV head) form one thread-block cluster) that
// keeps the (request, KV head, split) CTAs within about three per SM, with at
// most one split per started 64 selected tokens -- and, when the device can
// be queried, with every cluster resident at once (no second wave).
int decode_splits(const ds_shape* s, int k) {
  const long long rows = static_cast<long long>(s->batch) * s->num_kv_heads;
  if (rows <= 0 || k <= 64) return 1;
  const long long cap = (k + 63) / 64;
  int S = 1;
  while (S < 16 && 2 * S <= cap && rows * 2 * S <= kDecodeTargetCtas) S *= 2;
  const int G = s->num_q_heads / s->num_kv_heads;
  while (S > 1) {
    const int resident = sparse_attn_resident_clusters(G, 1, S, s->head_dim);
    if (resident == 0 || rows <= resident) break;   // unknown device, or every cluster resident at once
    S /= 2;
  }
  return S;
}

}  // namespace ds

using namespace ds;

extern "C" {

const char* ds_error_string(ds_status status) {
  switch (status) {
    case DS_OK: return "DS_OK";
    case DS_ERR_INVALID_ARG: return "DS_ERR_INVALID_ARG: null, negative, misaligned or inconsistent argument";
    case DS_ERR_UNSUPPORTED: return "DS_ERR_UNSUPPORTED: size not implemented by this library";
    case DS_ERR_CUDA: return "DS_ERR_CUDA: a CUDA runtime call or kernel launch failed";
    case DS_ERR_WORKSPACE: return "DS_ERR_WORKSPACE: workspace too small or misaligned";
    case DS_ERR_DEVICE_CHECK: return "DS_ERR_DEVICE_CHECK: a kernel flagged an out-of-range element";
  }
  return "unknown ds_status";
}

ds_status ds_device_errors(unsigned* flags) {
  unsigned v = 0;
  if (cudaDeviceSynchronize() != cudaSuccess) return DS_ERR_CUDA;
  if (cudaMemcpyFromSymbol(&v, g_ds_device_errors, sizeof v) != cudaSuccess) return DS_ERR_CUDA;
  const unsigned zero = 0;
  if (cudaMemcpyToSymbol(g_ds_device_errors, &zero, sizeof zero) != cudaSuccess) return DS_ERR_CUDA;
  if (flags) *flags = v;
  return v ? DS_ERR_DEVICE_CHECK : DS_OK;
}

ds_status ds_index_score(const ds_shape* shape, const void* qp, int proxy_dim, const void* label,
                         int label_heads, const int32_t* page_table, const int32_t* seq_lens,
                         float* scores, ds_stream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (proxy_dim != 16 && proxy_dim != 32 && proxy_dim != 64) return DS_ERR_UNSUPPORTED;
  if (label_heads != 1 && label_heads != shape->num_kv_heads) return DS_ERR_INVALID_ARG;
  if (!index_score_supported(proxy_dim, label_heads, shape->num_kv_heads,
                             shape->num_q_heads / shape->num_kv_heads))
    return DS_ERR_UNSUPPORTED;
  if (shape->batch == 0 || shape->max_seq_len == 0) return DS_OK;
  if (!qp || !label || !page_table || !seq_lens || !scores) return DS_ERR_INVALID_ARG;
  if (!aligned(qp, 16) || !aligned(label, 16) || !aligned(scores, 4)) return DS_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  ScoreArgs a{qp, label, page_table, seq_lens, scores, err, shape->batch, shape->num_q_heads,
              shape->num_kv_heads, label_heads, proxy_dim, shape->max_pages_per_req, shape->num_pages,
              shape->max_seq_len};
  return from_cuda(launch_index_score(a, reinterpret_cast<cudaStream_t>(stream)));
}

size_t ds_topk_workspace_bytes(const ds_shape* shape, int k) {
  if (check_shape(shape) != DS_OK || k < 0) return 0;
  return topk_layout(nullptr, shape->batch * shape->num_kv_heads, shape->max_seq_len).bytes;
}

ds_status ds_topk_select(const ds_shape* shape, const float* scores, const int32_t* seq_lens, int k,
                         int32_t* idx, void* workspace, size_t workspace_bytes, ds_stream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (k < 0) return DS_ERR_INVALID_ARG;
  if (shape->batch == 0 || k == 0) return DS_OK;
  if (!seq_lens || !idx || (shape->max_seq_len > 0 && !scores)) return DS_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || (scores && !aligned(scores, 4))) return DS_ERR_INVALID_ARG;
  const TopkLayout L = topk_layout(workspace, shape->batch * shape->num_kv_heads, shape->max_seq_len);
  if (!workspace || workspace_bytes < L.bytes || !aligned(workspace, 256)) return DS_ERR_WORKSPACE;
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  TopkArgs a{scores, seq_lens, idx, err, shape->batch, shape->num_kv_heads, shape->max_seq_len,
             shape->max_pages_per_req * shape->page_size, k, L, nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0, 0};
  return from_cuda(launch_topk(a, reinterpret_cast<cudaStream_t>(stream)));
}

static ds_status attn_common(const ds_shape* shape, const void* q, const void* k_cache, const void* v_cache,
                             ds_kv_dtype kv_dtype, const float* k_scale, const float* v_scale,
                             const int32_t* page_table, const int32_t* seq_lens, const int32_t* idx, int k,
                             float sm_scale, int num_splits, int split_mode, float* o_part, float* lse_part,
                             void* out, float* lse, const int32_t* slots, const float2* sscale, int n_from_seq_len,
                             int cluster_merge, int pre_wait, cudaStream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (kv_dtype != DS_KV_BF16 && kv_dtype != DS_KV_FP8_E4M3) return DS_ERR_INVALID_ARG;
  if (k < 0 || num_splits < 1 || (split_mode != DS_SPLIT_CONTIGUOUS && split_mode != DS_SPLIT_PAGE_INTERLEAVED))
    return DS_ERR_INVALID_ARG;
  if (!(sm_scale == sm_scale)) return DS_ERR_INVALID_ARG;
  if (!sparse_attn_supported(shape->num_q_heads / shape->num_kv_heads, shape->head_dim)) return DS_ERR_UNSUPPORTED;
  if (shape->batch == 0) return DS_OK;
  if (!q || !k_cache || !v_cache || !page_table || !seq_lens || (k > 0 && !idx)) return DS_ERR_INVALID_ARG;
  if (kv_dtype == DS_KV_FP8_E4M3 && (!k_scale || !v_scale)) return DS_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return DS_ERR_INVALID_ARG;
  if (num_splits == 1 || cluster_merge) {
    if (!out || !aligned(out, 4)) return DS_ERR_INVALID_ARG;
  }
  if (num_splits > 1 && !cluster_merge) {
    if (!o_part || !lse_part || !aligned(o_part, 4)) return DS_ERR_INVALID_ARG;
  }
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  AttnArgs a{q, k_cache, v_cache, k_scale, v_scale, page_table, seq_lens, idx, o_part, lse_part, out, lse, err,
             shape->batch, shape->num_q_heads, shape->num_kv_heads, shape->max_pages_per_req, shape->num_pages,
             shape->max_seq_len, k, num_splits, split_mode, kv_dtype == DS_KV_FP8_E4M3 ? 1 : 0, sm_scale,
             slots, sscale, n_from_seq_len, cluster_merge, pre_wait, shape->head_dim};
  return from_cuda(launch_sparse_attn(a, stream));
}

ds_status ds_sparse_decode_attn(const ds_shape* shape, const void* q, const void* k_cache,
                                const void* v_cache, ds_kv_dtype kv_dtype, const float* k_scale,
                                const float* v_scale, const int32_t* page_table,
                                const int32_t* seq_lens, const int32_t* idx, int k, float sm_scale,
                                int num_splits, ds_split_mode split_mode, float* o_part,
                                float* lse_part, void* out, float* lse, ds_stream_t stream) {
  return attn_common(shape, q, k_cache, v_cache, kv_dtype, k_scale, v_scale, page_table, seq_lens, idx, k,
                     sm_scale, num_splits, static_cast<int>(split_mode), o_part, lse_part, out, lse, nullptr, nullptr, 0,
                     0, 0,
                     reinterpret_cast<cudaStream_t>(stream));
}

ds_status ds_lse_merge(int num_splits, int rows, int head_dim, const float* o_part, const float* lse_part,
                       void* out, float* lse, ds_stream_t stream) {
  if (num_splits < 1 || rows < 0 || head_dim <= 0 || head_dim % 4) return DS_ERR_INVALID_ARG;
  if (rows == 0) return DS_OK;
  if (!o_part || !lse_part || !out) return DS_ERR_INVALID_ARG;
  if (!aligned(o_part, 16) || !aligned(out, 8) || !aligned(lse_part, 4)) return DS_ERR_INVALID_ARG;
  return from_cuda(launch_lse_merge(num_splits, rows, head_dim, o_part, lse_part, out, lse,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

size_t ds_topk_sharded_workspace_bytes(const ds_shape* shape, int k, int num_shards) {
  if (check_shape(shape) != DS_OK || k < 0 || num_shards < 1 || num_shards > kMaxShards) return 0;
  return topk_sharded_workspace_bytes(shape->batch * shape->num_kv_heads, shape->max_seq_len, k, num_shards);
}

ds_status ds_topk_select_sharded(const ds_shape* shape, const float* scores, const int32_t* seq_lens, int k,
                                 int num_shards, int32_t* idx, void* workspace, size_t workspace_bytes,
                                 ds_stream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (k < 0 || num_shards < 1) return DS_ERR_INVALID_ARG;
  if (num_shards > kMaxShards) return DS_ERR_UNSUPPORTED;
  if (shape->batch == 0 || k == 0) return DS_OK;
  if (!seq_lens || !idx || (shape->max_seq_len > 0 && !scores)) return DS_ERR_INVALID_ARG;
  if (!aligned(idx, 4) || (scores && !aligned(scores, 4))) return DS_ERR_INVALID_ARG;
  const size_t need = topk_sharded_workspace_bytes(shape->batch * shape->num_kv_heads, shape->max_seq_len, k,
                                                   num_shards);
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return DS_ERR_WORKSPACE;
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  return from_cuda(launch_topk_sharded(scores, seq_lens, shape->batch, shape->num_kv_heads, shape->max_seq_len,
                                       shape->max_pages_per_req * shape->page_size, k, num_shards, idx, workspace,
                                       err, reinterpret_cast<cudaStream_t>(stream)));
}

ds_status ds_cache_append(const ds_shape* shape, const void* k_new, const void* v_new, ds_kv_dtype kv_dtype,
                          void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                          const int32_t* page_table, const int32_t* positions, int proxy_dim, int label_heads,
                          const int32_t* channels, const void* index_key, void* label, ds_stream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (kv_dtype != DS_KV_BF16 && kv_dtype != DS_KV_FP8_E4M3) return DS_ERR_INVALID_ARG;
  if (shape->batch == 0) return DS_OK;
  if (!k_new || !v_new || !k_cache || !v_cache || !page_table || !positions) return DS_ERR_INVALID_ARG;
  if (kv_dtype == DS_KV_FP8_E4M3 && (!k_scale || !v_scale)) return DS_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return DS_ERR_INVALID_ARG;
  if (label) {
    if (proxy_dim != 16 && proxy_dim != 32 && proxy_dim != 64) return DS_ERR_UNSUPPORTED;
    if (channels) {
      if (label_heads != shape->num_kv_heads) return DS_ERR_INVALID_ARG;
    } else {
      if (label_heads != 1 || !index_key) return DS_ERR_INVALID_ARG;
    }
    if (!aligned(label, 16)) return DS_ERR_INVALID_ARG;
  }
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  AppendArgs a{k_new, v_new, k_cache, v_cache, k_scale, v_scale, page_table, positions,
               label ? channels : nullptr, label ? index_key : nullptr, label, err, shape->batch,
               shape->num_kv_heads, shape->max_pages_per_req, shape->num_pages,
               kv_dtype == DS_KV_FP8_E4M3 ? 1 : 0, label ? label_heads : 0, label ? proxy_dim : 0,
               shape->head_dim};
  return from_cuda(launch_cache_append(a, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

// Workspace of the chained call: the scores and their 16-token block maxima,
// the top-k overflow lists and the physical slots of the selection.
struct DecodeLayout {
  float* scores;
  float* bmax;      // [B, Hkv, ceil(max_seq_len / 16)]
  TopkLayout topk;
  int32_t* slots;   // [B, Hkv, k]
  float2* sscale;   // [B, Hkv, k] (K, V) page scales of the kept tokens (FP8 caches)
  size_t bytes;
};

DecodeLayout decode_layout(const ds_shape* s, int k, void* base) {
  DecodeLayout L;
  char* p = static_cast<char*>(base);
  const int R = s->batch * s->num_kv_heads;
  size_t off = 0;
  L.scores = reinterpret_cast<float*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (s->max_seq_len > 0 ? s->max_seq_len : 1) * 4);
  L.bmax = reinterpret_cast<float*>(p + off);
  const size_t nbr = static_cast<size_t>((s->max_seq_len > 0 ? s->max_seq_len : 1) + kMaxBlock - 1) / kMaxBlock;
  off = align256(off + static_cast<size_t>(R) * nbr * 4);
  L.topk = topk_layout(p + off, R, s->max_seq_len);
  off = align256(off + L.topk.bytes);
  L.slots = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (k > 0 ? k : 1) * 4);
  L.sscale = reinterpret_cast<float2*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (k > 0 ? k : 1) * 8);
  L.bytes = off;
  return L;
}

}  // namespace

size_t ds_decode_workspace_bytes(const ds_shape* shape, int proxy_dim, int k) {
  (void)proxy_dim;
  if (check_shape(shape) != DS_OK || k < 0) return 0;
  return decode_layout(shape, k, nullptr).bytes;
}

int ds_decode_num_splits(const ds_shape* shape, int k) {
  if (check_shape(shape) != DS_OK || k < 0) return 0;
  return decode_splits(shape, k);
}

int ds_decode_kernel_launches(const ds_shape* shape, int k) {
  if (check_shape(shape) != DS_OK || k < 0 || shape->batch == 0) return 0;
  int n = 0;
  if (shape->max_seq_len > 0) n += 1;       // scoring
  if (k > 0) n += 1;                   // top-k (one cluster per row)
  n += 1;                              // attention (splits merged inside their cluster)
  return n;
}

static ds_status decode_impl(const ds_shape* shape, const ds_decode_args* args, void* workspace,
                             size_t workspace_bytes, ds_stream_t stream, void* const* events) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (!args) return DS_ERR_INVALID_ARG;
  if (args->k < 0) return DS_ERR_INVALID_ARG;
  if (shape->batch == 0) return DS_OK;
  if (!args->idx || !args->out || !aligned(args->idx, 4)) return DS_ERR_INVALID_ARG;
  const DecodeLayout L = decode_layout(shape, args->k, workspace);
  if (!workspace || workspace_bytes < L.bytes || !aligned(workspace, 256)) return DS_ERR_WORKSPACE;
  const int pd = args->proxy_dim;
  if (pd != 16 && pd != 32 && pd != 64) return DS_ERR_UNSUPPORTED;
  if (args->label_heads != 1 && args->label_heads != shape->num_kv_heads) return DS_ERR_INVALID_ARG;
  if (!index_score_supported(pd, args->label_heads, shape->num_kv_heads, shape->num_q_heads / shape->num_kv_heads))
    return DS_ERR_UNSUPPORTED;
  if (!args->qp || !args->label || !args->page_table || !args->seq_lens) return DS_ERR_INVALID_ARG;
  if (!aligned(args->qp, 16) || !aligned(args->label, 16)) return DS_ERR_INVALID_ARG;
  // The cache arguments (and the FP8 page scales, which the top-k stage reads)
  // are checked before anything is launched.
  if (args->kv_dtype != DS_KV_BF16 && args->kv_dtype != DS_KV_FP8_E4M3) return DS_ERR_INVALID_ARG;
  if (!args->q || !args->k_cache || !args->v_cache) return DS_ERR_INVALID_ARG;
  if (!aligned(args->q, 16) || !aligned(args->k_cache, 16) || !aligned(args->v_cache, 16)) return DS_ERR_INVALID_ARG;
  if (args->kv_dtype == DS_KV_FP8_E4M3 && (!args->k_scale || !args->v_scale)) return DS_ERR_INVALID_ARG;
  if (!sparse_attn_supported(shape->num_q_heads / shape->num_kv_heads, shape->head_dim)) return DS_ERR_UNSUPPORTED;
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int S = decode_splits(shape, args->k);
  const int k = args->k;
  auto mark = [&](int i) {
    return events ? cudaEventRecord(static_cast<cudaEvent_t>(events[i]), s) : cudaSuccess;
  };
  if (mark(0) != cudaSuccess) return DS_ERR_CUDA;
  if (shape->max_seq_len > 0) {
    ScoreArgs sa{args->qp, args->label, args->page_table, args->seq_lens, L.scores, err, shape->batch,
                 shape->num_q_heads, shape->num_kv_heads, args->label_heads, pd, shape->max_pages_per_req,
                 shape->num_pages, shape->max_seq_len, L.bmax};
    st = from_cuda(launch_index_score(sa, s));
    if (st != DS_OK) return st;
  }
  if (mark(1) != cudaSuccess) return DS_ERR_CUDA;
  if (k > 0) {
    const bool fp8 = args->kv_dtype == DS_KV_FP8_E4M3;
    TopkArgs ta{L.scores, args->seq_lens, args->idx, err, shape->batch, shape->num_kv_heads, shape->max_seq_len,
                shape->max_pages_per_req * shape->page_size, k, L.topk, L.slots, args->page_table,
                fp8 ? args->k_scale : nullptr, fp8 ? args->v_scale : nullptr, fp8 ? L.sscale : nullptr,
                shape->max_pages_per_req, shape->num_pages, shape->max_seq_len > 0 ? 1 : 0,
                (shape->max_seq_len > 0 && index_score_block_maxima(pd, args->label_heads, shape->num_kv_heads))
                    ? L.bmax
                    : nullptr};
    st = from_cuda(launch_topk(ta, s));
    if (st != DS_OK) return st;
  }
  if (mark(2) != cudaSuccess) return DS_ERR_CUDA;
  st = attn_common(shape, args->q, args->k_cache, args->v_cache, args->kv_dtype, args->k_scale, args->v_scale,
                   args->page_table, args->seq_lens, args->idx, k, args->sm_scale, S, DS_SPLIT_CONTIGUOUS,
                   nullptr, nullptr, args->out, args->lse, k > 0 ? L.slots : nullptr,
                   (k > 0 && args->kv_dtype == DS_KV_FP8_E4M3) ? L.sscale : nullptr, 1, S > 1 ? 1 : 0,
                   (shape->max_seq_len > 0 || k > 0) ? 1 : 0, s);
  if (st != DS_OK) return st;
  return mark(3) == cudaSuccess ? DS_OK : DS_ERR_CUDA;
}

ds_status ds_sparse_decode(const ds_shape* shape, const ds_decode_args* args, void* workspace,
                           size_t workspace_bytes, ds_stream_t stream) {
  return decode_impl(shape, args, workspace, workspace_bytes, stream, nullptr);
}

// ---- block-compressed selection

ds_status ds_block_compress(const ds_shape* shape, const void* index_key, int proxy_dim, const int32_t* page_table,
                            const int32_t* seq_lens, int last_page_only, void* block_keys, ds_stream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (proxy_dim != 16 && proxy_dim != 32 && proxy_dim != 64) return DS_ERR_UNSUPPORTED;
  if (shape->batch == 0) return DS_OK;
  if (!index_key || !page_table || !seq_lens || !block_keys) return DS_ERR_INVALID_ARG;
  if (!aligned(index_key, 16) || !aligned(block_keys, 16)) return DS_ERR_INVALID_ARG;
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  return from_cuda(launch_block_compress(index_key, page_table, seq_lens, shape->batch, proxy_dim,
                                         shape->max_pages_per_req, shape->num_pages, last_page_only ? 1 : 0,
                                         block_keys, err, reinterpret_cast<cudaStream_t>(stream)));
}

namespace {

// Workspace of the block decode: block scores, block counts, the top-k's
// overflow lists and the expanded token lists.
struct BlockLayout {
  float* scores;     // [R, maxp]
  int32_t* nblocks;  // [B]
  TopkLayout topk;
  int32_t* tokens;   // [R, kb * 64]
  size_t bytes;
};

BlockLayout block_layout(const ds_shape* s, int kb, void* base) {
  BlockLayout L;
  char* p = static_cast<char*>(base);
  const int R = s->batch * s->num_kv_heads;
  const int nbm = s->max_pages_per_req;
  size_t off = 0;
  L.scores = reinterpret_cast<float*>(p + off);
  off = align256(off + static_cast<size_t>(R) * nbm * 4);
  L.nblocks = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + static_cast<size_t>(s->batch > 0 ? s->batch : 1) * 4);
  L.topk = topk_layout(p + off, R, nbm);
  off = align256(off + L.topk.bytes);
  L.tokens = reinterpret_cast<int32_t*>(p + off);
  off = align256(off + static_cast<size_t>(R) * (kb > 0 ? kb : 1) * s->page_size * 4);
  L.bytes = off;
  return L;
}

}  // namespace

size_t ds_block_decode_workspace_bytes(const ds_shape* shape, int kb) {
  if (check_shape(shape) != DS_OK || kb < 0) return 0;
  return block_layout(shape, kb, nullptr).bytes;
}

ds_status ds_sparse_decode_blocks(const ds_shape* shape, const ds_block_decode_args* args, void* workspace,
                                  size_t workspace_bytes, ds_stream_t stream) {
  ds_status st = check_shape(shape);
  if (st != DS_OK) return st;
  if (!args || args->kb < 0) return DS_ERR_INVALID_ARG;
  if (shape->batch == 0) return DS_OK;
  const int pd = args->proxy_dim;
  if (pd != 16 && pd != 32 && pd != 64) return DS_ERR_UNSUPPORTED;
  if (static_cast<long long>(args->kb) * shape->page_size > 0x7fffffffLL / 2) return DS_ERR_UNSUPPORTED;
  if (!args->qp || !args->block_keys || !args->page_table || !args->seq_lens || (args->kb > 0 && !args->blocks) ||
      !args->out)
    return DS_ERR_INVALID_ARG;
  if (!aligned(args->qp, 4) || !aligned(args->block_keys, 16) || !aligned(args->blocks, 4)) return DS_ERR_INVALID_ARG;
  const BlockLayout L = block_layout(shape, args->kb, workspace);
  if (!workspace || workspace_bytes < L.bytes || !aligned(workspace, 256)) return DS_ERR_WORKSPACE;
  unsigned* err = error_word();
  if (!err) return DS_ERR_CUDA;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const int kb = args->kb;
  const int ktok = kb * shape->page_size;
  const int nbm = shape->max_pages_per_req;
  const int lim = static_cast<int>(std::min<long long>(shape->max_seq_len, static_cast<long long>(nbm) * shape->page_size));
  st = from_cuda(launch_block_score(args->qp, args->block_keys, args->page_table, args->seq_lens, shape->batch,
                                    shape->num_q_heads, shape->num_kv_heads, pd, nbm, shape->num_pages, lim, L.scores,
                                    L.nblocks, err, s));
  if (st != DS_OK) return st;
  if (kb > 0) {
    // pre_wait 0: the block counts come from the block scores' kernel.
    TopkArgs ta{L.scores, L.nblocks, args->blocks, err, shape->batch, shape->num_kv_heads, nbm, nbm, kb, L.topk,
                nullptr, nullptr, nullptr, nullptr, nullptr, 0, 0, 0};
    st = from_cuda(launch_topk(ta, s));
    if (st != DS_OK) return st;
    st = from_cuda(launch_block_expand(args->blocks, args->seq_lens, shape->batch, shape->num_kv_heads, kb, lim,
                                       L.tokens, s));
    if (st != DS_OK) return st;
  }
  const int S = decode_splits(shape, ktok);
  return attn_common(shape, args->q, args->k_cache, args->v_cache, args->kv_dtype, args->k_scale, args->v_scale,
                     args->page_table, args->seq_lens, L.tokens, ktok, args->sm_scale, S, DS_SPLIT_CONTIGUOUS,
                     nullptr, nullptr, args->out, args->lse, nullptr, nullptr, 0, S > 1 ? 1 : 0, 1, s);
}

ds_status ds_sparse_decode_profiled(const ds_shape* shape, const ds_decode_args* args, void* workspace,
                                    size_t workspace_bytes, ds_stream_t stream, void* const* events) {
  return decode_impl(shape, args, workspace, workspace_bytes, stream, events);
}

}  // extern "C"
