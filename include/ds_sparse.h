/*
 * ds_sparse.h -- C ABI of the decode-step top-k sparse attention library
 * (libdssparse.so, CUDA, sm_103a).
 *
 * One decode step of Double-Sparsity / QSA-style attention runs in four stages:
 *   1. ds_index_score        score every cached token with a cheap proxy
 *   2. ds_topk_select        keep the exact top-k tokens per (request, KV head)
 *   3. ds_sparse_decode_attn GQA attention over the kept tokens only, gathered
 *                            from a paged bf16 or FP8-E4M3 KV cache
 *   4. ds_lse_merge          merge split-KV partial outputs by log-sum-exp
 * and ds_sparse_decode chains all four on one stream.
 *
 * Sources: "Support double sparsity" (sglang PR #1459: label cache of heavy
 * channels, heavy-token selection, sparse decode attention); sglang PR #43527
 * "QSA cache sharding", sections "Distributed QSA execution" (exact Top-K with
 * deterministic global token-ID tie-breaking, owner-side sparse attention,
 * FP32 log-sum-exp merge), "CUDA Graph buffers" and "CUDA Graph metadata";
 * "QSA HiSparse - SGLang plugin", "Supported versions" (FP8 E4M3 KV cache,
 * page size 64).
 *
 * Conventions for every entry point:
 *  - All pointers are DEVICE pointers on the current device unless stated.
 *    The caller owns all memory; the library never allocates or frees.
 *  - Calls are asynchronous on `stream` and never synchronise the host
 *    (ds_device_errors, the explicit check, is the one exception).
 *    Arguments are validated on the host before any launch; a call that
 *    returns an error has launched nothing.
 *  - Make calls from one host thread at a time: the entry points set kernel
 *    attributes and cache device queries (SM count, resident clusters) in
 *    process-wide tables without a lock.
 *  - Problems the host cannot see (a seq_len, page id or token index outside
 *    its range) never cause an out-of-bounds access: the kernel skips the bad
 *    element and sets a bit in a sticky device error word, read back with
 *    ds_device_errors(). Results of such a call are unspecified.
 *  - Tensor layouts are row-major and dense; base pointers are 16-byte aligned.
 *  - GQA grouping is contiguous: query head h uses KV head h / (Hq / Hkv).
 *  - Logical token t of request b lives in physical slot
 *        page_table[b][t / page_size] * page_size + t % page_size.
 *    Page-table entries at or past ceil(seq_lens[b] / page_size) are never read.
 */
#ifndef DS_SPARSE_H
#define DS_SPARSE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL means the legacy default stream. */
typedef struct CUstream_st* ds_stream_t;

typedef enum {
  DS_OK = 0,
  DS_ERR_INVALID_ARG = -1,   /* null pointer, negative size, misaligned pointer, too-small buffer */
  DS_ERR_UNSUPPORTED = -2,   /* a size this library does not implement (head_dim, page_size, group, ...) */
  DS_ERR_CUDA = -3,          /* a CUDA runtime call or launch failed */
  DS_ERR_WORKSPACE = -4,     /* workspace too small (see the *_workspace_bytes queries) */
  DS_ERR_DEVICE_CHECK = -5   /* ds_device_errors found a flagged element */
} ds_status;

typedef enum { DS_KV_BF16 = 0, DS_KV_FP8_E4M3 = 1 } ds_kv_dtype;

/* How stage 3 cuts a row's selected tokens into num_splits chunks. */
typedef enum {
  DS_SPLIT_CONTIGUOUS = 0,       /* chunk j = positions [j*n/S, (j+1)*n/S) of the n selected tokens */
  DS_SPLIT_PAGE_INTERLEAVED = 1  /* chunk j = selected tokens whose logical page % S == j (page owners) */
} ds_split_mode;

/* Bits of the device error word. */
#define DS_DEVERR_SEQ_LEN   1u   /* seq_lens[b] < 0 or > min(max_seq_len, max_pages_per_req*page_size); clamped */
#define DS_DEVERR_PAGE_ID   2u   /* a page-table entry outside [0, num_pages); its tokens were skipped */
#define DS_DEVERR_TOKEN_IDX 4u   /* an index entry outside [0, seq_lens[b]) before the -1 padding; skipped */
#define DS_DEVERR_TIMEOUT   8u   /* a bounded wait for an asynchronous copy gave up; the call's results are invalid */
#define DS_DEVERR_CHANNEL   16u  /* ds_cache_append: a heavy-channel id outside [0, head_dim); that label entry skipped */

typedef struct {
  int batch;             /* B, requests in the step (>= 0) */
  int num_q_heads;       /* Hq, a multiple of num_kv_heads; Hq / Hkv in {1, 2, 4, 8} */
  int num_kv_heads;      /* Hkv (>= 1) */
  int head_dim;          /* D; the library supports 128 and 256 (the QSA model's shape on Blackwell,
                            sglang PR #43527 review thread: BF16 queries, head dimension 256) */
  int page_size;         /* P; the library supports 64 */
  int max_pages_per_req; /* row stride of page_table (>= 1) */
  int num_pages;         /* physical pages in the pool; valid page ids are [0, num_pages) */
  int max_seq_len;       /* Tmax, row stride of the score buffer; every seq_lens[b] must be <= it */
} ds_shape;

/*
 * Stage 1: proxy scores ("Support double sparsity": the query's heavy channels
 * against a label cache of heavy K channels; PR #39721 / #43527: the QSA
 * indexer scans per-token index keys and scores them).
 *
 *   s[b, g, t] = sum over q-heads h of group g, sum_c qp[b, h, c] * label[slot(b,t), gL, c]
 *
 * for t < seq_lens[b], with gL = g when label_heads == Hkv (a per-head label
 * cache) and gL = 0 when label_heads == 1 (one index key per token shared by
 * all heads). Accumulated in fp32; exact whenever every partial sum is an
 * integer below 2^24 in magnitude (e.g. integer-valued inputs).
 *
 *   qp          bf16  [B, Hq, proxy_dim]                      proxy query
 *   proxy_dim   C in {16, 32, 64}
 *   label       bf16  [num_pages * P, label_heads, proxy_dim] label cache / index keys
 *   label_heads Hkv or 1
 *   page_table  int32 [B, max_pages_per_req]
 *   seq_lens    int32 [B]
 *   scores      fp32  [B, Hkv, max_seq_len]; positions t >= seq_lens[b] are not written
 */
ds_status ds_index_score(const ds_shape* shape, const void* qp, int proxy_dim, const void* label,
                         int label_heads, const int32_t* page_table, const int32_t* seq_lens,
                         float* scores, ds_stream_t stream);

/*
 * Stage 2: exact top-k (PR #43527, "Distributed QSA execution": exact Top-K
 * with deterministic token-ID tie-breaking; PR #1459 heavy-token count).
 *
 * For each row (b, g) keeps the K_eff = min(k, seq_lens[b]) tokens that come
 * first in the order (score descending, token index ascending): equal scores
 * go to the smaller token index, -0.0 equals +0.0, NaN ranks below every
 * number. The result is unique. idx[b, g, :] holds the kept token indices in
 * ascending order followed by -1 up to k. k == 0 or seq_lens[b] == 0 gives
 * an all -1 row.
 *
 *   scores     fp32  [B, Hkv, max_seq_len] (only t < seq_lens[b] is read)
 *   idx        int32 [B, Hkv, k]
 *   workspace  device scratch of at least ds_topk_workspace_bytes(shape, k)
 *              bytes, 256-byte aligned; its contents need no initialisation and
 *              are overwritten. Two calls in flight at once need two workspaces.
 */
size_t ds_topk_workspace_bytes(const ds_shape* shape, int k);
ds_status ds_topk_select(const ds_shape* shape, const float* scores, const int32_t* seq_lens, int k,
                         int32_t* idx, void* workspace, size_t workspace_bytes, ds_stream_t stream);

/*
 * ds_topk_select without a workspace argument, for callers that cannot
 * allocate device memory: a plugin whose host framework owns every device
 * allocation and hands it only the tensors of the call, or a latency-critical
 * serving thread that must not wait on an allocator's lock. The pages
 * describe no such entry point; it exists for these callers only. Same
 * arguments and results as ds_topk_select, and nothing is allocated or freed.
 *
 * Scratch comes from an array of DS_TOPK_STATIC_SCRATCH_BYTES (16 MiB)
 * compiled into the library; each GPU that loads the library holds one until
 * the process exits. A (shape, k) needing more scratch than that (see
 * ds_topk_workspace_bytes) returns DS_ERR_WORKSPACE and launches nothing.
 * The first call on a device looks up the array's device address (once per
 * device, with that device current) and caches it; make that first call
 * before any stream capture, and note that cudaDeviceReset invalidates the
 * cached address. All calls share the one array, so calls whose work
 * overlaps on the GPU (other streams, other host threads) race and corrupt
 * each other's results: serialise them. The array needs no clearing: the
 * top-k only spills candidate lists there, writing before it reads.
 */
#define DS_TOPK_STATIC_SCRATCH_BYTES (16u << 20)
ds_status ds_topk_select_static(const ds_shape* shape, const float* scores, const int32_t* seq_lens, int k,
                                int32_t* idx, ds_stream_t stream);

/*
 * ds_topk_select computed the way the QSA cache-sharding page distributes it
 * (sglang PR #43527, "QSA cache placement": each cache page has one owner;
 * "Distributed QSA execution": each shard selects local candidates, merged
 * into an exact global Top-K with deterministic global token-ID
 * tie-breaking), emulated on one GPU: logical page p of a request belongs to
 * shard p mod num_shards; each shard takes the local top-k of its tokens; the
 * merge takes the top-k of the union, equal scores to the smaller token
 * index. The result equals ds_topk_select's (same arguments and layout).
 *
 *   num_shards  1 .. 64 (num_shards * B * Hkv <= 65535)
 *   workspace   at least ds_topk_sharded_workspace_bytes(shape, k, num_shards)
 *               bytes, 256-byte aligned; needs no initialisation (the call
 *               clears what it needs with an asynchronous memset)
 */
size_t ds_topk_sharded_workspace_bytes(const ds_shape* shape, int k, int num_shards);
ds_status ds_topk_select_sharded(const ds_shape* shape, const float* scores, const int32_t* seq_lens, int k,
                                 int num_shards, int32_t* idx, void* workspace, size_t workspace_bytes,
                                 ds_stream_t stream);

/*
 * Stage 3: sparse GQA decode attention over the selected tokens (PR #1459
 * sparse decode attention; PR #39721 sparse_gqa; FP8 E4M3 paged KV of the
 * QSA HiSparse plugin).
 *
 * For query head h of request b, with g = h / G and I the valid entries of
 * idx[b, g, :] (a prefix of token indices, then -1):
 *   z_t = sm_scale * q[b,h,:] . K[slot(b,t), g, :]
 *   o   = sum_{t in I} softmax(z)_t * V[slot(b,t), g, :],  lse = ln sum_{t in I} exp(z_t)
 * FP8 values are e4m3 times one fp32 scale per physical page (k_scale for K,
 * v_scale for V). Math is fp32.
 *
 * num_splits == 1: writes out (bf16 [B, Hq, D]) and lse (fp32 [B, Hq]).
 * num_splits  > 1: cuts I into S chunks by split_mode and writes, per chunk j,
 *   the normalised partial o_part[j] (fp32 [S, B, Hq, D]) and its
 *   lse_part[j] (fp32 [S, B, Hq]); an empty chunk gives o = 0, lse = -inf.
 *   out / lse are not touched (merge with ds_lse_merge).
 * An empty row gives o = 0 and lse = -inf.
 *
 *   q         bf16 [B, Hq, D]
 *   k_cache   [num_pages * P, Hkv, D], bf16 or e4m3 bytes per kv_dtype; v_cache likewise
 *   k_scale   fp32 [num_pages] (FP8 only; NULL for bf16); v_scale likewise
 *   idx       int32 [B, Hkv, k]
 *   sm_scale  softmax scale, normally 1/sqrt(D)
 */
ds_status ds_sparse_decode_attn(const ds_shape* shape, const void* q, const void* k_cache,
                                const void* v_cache, ds_kv_dtype kv_dtype, const float* k_scale,
                                const float* v_scale, const int32_t* page_table,
                                const int32_t* seq_lens, const int32_t* idx, int k, float sm_scale,
                                int num_splits, ds_split_mode split_mode, float* o_part,
                                float* lse_part, void* out, float* lse, ds_stream_t stream);

/*
 * Stage 4: log-sum-exp merge of split partials (PR #43527: owner-side
 * partial outputs merged with FP32 log-sum-exp normalisation).
 *   lse = ln sum_j exp(lse_j);  out = sum_j exp(lse_j - lse) * o_j
 * Chunks with lse_j = -inf weigh nothing; if all are -inf, out = 0 and
 * lse = -inf.
 *
 *   o_part   fp32 [num_splits, rows, head_dim]; lse_part fp32 [num_splits, rows]
 *   out      bf16 [rows, head_dim];             lse      fp32 [rows] (may be NULL)
 *   head_dim a multiple of 4
 */
ds_status ds_lse_merge(int num_splits, int rows, int head_dim, const float* o_part,
                       const float* lse_part, void* out, float* lse, ds_stream_t stream);

/*
 * The step before the path: append each request's new token to the caches
 * ("Support double sparsity", review thread: the label cache is the per-head
 * gather of K at the heavy channels; "QSA HiSparse - SGLang plugin",
 * "Supported versions": FP8 E4M3 paged KV, page size 64; sglang PR #39721:
 * the indexer stores each token's raw index key).
 *
 * Request b's new token sits at logical position t = positions[b] (usually
 * the sequence length before this step; negative: the request is skipped)
 * and goes to slot page_table[b][t / 64] * 64 + t % 64, whose page the
 * caller has allocated (and, for FP8, given its scales):
 *   K, V rows  bf16 copied; e4m3 = the fp32 quotient x / k_scale[page]
 *              (v_scale for V) rounded to nearest even, saturated to +-448
 *   label row  label_heads == Hkv: label[slot, g, c] = k_new[b, g, channels[g, c]]
 *              (the bf16 K, before any FP8 rounding);
 *              label_heads == 1:   label[slot, 0, :] = index_key[b, :]
 *
 *   k_new, v_new  bf16 [B, Hkv, D]
 *   k_cache, v_cache, k_scale, v_scale  as in ds_sparse_decode_attn (written)
 *   page_table    int32 [B, max_pages_per_req]; positions int32 [B]
 *   label         bf16 [num_pages * 64, label_heads, proxy_dim], or NULL to
 *                 write K and V only
 *   channels      int32 [Hkv, proxy_dim], each in [0, D) (per-head label), or NULL
 *   index_key     bf16 [B, proxy_dim] (shared key; used when channels is NULL)
 * A position at or past max_pages_per_req * 64 (DS_DEVERR_SEQ_LEN), a page id
 * outside [0, num_pages) (DS_DEVERR_PAGE_ID) or a channel outside [0, D)
 * (DS_DEVERR_CHANNEL) is skipped and flagged. Requests must not share a slot.
 */
ds_status ds_cache_append(const ds_shape* shape, const void* k_new, const void* v_new, ds_kv_dtype kv_dtype,
                          void* k_cache, void* v_cache, const float* k_scale, const float* v_scale,
                          const int32_t* page_table, const int32_t* positions, int proxy_dim, int label_heads,
                          const int32_t* channels, const void* index_key, void* label, ds_stream_t stream);

/* Arguments of the chained call (meanings as in the stages above). */
typedef struct {
  const void* q;             /* bf16 [B, Hq, D] */
  const void* qp;            /* bf16 [B, Hq, proxy_dim] */
  int proxy_dim;
  const void* label;         /* bf16 [num_pages * P, label_heads, proxy_dim] */
  int label_heads;
  const void* k_cache;
  const void* v_cache;
  ds_kv_dtype kv_dtype;
  const float* k_scale;
  const float* v_scale;
  const int32_t* page_table;
  const int32_t* seq_lens;
  int k;
  float sm_scale;
  int32_t* idx;              /* out: int32 [B, Hkv, k] selected tokens */
  void* out;                 /* out: bf16 [B, Hq, D] */
  float* lse;                /* out: fp32 [B, Hq] (may be NULL) */
} ds_decode_args;

/*
 * The whole decode step: ds_index_score -> ds_topk_select ->
 * ds_sparse_decode_attn (internal split-KV chosen for occupancy) ->
 * ds_lse_merge, on one stream, with scores in `workspace`
 * (at least ds_decode_workspace_bytes bytes, 256-byte aligned; its contents
 * need no initialisation). The splits of each (request, KV head) run as one
 * thread-block cluster and merge in on-chip shared memory. Calls sharing one
 * workspace must not overlap on the GPU. No host synchronisation and no
 * allocation.
 */
size_t ds_decode_workspace_bytes(const ds_shape* shape, int proxy_dim, int k);
ds_status ds_sparse_decode(const ds_shape* shape, const ds_decode_args* args, void* workspace,
                           size_t workspace_bytes, ds_stream_t stream);

/*
 * ds_sparse_decode, instrumented: when `events` is not NULL it must hold four
 * created cudaEvent_t handles, recorded on `stream` before the scoring stage,
 * after it, after the top-k stage and after the attention stage (which
 * includes the fused merge), so a caller can time each stage of the very
 * same launches. Results and requirements are those of ds_sparse_decode.
 */
ds_status ds_sparse_decode_profiled(const ds_shape* shape, const ds_decode_args* args, void* workspace,
                                    size_t workspace_bytes, ds_stream_t stream, void* const* events);

/* ------------------------------------------------------------------------
 * Block-compressed selection (sglang PR #43527 "QSA cache sharding",
 * "Summary": the QSA state keeps a compressed cache beside the raw K/V
 * history, and the review thread has the merge "choose 512 of 1024 blocks").
 * The pages do not define a block or its compressed key; this library's
 * reading: a block is one 64-token page of a request, and its key is the
 * per-channel mean of its tokens' index keys (summed in double in token
 * order, divided by the tokens present, rounded to nearest-even bf16).
 * ------------------------------------------------------------------------ */

/*
 * Compressed keys of the blocks of every request, written at each block's
 * physical page:
 *   index_key   bf16 [num_pages * page_size, 1, proxy_dim], the shared
 *               per-token index keys (16-byte aligned); proxy_dim 16, 32, 64
 *   page_table  int32 [B, max_pages_per_req]; seq_lens int32 [B]
 *   block_keys  out: bf16 [num_pages, proxy_dim] (16-byte aligned); entries of
 *               pages outside every request's first ceil(T_b / 64) pages are
 *               not written
 *   last_page_only  nonzero: only the page holding token T_b - 1 of each
 *               request (the one an append changes)
 * A sequence length outside [0, max_pages_per_req * 64] is flagged
 * (DS_DEVERR_SEQ_LEN) and its request skipped; a page id outside
 * [0, num_pages) is flagged (DS_DEVERR_PAGE_ID) and its block skipped.
 */
ds_status ds_block_compress(const ds_shape* shape, const void* index_key, int proxy_dim, const int32_t* page_table,
                            const int32_t* seq_lens, int last_page_only, void* block_keys, ds_stream_t stream);

typedef struct ds_block_decode_args {
  const void* q;             /* bf16 [B, Hq, D] attention queries */
  const void* qp;            /* bf16 [B, Hq, proxy_dim] index queries */
  int proxy_dim;             /* 16, 32 or 64 */
  const void* block_keys;    /* bf16 [num_pages, proxy_dim], from ds_block_compress */
  const void* k_cache;       /* [num_pages * 64, Hkv, D] bf16 or e4m3 */
  const void* v_cache;
  ds_kv_dtype kv_dtype;
  const float* k_scale;      /* fp32 [num_pages] (e4m3 only) */
  const float* v_scale;
  const int32_t* page_table; /* int32 [B, max_pages_per_req] */
  const int32_t* seq_lens;   /* int32 [B] */
  int kb;                    /* blocks kept per (request, KV head) */
  float sm_scale;
  int32_t* blocks;           /* out: int32 [B, Hkv, kb] kept blocks, ascending, -1 padded (NULL when kb = 0) */
  void* out;                 /* out: bf16 [B, Hq, D] */
  float* lse;                /* out: fp32 [B, Hq] (may be NULL) */
} ds_block_decode_args;

/*
 * The block-level decode step: block scores s[b,g,j] = sum over the group's
 * query heads and channels of qp * block key (the ds_index_score sum with the
 * block key in place of the token key), the exact top-kb blocks of each
 * (request, KV head) with ties to the lower block index (the ds_topk_select
 * rule on block rows of ceil(T_b / 64) entries), then sparse attention with
 * the fused LSE merge over every token below T_b of the kept blocks (at most
 * kb * 64 tokens). `workspace`: at least ds_block_decode_workspace_bytes
 * bytes, 256-byte aligned, no initialisation; calls sharing it must not
 * overlap. No host synchronisation, no allocation.
 */
size_t ds_block_decode_workspace_bytes(const ds_shape* shape, int kb);
ds_status ds_sparse_decode_blocks(const ds_shape* shape, const ds_block_decode_args* args, void* workspace,
                                  size_t workspace_bytes, ds_stream_t stream);

/*
 * Kernel launches one ds_sparse_decode call makes for this shape and k (it
 * issues no other device work: no copies, no memsets); 0 when the arguments
 * are invalid or there is nothing to do. Host-only query.
 */
int ds_decode_kernel_launches(const ds_shape* shape, int k);

/*
 * Split-KV count the chained call uses internally for this shape and k (so a
 * caller running the four stages one by one can reproduce it): the largest
 * power of two up to 16 with at most one split per started 64 selected
 * tokens and at most 456 (request, KV head, split) CTAs, lowered on a device
 * until every cluster of splits is resident at once. 0 for an invalid shape.
 * Host-only.
 */
int ds_decode_num_splits(const ds_shape* shape, int k);

/* Human-readable name of a status. */
const char* ds_error_string(ds_status status);

/*
 * Synchronises the current device, returns the sticky device error word in
 * *flags (DS_DEVERR_* bits) and clears it. Returns DS_ERR_DEVICE_CHECK when
 * any bit was set, DS_OK otherwise.
 */
ds_status ds_device_errors(unsigned* flags);

#ifdef __cplusplus
}
#endif

#endif /* DS_SPARSE_H */
