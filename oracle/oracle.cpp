// Oracle for decode-step top-k sparse attention -- TEST INFRASTRUCTURE ONLY.
//
// A plain, slow, single-threaded CPU restatement of the four stages, written
// for a reader to check by eye. Only the tests, the smoke check and the
// benchmark's CPU-baseline leg load it; the library never calls it, and it
// shares no code, header or table with the CUDA path.
//
// Sources (the pages give prose, no formulas or code):
//   [DS]   "Support double sparsity" (sglang PR #1459): sections "Motivation",
//          "Modifications" (a Triton sparse decode attention) and "Speedup
//          Evaluation" (heavy channels, heavy tokens); the review thread's
//          forward_extend traceback shows the label cache as a per-token,
//          per-head gather of K channels (index [tokens, heads, channels]).
//   [QSA]  sglang PR #43527 "QSA cache sharding": section "Distributed QSA
//          execution" (scan, exact Top-K with deterministic global token-ID
//          tie-breaking, owner-side sparse attention, FP32 log-sum-exp merge
//          of partial outputs) and "CUDA Graph metadata" (page-table tails are
//          not cleared; consumers stop at the sequence length).
//   [PLG]  "QSA HiSparse - SGLang plugin", section "Supported versions": FP8
//          E4M3 KV cache, page size 64.
//   [CP]   sglang PR #39721, "Motivation": the QSA indexer scores and selects
//          top-k; sparse_gqa attends over the selection.
//
// Readings taken where the pages are silent (each one is a choice):
//   R1 proxy score of KV head g = sum over the query heads h of g's group of
//      sum_c qp[b,h,c] * L[slot(b,t), gL, c]; no scale, no activation.
//      gL = g for a per-head label cache, 0 for a shared index key.
//   R2 GQA grouping is contiguous: query head h belongs to KV head h / G.
//   R3 slot(b,t) = page_table[b][t / P] * P + t % P.
//   R4 top-k order: larger score first, equal scores by smaller token index;
//      NaN ranks below every number. Output ascending by token index, padded
//      with -1 after min(k, T_b) entries.
//   R5 attention scale is a caller argument (1/sqrt(D) by default); logs are
//      natural logs.
//   R6 split-KV: contiguous balanced chunks of the selected list, or chunk =
//      logical page mod S (the page-owner placement); an empty chunk has
//      lse = -inf and o = 0.
//   R7 FP8 values are e4m3 (1 sign, 4 exponent bits with bias 7, 3 mantissa
//      bits, subnormals, S.1111.111 = NaN, no infinities) times one fp32 scale
//      per physical page, separate for K and V.
//   R8 appending a token to an FP8 cache stores e4m3(x / scale) with the
//      page's scale: the fp32 quotient rounded to nearest even, saturated to
//      +-448. The page's scale is set by whoever allocates the page.
//   R9 the new token of request b goes to logical position positions[b]
//      (a negative position skips the row); the DS label of a token is the
//      per-head gather of its K at the heavy channels, taken from the bf16 K
//      before any FP8 rounding; the QSA index key is an input, copied.
//   R14 shard ownership of pages is page-interleaved: logical page p of a
//      request belongs to shard p mod S (the placement the attention's split
//      mode 1 also uses).
//   R15 a compressed block of [QSA] "Summary" (the QSA compressed cache) and
//      the review thread ("choose 512 of 1024 blocks") is one KV page of a
//      request: block j covers logical tokens [64j, 64j + 64) below T_b.
//   R16 a block's compressed index key is the per-channel mean of its tokens'
//      index keys: their sum in double in token order, divided by the number
//      of tokens present, rounded to bfloat16 (nearest, ties to even), stored
//      per physical page. A block is scored like a token (R1) with its key.
//   R17 block selection keeps the top-k blocks of each (request, KV head) by
//      the R4 rule (ties to the lower block index); the attended tokens are
//      every token below T_b of the kept blocks, ascending, then -1.
//
// All arithmetic is in double; the scores are rounded to float once, at the
// end (the top-k ranks float scores, as the CUDA path does).

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <limits>
#include <vector>

namespace {

// bfloat16 is the upper half of an IEEE binary32.
double bf16_value(uint16_t bits) {
  uint32_t u = static_cast<uint32_t>(bits) << 16;
  float f;
  std::memcpy(&f, &u, sizeof f);
  return static_cast<double>(f);
}

// OCP FP8 E4M3 (reading R7), decoded from the bit fields.
double e4m3_value(uint8_t byte) {
  const int sign = (byte >> 7) & 1;
  const int exp = (byte >> 3) & 0xF;
  const int man = byte & 0x7;
  double mag;
  if (exp == 0xF && man == 0x7) return std::numeric_limits<double>::quiet_NaN();
  if (exp == 0)
    mag = std::ldexp(static_cast<double>(man) / 8.0, 1 - 7);        // subnormal
  else
    mag = std::ldexp(1.0 + static_cast<double>(man) / 8.0, exp - 7);  // normal
  return sign ? -mag : mag;
}

// E4M3 encoding of x (reading R8): the finite code whose value (R7) is
// nearest to x, ties to the code with an even last mantissa bit (round to
// nearest even); magnitudes past 448, the largest finite value, give 448
// (saturation); NaN gives S.1111.111. Found by comparing against all 127
// non-negative finite codes, in increasing order of value.
uint8_t e4m3_encode(double x) {
  if (std::isnan(x)) return 0x7F;
  const uint8_t sign = std::signbit(x) ? 0x80 : 0x00;
  const double a = std::fabs(x);
  uint8_t best = 0;
  double best_err = std::numeric_limits<double>::infinity();
  for (int c = 0; c <= 0x7E; ++c) {
    const double err = std::fabs(a - e4m3_value(static_cast<uint8_t>(c)));
    if (err < best_err || (err == best_err && (c & 1) == 0)) {
      best = static_cast<uint8_t>(c);
      best_err = err;
    }
  }
  return sign | best;
}

long long slot_of(const int32_t* page_table, int max_pages, int page_size, int b, long long t) {
  const long long page = page_table[static_cast<long long>(b) * max_pages + t / page_size];
  return page * page_size + t % page_size;
}

// Nearest bfloat16 to x, ties to the even significand (R16): bfloat16 has the
// exponent range of binary32 and 8 significant bits, so the spacing of values
// near x = m 2^e (0.5 <= |m| < 1) is 2^(e-8), and never below 2^-133, the
// smallest subnormal. Finite results only (block means of finite keys).
uint16_t bf16_round(double x) {
  if (x == 0.0) return std::signbit(x) ? 0x8000u : 0u;
  int e = 0;
  std::frexp(x, &e);
  const int qexp = std::max(e - 8, -133);
  const double r = std::nearbyint(std::ldexp(x, -qexp));   // default rounding: nearest, ties to even
  const float v = static_cast<float>(std::ldexp(r, qexp));  // exact: r has at most 8 significant bits
  uint32_t u;
  std::memcpy(&u, &v, 4);
  return static_cast<uint16_t>(u >> 16);
}

}  // namespace

extern "C" {

double oracle_bf16_value(uint16_t bits) { return bf16_value(bits); }
double oracle_e4m3_value(uint8_t byte) { return e4m3_value(byte); }

// Stage 1, proxy scoring ([DS] label cache, [QSA]/[CP] index scan; R1-R3).
//   qp      bf16 bits [B, Hq, C]
//   label   bf16 bits [num_slots, HL, C], HL = Hkv (per-head label) or 1 (shared key)
//   scores  float [B, Hkv, Tmax]; only t < seq_lens[b] is written.
//   row_mask (may be null) uint8 [B, Hkv]: compute only rows with a nonzero mask.
// Returns 0, or -1 on an argument outside the definition.
int oracle_index_score(int B, int Hq, int Hkv, int HL, int C, int page_size, int max_pages,
                       int Tmax, const uint16_t* qp, const uint16_t* label,
                       const int32_t* page_table, const int32_t* seq_lens,
                       const uint8_t* row_mask, float* scores) {
  if (Hkv <= 0 || Hq % Hkv != 0 || !(HL == Hkv || HL == 1)) return -1;
  const int G = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    const long long T = seq_lens[b];
    if (T < 0 || T > Tmax || T > static_cast<long long>(max_pages) * page_size) return -1;
    for (int g = 0; g < Hkv; ++g) {
      if (row_mask && !row_mask[b * Hkv + g]) continue;
      const int gL = (HL == 1) ? 0 : g;
      for (long long t = 0; t < T; ++t) {
        const long long slot = slot_of(page_table, max_pages, page_size, b, t);
        double s = 0.0;
        for (int h = g * G; h < (g + 1) * G; ++h) {
          for (int c = 0; c < C; ++c) {
            const double qv = bf16_value(qp[(static_cast<long long>(b) * Hq + h) * C + c]);
            const double lv = bf16_value(label[(slot * HL + gL) * C + c]);
            s += qv * lv;
          }
        }
        scores[(static_cast<long long>(b) * Hkv + g) * Tmax + t] = static_cast<float>(s);
      }
    }
  }
  return 0;
}

// Stage 2, exact top-k with lowest-token-index tie-breaking ([QSA] "Distributed
// QSA execution"; R4). Sorts every token of the row by the total order, keeps
// the first min(k, T_b), and writes them ascending by token index.
//   scores float [B, Hkv, Tmax];  idx int32 [B, Hkv, k]
int oracle_topk(int B, int Hkv, int Tmax, const float* scores, const int32_t* seq_lens, int k,
                const uint8_t* row_mask, int32_t* idx) {
  if (k < 0) return -1;
  for (int b = 0; b < B; ++b) {
    const int T = seq_lens[b];
    if (T < 0 || T > Tmax) return -1;
    for (int g = 0; g < Hkv; ++g) {
      if (row_mask && !row_mask[b * Hkv + g]) continue;
      const float* s = scores + (static_cast<long long>(b) * Hkv + g) * Tmax;
      std::vector<int32_t> order(T);
      for (int t = 0; t < T; ++t) order[t] = t;
      auto before = [s](int32_t x, int32_t y) {
        const bool nx = std::isnan(s[x]), ny = std::isnan(s[y]);
        if (nx != ny) return ny;             // a number ranks above NaN
        if (!nx && s[x] != s[y]) return s[x] > s[y];
        return x < y;                        // equal scores: smaller token index first
      };
      std::sort(order.begin(), order.end(), before);
      const int keff = std::min(k, T);
      std::vector<int32_t> chosen(order.begin(), order.begin() + keff);
      std::sort(chosen.begin(), chosen.end());
      int32_t* out = idx + (static_cast<long long>(b) * Hkv + g) * k;
      for (int i = 0; i < k; ++i) out[i] = (i < keff) ? chosen[i] : -1;
    }
  }
  return 0;
}

// Stage 3, sparse GQA decode attention over the selected tokens ([DS]
// "Modifications", [CP] sparse_gqa, [PLG] paged FP8 KV; R2, R3, R5-R7).
//   q        bf16 bits [B, Hq, D]
//   k_cache  [num_slots, Hkv, D], bf16 bits (kv_fp8 == 0) or e4m3 bytes (kv_fp8 == 1)
//   k_scale  float [num_pages] (FP8 only)
//   idx      int32 [B, Hkv, k]: a prefix of valid token indices, then -1
//   o_part   double [S, B, Hq, D]; lse_part double [S, B, Hq]
// Chunk j of the valid list is positions [j*n/S, (j+1)*n/S) (split_mode 0), or
// the tokens whose logical page mod S equals j (split_mode 1).
int oracle_sparse_attn(int B, int Hq, int Hkv, int D, int page_size, int max_pages, int kv_fp8,
                       const uint16_t* q, const void* k_cache, const void* v_cache,
                       const float* k_scale, const float* v_scale, const int32_t* page_table,
                       const int32_t* seq_lens, const int32_t* idx, int k, double sm_scale,
                       int num_splits, int split_mode, const uint8_t* row_mask,
                       double* o_part, double* lse_part) {
  if (Hkv <= 0 || Hq % Hkv != 0 || num_splits < 1 || k < 0) return -1;
  const int G = Hq / Hkv;
  const int S = num_splits;
  const double NEG_INF = -std::numeric_limits<double>::infinity();
  auto kval = [&](long long slot, int g, int d) {
    const long long e = (slot * Hkv + g) * D + d;
    if (!kv_fp8) return bf16_value(static_cast<const uint16_t*>(k_cache)[e]);
    return e4m3_value(static_cast<const uint8_t*>(k_cache)[e]) * k_scale[slot / page_size];
  };
  auto vval = [&](long long slot, int g, int d) {
    const long long e = (slot * Hkv + g) * D + d;
    if (!kv_fp8) return bf16_value(static_cast<const uint16_t*>(v_cache)[e]);
    return e4m3_value(static_cast<const uint8_t*>(v_cache)[e]) * v_scale[slot / page_size];
  };
  for (int b = 0; b < B; ++b) {
    const int T = seq_lens[b];
    for (int g = 0; g < Hkv; ++g) {
      if (row_mask && !row_mask[b * Hkv + g]) continue;
      const int32_t* row = idx + (static_cast<long long>(b) * Hkv + g) * k;
      int n = 0;
      while (n < k && row[n] >= 0) ++n;
      for (int i = 0; i < n; ++i)
        if (row[i] >= T) return -1;
      for (int h = g * G; h < (g + 1) * G; ++h) {
        const uint16_t* qh = q + (static_cast<long long>(b) * Hq + h) * D;
        for (int j = 0; j < S; ++j) {
          std::vector<int32_t> chunk;
          for (int i = 0; i < n; ++i) {
            const bool mine = (split_mode == 0)
                                  ? (i >= static_cast<long long>(j) * n / S &&
                                     i < static_cast<long long>(j + 1) * n / S)
                                  : ((row[i] / page_size) % S == j);
            if (mine) chunk.push_back(row[i]);
          }
          double* o = o_part + ((static_cast<long long>(j) * B + b) * Hq + h) * D;
          double& lse = lse_part[(static_cast<long long>(j) * B + b) * Hq + h];
          for (int d = 0; d < D; ++d) o[d] = 0.0;
          if (chunk.empty()) {
            lse = NEG_INF;
            continue;
          }
          std::vector<double> z(chunk.size());
          double m = NEG_INF;
          for (size_t i = 0; i < chunk.size(); ++i) {
            const long long slot = slot_of(page_table, max_pages, page_size, b, chunk[i]);
            double dot = 0.0;
            for (int d = 0; d < D; ++d) dot += bf16_value(qh[d]) * kval(slot, g, d);
            z[i] = sm_scale * dot;
            m = std::max(m, z[i]);
          }
          double l = 0.0;
          for (size_t i = 0; i < chunk.size(); ++i) {
            const long long slot = slot_of(page_table, max_pages, page_size, b, chunk[i]);
            const double w = std::exp(z[i] - m);
            l += w;
            for (int d = 0; d < D; ++d) o[d] += w * vval(slot, g, d);
          }
          for (int d = 0; d < D; ++d) o[d] /= l;
          lse = m + std::log(l);
        }
      }
    }
  }
  return 0;
}

// Stage 4, log-sum-exp merge of split partials ([QSA] "Distributed QSA
// execution": partial outputs merged with FP32 log-sum-exp normalisation; here
// in double). lse = log sum_j exp(lse_j); o = sum_j exp(lse_j - lse) * o_j.
//   o_part [S, rows, D]; lse_part [S, rows] -> out [rows, D]; lse [rows]
int oracle_lse_merge(int S, long long rows, int D, const double* o_part, const double* lse_part,
                     double* out, double* lse) {
  if (S < 1) return -1;
  const double NEG_INF = -std::numeric_limits<double>::infinity();
  for (long long r = 0; r < rows; ++r) {
    double m = NEG_INF;
    for (int j = 0; j < S; ++j) m = std::max(m, lse_part[j * rows + r]);
    double* o = out + r * D;
    for (int d = 0; d < D; ++d) o[d] = 0.0;
    if (m == NEG_INF) {
      lse[r] = NEG_INF;
      continue;
    }
    double sum = 0.0;
    for (int j = 0; j < S; ++j) sum += std::exp(lse_part[j * rows + r] - m);
    lse[r] = m + std::log(sum);
    for (int j = 0; j < S; ++j) {
      const double w = std::exp(lse_part[j * rows + r] - lse[r]);
      if (w == 0.0) continue;
      for (int d = 0; d < D; ++d) o[d] += w * o_part[(j * rows + r) * D + d];
    }
  }
  return 0;
}

// Cache append, the step before the path ([DS] review thread: the label is a
// per-head gather of K's channels; [PLG] FP8 E4M3 paged KV; R3, R8, R9).
//   k_new, v_new  bf16 bits [B, Hkv, D]
//   k_cache, v_cache  [num_slots, Hkv, D]: bf16 bits (kv_fp8 = 0) or e4m3 bytes
//   k_scale, v_scale  float [num_pages] (FP8 only)
//   positions     int32 [B]: logical token index to write, < 0 skips the row
//   label         bf16 bits [num_slots, HL, C]: HL == Hkv gathers
//                 k_new[b, g, channels[g, c]]; HL == 1 copies index_key[b, c]
// Rows whose position is past the page table or whose page id is outside
// [0, num_pages) are skipped. Returns 0, or -1 on an argument outside the
// definition.
int oracle_cache_append(int B, int Hkv, int D, int page_size, int max_pages, int num_pages, int kv_fp8,
                        const uint16_t* k_new, const uint16_t* v_new, void* k_cache, void* v_cache,
                        const float* k_scale, const float* v_scale, const int32_t* page_table,
                        const int32_t* positions, int HL, int C, const int32_t* channels,
                        const uint16_t* index_key, uint16_t* label) {
  if (HL != Hkv && HL != 1) return -1;
  for (int b = 0; b < B; ++b) {
    const long long t = positions[b];
    if (t < 0 || t >= static_cast<long long>(max_pages) * page_size) continue;
    const int page = page_table[static_cast<long long>(b) * max_pages + t / page_size];
    if (page < 0 || page >= num_pages) continue;
    const long long slot = slot_of(page_table, max_pages, page_size, b, t);
    for (int g = 0; g < Hkv; ++g) {
      for (int d = 0; d < D; ++d) {
        const long long src = (static_cast<long long>(b) * Hkv + g) * D + d;
        const long long dst = (slot * Hkv + g) * D + d;
        if (kv_fp8) {
          const float kq = static_cast<float>(bf16_value(k_new[src])) / k_scale[page];
          const float vq = static_cast<float>(bf16_value(v_new[src])) / v_scale[page];
          static_cast<uint8_t*>(k_cache)[dst] = e4m3_encode(kq);
          static_cast<uint8_t*>(v_cache)[dst] = e4m3_encode(vq);
        } else {
          static_cast<uint16_t*>(k_cache)[dst] = k_new[src];
          static_cast<uint16_t*>(v_cache)[dst] = v_new[src];
        }
      }
    }
    if (!label) continue;
    for (int g = 0; g < HL; ++g) {
      for (int c = 0; c < C; ++c) {
        uint16_t v;
        if (HL == Hkv && channels) {
          const int ch = channels[g * C + c];
          if (ch < 0 || ch >= D) return -1;
          v = k_new[(static_cast<long long>(b) * Hkv + g) * D + ch];
        } else {
          v = index_key[static_cast<long long>(b) * C + c];
        }
        label[(slot * HL + g) * C + c] = v;
      }
    }
  }
  return 0;
}

// Exact top-k computed as the cache-sharding page describes it ([QSA]
// "QSA cache placement", "Distributed QSA execution"; reading R14): every
// page of a request is owned by one of S shards (logical page p by shard
// p mod S); each shard takes the local top-k of its own tokens; the local
// candidates are merged into the global top-k, equal scores going to the
// smaller global token index. Same output layout as oracle_topk.
int oracle_topk_sharded(int B, int Hkv, int Tmax, const float* scores, const int32_t* seq_lens, int k,
                        int num_shards, int page_size, int32_t* idx) {
  if (k < 0 || num_shards < 1 || page_size < 1) return -1;
  for (int b = 0; b < B; ++b) {
    const int T = seq_lens[b];
    if (T < 0 || T > Tmax) return -1;
    for (int g = 0; g < Hkv; ++g) {
      const float* s = scores + (static_cast<long long>(b) * Hkv + g) * Tmax;
      auto before = [s](int32_t x, int32_t y) {   // (score descending, token ascending), NaN last
        const bool nx = std::isnan(s[x]), ny = std::isnan(s[y]);
        if (nx != ny) return ny;
        if (!nx && s[x] != s[y]) return s[x] > s[y];
        return x < y;
      };
      std::vector<int32_t> candidates;
      for (int j = 0; j < num_shards; ++j) {
        std::vector<int32_t> local;   // this shard's tokens
        for (int t = 0; t < T; ++t)
          if ((t / page_size) % num_shards == j) local.push_back(t);
        std::sort(local.begin(), local.end(), before);
        const int kj = std::min(k, static_cast<int>(local.size()));
        candidates.insert(candidates.end(), local.begin(), local.begin() + kj);
      }
      std::sort(candidates.begin(), candidates.end(), before);
      const int keff = std::min(k, static_cast<int>(candidates.size()));
      std::vector<int32_t> chosen(candidates.begin(), candidates.begin() + keff);
      std::sort(chosen.begin(), chosen.end());
      int32_t* out = idx + (static_cast<long long>(b) * Hkv + g) * k;
      for (int i = 0; i < k; ++i) out[i] = (i < keff) ? chosen[i] : -1;
    }
  }
  return 0;
}

uint8_t oracle_e4m3_encode(double x) { return e4m3_encode(x); }

// f3, block compression (R15, R16): the compressed key of every logical page
// j < ceil(T_b / 64) of every request, written at its physical page.
//   keys        bf16 bits [num_slots, 1, C] (the shared index-key cache)
//   block_keys  bf16 bits [num_pages, C]; pages outside every request untouched
int oracle_block_compress(int B, int C, int page_size, int max_pages, int num_pages, const uint16_t* keys,
                          const int32_t* page_table, const int32_t* seq_lens, uint16_t* block_keys) {
  for (int b = 0; b < B; ++b) {
    const long long T = seq_lens[b];
    if (T < 0 || T > static_cast<long long>(max_pages) * page_size) return -1;
    for (long long j = 0; j * page_size < T; ++j) {
      const int32_t pid = page_table[static_cast<long long>(b) * max_pages + j];
      if (pid < 0 || pid >= num_pages) return -1;
      const long long t0 = j * page_size, t1 = std::min(T, t0 + page_size);
      for (int c = 0; c < C; ++c) {
        double sum = 0.0;
        for (long long t = t0; t < t1; ++t) sum += bf16_value(keys[slot_of(page_table, max_pages, page_size, b, t) * C + c]);
        block_keys[static_cast<long long>(pid) * C + c] = bf16_round(sum / static_cast<double>(t1 - t0));
      }
    }
  }
  return 0;
}

// f3, block scores (R1 with the block key, R15): scores float [B, Hkv, nb_max]
// for blocks j < ceil(T_b / 64).
int oracle_block_score(int B, int Hq, int Hkv, int C, int page_size, int max_pages, int nb_max, const uint16_t* qp,
                       const uint16_t* block_keys, const int32_t* page_table, const int32_t* seq_lens,
                       float* scores) {
  if (Hkv <= 0 || Hq % Hkv != 0) return -1;
  const int G = Hq / Hkv;
  for (int b = 0; b < B; ++b) {
    const long long T = seq_lens[b];
    const long long nb = (T + page_size - 1) / page_size;
    if (T < 0 || nb > nb_max || nb > max_pages) return -1;
    for (int g = 0; g < Hkv; ++g) {
      for (long long j = 0; j < nb; ++j) {
        const long long pid = page_table[static_cast<long long>(b) * max_pages + j];
        double s = 0.0;
        for (int h = g * G; h < (g + 1) * G; ++h)
          for (int c = 0; c < C; ++c)
            s += bf16_value(qp[(static_cast<long long>(b) * Hq + h) * C + c]) * bf16_value(block_keys[pid * C + c]);
        scores[(static_cast<long long>(b) * Hkv + g) * nb_max + j] = static_cast<float>(s);
      }
    }
  }
  return 0;
}

// f3, the tokens of the kept blocks (R17): blocks int32 [B, Hkv, kb] (ascending,
// -1 padded) -> idx int32 [B, Hkv, kb * 64]: the tokens below T_b of each kept
// block in ascending order, then -1.
int oracle_block_expand(int B, int Hkv, int kb, int page_size, const int32_t* blocks, const int32_t* seq_lens,
                        int32_t* idx) {
  const long long width = static_cast<long long>(kb) * page_size;
  for (int b = 0; b < B; ++b) {
    const long long T = seq_lens[b];
    for (int g = 0; g < Hkv; ++g) {
      const int32_t* blk = blocks + (static_cast<long long>(b) * Hkv + g) * kb;
      int32_t* out = idx + (static_cast<long long>(b) * Hkv + g) * width;
      long long n = 0;
      for (int i = 0; i < kb; ++i) {
        if (blk[i] < 0) continue;
        for (long long t = static_cast<long long>(blk[i]) * page_size; t < (blk[i] + 1LL) * page_size && t < T; ++t)
          out[n++] = static_cast<int32_t>(t);
      }
      for (; n < width; ++n) out[n] = -1;
    }
  }
  return 0;
}

}  // extern "C"
