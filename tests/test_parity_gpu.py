"""GPU parity: every stage of libdssparse, called through its C ABI, against
the oracle on the same seeded inputs.

Top-k indices and integer-valued proxy scores must be bit-exact; attention
outputs within |gpu - ref| <= atol + 1e-2 |ref| (atol 2e-3 for a bf16 KV cache,
2e-2 for FP8), lse within 1e-3. Sizes span several tiles and a ragged tail.
"""
import math

import pytest
import torch

import dsgen
import oracle
from gpu_helpers import (ATOL_BF16, ATOL_FP8, assert_close, assert_lse_close, atol_for, default_scale,
                         oracle_every_row, run_decode, shape_of, workload)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ds():
    import top_sparse_decode_label_gb300 as ds
    return ds


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    if torch.cuda.is_available():
        assert _ds().ds_device_errors() == 0


# --------------------------------------------------------------------- stage 1

SCORE_CASES = [
    # name, B, Hq, Hkv, T, C, HL
    ("ds_c16_single_kv", 1, 4, 1, [1000], 16, 1),
    ("ds_c32_hkv8", 3, 32, 8, [3000, 1777, 64], 32, 8),
    ("ds_c16_hkv32_two_head_blocks", 3, 32, 32, [1500, 999, 1], 16, 32),
    ("ds_c16_hkv2_tpi8", 2, 8, 2, [700, 130], 16, 2),
    ("ds_c64_hkv8_two_head_blocks", 2, 16, 8, [650, 65], 64, 8),
    ("ds_c32_hkv2", 2, 16, 2, [333, 1000], 32, 2),
    ("qsa_c64_hkv4", 2, 32, 4, [2000, 333], 64, 1),
    ("qsa_c64_hkv8_g1", 2, 8, 8, [257, 129], 64, 1),
    ("qsa_c32_hkv2", 1, 16, 2, [515], 32, 1),
    ("qsa_c16_hkv2", 1, 16, 2, [515], 16, 1),
]


@pytest.mark.parametrize("case", SCORE_CASES, ids=[c[0] for c in SCORE_CASES])
def test_index_score_bit_exact(case):
    name, B, Hq, Hkv, T, C, HL = case
    w = workload(name, B, Hq, Hkv, T, C, HL, k=16)
    inp = dsgen.make_inputs(w)
    g = inp.to(DEV)
    shape = shape_of(inp)
    scores = torch.full((B, Hkv, w.max_seq_len), float("nan"), device=DEV)
    _ds().ds_index_score(shape, g.qp, g.label, g.page_table, g.seq_lens, scores)
    ref = oracle.index_score(inp.qp, inp.label, inp.page_table, inp.seq_lens, Hkv, w.max_seq_len)
    got = scores.cpu()
    for b in range(B):
        Tb = w.seq_lens[b]
        assert torch.equal(got[b, :, :Tb], ref[b, :, :Tb]), f"request {b}"
        assert torch.isnan(got[b, :, Tb:]).all(), "wrote past the request's length"


# --------------------------------------------------------------------- stage 2

def _topk_gpu(scores, seq, k, Tmax=None):
    ds = _ds()
    B, H, Tm = scores.shape
    shape = ds.Shape(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, page_size=64,
                     max_pages_per_req=max(1, -(-Tm // 64)), num_pages=1, max_seq_len=Tm)
    idx = torch.full((B, H, k), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(1, ds.ds_topk_workspace_bytes(shape, k)), dtype=torch.uint8, device=DEV)
    ds.ds_topk_select(shape, scores.to(DEV).contiguous(), seq.to(DEV), k, idx, ws)
    return idx.cpu()


def _int_scores(B, H, T, lo, hi, seed):
    return dsgen.uniform_int((B, H, T), lo, hi, seed, 3, dtype=torch.float32)


TOPK_CASES = [
    # B, H, T, seq_lens, k, lo, hi
    (1, 1, 100, [100], 10, -3, 3),
    (2, 3, 5000, [5000, 4097], 300, -40, 40),
    (1, 2, 20000, [20000], 1024, -500, 500),
    (3, 2, 9000, [9000, 0, 8191], 256, -2, 2),         # empty row, heavy ties
    (1, 1, 4096, [4096], 4096, -5, 5),                 # k == T
    (1, 1, 3000, [3000], 5000, -5, 5),                 # k > T: pad with -1
    (2, 1, 70000, [70000, 65536], 3000, -1000, 1000),
    (1, 4, 12000, [12000], 2048, 0, 0),                 # all equal: lowest indices
    (1, 1, 12000, [11999], 1, -100000, 100000),
]


@pytest.mark.parametrize("case", TOPK_CASES)
def test_topk_bit_exact_on_integer_scores(case):
    B, H, T, seq, k, lo, hi = case
    s = _int_scores(B, H, T, lo, hi, T + k)
    seq_t = torch.tensor(seq, dtype=torch.int32)
    got = _topk_gpu(s, seq_t, k)
    ref = oracle.topk(s, seq_t, k)
    assert torch.equal(got, ref)


def test_topk_real_valued_scores_with_nan_and_signed_zero():
    s = dsgen.normal((2, 2, 30000), 9, 4, dtype=torch.float32)
    s[0, 0, 100:200] = float("nan")
    s[0, 1, :5000] = 0.0
    s[0, 1, 5000:10000] = -0.0
    s[1, 0, ::7] = 2.5
    seq = torch.tensor([30000, 29999], dtype=torch.int32)
    for k in (1, 777, 5000, 29990):
        assert torch.equal(_topk_gpu(s, seq, k), oracle.topk(s, seq, k)), k


def test_topk_periodic_blocks_of_ties():
    # Blocks of 16 equal high scores every 400 tokens over a background of
    # equal low scores: the k-th largest falls inside a tie class for k above
    # and below the number of high scores (4096), so the lowest-index rule
    # decides which ties are kept.
    T = 512 * 200
    s = torch.zeros((1, 1, T))
    for j in range(256):
        s[0, 0, 400 * j + 192:400 * j + 208] = 1.0
    seq = torch.tensor([T], dtype=torch.int32)
    for k in (5000, 4097, 4096, 100):
        assert torch.equal(_topk_gpu(s, seq, k), oracle.topk(s, seq, k)), k


def test_topk_rows_longer_than_one_bitmap_window():
    T = (1 << 20) + 70000
    s = _int_scores(1, 2, T, -3000, 3000, 11)
    seq = torch.tensor([T], dtype=torch.int32)
    assert torch.equal(_topk_gpu(s, seq, 2048), oracle.topk(s, seq, 2048))
    ties = torch.zeros((1, 1, T))
    ties[0, 0, (1 << 20) - 5:] = 1.0     # ties straddle the window edge
    assert torch.equal(_topk_gpu(ties, seq, 100), oracle.topk(ties, seq, 100))


# --------------------------------------------------------------------- stage 3 + 4

ATTN_CASES = [
    # name, B, Hq, Hkv, T, kv, k
    ("g4_bf16", 2, 16, 4, [1500, 333], "bf16", 200),
    ("g1_bf16", 2, 4, 4, [900, 100], "bf16", 150),
    ("g2_bf16", 1, 8, 4, [700], "bf16", 64),
    ("g8_fp8", 2, 32, 4, [2000, 700], "fp8_e4m3", 300),
    ("g4_fp8", 1, 8, 2, [515], "fp8_e4m3", 40),
    ("g1_fp8", 1, 2, 2, [515], "fp8_e4m3", 97),
]


def _attn_inputs(case):
    name, B, Hq, Hkv, T, kv, k = case
    HL = 1 if kv == "fp8_e4m3" else Hkv
    C = 64 if HL == 1 else 32
    w = workload(name, B, Hq, Hkv, T, C, HL, k, kv)
    inp = dsgen.make_inputs(w)
    _, idx, _, _ = oracle.decode(inp, k=k)
    return w, inp, idx


@pytest.mark.parametrize("case", ATTN_CASES, ids=[c[0] for c in ATTN_CASES])
@pytest.mark.parametrize("S,mode", [(1, 0), (3, 0), (16, 0), (4, 1), (5, 1)])
def test_sparse_attention_partials_match_oracle(case, S, mode):
    w, inp, idx = _attn_inputs(case)
    g = inp.to(DEV)
    shape = shape_of(inp)
    B, Hq, D = w.batch, w.num_q_heads, w.head_dim
    o_ref, l_ref = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                                      inp.seq_lens, idx, None, S, mode)
    atol = atol_for(w)
    if S == 1:
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, Hq), float("nan"), device=DEV)
        _ds().ds_sparse_decode_attn(shape, g.q, g.k_cache, g.v_cache, g.k_scale, g.v_scale, g.page_table,
                                    g.seq_lens, idx.to(DEV), out=out, lse=lse)
        assert_close(out, o_ref[0], atol, "out")
        assert_lse_close(lse, l_ref[0], "lse")
    else:
        o_part = torch.full((S, B, Hq, D), float("nan"), device=DEV)
        l_part = torch.full((S, B, Hq), float("nan"), device=DEV)
        _ds().ds_sparse_decode_attn(shape, g.q, g.k_cache, g.v_cache, g.k_scale, g.v_scale, g.page_table,
                                    g.seq_lens, idx.to(DEV), num_splits=S, split_mode=mode, o_part=o_part,
                                    lse_part=l_part)
        assert_close(o_part, o_ref, atol, "o_part")
        assert_lse_close(l_part, l_ref, "lse_part")
        # Merging the GPU partials on the GPU gives the unsplit oracle result.
        out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=DEV)
        lse = torch.empty((B, Hq), device=DEV)
        _ds().ds_lse_merge(o_part, l_part, out, lse)
        o1, l1 = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                                    inp.seq_lens, idx, None, 1, 0)
        assert_close(out, o1[0], atol, "merged out")
        assert_lse_close(lse, l1[0], "merged lse")


ATTN_CASES_256 = [
    # name, B, Hq, Hkv, T, kv, k -- head dimension 256 (the QSA model's shape on Blackwell)
    ("d256_g8_fp8", 2, 32, 4, [2000, 700], "fp8_e4m3", 300),
    ("d256_g4_bf16", 2, 16, 4, [1000, 333], "bf16", 200),
    ("d256_g1_bf16", 1, 2, 2, [515], "bf16", 97),
]


@pytest.mark.parametrize("case", ATTN_CASES_256, ids=[c[0] for c in ATTN_CASES_256])
@pytest.mark.parametrize("S,mode", [(1, 0), (3, 0), (4, 1)])
def test_sparse_attention_head_dim_256(case, S, mode):
    name, B, Hq, Hkv, T, kv, k = case
    HL = 1 if kv == "fp8_e4m3" else Hkv
    w = workload(name, B, Hq, Hkv, T, 64 if HL == 1 else 32, HL, k, kv, head_dim=256)
    inp = dsgen.make_inputs(w)
    _, idx, _, _ = oracle.decode(inp, k=k)
    g = inp.to(DEV)
    D = 256
    o_ref, l_ref = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                                      inp.seq_lens, idx, None, S, mode)
    o_part = torch.full((S, B, Hq, D), float("nan"), device=DEV)
    l_part = torch.full((S, B, Hq), float("nan"), device=DEV)
    if S == 1:
        out = torch.full((B, Hq, D), float("nan"), dtype=torch.bfloat16, device=DEV)
        lse = torch.full((B, Hq), float("nan"), device=DEV)
        _ds().ds_sparse_decode_attn(shape_of(inp), g.q, g.k_cache, g.v_cache, g.k_scale, g.v_scale, g.page_table,
                                    g.seq_lens, idx.to(DEV), out=out, lse=lse)
        assert_close(out, o_ref[0], atol_for(w), "out")
        assert_lse_close(lse, l_ref[0], "lse")
    else:
        _ds().ds_sparse_decode_attn(shape_of(inp), g.q, g.k_cache, g.v_cache, g.k_scale, g.v_scale, g.page_table,
                                    g.seq_lens, idx.to(DEV), num_splits=S, split_mode=mode, o_part=o_part,
                                    lse_part=l_part)
        assert_close(o_part, o_ref, atol_for(w), "o_part")
        assert_lse_close(l_part, l_ref, "lse_part")


def test_attention_with_padded_and_empty_rows():
    w = workload("pad", 3, 8, 2, [100, 0, 37], 32, 2, 64)
    inp = dsgen.make_inputs(w)
    _, idx, _, _ = oracle.decode(inp)
    assert (idx[2] == -1).any() and (idx[1] == -1).all() and not (idx[0] == -1).any()
    g = inp.to(DEV)
    out = torch.full((3, 8, 128), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((3, 8), float("nan"), device=DEV)
    _ds().ds_sparse_decode_attn(shape_of(inp), g.q, g.k_cache, g.v_cache, None, None, g.page_table, g.seq_lens,
                                idx.to(DEV), out=out, lse=lse)
    o_ref, l_ref = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, None, None, inp.page_table, inp.seq_lens,
                                      idx)
    assert_close(out, o_ref[0], ATOL_BF16, "out")
    assert_lse_close(lse, l_ref[0], "lse")
    assert torch.equal(out[1].cpu(), torch.zeros(8, 128, dtype=torch.bfloat16))


def test_lse_merge_matches_oracle_with_empty_chunks():
    S, rows, D = 7, 300, 128
    o = dsgen.normal((S, rows, D), 3, 1, dtype=torch.float32)
    l = dsgen.normal((S, rows), 3, 2, dtype=torch.float32) * 5
    l[2] = -math.inf
    l[:, 17] = -math.inf
    out = torch.empty((rows, D), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((rows,), device=DEV)
    _ds().ds_lse_merge(o.to(DEV), l.to(DEV), out, lse)
    ro, rl = oracle.lse_merge(o.double(), l.double())
    assert_close(out, ro, ATOL_BF16, "merge out")
    assert_lse_close(lse, rl, "merge lse")


# --------------------------------------------------------------------- chained

CHAIN_CASES = [
    ("tiny_ds", dsgen.WORKLOADS[0].scaled(seq_lens=[4096])),
    ("llama_ds_small", dsgen.WORKLOADS[1].scaled(seq_lens=[6000, 5001, 77], top_k=300)),
    ("longchat_ds_small", dsgen.WORKLOADS[2].scaled(batch=2, seq_lens=[2000, 1999], top_k=128)),
    ("qsa_small", dsgen.WORKLOADS[3].scaled(batch=3, seq_lens=[9000, 6401, 4096], top_k=512)),
    ("qsa_1m_small", dsgen.WORKLOADS[4].scaled(seq_lens=[40000], top_k=2048)),
    ("qsa_d256_small", dsgen.WORKLOADS[3].scaled(batch=2, seq_lens=[9000, 4097], top_k=512, head_dim=256)),
    ("llama_ds_d256_small", dsgen.WORKLOADS[1].scaled(batch=2, seq_lens=[5000, 77], top_k=300, head_dim=256)),
    # Rows of one call whose k is small, large and equal against their length.
    ("mixed_rows", dsgen.WORKLOADS[1].scaled(seq_lens=[6000, 1000, 300], top_k=300)),
    # 96 rows of up to 20,000 tokens: two-CTA clusters whose full slices take one pass of 20 keys per thread.
    ("longchat_one_wide_pass", dsgen.WORKLOADS[2].scaled(seq_lens=[20000, 17001, 9000], top_k=1024)),
]


@pytest.mark.parametrize("name,w", CHAIN_CASES, ids=[c[0] for c in CHAIN_CASES])
def test_chained_decode_matches_oracle(name, w):
    inp = dsgen.make_inputs(w)
    g = inp.to(DEV)
    idx, out, lse = run_decode(g, shape_of(inp), w.top_k)
    _, ridx, rout, rlse = oracle.decode(inp)
    assert torch.equal(idx.cpu(), ridx)
    assert_close(out, rout, atol_for(w), "out")
    assert_lse_close(lse, rlse, "lse")


def _one_token_per_page(T):
    """One token of every 64-token page of a row of T tokens, at an offset that varies from page to page (the
    page's first token when that offset lies past T)."""
    out = []
    for i in range(-(-T // 64)):
        t = i * 64 + ((i * 37 + 11) & 63)
        out.append(t if t < T else i * 64)
    return out


@pytest.mark.parametrize("layout", ["per_head_label", "shared_index_key"])
def test_chained_decode_with_a_few_high_tokens_and_ties_below_them(layout):
    # Only one token per page scores high (all equally), every other token scores 0: the top-k keeps the high
    # tokens and then the lowest-index tokens of score 0, through the chained call on both label layouts.
    T, k = 20000, 1000
    if layout == "per_head_label":
        w = workload("sparse_high_ds", 1, 8, 2, [T], 32, 2, k)
    else:
        w = workload("sparse_high_qsa", 1, 16, 2, [T], 64, 1, k, kv="fp8_e4m3", from_q=False)
    inp = dsgen.make_inputs(w)
    inp.qp = torch.ones_like(inp.qp)
    lab = torch.zeros_like(inp.label)
    pt = inp.page_table[0].long()
    high = _one_token_per_page(T)
    for t in high:
        lab[pt[t // 64] * 64 + t % 64] = 8
    inp.label = lab
    g = inp.to(DEV)
    idx, out, lse = run_decode(g, shape_of(inp), k)
    _, ridx, rout, rlse = oracle.decode(inp)
    assert torch.equal(idx.cpu(), ridx)
    assert set(high) <= set(ridx[0, 0].tolist()) and len(high) < k
    assert_close(out, rout, atol_for(w), "out")
    assert_lse_close(lse, rlse, "lse")


@pytest.mark.parametrize("pattern", ["iid", "high_per_page", "negative", "all_tied"])
def test_chained_decode_with_the_block_maxima_filter(pattern):
    # Shared 64-wide index keys, rows long enough and k small enough (at most 1/128 of the row) for the top-k to
    # bound its threshold with the scan's 16-token block maxima and read only the blocks that can hold a kept
    # token; the second request is ragged (a partial last block). Patterns: iid scores; one high token per
    # page, all equal and more of them than k (ties at the threshold); every score negative; every score tied
    # (the candidates overflow and the exact two-pass selection takes over).
    T, k = [300001, 280003], 2048
    w = workload("bm_" + pattern, 2, 16, 2, T, 64, 1, k, kv="fp8_e4m3", from_q=False)
    inp = dsgen.make_inputs(w)
    if pattern == "high_per_page":
        inp.qp = torch.ones_like(inp.qp)
        lab = torch.zeros_like(inp.label)
        for b in range(2):
            pt = inp.page_table[b].long()
            for t in _one_token_per_page(T[b]):
                lab[pt[t // 64] * 64 + t % 64] = 8
        inp.label = lab
    elif pattern == "negative":
        inp.qp = -inp.qp.abs()
        inp.label = inp.label.abs()
    elif pattern == "all_tied":
        inp.qp = torch.zeros_like(inp.qp)
    g = inp.to(DEV)
    idx, out, lse = run_decode(g, shape_of(inp), k)
    ridx, rout, rlse = oracle_every_row(inp)
    assert torch.equal(idx.cpu(), ridx)
    if pattern == "high_per_page":
        assert all(ridx[b, h].tolist() == _one_token_per_page(T[b])[:k] for b in range(2) for h in range(2))
    if pattern == "all_tied":
        assert ridx.eq(torch.arange(k, dtype=torch.int32)).all()
    assert_close(out, rout, ATOL_FP8, "out")
    assert_lse_close(lse, rlse, "lse")


@pytest.mark.parametrize("pattern", ["iid", "all_tied"])
def test_chained_decode_long_rows_with_a_per_head_label(pattern):
    # The same long rows and small k with a per-head label cache (no block maxima from that scan): the top-k
    # guesses its filter bin from a sample of the scores; with every score tied the guess fails and the exact
    # two-pass selection takes over.
    T, k = [300001, 280003], 2048
    w = workload("long_ds_" + pattern, 2, 8, 2, T, 32, 2, k)
    inp = dsgen.make_inputs(w)
    if pattern == "all_tied":
        inp.qp = torch.zeros_like(inp.qp)
    g = inp.to(DEV)
    idx, out, lse = run_decode(g, shape_of(inp), k)
    ridx, rout, rlse = oracle_every_row(inp)
    assert torch.equal(idx.cpu(), ridx)
    if pattern == "all_tied":
        assert ridx.eq(torch.arange(k, dtype=torch.int32)).all()
    assert_close(out, rout, ATOL_BF16, "out")
    assert_lse_close(lse, rlse, "lse")


def test_chained_decode_is_exact_when_every_score_ties():
    # A zero proxy query: every score is 0 and the top-k keeps the lowest token indices, on a long and a short
    # row of one call.
    w = dsgen.WORKLOADS[1].scaled(batch=2, seq_lens=[20000, 5000], top_k=600)
    inp = dsgen.make_inputs(w)
    inp.qp = torch.zeros_like(inp.qp)
    g = inp.to(DEV)
    idx, out, lse = run_decode(g, shape_of(inp), w.top_k)
    _, ridx, rout, rlse = oracle.decode(inp)
    assert torch.equal(idx.cpu(), ridx)
    assert idx.cpu().eq(torch.arange(600, dtype=torch.int32)).all()
    assert_close(out, rout, ATOL_BF16, "out")
    assert_lse_close(lse, rlse, "lse")


def test_chained_decode_on_long_rows_reuses_its_workspace():
    # Rows of 200,000 and 150,001 tokens, two calls with different inputs on one workspace: the second call must
    # not see the first one's state.
    w = dsgen.WORKLOADS[3].scaled(batch=2, seq_lens=[200000, 150001], top_k=2048)
    a = dsgen.make_inputs(w, seed=31)
    b = dsgen.make_inputs(w, seed=32)
    g = a.to(DEV)
    shape = shape_of(a)
    ds = _ds()
    ws = torch.zeros(ds.ds_decode_workspace_bytes(shape, w.proxy_dim, w.top_k), dtype=torch.uint8, device=DEV)
    idx = torch.empty((w.batch, w.num_kv_heads, w.top_k), dtype=torch.int32, device=DEV)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.batch, w.num_q_heads), device=DEV)
    for src in (a, b):
        for name in ("q", "qp", "label", "k_cache", "v_cache", "k_scale", "v_scale", "page_table"):
            getattr(g, name).copy_(getattr(src, name).to(DEV))
        ds.ds_sparse_decode(shape, g.q, g.qp, g.label, g.k_cache, g.v_cache, g.k_scale, g.v_scale, g.page_table,
                            g.seq_lens, w.top_k, idx, out, lse, ws)
        torch.cuda.synchronize()
        ridx, rout, rlse = oracle_every_row(src)
        assert torch.equal(idx.cpu(), ridx)
        assert_close(out, rout, ATOL_FP8, "out")
        assert_lse_close(lse, rlse, "lse")


def test_k_at_least_seq_len_is_dense_attention():
    w = dsgen.WORKLOADS[2].scaled(batch=2, seq_lens=[1500, 900])
    inp = dsgen.make_inputs(w)
    g = inp.to(DEV)
    k = 1500
    idx, out, lse = run_decode(g, shape_of(inp), k)
    _, ridx, rout, rlse = oracle.decode(inp, k=k)
    assert torch.equal(idx.cpu(), ridx)
    assert idx[0, :, :1500].cpu().eq(torch.arange(1500, dtype=torch.int32)).all()
    assert_close(out, rout, ATOL_BF16, "dense out")
    assert_lse_close(lse, rlse, "dense lse")


def test_replay_after_input_mutation_reuses_workspace():
    # The same buffers, new contents: the second call must not see the first one's state.
    w = dsgen.WORKLOADS[1].scaled(seq_lens=[5000, 3000, 4000], top_k=256)
    a = dsgen.make_inputs(w, seed=21)
    b = dsgen.make_inputs(w, seed=22)
    ga = a.to(DEV)
    shape = shape_of(a)
    ws = torch.zeros(_ds().ds_decode_workspace_bytes(shape, w.proxy_dim, w.top_k), dtype=torch.uint8, device=DEV)
    idx = torch.empty((w.batch, w.num_kv_heads, w.top_k), dtype=torch.int32, device=DEV)
    out = torch.empty((w.batch, w.num_q_heads, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((w.batch, w.num_q_heads), device=DEV)
    for src in (a, b, a):
        ga.qp.copy_(src.qp.to(DEV))
        ga.label.copy_(src.label.to(DEV))
        ga.q.copy_(src.q.to(DEV))
        ga.k_cache.copy_(src.k_cache.to(DEV))
        ga.v_cache.copy_(src.v_cache.to(DEV))
        _ds().ds_sparse_decode(shape, ga.q, ga.qp, ga.label, ga.k_cache, ga.v_cache, None, None, ga.page_table,
                               ga.seq_lens, w.top_k, idx, out, lse, ws)
        _, ridx, rout, rlse = oracle.decode(src)
        assert torch.equal(idx.cpu(), ridx)
        assert_close(out, rout, ATOL_BF16, "out")


def test_bad_page_id_is_flagged_not_read():
    w = workload("badpage", 1, 8, 2, [300], 32, 2, 32)
    inp = dsgen.make_inputs(w)
    inp.page_table[0, 2] = 10 ** 6
    g = inp.to(DEV)
    run_decode(g, shape_of(inp), 32)
    flags = _ds().ds_device_errors()
    assert flags & 2


# --------------------------------------------------------------------- full size, every row

@pytest.mark.parametrize("ci,D", [(1, 128), (2, 128), (3, 128), (4, 128), (1, 256), (3, 256)])
def test_full_size_workload_every_row(ci, D):
    # The four full-size workloads through the chained call the bench times, every (request, KV head) row
    # against the oracle (indices bit-exact, out and lse element by element); head dimension 256 for the
    # Llama-8B DS and QSA shapes as `bench.py --head-dim 256` times them.
    w = dsgen.WORKLOADS[ci]
    if D != w.head_dim:
        w = w.scaled(head_dim=D, name=f"{w.name}_d{D}")
    g = dsgen.make_inputs(w, device=DEV)
    shape = shape_of(g)
    idx, out, lse = run_decode(g, shape, w.top_k)
    torch.cuda.synchronize()
    inp = g.to("cpu")
    ridx, rout, rlse = oracle_every_row(inp)
    gi = idx.cpu()
    for b in range(w.batch):
        for gg in range(w.num_kv_heads):
            assert torch.equal(gi[b, gg], ridx[b, gg]), f"indices of row (b{b}, g{gg})"
    assert_close(out, rout, atol_for(w), "out")
    assert_lse_close(lse, rlse, "lse")
    if ci == 4:
        # Split-KV over 4 and 16 chunks, merged, equals the unsplit result and the oracle's split merge.
        ds = _ds()
        for S in (4, 16):
            o_part = torch.empty((S, w.batch, w.num_q_heads, w.head_dim), device=DEV)
            l_part = torch.empty((S, w.batch, w.num_q_heads), device=DEV)
            ds.ds_sparse_decode_attn(shape, g.q, g.k_cache, g.v_cache, g.k_scale, g.v_scale, g.page_table,
                                     g.seq_lens, idx, num_splits=S, o_part=o_part, lse_part=l_part)
            mo = torch.empty_like(out)
            ml = torch.empty_like(lse)
            ds.ds_lse_merge(o_part, l_part, mo, ml)
            assert_close(mo, out.float(), ATOL_FP8, f"merged S={S} vs unsplit")
            assert_lse_close(ml, lse.double(), f"merged lse S={S}")
            os_, ls_ = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                                          inp.page_table, inp.seq_lens, ridx, None, S, 0)
            mo2, ml2 = oracle.lse_merge(os_, ls_)
            assert_close(mo, mo2, ATOL_FP8, f"merged S={S} vs the oracle's split merge")
            assert_lse_close(ml, ml2, f"merged lse S={S} vs the oracle's")


def test_k_equal_to_seq_len_is_dense_attention_at_the_longchat_size():
    # The longchat workload's own size (3 requests x 20000 tokens, 32 KV heads) with k = T = 20000: every
    # token is kept, so the call is dense softmax attention over the whole cache, split and merged inside
    # the attention's clusters at that size.
    w = dsgen.WORKLOADS[2]
    T = w.max_seq_len
    g = dsgen.make_inputs(w, device=DEV)
    idx, out, lse = run_decode(g, shape_of(g), T)
    torch.cuda.synchronize()
    inp = g.to("cpu")
    ridx, rout, rlse = oracle_every_row(inp, k=T)
    assert torch.equal(idx.cpu(), ridx)
    assert idx.cpu().eq(torch.arange(T, dtype=torch.int32)).all()
    assert_close(out, rout, ATOL_BF16, "dense out")
    assert_lse_close(lse, rlse, "dense lse")
