"""GPU parity of the block-compressed selection (ds_block_compress,
ds_sparse_decode_blocks) against the oracle.

Block keys must equal the oracle's bit for bit (both sides: the sum in double
in token order, one division, one rounding to nearest-even bf16). The kept
blocks must equal the oracle's top-k of its block scores exactly where those
scores are exact in fp32 (small integer keys and queries, pages whose token
counts are powers of two); on real-valued keys they must be a valid top-k up
to the rounding of the scores. The attention output is held to the
tolerances of the token path.
"""
import pytest
import torch

import dsgen
import oracle
from gpu_helpers import assert_close, assert_lse_close, atol_for, shape_of, workload

pytestmark = pytest.mark.gpu
DEV = "cuda"
P = 64


def _ds():
    import top_sparse_decode_label_gb300 as ds
    return ds


@pytest.fixture(autouse=True)
def _no_device_errors():
    yield
    if torch.cuda.is_available():
        assert _ds().ds_device_errors() == 0


def _inputs(name, B, Hq, Hkv, T, C, kv, seed, key_range=None, head_dim=128):
    w = workload(name, B, Hq, Hkv, T, C, 1, 64, kv=kv, seed=seed, head_dim=head_dim)
    inp = dsgen.make_inputs(w)
    if key_range is not None:      # small integer index keys: block means exact in bf16
        inp.label = dsgen.uniform_int(tuple(inp.label.shape), -key_range, key_range, seed, 77)
    else:                          # real-valued keys
        inp.label = dsgen.normal(tuple(inp.label.shape), seed, 78)
    return w, inp


def _compress(inp, last_only=False, init=None):
    ds = _ds()
    g = inp.to(DEV)
    C = inp.label.shape[-1]
    bk = (init.clone() if init is not None else torch.zeros((inp.num_pages, C), dtype=torch.bfloat16)).to(DEV)
    ds.ds_block_compress(shape_of(inp), g.label, g.page_table, g.seq_lens, bk, last_page_only=last_only)
    return bk.cpu()


def _decode_blocks(inp, bk, kb):
    ds = _ds()
    w = inp.w
    g = inp.to(DEV)
    shape = shape_of(inp)
    blocks = torch.full((w.batch, w.num_kv_heads, kb), -7, dtype=torch.int32, device=DEV)
    out = torch.full((w.batch, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full((w.batch, w.num_q_heads), float("nan"), dtype=torch.float32, device=DEV)
    ws = torch.empty(ds.ds_block_decode_workspace_bytes(shape, kb), dtype=torch.uint8, device=DEV)
    ds.ds_sparse_decode_blocks(shape, g.q, g.qp, bk.to(DEV), g.k_cache, g.v_cache, g.k_scale, g.v_scale,
                               g.page_table, g.seq_lens, kb, blocks, out, lse, ws)
    torch.cuda.synchronize()
    return blocks.cpu(), out.cpu(), lse.cpu()


def _reference(inp, bk, kb):
    w = inp.w
    scores = oracle.block_score(inp.qp, bk, inp.page_table, inp.seq_lens, w.num_kv_heads)
    nblocks = ((inp.seq_lens + P - 1) // P).to(torch.int32)
    blocks = oracle.topk(scores, nblocks, kb)
    idx = oracle.block_expand(blocks, inp.seq_lens)
    o, l = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                              inp.seq_lens, idx)
    rout, rlse = oracle.lse_merge(o, l)
    return scores, blocks, rout, rlse


COMPRESS_CASES = [
    # name, B, Hq, Hkv, T, C
    ("qsa_c64", 3, 32, 4, [1000, 64, 1], 64),
    ("c32_ragged", 2, 8, 2, [4097, 300], 32),
    ("c16", 2, 8, 8, [130, 2000], 16),
]


@pytest.mark.parametrize("case", COMPRESS_CASES, ids=[c[0] for c in COMPRESS_CASES])
def test_block_compress_bit_exact(case):
    name, B, Hq, Hkv, T, C = case
    w, inp = _inputs(name, B, Hq, Hkv, T, C, "bf16", 21)
    got = _compress(inp)
    ref = oracle.block_compress(inp.label, inp.page_table, inp.seq_lens, inp.num_pages)
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))


def test_block_compress_last_page_only_touches_only_the_last_pages():
    w, inp = _inputs("last", 3, 8, 2, [1000, 64, 129], 64, "bf16", 23)
    init = torch.full((inp.num_pages, 64), 0.5, dtype=torch.bfloat16)
    got = _compress(inp, last_only=True, init=init)
    ref = oracle.block_compress(inp.label, inp.page_table, inp.seq_lens, inp.num_pages)
    last = {int(inp.page_table[b, (int(T) - 1) // P]) for b, T in enumerate(inp.seq_lens.tolist())}
    for p in range(inp.num_pages):
        want = ref[p] if p in last else init[p]
        assert torch.equal(got[p].view(torch.int16), want.view(torch.int16)), p


BLOCK_CASES = [
    # name, B, Hq, Hkv, T, C, kb, kv
    ("qsa_bf16", 2, 32, 4, [64 * 40, 64 * 17 + 32], 64, 8, "bf16"),
    ("qsa_fp8", 3, 32, 4, [64 * 100, 64 * 3 + 16, 64 * 64], 64, 16, "fp8_e4m3"),
    ("all_blocks", 2, 8, 2, [64 * 5 + 8, 64 * 2], 32, 9, "bf16"),     # kb above the block count: dense
    ("one_block", 2, 16, 2, [64 * 30, 4], 64, 1, "fp8_e4m3"),
    ("empty_row", 2, 8, 1, [0, 64 * 7 + 2], 16, 3, "bf16"),
    ("qsa_d256_fp8", 2, 16, 2, [64 * 30 + 16, 64 * 9], 64, 5, "fp8_e4m3", 256),
]


@pytest.mark.parametrize("case", BLOCK_CASES, ids=[c[0] for c in BLOCK_CASES])
def test_block_decode_matches_the_oracle(case):
    name, B, Hq, Hkv, T, C, kb, kv = case[:8]
    D = case[8] if len(case) > 8 else 128
    w, inp = _inputs(name, B, Hq, Hkv, T, C, kv, 31, key_range=2, head_dim=D)
    bk = oracle.block_compress(inp.label, inp.page_table, inp.seq_lens, inp.num_pages)
    blocks, out, lse = _decode_blocks(inp, bk, kb)
    _, rblocks, rout, rlse = _reference(inp, bk, kb)
    assert torch.equal(blocks, rblocks)
    assert_close(out, rout, atol_for(w), "block decode out")
    assert_lse_close(lse, rlse, "block decode lse")


def _assert_valid_top_k(blocks, rblocks, scores):
    """Kept blocks equal the oracle's, except for swaps of blocks whose oracle scores lie within fp32
    rounding of the threshold; the list is ascending and -1 padded like the oracle's."""
    for b in range(blocks.shape[0]):
        for g in range(blocks.shape[1]):
            row = blocks[b, g].tolist()
            n = sum(1 for j in row if j >= 0)
            assert row[:n] == sorted(row[:n]) and all(j == -1 for j in row[n:])
            assert n == sum(1 for j in rblocks[b, g].tolist() if j >= 0)
            got, ref = set(row), set(rblocks[b, g].tolist())
            if got == ref:
                continue
            s = scores[b, g]
            thr = min(float(s[j]) for j in ref if j >= 0)
            for j in got ^ ref:
                assert abs(float(s[j]) - thr) <= 1e-5 * max(1.0, abs(thr)), (b, g, j)


def test_block_decode_on_real_valued_keys_keeps_a_valid_top_k():
    # Keys N(0, 1): block scores round differently in fp32 and in double, so a
    # block may swap with one whose score is within rounding of the threshold.
    w, inp = _inputs("real", 2, 32, 4, [64 * 200 + 7, 64 * 90], 64, "bf16", 41)
    kb = 12
    bk = _compress(inp)
    blocks, out, lse = _decode_blocks(inp, bk, kb)
    scores, rblocks, _, _ = _reference(inp, bk, kb)
    _assert_valid_top_k(blocks, rblocks, scores)
    # Attention over what the GPU kept equals the oracle's attention over the same blocks.
    idx = oracle.block_expand(blocks, inp.seq_lens)
    o, l = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                              inp.seq_lens, idx)
    rout, rlse = oracle.lse_merge(o, l)
    assert_close(out, rout, atol_for(w), "block decode out")
    assert_lse_close(lse, rlse, "block decode lse")


def test_block_decode_at_the_qsa_1m_shape():
    # One request of 1,048,576 tokens (16,384 blocks), 32 of them kept (2048 tokens), FP8 cache.
    w = dsgen.WORKLOADS[4]
    g = dsgen.make_inputs(w, device=DEV)
    shape = shape_of(g)
    ds = _ds()
    bk = torch.empty((g.num_pages, w.proxy_dim), dtype=torch.bfloat16, device=DEV)
    ds.ds_block_compress(shape, g.label, g.page_table, g.seq_lens, bk)
    blocks, out, lse = _decode_blocks(g, bk, 32)
    inp = g.to("cpu")
    bkc = bk.cpu()
    # Every block key of the request, bit for bit.
    ref_keys = oracle.block_compress(inp.label, inp.page_table, inp.seq_lens, inp.num_pages)
    used = inp.page_table[0, : w.seq_lens[0] // P].long()
    assert torch.equal(bkc[used].view(torch.int16), ref_keys[used].view(torch.int16))
    # The kept blocks are the oracle's top 32 of the block scores (up to score rounding: the keys' means
    # are not exact in bf16 here).
    scores = oracle.block_score(inp.qp, bkc, inp.page_table, inp.seq_lens, w.num_kv_heads)
    rblocks = oracle.topk(scores, torch.tensor([w.seq_lens[0] // P], dtype=torch.int32), 32)
    _assert_valid_top_k(blocks, rblocks, scores)
    # The attention over the tokens of the blocks the GPU kept, against the oracle's attention over them.
    idx = oracle.block_expand(blocks, inp.seq_lens)
    o, l = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                              inp.seq_lens, idx)
    rout, rlse = oracle.lse_merge(o, l)
    assert_close(out, rout, atol_for(w), "out over the kept blocks")
    assert_lse_close(lse, rlse, "lse over the kept blocks")


def test_block_decode_replays_in_a_cuda_graph_with_new_inputs():
    # No host synchronisation and no allocation: the block-level step is captured once and replayed after
    # the caches and queries change in place; each replay matches the oracle on the new contents.
    ds = _ds()
    kb = 6
    wa, a = _inputs("graph", 2, 32, 4, [64 * 50, 64 * 21 + 8], 64, "bf16", 51, key_range=2)
    _, b_ = _inputs("graph", 2, 32, 4, [64 * 50, 64 * 21 + 8], 64, "bf16", 52, key_range=2)
    g = a.to(DEV)
    shape = shape_of(a)
    bk = torch.zeros((a.num_pages, 64), dtype=torch.bfloat16, device=DEV)
    blocks = torch.empty((wa.batch, wa.num_kv_heads, kb), dtype=torch.int32, device=DEV)
    out = torch.empty((wa.batch, wa.num_q_heads, 128), dtype=torch.bfloat16, device=DEV)
    lse = torch.empty((wa.batch, wa.num_q_heads), dtype=torch.float32, device=DEV)
    ws = torch.empty(ds.ds_block_decode_workspace_bytes(shape, kb), dtype=torch.uint8, device=DEV)
    stream = torch.cuda.Stream()

    def step():
        ds.ds_block_compress(shape, g.label, g.page_table, g.seq_lens, bk, stream=stream)
        ds.ds_sparse_decode_blocks(shape, g.q, g.qp, bk, g.k_cache, g.v_cache, None, None, g.page_table,
                                   g.seq_lens, kb, blocks, out, lse, ws, stream=stream)

    with torch.cuda.stream(stream):
        step()                       # warm-up outside the capture (sets kernel attributes)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        step()
    for src in (a, b_, a):
        for name in ("q", "qp", "label", "k_cache", "v_cache", "page_table"):
            getattr(g, name).copy_(getattr(src, name).to(DEV))
        graph.replay()
        torch.cuda.synchronize()
        bkr = oracle.block_compress(src.label, src.page_table, src.seq_lens, src.num_pages)
        assert torch.equal(bk.cpu().view(torch.int16), bkr.view(torch.int16))
        _, rblocks, rout, rlse = _reference(src, bkr, kb)
        assert torch.equal(blocks.cpu(), rblocks)
        assert_close(out, rout, atol_for(wa), "graph replay out")


def test_append_then_last_page_compress_equals_a_full_compress():
    # The maintenance sequence a decoder runs per step: append each request's new token (its index key
    # included), then refresh only the page that changed; the compressed cache must equal a full rebuild.
    ds = _ds()
    w, inp = _inputs("append_blocks", 3, 32, 4, [64 * 9 + 10, 64 * 3, 64 * 20 - 1], 64, "fp8_e4m3", 61)
    g = inp.to(DEV)
    shape = shape_of(inp)
    bk = torch.zeros((inp.num_pages, 64), dtype=torch.bfloat16, device=DEV)
    ds.ds_block_compress(shape, g.label, g.page_table, g.seq_lens, bk)
    pos = torch.tensor([64 * 9 + 10, 64 * 3 - 1, 64 * 20 - 1], dtype=torch.int32)   # next token, last token, last
    k_new = dsgen.normal((w.batch, w.num_kv_heads, 128), 61, 101)
    v_new = dsgen.normal((w.batch, w.num_kv_heads, 128), 61, 102)
    ikey = dsgen.uniform_int((w.batch, 64), -2, 2, 61, 103)
    ds.ds_cache_append(shape, k_new.to(DEV), v_new.to(DEV), g.k_cache, g.v_cache, g.k_scale, g.v_scale,
                       g.page_table, pos.to(DEV), label=g.label, index_key=ikey.to(DEV))
    seq = torch.maximum(inp.seq_lens, pos + 1).to(torch.int32)
    g.seq_lens.copy_(seq.to(DEV))
    ds.ds_block_compress(shape, g.label, g.page_table, g.seq_lens, bk, last_page_only=True)
    full = torch.zeros_like(bk)
    ds.ds_block_compress(shape, g.label, g.page_table, g.seq_lens, full)
    torch.cuda.synchronize()
    assert torch.equal(bk.view(torch.int16), full.view(torch.int16))
    ref = oracle.block_compress(g.label.cpu(), inp.page_table, seq, inp.num_pages)
    assert torch.equal(bk.cpu().view(torch.int16), ref.view(torch.int16))


def test_block_decode_with_no_kept_blocks_is_an_empty_attention():
    w, inp = _inputs("kb0", 2, 8, 2, [64 * 4, 64 * 2], 32, "bf16", 71, key_range=2)
    bk = oracle.block_compress(inp.label, inp.page_table, inp.seq_lens, inp.num_pages)
    blocks, out, lse = _decode_blocks(inp, bk, 0)
    assert blocks.numel() == 0
    assert (out.float() == 0).all() and torch.isinf(lse).all() and (lse < 0).all()
