"""The seeded input generator (``dsgen``) does what its recipe says.

Both the library's tests and the oracle's draw their inputs here, so the
recipe is checked on its own: the counter-based hash written with int64 torch
ops equals the same hash in exact integer arithmetic, any chunk of a stream
can be drawn on its own, the value ranges and distributions are the stated
ones, the FP8 pages hold e4m3 codes of x / scale (never the NaN code), and the
page tables place every page of every request exactly once.
"""
import math

import pytest
import torch

import dsgen

P = dsgen.PAGE_SIZE


def test_tensor_hash_equals_the_integer_hash():
    xs = [0, 1, 2, 0x7FFFFFFF, 0x80000000, 0xFFFFFFFE, 0xFFFFFFFF, 0x12345678, 0x9E3779B9]
    xs += dsgen.hash_u32(dsgen.stream_key(3, 4), 0, 2000, "cpu").tolist()
    got = dsgen._fmix32(torch.tensor(xs, dtype=torch.int64)).tolist()
    assert got == [dsgen._fmix32_int(x) for x in xs]
    assert all(0 <= v <= 0xFFFFFFFF for v in got)


def test_streams_are_deterministic_chunkable_and_distinct():
    key = dsgen.stream_key(11, 5)
    whole = dsgen.hash_u32(key, 0, 10000, "cpu")
    assert torch.equal(whole, dsgen.hash_u32(key, 0, 10000, "cpu"))
    assert torch.equal(whole[3000:7000], dsgen.hash_u32(key, 3000, 4000, "cpu"))
    # counters past 2^32 use the high word
    far = dsgen.hash_u32(key, (1 << 32) - 5, 10, "cpu")
    assert torch.equal(far[:5], dsgen.hash_u32(key, (1 << 32) - 5, 5, "cpu"))
    assert not torch.equal(far[5:], dsgen.hash_u32(key, 0, 5, "cpu"))
    other = dsgen.hash_u32(dsgen.stream_key(11, 6), 0, 10000, "cpu")
    assert (whole == other).float().mean() < 1e-3
    assert dsgen.stream_key(11, 5) != dsgen.stream_key(12, 5)


def test_uniform_integers_cover_their_range_evenly():
    x = dsgen.uniform_int((170000,), -8, 8, 7, 1, dtype=torch.int32)
    assert int(x.min()) == -8 and int(x.max()) == 8
    counts = torch.bincount(x + 8, minlength=17).double()
    expect = x.numel() / 17
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 60.0        # 16 degrees of freedom: p < 1e-6 above this


def test_normal_draws_are_standard_and_rounded_to_nearest_bf16():
    x32 = dsgen.normal((400000,), 9, 2, dtype=torch.float32)
    assert abs(float(x32.mean())) < 0.01 and abs(float(x32.std()) - 1.0) < 0.01
    assert float((x32.abs() > 3).double().mean()) == pytest.approx(0.0027, abs=0.0006)
    xb = dsgen.normal((400000,), 9, 2, dtype=torch.bfloat16)
    assert torch.equal(xb, x32.to(torch.bfloat16))
    assert torch.equal(dsgen._normal_at(9, 2, 123456, (1000,), "cpu"), x32[123456:124456])


def test_uniform_floats_and_permutations():
    s = dsgen.uniform_float((50000,), 0.25, 4.0, 3, 7)
    assert float(s.min()) >= 0.25 and float(s.max()) <= 4.0 and abs(float(s.mean()) - 2.125) < 0.02
    p = dsgen.permutation(1000, 3, 8)
    assert sorted(p.tolist()) == list(range(1000)) and p.tolist() != list(range(1000))
    assert torch.equal(p, dsgen.permutation(1000, 3, 8))


def _small(kind):
    if kind == "ds":
        return dsgen.WORKLOADS[1].scaled(seq_lens=[700, 64, 1], name="ds_small")
    return dsgen.WORKLOADS[3].scaled(batch=3, seq_lens=[700, 64, 129], name="qsa_small")


@pytest.mark.parametrize("kind", ["ds", "qsa"])
def test_decode_inputs_follow_the_recipe(kind):
    w = _small(kind)
    inp = dsgen.make_inputs(w)
    B, Hq, Hkv, D, C, HL = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim, w.proxy_dim, w.label_heads
    slots = inp.num_pages * P
    assert inp.q.shape == (B, Hq, D) and inp.qp.shape == (B, Hq, C) and inp.label.shape == (slots, HL, C)
    assert inp.k_cache.shape == (slots, Hkv, D) and inp.v_cache.shape == (slots, Hkv, D)
    # integer-valued queries in [-4, 4] and labels in [-8, 8]
    for t, lim in ((inp.q, 4), (inp.qp, 4), (inp.label, 8)):
        v = t.double()
        assert torch.equal(v, v.round()) and float(v.abs().max()) == lim
    if w.proxy_from_query:
        # the proxy query is q at C distinct heavy channels, the same for the query heads of one KV head
        for b in range(B):
            for h in range(Hq):
                row = inp.q[b, h].tolist()
                assert all(x in row for x in inp.qp[b, h].tolist())
    # page table: each request's ceil(T/64) pages, every physical page exactly once, -1 after
    counts = [-(-T // P) for T in w.seq_lens]
    used = []
    for b, c in enumerate(counts):
        used += inp.page_table[b, :c].tolist()
        assert (inp.page_table[b, c:] == -1).all()
    assert sorted(used) == list(range(inp.num_pages)) and inp.num_pages == sum(counts)
    assert used != sorted(used) or not w.shuffle_pages
    if w.kv_dtype == "fp8_e4m3":
        for cache, scale in ((inp.k_cache, inp.k_scale), (inp.v_cache, inp.v_scale)):
            assert cache.dtype == torch.uint8
            assert not ((cache & 0x7F) == 0x7F).any()          # never the NaN code
            assert float(scale.min()) >= 0.25 and float(scale.max()) <= 4.0
        # K bytes are e4m3(x / scale[page]) of the K stream's normal draws
        x = dsgen._normal_at(w.seed, 5, 0, (slots, Hkv, D), "cpu")
        sc = inp.k_scale.repeat_interleave(P).view(-1, 1, 1)
        want = torch.clamp(x / sc, -448, 448).to(torch.float8_e4m3fn).view(torch.uint8)
        assert torch.equal(inp.k_cache, want)
        dec = inp.k_cache.view(torch.float8_e4m3fn).double() * sc.double()
        small = (x / sc).abs() >= 2.0 ** -6                # normal e4m3 range: 3 mantissa bits
        rel = ((dec - x.double()) / x.double()).abs()[small]
        assert float(rel.max()) <= 2.0 ** -4 + 1e-6
    else:
        assert inp.k_cache.dtype == torch.bfloat16 and inp.k_scale is None
        assert abs(float(inp.k_cache.double().mean())) < 0.02 and abs(float(inp.k_cache.double().std()) - 1) < 0.02


def test_workload_shapes_are_the_pages_workloads():
    # "Support double sparsity", "Speedup Evaluation": longchat-7b batch 3 x 20000 tokens, 16 heavy channels,
    # 1024 heavy tokens; Llama-3.1-8B batch 3 x 60000 tokens, 32 K-type channels, 3000 heavy tokens.
    # "QSA HiSparse - SGLang plugin", "Supported versions": FP8 E4M3, page 64, 262,144 tokens, 8 requests;
    # PR #43527 "Performance": 1M-token requests; top_k 2048.
    by = {w.name: w for w in dsgen.WORKLOADS}
    l8 = by["llama8b_ds_b3_h32kv8_t60000_c32_k3000"]
    assert (l8.batch, l8.seq_lens, l8.proxy_dim, l8.top_k, l8.num_q_heads, l8.num_kv_heads) == \
        (3, [60000] * 3, 32, 3000, 32, 8)
    assert l8.seq_lens[0] % P != 0                         # the last page is partial
    lc = by["longchat7b_ds_b3_h32kv32_t20000_c16_k1024"]
    assert (lc.batch, lc.seq_lens, lc.proxy_dim, lc.top_k, lc.num_kv_heads) == (3, [20000] * 3, 16, 1024, 32)
    q8 = by["qsa_b8_h32kv4_t262144_idx64_k2048_fp8"]
    assert (q8.batch, q8.seq_lens[0], q8.kv_dtype, q8.page_size, q8.top_k, q8.label_heads) == \
        (8, 262144, "fp8_e4m3", 64, 2048, 1)
    q1 = by["qsa_1m_b1_h32kv4_t1048576_idx64_k2048_fp8"]
    assert (q1.batch, q1.seq_lens[0], q1.top_k) == (1, 1 << 20, 2048) and 4 in q1.splits
    assert [w.seed for w in dsgen.WORKLOADS] == [1000 + i for i in range(len(dsgen.WORKLOADS))]
    assert all(math.log2(w.page_size) == 6 for w in dsgen.WORKLOADS)
