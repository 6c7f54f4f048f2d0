"""Pins of the oracle against what the pages and the mathematics fix.

None of these tests compares the oracle with a retyped copy of itself. Each
one checks it against a library routine on a special case (torch matmul and
scaled_dot_product_attention, torch's bf16 / e4m3 conversions), a closed form,
an invariant the definition implies (GQA decomposition, page relocation,
split/unsplit equality), or brute force on tiny inputs.
"""
import math

import pytest
import torch
import torch.nn.functional as F

import dsgen
import oracle

P = 64


# ---------------------------------------------------------------- decoders

def test_bf16_decoder_matches_torch_on_every_code():
    bits = torch.arange(0, 1 << 16, dtype=torch.int32).to(torch.int16)
    ref = bits.view(torch.bfloat16).double()
    got = torch.tensor([oracle.bf16_value(int(b) & 0xFFFF) for b in bits.tolist()], dtype=torch.float64)
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan], ref[~nan])


def test_e4m3_decoder_matches_torch_on_every_code():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).double()
    got = torch.tensor([oracle.e4m3_value(c) for c in range(256)], dtype=torch.float64)
    nan = torch.isnan(ref)
    assert nan.sum() == 2                      # S.1111.111 only: the format has no infinities
    assert torch.equal(torch.isnan(got), nan)
    assert torch.equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9 and got[0x80] == 0.0


def test_e4m3_encoder_matches_torch_rounding_within_range():
    # Every code's value, every midpoint between neighbouring codes (the
    # ties), and random values across the range including subnormals.
    vals = sorted({oracle.e4m3_value(c) for c in range(0x7F)})
    mids = [(a + b) / 2 for a, b in zip(vals, vals[1:])]
    rnd = (dsgen.normal((4000,), 5, 1, dtype=torch.float32) * 60).clamp(-448, 448).tolist()
    tiny = (dsgen.normal((1000,), 5, 2, dtype=torch.float32) * 2.0 ** -8).tolist()
    xs = torch.tensor(vals + mids + [-v for v in vals + mids] + rnd + tiny, dtype=torch.float32)
    ref = xs.to(torch.float8_e4m3fn).view(torch.uint8)
    got = torch.tensor([oracle.e4m3_encode(float(x)) for x in xs.tolist()], dtype=torch.uint8)
    assert torch.equal(got, ref)


def test_e4m3_encoder_saturates_and_keeps_sign_zero_and_nan():
    assert oracle.e4m3_encode(448.0) == 0x7E and oracle.e4m3_encode(449.0) == 0x7E
    assert oracle.e4m3_encode(1e30) == 0x7E and oracle.e4m3_encode(-1e30) == 0xFE
    assert oracle.e4m3_encode(0.0) == 0x00 and oracle.e4m3_encode(-0.0) == 0x80
    assert oracle.e4m3_encode(float("nan")) == 0x7F
    for c in range(256):                        # every finite code round-trips
        v = oracle.e4m3_value(c)
        if not math.isnan(v):
            assert oracle.e4m3_encode(v) == c, c


# ---------------------------------------------------------------- cache append

def _append_case(kv_fp8: bool, per_head: bool, seed: int):
    B, Hkv, D, C = 3, 2, 128, 16
    pages_per_req = 3
    pt, num_pages = _shuffled_table(B, pages_per_req, seed)
    k_new = dsgen.normal((B, Hkv, D), seed, 1, dtype=torch.bfloat16)
    v_new = dsgen.normal((B, Hkv, D), seed, 2, dtype=torch.bfloat16)
    slots = num_pages * P
    if kv_fp8:
        kc = dsgen.uniform_int((slots, Hkv, D), 0, 126, seed, 3, dtype=torch.int32).to(torch.uint8)
        vc = dsgen.uniform_int((slots, Hkv, D), 0, 126, seed, 4, dtype=torch.int32).to(torch.uint8)
        ks = dsgen.uniform_float((num_pages,), 0.25, 4.0, seed, 5)
        vs = dsgen.uniform_float((num_pages,), 0.25, 4.0, seed, 6)
    else:
        kc = dsgen.normal((slots, Hkv, D), seed, 3, dtype=torch.bfloat16)
        vc = dsgen.normal((slots, Hkv, D), seed, 4, dtype=torch.bfloat16)
        ks = vs = None
    HL = Hkv if per_head else 1
    label = dsgen.normal((slots, HL, C), seed, 7, dtype=torch.bfloat16)
    channels = dsgen.uniform_int((Hkv, C), 0, D - 1, seed, 8, dtype=torch.int32) if per_head else None
    index_key = None if per_head else dsgen.normal((B, C), seed, 9, dtype=torch.bfloat16)
    positions = torch.tensor([63, 64, -1], dtype=torch.int32)        # last slot of a page, first of the next, skipped
    return dict(k_new=k_new, v_new=v_new, kc=kc, vc=vc, ks=ks, vs=vs, pt=pt, positions=positions, label=label,
                channels=channels, index_key=index_key)


@pytest.mark.parametrize("kv_fp8", [False, True])
@pytest.mark.parametrize("per_head", [True, False])
def test_cache_append_writes_the_slot_and_gathers_the_label(kv_fp8, per_head):
    c = _append_case(kv_fp8, per_head, 40 + 2 * kv_fp8 + per_head)
    kc, vc, lb = oracle.cache_append(c["k_new"], c["v_new"], c["kc"], c["vc"], c["ks"], c["vs"], c["pt"],
                                     c["positions"], c["label"], channels=c["channels"], index_key=c["index_key"])
    touched = set()
    for b in range(c["k_new"].shape[0]):
        t = int(c["positions"][b])
        if t < 0:
            continue
        page = int(c["pt"][b, t // P])
        slot = page * P + t % P
        touched.add(slot)
        if kv_fp8:
            # torch's own float -> e4m3 conversion of the fp32 quotient (|x / scale| < 448 here)
            kq = (c["k_new"][b].float() / c["ks"][page]).to(torch.float8_e4m3fn).view(torch.uint8)
            vq = (c["v_new"][b].float() / c["vs"][page]).to(torch.float8_e4m3fn).view(torch.uint8)
            assert torch.equal(kc[slot], kq) and torch.equal(vc[slot], vq)
        else:
            assert torch.equal(kc[slot], c["k_new"][b]) and torch.equal(vc[slot], c["v_new"][b])
        if per_head:
            ref = torch.gather(c["k_new"][b], 1, c["channels"].long())
            assert torch.equal(lb[slot], ref)
        else:
            assert torch.equal(lb[slot, 0], c["index_key"][b])
    others = torch.tensor([s for s in range(kc.shape[0]) if s not in touched])
    assert torch.equal(kc[others].view(torch.uint8), c["kc"][others].view(torch.uint8))
    assert torch.equal(lb[others].view(torch.int16), c["label"][others].view(torch.int16))


# ---------------------------------------------------------------- helpers

def _paged(dense: torch.Tensor, page_table: torch.Tensor, num_pages: int) -> torch.Tensor:
    """Scatter per-request rows dense[b, t, ...] into a page pool via the page table."""
    B, T = dense.shape[:2]
    pool = torch.zeros((num_pages * P,) + tuple(dense.shape[2:]), dtype=dense.dtype)
    for b in range(B):
        for t in range(T):
            pool[int(page_table[b, t // P]) * P + t % P] = dense[b, t]
    return pool


def _shuffled_table(B, pages_per_req, seed):
    total = B * pages_per_req
    perm = dsgen.permutation(total, seed, 7)
    return perm.view(B, pages_per_req).clone(), total


def _ints(shape, lo, hi, seed, tid):
    return dsgen.uniform_int(shape, lo, hi, seed, tid)


# ---------------------------------------------------------------- stage 1: scores

def test_score_is_matmul_when_label_is_the_key_and_group_is_one():
    # With G = 1 and C = D, the label row of head g is K itself and qp is q:
    # the proxy score is the plain dot product q . K_t, i.e. a matmul.
    B, H, C, T = 2, 3, 16, 150
    pt, npages = _shuffled_table(B, 3, 11)
    dense = _ints((B, T, H, C), -8, 8, 11, 1)
    label = _paged(dense, pt, npages)
    qp = _ints((B, H, C), -4, 4, 11, 2)
    seq = torch.tensor([150, 97], dtype=torch.int32)
    s = oracle.index_score(qp, label, pt, seq, H, T)
    for b in range(B):
        Tb = int(seq[b])
        ref = torch.matmul(dense[b, :Tb].double().permute(1, 0, 2), qp[b].double().unsqueeze(-1)).squeeze(-1)
        assert torch.equal(s[b, :, :Tb].double(), ref)
        assert torch.isnan(s[b, :, Tb:]).all()     # nothing written past the length


def test_score_group_is_the_sum_of_its_query_heads():
    # Contiguous GQA grouping: KV head g scores with query heads g*G .. g*G+G-1.
    B, Hq, Hkv, C, T = 1, 8, 2, 32, 130
    G = Hq // Hkv
    pt, npages = _shuffled_table(B, 3, 12)
    label = _ints((npages * P, Hkv, C), -8, 8, 12, 1)
    qp = _ints((B, Hq, C), -4, 4, 12, 2)
    seq = torch.tensor([T], dtype=torch.int32)
    grouped = oracle.index_score(qp, label, pt, seq, Hkv, T)
    per_head = oracle.index_score(qp, label.repeat_interleave(G, dim=1), pt, seq, Hq, T)
    ref = per_head.view(B, Hkv, G, T).double().sum(2)
    assert torch.equal(grouped.double(), ref)


def test_shared_index_key_equals_a_replicated_per_head_label():
    B, Hq, Hkv, C, T = 2, 8, 4, 64, 100
    pt, npages = _shuffled_table(B, 2, 13)
    keys = _ints((npages * P, 1, C), -8, 8, 13, 1)
    qp = _ints((B, Hq, C), -4, 4, 13, 2)
    seq = torch.tensor([100, 65], dtype=torch.int32)
    shared = oracle.index_score(qp, keys, pt, seq, Hkv, T)
    repl = oracle.index_score(qp, keys.expand(-1, Hkv, -1).contiguous(), pt, seq, Hkv, T)
    assert torch.equal(torch.nan_to_num(shared, 7.5), torch.nan_to_num(repl, 7.5))


def test_score_does_not_depend_on_where_pages_live():
    B, Hq, Hkv, C, T = 2, 4, 2, 16, 200
    pt, npages = _shuffled_table(B, 4, 14)
    dense = _ints((B, T, Hkv, C), -8, 8, 14, 1)
    qp = _ints((B, Hq, C), -4, 4, 14, 2)
    seq = torch.tensor([200, 129], dtype=torch.int32)
    a = oracle.index_score(qp, _paged(dense, pt, npages), pt, seq, Hkv, T)
    pt2 = pt.flip(1).roll(1, 0).contiguous()        # another placement of the same pages
    b = oracle.index_score(qp, _paged(dense, pt2, npages), pt2, seq, Hkv, T)
    assert torch.equal(torch.nan_to_num(a, 7.5), torch.nan_to_num(b, 7.5))


def test_score_worked_example_by_hand():
    # One request, one KV head of two query heads, C = 2, pages of 64 with the
    # request's single page stored at physical page 1. Token 0 has label
    # (1, 2), token 1 has (-3, 4); queries (1, 1) and (2, -1) sum to (3, 0):
    # scores 3*1 + 0*2 = 3 and 3*(-3) + 0*4 = -9.
    label = torch.zeros((2 * P, 1, 2), dtype=torch.bfloat16)
    label[P + 0, 0] = torch.tensor([1.0, 2.0])
    label[P + 1, 0] = torch.tensor([-3.0, 4.0])
    qp = torch.tensor([[[1.0, 1.0], [2.0, -1.0]]], dtype=torch.bfloat16)
    pt = torch.tensor([[1]], dtype=torch.int32)
    s = oracle.index_score(qp, label, pt, torch.tensor([2], dtype=torch.int32), 1, 2)
    assert s[0, 0].tolist() == [3.0, -9.0]


# ---------------------------------------------------------------- stage 2: top-k

def _brute_topk(s, T, k):
    keyed = sorted(range(T), key=lambda t: (-s[t], t))
    return sorted(keyed[:min(k, T)]) + [-1] * (k - min(k, T))


@pytest.mark.parametrize("T,k,lo,hi", [(1, 1, -2, 2), (17, 5, -2, 2), (64, 64, -1, 1), (100, 7, 0, 0),
                                       (250, 40, -3, 3), (33, 50, -5, 5), (513, 128, -50, 50)])
def test_topk_equals_brute_force_sort(T, k, lo, hi):
    B, H = 2, 3
    s = _ints((B, H, T), lo, hi, T * 31 + k, 1).float()
    seq = torch.tensor([T, max(0, T - 9)], dtype=torch.int32)
    idx = oracle.topk(s, seq, k)
    for b in range(B):
        for g in range(H):
            assert idx[b, g].tolist() == _brute_topk(s[b, g].tolist(), int(seq[b]), k)


@pytest.mark.parametrize("S", [1, 2, 3, 4, 16])
def test_sharded_topk_equals_the_unsharded_topk(S):
    # The page's claim for its distributed selection: shard-local top-k plus
    # a merge with token-id tie-breaking gives the unsharded result. Integer
    # scores with many ties, ragged lengths, k above and below a shard's size.
    s = dsgen.uniform_int((2, 3, 1500), -6, 6, 17, S, dtype=torch.float32)
    s[1, 2, ::5] = float("nan")
    seq = torch.tensor([1500, 611], dtype=torch.int32)
    for k in (1, 64, 130, 700, 1499, 2000):
        assert torch.equal(oracle.topk_sharded(s, seq, k, S), oracle.topk(s, seq, k)), (S, k)


def test_topk_all_ties_take_the_lowest_indices():
    s = torch.full((1, 1, 1000), 3.0)
    idx = oracle.topk(s, torch.tensor([1000], dtype=torch.int32), 10)
    assert idx[0, 0].tolist() == list(range(10))


def test_topk_negative_zero_ties_with_zero():
    s = torch.tensor([[[-0.0, 0.0, -0.0, 1.0, -1.0]]])
    idx = oracle.topk(s, torch.tensor([5], dtype=torch.int32), 3)
    assert idx[0, 0].tolist() == [0, 1, 3]


def test_topk_nan_ranks_last_and_empty_rows_pad():
    s = torch.tensor([[[float("nan"), -100.0, float("nan"), 5.0]]])
    assert oracle.topk(s, torch.tensor([4], dtype=torch.int32), 3)[0, 0].tolist() == [0, 1, 3]
    assert oracle.topk(s, torch.tensor([0], dtype=torch.int32), 3)[0, 0].tolist() == [-1, -1, -1]
    assert oracle.topk(s, torch.tensor([4], dtype=torch.int32), 0).shape == (1, 1, 0)


# ---------------------------------------------------------------- stage 3: attention

def _dequant(inp, cache, scale):
    if cache.dtype == torch.uint8:
        vals = cache.view(torch.float8_e4m3fn).double()
        return vals * scale.double().repeat_interleave(P).view(-1, 1, 1)
    return cache.double()


def _sdpa_rows(q_bh, K_rows, V_rows, scale):
    """Library attention of one query over given rows, with its lse."""
    o = F.scaled_dot_product_attention(q_bh.view(1, 1, 1, -1), K_rows.unsqueeze(0).unsqueeze(0),
                                       V_rows.unsqueeze(0).unsqueeze(0), scale=scale).view(-1)
    lse = torch.logsumexp(scale * (K_rows @ q_bh), 0)
    return o, lse


def _small_workload(kv_dtype, B=2, Hq=8, Hkv=2, T=(300, 131), C=16, HL=None, k=40, shuffle=True):
    return dsgen.Workload(name="pin", batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=32,
                          seq_lens=list(T), proxy_dim=C, label_heads=Hkv if HL is None else HL,
                          top_k=k, kv_dtype=kv_dtype, shuffle_pages=shuffle, seed=77,
                          proxy_from_query=False)


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_attention_with_k_at_least_T_is_dense_softmax_attention(kv_dtype):
    w = _small_workload(kv_dtype)
    inp = dsgen.make_inputs(w)
    k = w.max_seq_len + 5
    _, idx, out, lse = oracle.decode(inp, k=k)
    Kd = _dequant(inp, inp.k_cache, inp.k_scale)
    Vd = _dequant(inp, inp.v_cache, inp.v_scale)
    scale = 1.0 / math.sqrt(w.head_dim)
    for b in range(w.batch):
        Tb = w.seq_lens[b]
        assert idx[b, :, :Tb].tolist() == [list(range(Tb))] * w.num_kv_heads
        slots = inp.page_table[b, torch.arange(Tb) // P].long() * P + torch.arange(Tb) % P
        for h in range(w.num_q_heads):
            g = h // w.group
            o_ref, lse_ref = _sdpa_rows(inp.q[b, h].double(), Kd[slots, g], Vd[slots, g], scale)
            assert torch.allclose(out[b, h], o_ref, rtol=0, atol=1e-12)
            assert abs(float(lse[b, h]) - float(lse_ref)) < 1e-12


@pytest.mark.parametrize("kv_dtype", ["bf16", "fp8_e4m3"])
def test_sparse_attention_equals_library_attention_over_the_selected_rows(kv_dtype):
    w = _small_workload(kv_dtype)
    inp = dsgen.make_inputs(w)
    _, idx, out, lse = oracle.decode(inp)
    Kd = _dequant(inp, inp.k_cache, inp.k_scale)
    Vd = _dequant(inp, inp.v_cache, inp.v_scale)
    scale = 1.0 / math.sqrt(w.head_dim)
    for b in range(w.batch):
        for h in range(w.num_q_heads):
            g = h // w.group
            sel = idx[b, g][idx[b, g] >= 0].long()
            assert len(sel) == min(w.top_k, w.seq_lens[b])
            slots = inp.page_table[b, sel // P].long() * P + sel % P
            o_ref, lse_ref = _sdpa_rows(inp.q[b, h].double(), Kd[slots, g], Vd[slots, g], scale)
            assert torch.allclose(out[b, h], o_ref, rtol=0, atol=1e-12)
            assert abs(float(lse[b, h]) - float(lse_ref)) < 1e-12


def test_single_selected_token_returns_its_value_row():
    w = _small_workload("bf16", k=1)
    inp = dsgen.make_inputs(w)
    _, idx, out, _ = oracle.decode(inp)
    for b in range(w.batch):
        for h in range(w.num_q_heads):
            t = int(idx[b, h // w.group, 0])
            slot = int(inp.page_table[b, t // P]) * P + t % P
            assert torch.equal(out[b, h], inp.v_cache[slot, h // w.group].double())


def test_empty_rows_give_zero_output_and_minus_infinity_lse():
    w = _small_workload("bf16", T=(0, 70))
    inp = dsgen.make_inputs(w)
    _, idx, out, lse = oracle.decode(inp)
    assert (idx[0] == -1).all()
    assert torch.equal(out[0], torch.zeros_like(out[0]))
    assert torch.isinf(lse[0]).all() and (lse[0] < 0).all()
    _, _, out0, lse0 = oracle.decode(inp, k=0)
    assert torch.equal(out0, torch.zeros_like(out0)) and torch.isinf(lse0).all()


# ---------------------------------------------------------------- stage 4: merge

@pytest.mark.parametrize("S", [2, 3, 4, 16, 64])
@pytest.mark.parametrize("split_mode", [0, 1])
def test_merge_of_any_split_equals_the_unsplit_result(S, split_mode):
    w = _small_workload("fp8_e4m3", T=(700, 45), k=90)
    inp = dsgen.make_inputs(w)
    _, idx, out1, lse1 = oracle.decode(inp)
    o, l = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                              inp.page_table, inp.seq_lens, idx, None, S, split_mode)
    if S > 45:
        assert torch.isinf(l[:, 1]).any()               # some chunks of the short request are empty
    out, lse = oracle.lse_merge(o, l)
    assert torch.allclose(out, out1, rtol=0, atol=1e-12)
    assert torch.allclose(lse, lse1, rtol=0, atol=1e-12)


@pytest.mark.parametrize("S,split_mode", [(3, 0), (7, 0), (4, 1), (5, 1)])
def test_each_split_chunk_is_attention_over_its_own_tokens(S, split_mode):
    # Reading R6 fixes which selected tokens each chunk holds: contiguous
    # splitting gives chunk j the positions [j n / S, (j + 1) n / S) of the n
    # selected tokens, page-interleaved splitting the tokens whose logical page
    # is j mod S. Each chunk's partial must be library attention over exactly
    # those tokens, and a chunk without tokens has o = 0 and lse = -inf. (The
    # merge test above cannot see a wrong assignment: any partition merges to
    # the same result.)
    w = _small_workload("bf16", T=(700, 45), k=90)
    inp = dsgen.make_inputs(w)
    _, idx, _, _ = oracle.decode(inp)
    o, l = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                              inp.page_table, inp.seq_lens, idx, None, S, split_mode)
    Kd = _dequant(inp, inp.k_cache, inp.k_scale)
    Vd = _dequant(inp, inp.v_cache, inp.v_scale)
    scale = 1.0 / math.sqrt(w.head_dim)
    empty = 0
    for b in range(w.batch):
        for h in range(w.num_q_heads):
            g = h // w.group
            sel = idx[b, g][idx[b, g] >= 0].long()
            n = len(sel)
            for j in range(S):
                mine = sel[j * n // S:(j + 1) * n // S] if split_mode == 0 else sel[(sel // P) % S == j]
                if len(mine) == 0:
                    empty += 1
                    assert torch.equal(o[j, b, h], torch.zeros_like(o[j, b, h]))
                    assert math.isinf(float(l[j, b, h])) and float(l[j, b, h]) < 0
                    continue
                slots = inp.page_table[b, mine // P].long() * P + mine % P
                o_ref, lse_ref = _sdpa_rows(inp.q[b, h].double(), Kd[slots, g], Vd[slots, g], scale)
                assert torch.allclose(o[j, b, h], o_ref, rtol=0, atol=1e-12), (b, h, j)
                assert abs(float(l[j, b, h]) - float(lse_ref)) < 1e-12, (b, h, j)
    if split_mode == 1:
        assert empty > 0          # the 45-token request has one page: every other chunk is empty


def test_merge_closed_form_two_partials():
    # lse_1 = 0, lse_2 = ln 3: total lse = ln 4, weights 1/4 and 3/4.
    o = torch.tensor([[[1.0, 0.0]], [[0.0, 2.0]]], dtype=torch.float64)
    l = torch.tensor([[0.0], [math.log(3.0)]], dtype=torch.float64)
    out, lse = oracle.lse_merge(o, l)
    assert torch.allclose(out, torch.tensor([[0.25, 1.5]], dtype=torch.float64), atol=1e-15)
    assert abs(float(lse[0]) - math.log(4.0)) < 1e-15


def test_merge_single_split_is_identity_and_all_empty_is_empty():
    o = torch.randn(1, 5, 8, dtype=torch.float64)
    l = torch.randn(1, 5, dtype=torch.float64)
    out, lse = oracle.lse_merge(o, l)
    assert torch.allclose(out, o[0], atol=1e-15) and torch.allclose(lse, l[0], atol=1e-15)
    out, lse = oracle.lse_merge(torch.zeros(3, 2, 4, dtype=torch.float64),
                                torch.full((3, 2), -math.inf, dtype=torch.float64))
    assert torch.equal(out, torch.zeros(2, 4, dtype=torch.float64)) and torch.isinf(lse).all()


# ---------------------------------------------------------------- block-compressed selection (f3)

def _nearest_bf16_exact(x):
    """Nearest bfloat16 to the rational x, ties to the even code, by exact comparison of its two neighbours."""
    from fractions import Fraction
    import struct
    if x == 0:
        return 0
    f = float(x)                                   # within a float ulp of x
    bits = struct.unpack("<I", struct.pack("<f", f))[0] >> 16
    cands = []
    for d in (-2, -1, 0, 1, 2):
        c = (bits + d) & 0xFFFF
        v = struct.unpack("<f", struct.pack("<I", c << 16))[0]
        if math.isfinite(v) and (v > 0) == (x > 0):
            cands.append((abs(Fraction(v) - x), c & 1, c))
    cands.sort()
    best = [c for c in cands if c[0] == cands[0][0]]
    return min(best, key=lambda c: c[1])[2]        # a tie goes to the even significand


def _block_case(seed, B=2, T=(200, 64 * 3), C=16, scale=1.0):
    P_ = (max(T) + P - 1) // P
    pt = torch.stack([dsgen.permutation(P_ * B, seed, 50)[b * P_:(b + 1) * P_] for b in range(B)]).to(torch.int32)
    keys = (dsgen.normal((P_ * B * P, 1, C), seed, 51, dtype=torch.float32) * scale).to(torch.bfloat16)
    return keys, pt, torch.tensor(T, dtype=torch.int32), P_ * B


def test_block_keys_are_the_exactly_rounded_means_of_their_tokens():
    from fractions import Fraction
    keys, pt, sl, npages = _block_case(3)
    bk = oracle.block_compress(keys, pt, sl, npages)
    kb = keys.view(torch.int16)
    for b in range(pt.shape[0]):
        T = int(sl[b])
        for j in range((T + P - 1) // P):
            pid = int(pt[b, j])
            toks = range(j * P, min(T, j * P + P))
            for c in range(keys.shape[-1]):
                mean = sum(Fraction(float(keys[pid * P + t % P, 0, c])) for t in toks) / len(toks)
                assert int(bk[pid, c].view(torch.int16)) & 0xFFFF == _nearest_bf16_exact(mean), (b, j, c)


def test_block_key_rounding_ties_go_to_the_even_code():
    # Pages holding two tokens: the means 1 + 2^-8 and 1 + 3 * 2^-8 lie halfway between neighbouring bfloat16
    # values; the even significands are 1.0 and 1 + 2^-6.
    keys = torch.zeros((2 * P, 1, 2), dtype=torch.bfloat16)
    keys[0, 0, 0], keys[1, 0, 0] = 1.0, 1.0 + 2 ** -7
    keys[0, 0, 1], keys[1, 0, 1] = 1.0 + 2 ** -7, 1.0 + 2 ** -6
    keys[P, 0, 0], keys[P + 1, 0, 0] = -1.0, -(1.0 + 2 ** -7)
    pt = torch.tensor([[0], [1]], dtype=torch.int32)
    bk = oracle.block_compress(keys, pt, torch.tensor([2, 2], dtype=torch.int32), 2).float()
    assert bk[0, 0] == 1.0 and bk[0, 1] == 1.0 + 2 ** -6 and bk[1, 0] == -1.0


def test_block_key_of_a_constant_page_is_that_key():
    keys = torch.zeros((3 * P, 1, 4), dtype=torch.bfloat16)
    keys[:P] = 0.3
    keys[P:2 * P] = -7.5
    keys[2 * P:] = 1e-30
    pt = torch.tensor([[2, 0, 1]], dtype=torch.int32)   # logical pages 0, 1, 2 -> physical 2, 0, 1 (5 tokens in 2)
    bk = oracle.block_compress(keys, pt, torch.tensor([2 * P + 5], dtype=torch.int32), 3)
    assert torch.equal(bk[0], keys[0, 0]) and torch.equal(bk[1], keys[P, 0]) and torch.equal(bk[2], keys[2 * P, 0])


def test_block_scores_match_a_library_contraction_of_the_block_keys():
    keys, pt, sl, npages = _block_case(5, C=64)
    bk = oracle.block_compress(keys, pt, sl, npages)
    B, Hq, Hkv = 2, 8, 2
    qp = dsgen.normal((B, Hq, 64), 5, 52)
    s = oracle.block_score(qp, bk, pt, sl, Hkv)
    qg = qp.double().view(B, Hkv, Hq // Hkv, 64).sum(2)
    for b in range(B):
        nb = (int(sl[b]) + P - 1) // P
        ref = torch.einsum("gc,jc->gj", qg[b], bk[pt[b, :nb].long()].double()).float()
        assert torch.equal(s[b, :, :nb], ref)
        assert torch.isnan(s[b, :, nb:]).all()


def test_block_expansion_lists_the_kept_blocks_tokens_below_the_length():
    blocks = torch.tensor([[[0, 2, 3, -1]], [[1, -1, -1, -1]]], dtype=torch.int32)
    sl = torch.tensor([3 * P + 10, 64], dtype=torch.int32)
    idx = oracle.block_expand(blocks, sl)
    want0 = list(range(0, P)) + list(range(2 * P, 3 * P)) + list(range(3 * P, 3 * P + 10))
    assert idx[0, 0, :len(want0)].tolist() == want0 and (idx[0, 0, len(want0):] == -1).all()
    assert (idx[1, 0] == -1).all()          # block 1 lies past the 64-token sequence
    all_blocks = torch.arange(4, dtype=torch.int32).view(1, 1, 4)
    assert torch.equal(oracle.block_expand(all_blocks, sl[:1])[0, 0, :3 * P + 10], torch.arange(3 * P + 10, dtype=torch.int32))
