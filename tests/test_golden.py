"""The oracle on small cases worked by hand (tests/golden/*.json).

Each fixture states its inputs, the page sections that define each step, a
derivation of every expected value from those definitions, and the values;
none of them was produced by running code. Tolerances: 1e-12 (the oracle
computes in double; the hand values are rounded to 16 digits).
"""
import json
import math
import os

import torch

import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
P = 64


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def _bf16(x):
    return torch.tensor(x, dtype=torch.float64).to(torch.bfloat16)


def test_tiny_decode_step_by_hand():
    g = _load("tiny_decode_step.json")
    inp, exp = g["inputs"], g["expected"]
    pid, npages, T = inp["physical_page"], inp["num_pages"], inp["seq_len"]
    slots = npages * P
    label = torch.zeros((slots, 1, 2), dtype=torch.bfloat16)
    K = torch.zeros((slots, 1, 4), dtype=torch.bfloat16)
    V = torch.zeros((slots, 1, 4), dtype=torch.bfloat16)
    for t in range(T):
        label[pid * P + t, 0] = _bf16(inp["label"][t])
        K[pid * P + t, 0] = _bf16(inp["K"][t])
        V[pid * P + t, 0] = _bf16(inp["V"][t])
    qp = _bf16([inp["qp"]])
    q = _bf16([inp["q"]])
    pt = torch.tensor([[pid]], dtype=torch.int32)
    sl = torch.tensor([T], dtype=torch.int32)

    s = oracle.index_score(qp, label, pt, sl, 1, T)
    assert s[0, 0].tolist() == exp["scores"]
    idx2 = oracle.topk(s, sl, 2)
    idx1 = oracle.topk(s, sl, 1)
    assert idx2[0, 0].tolist() == exp["topk_k2"] and idx1[0, 0].tolist() == exp["topk_k1"]

    for idx, out_key, lse_key in ((idx2, "out_k2", "lse_k2"), (idx1, "out_k1", "lse_k1")):
        o, l = oracle.sparse_attn(q, K, V, None, None, pt, sl, idx)
        out, lse = oracle.lse_merge(o, l)
        assert torch.allclose(out[0], torch.tensor(exp[out_key], dtype=torch.float64), atol=1e-12, rtol=0)
        assert torch.allclose(lse[0], torch.tensor(exp[lse_key], dtype=torch.float64), atol=1e-12, rtol=0)
    # The hand values themselves: e/(e+1), ln(e+1), ln 2.
    e = math.e
    assert abs(exp["out_k2"][0][0] - e / (e + 1)) < 1e-15 and abs(exp["lse_k2"][0] - math.log(e + 1)) < 1e-15
    # Two splits of the k = 2 list merge to the one-split result.
    o, l = oracle.sparse_attn(q, K, V, None, None, pt, sl, idx2, num_splits=2)
    out, lse = oracle.lse_merge(o, l)
    assert torch.allclose(out[0], torch.tensor(exp["out_k2"], dtype=torch.float64), atol=1e-12, rtol=0)
    assert torch.allclose(lse[0], torch.tensor(exp["lse_k2"], dtype=torch.float64), atol=1e-12, rtol=0)


def test_block_keys_and_selection_by_hand():
    g = _load("block_keys_by_hand.json")
    # Three requests of one page each, pages 0, 1, 2 physical.
    keys = torch.zeros((3 * P, 1, 2), dtype=torch.float64)
    keys[0:32, 0, 0], keys[32:64, 0, 0], keys[0:64, 0, 1] = 1.0, 3.0, 0.5
    keys[P + 0, 0], keys[P + 1, 0], keys[P + 2, 0] = torch.tensor([1.0, 1.0]), torch.tensor([1.0, 1 + 2 ** -7]), \
        torch.tensor([2.0, 1 + 2 ** -7])
    keys[2 * P + 0, 0], keys[2 * P + 1, 0] = torch.tensor([1.0, -1.0]), torch.tensor([1 + 2 ** -7, -(1 + 2 ** -7)])
    pt = torch.tensor([[0], [1], [2]], dtype=torch.int32)
    sl = torch.tensor([c["tokens"] for c in g["key_cases"]], dtype=torch.int32)
    bk = oracle.block_compress(keys.to(torch.bfloat16), pt, sl, 3)
    for p, c in enumerate(g["key_cases"]):
        assert bk[p].double().tolist() == c["expected_key"], p

    # One request of three full pages with constant keys; group query [1, 1] from two heads.
    sel = g["selection_case"]
    consts = [[2.0, 0.5], [1.3359375, 1.0078125], [0.0, 0.0]]
    keys2 = torch.zeros((3 * P, 1, 2), dtype=torch.float64)
    for p, c in enumerate(consts):
        keys2[p * P:(p + 1) * P, 0] = torch.tensor(c)
    pt2 = torch.tensor([[0, 1, 2]], dtype=torch.int32)
    sl2 = torch.tensor([3 * P], dtype=torch.int32)
    bk2 = oracle.block_compress(keys2.to(torch.bfloat16), pt2, sl2, 3)
    assert bk2.double().tolist() == consts
    qp = _bf16([[[1, 0], [0, 1]]])
    assert qp[0].double().sum(0).tolist() == sel["group_query"]
    s = oracle.block_score(qp, bk2, pt2, sl2, 1)
    assert s[0, 0].tolist() == g["expected_scores"]
    top = oracle.topk(s, torch.tensor([3], dtype=torch.int32), sel["kb"])
    assert top[0, 0].tolist() == g["expected_top2"]
    toks = oracle.block_expand(top, sl2)[0, 0]
    valid = toks[toks >= 0]
    want = g["expected_tokens_top2"]
    assert valid.numel() == want["count"] and int(valid[0]) == want["first"] and int(valid[-1]) == want["last"]
    assert torch.equal(valid, torch.arange(want["count"], dtype=torch.int32))
