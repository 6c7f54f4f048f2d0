"""GPU parity of the cache-append step (ds_cache_append) against the oracle.

Every byte of the K and V caches and of the label cache must equal the
oracle's after the append: bf16 rows are copied, e4m3 rows are the fp32
quotient by the page scale rounded to nearest even (both sides take that
decision from the same fp32 value), label rows are gathered or copied.
"""
import pytest
import torch

import dsgen
import oracle
from gpu_helpers import assert_close, atol_for, run_decode, shape_of, workload

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


def _new_token(w, seed):
    B, Hkv, D, C = w.batch, w.num_kv_heads, w.head_dim, w.proxy_dim
    k_new = dsgen.normal((B, Hkv, D), seed, 101)
    v_new = dsgen.normal((B, Hkv, D), seed, 102)
    if w.label_heads == 1 and not (w.num_kv_heads == 1 and w.proxy_from_query):
        return k_new, v_new, None, dsgen.normal((B, C), seed, 103)
    # Heavy channels: C distinct channels per KV head.
    ch = torch.stack([dsgen.permutation(D, seed, 104 + g)[:C] for g in range(Hkv)]).to(torch.int32)
    return k_new, v_new, ch, None


def _positions(w, skip_row=None):
    # The next token when the request's last page has room, else its last
    # token again (the generator allocates only the pages a request uses).
    pos = []
    for b, T in enumerate(w.seq_lens):
        t = T if T % w.page_size else T - 1
        pos.append(-1 if b == skip_row else t)
    return torch.tensor(pos, dtype=torch.int32)


APPEND_CASES = [
    # name, B, Hq, Hkv, T, C, HL, kv
    ("ds_bf16_hkv8_c32", 3, 32, 8, [1000, 640, 63], 32, 8, "bf16"),
    ("ds_bf16_hkv32_c16", 2, 32, 32, [700, 1], 16, 32, "bf16"),
    ("ds_bf16_single_kv", 2, 4, 1, [128, 77], 16, 1, "bf16"),
    ("qsa_fp8_hkv4_c64", 4, 32, 4, [2000, 1024, 5, 4095], 64, 1, "fp8_e4m3"),
    ("ds_fp8_hkv2_c32", 2, 8, 2, [300, 257], 32, 2, "fp8_e4m3"),
    ("qsa_fp8_d256", 2, 16, 2, [700, 64], 64, 1, "fp8_e4m3", 256),
    ("ds_bf16_d256", 2, 8, 4, [300, 129], 32, 4, "bf16", 256),
]


@pytest.mark.parametrize("case", APPEND_CASES, ids=[c[0] for c in APPEND_CASES])
def test_cache_append_bit_exact(case):
    name, B, Hq, Hkv, T, C, HL, kv = case[:8]
    D = case[8] if len(case) > 8 else 128
    w = workload(name, B, Hq, Hkv, T, C, HL, 16, kv=kv, seed=77, head_dim=D)
    inp = dsgen.make_inputs(w)
    g = inp.to(DEV)
    k_new, v_new, ch, ikey = _new_token(w, 31)
    pos = _positions(w, skip_row=1 if B > 2 else None)
    ds = _ds()
    ds.ds_cache_append(shape_of(inp), k_new.to(DEV), v_new.to(DEV), g.k_cache, g.v_cache, g.k_scale, g.v_scale,
                       g.page_table, pos.to(DEV), label=g.label,
                       channels=None if ch is None else ch.to(DEV),
                       index_key=None if ikey is None else ikey.to(DEV))
    torch.cuda.synchronize()
    rk, rv, rl = oracle.cache_append(k_new, v_new, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                                     inp.page_table, pos, inp.label, channels=ch, index_key=ikey)
    as_bytes = lambda t: t.contiguous().view(torch.uint8).cpu()
    assert torch.equal(as_bytes(g.k_cache), as_bytes(rk)), "K cache"
    assert torch.equal(as_bytes(g.v_cache), as_bytes(rv)), "V cache"
    assert torch.equal(as_bytes(g.label), as_bytes(rl)), "label cache"


@pytest.mark.parametrize("k", [64, 4096])
def test_append_then_decode_over_the_extended_sequences(k):
    # Append every request's next token, extend the sequences by one, and the
    # chained decode step must match the oracle on the appended caches (with
    # k = 4096 every token, the new one included, is attended).
    w = workload("append_decode", 2, 8, 2, [1501, 701], 32, 2, k, seed=91)
    inp = dsgen.make_inputs(w)
    k_new, v_new, ch, ikey = _new_token(w, 33)
    pos = torch.tensor([1500, 700], dtype=torch.int32)    # sequences of 1500 and 700 tokens grow by one
    g = inp.to(DEV)
    ds = _ds()
    ds.ds_cache_append(shape_of(inp), k_new.to(DEV), v_new.to(DEV), g.k_cache, g.v_cache, g.k_scale, g.v_scale,
                       g.page_table, pos.to(DEV), label=g.label, channels=ch.to(DEV))
    seq = (pos + 1).to(torch.int32)
    g.seq_lens.copy_(seq.to(DEV))
    idx, out, lse = run_decode(g, shape_of(inp), w.top_k)
    torch.cuda.synchronize()
    rk, rv, rl = oracle.cache_append(k_new, v_new, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                                     inp.page_table, pos, inp.label, channels=ch)
    inp.k_cache, inp.v_cache, inp.label, inp.seq_lens = rk, rv, rl, seq
    _, ridx, rout, rlse = oracle.decode(inp)
    assert torch.equal(idx.cpu(), ridx)
    if k >= max(w.seq_lens) + 1:
        for b in range(w.batch):
            assert (idx[b] == int(pos[b])).any(dim=-1).all(), "the appended token was not attended"
    assert_close(out, rout, atol_for(w), "decode after append")


def test_append_flags_positions_past_the_page_table():
    w = workload("append_oob", 2, 4, 1, [64, 10], 16, 1, 8, seed=5)
    inp = dsgen.make_inputs(w)
    g = inp.to(DEV)
    k_new, v_new, ch, ikey = _new_token(w, 35)
    before = g.k_cache.clone()
    pos = torch.tensor([64, 10], dtype=torch.int32)       # request 0 has one page: position 64 is outside
    ds = _ds()
    ds.ds_cache_append(shape_of(inp), k_new.to(DEV), v_new.to(DEV), g.k_cache, g.v_cache, g.k_scale, g.v_scale,
                       g.page_table, pos.to(DEV), label=g.label, channels=ch.to(DEV))
    torch.cuda.synchronize()
    assert ds.ds_device_errors() == 1          # DS_DEVERR_SEQ_LEN, read and cleared
    slot1 = int(inp.page_table[1, 0]) * 64 + 10
    changed = (g.k_cache != before).any(dim=-1).any(dim=-1).nonzero().flatten().tolist()
    assert changed == [slot1] or changed == []   # request 1 written (unless its row was equal), request 0 not
