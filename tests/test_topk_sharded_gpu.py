"""GPU parity of the shard-emulated top-k (ds_topk_select_sharded): it must
equal the oracle's top-k (and so the unsharded ds_topk_select) bit-exactly,
whatever the number of shards."""
import pytest
import torch

import dsgen
import oracle

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


def _shape(ds, B, H, T):
    return ds.Shape(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, page_size=64,
                    max_pages_per_req=-(-T // 64), num_pages=1, max_seq_len=T)


def _sharded(scores, seq, k, S):
    ds = _ds()
    B, H, T = scores.shape
    shape = _shape(ds, B, H, T)
    idx = torch.full((B, H, k), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(1, ds.ds_topk_sharded_workspace_bytes(shape, k, S)), dtype=torch.uint8, device=DEV)
    ds.ds_topk_select_sharded(shape, scores.to(DEV).contiguous(), seq.to(DEV), k, S, idx, ws)
    return idx.cpu()


CASES = [
    # B, H, T, seq_lens, k, lo, hi
    (1, 1, 100, [100], 10, -3, 3),
    (2, 3, 5000, [5000, 4097], 300, -40, 40),
    (3, 2, 9000, [9000, 0, 8191], 256, -2, 2),          # an empty row, heavy ties
    (1, 1, 3000, [3000], 5000, -5, 5),                  # k > T
    (1, 4, 12000, [12000], 2048, 0, 0),                  # all equal
    (2, 1, 70000, [70000, 65], 3000, -1000, 1000),       # a shard shorter than k
]


@pytest.mark.parametrize("S", [1, 2, 4, 16])
@pytest.mark.parametrize("case", CASES)
def test_sharded_topk_bit_exact(case, S):
    B, H, T, seq, k, lo, hi = case
    s = dsgen.uniform_int((B, H, T), lo, hi, T + k + S, 3, dtype=torch.float32)
    seq_t = torch.tensor(seq, dtype=torch.int32)
    assert torch.equal(_sharded(s, seq_t, k, S), oracle.topk(s, seq_t, k))


def test_sharded_topk_real_valued_with_nan_and_signed_zero():
    s = dsgen.normal((2, 2, 30000), 9, 4, dtype=torch.float32)
    s[0, 0, 100:200] = float("nan")
    s[0, 1, :5000] = 0.0
    s[0, 1, 5000:10000] = -0.0
    seq = torch.tensor([30000, 29999], dtype=torch.int32)
    for k in (1, 777, 5000):
        assert torch.equal(_sharded(s, seq, k, 4), oracle.topk(s, seq, k)), k


def test_sharded_topk_equals_unsharded_on_the_1m_token_row():
    # QSA-shaped: 4 rows of 1,048,576 integer scores, 16 shards, k = 2048.
    ds = _ds()
    T, k = 1 << 20, 2048
    s = dsgen.uniform_int((1, 4, T), -3000, 3000, 21, 1, device=DEV, dtype=torch.float32)
    seq = torch.tensor([T], dtype=torch.int32, device=DEV)
    shape = _shape(ds, 1, 4, T)
    ref = torch.empty((1, 4, k), dtype=torch.int32, device=DEV)
    ws = torch.empty(ds.ds_topk_workspace_bytes(shape, k), dtype=torch.uint8, device=DEV)
    ds.ds_topk_select(shape, s, seq, k, ref, ws)
    got = _sharded(s, seq.cpu(), k, 16)
    assert torch.equal(got, ref.cpu())
    assert torch.equal(got[:, :1], oracle.topk(s[:, :1].cpu(), seq.cpu(), k))
