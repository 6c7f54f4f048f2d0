"""ds_topk_select_static: the top-k entry point for callers that cannot
allocate device memory (a plugin whose host framework owns every device
allocation and hands it only the call's tensors, or a serving thread that must
not wait on an allocator's lock). It uses a fixed scratch array inside the
library instead of a workspace; its results must be identical to
ds_topk_select's.

Kept in a file that pytest collects last, so that a run stopping at the first
failure has already run every other test.
"""
import pytest
import torch

import dsgen

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _shape(ds, B, H, T):
    return ds.Shape(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, page_size=64,
                    max_pages_per_req=-(-T // 64), num_pages=1, max_seq_len=T)


def _with_workspace(ds, shape, scores, seq, k):
    idx = torch.full((shape.batch, shape.num_kv_heads, k), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(ds.ds_topk_workspace_bytes(shape, k), dtype=torch.uint8, device=DEV)
    ds.ds_topk_select(shape, scores, seq, k, idx, ws)
    return idx


def _static(ds, shape, scores, seq, k):
    idx = torch.full((shape.batch, shape.num_kv_heads, k), -7, dtype=torch.int32, device=DEV)
    ds.ds_topk_select_static(shape, scores, seq, k, idx)
    return idx


def test_static_scratch_topk_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    import top_sparse_decode_label_gb300 as ds
    B, H, T, k = 3, 4, 50000, 1500
    shape = _shape(ds, B, H, T)
    assert ds.ds_topk_workspace_bytes(shape, k) <= 16 << 20
    seq = torch.tensor([50000, 31111, 7], dtype=torch.int32, device=DEV)
    # Two different inputs back to back: the second call must not see the
    # first one's leftovers in the shared scratch. Integer scores give many ties.
    for seed in (1, 2):
        scores = dsgen.uniform_int((B, H, T), -300, 300, seed, 5, device=DEV, dtype=torch.float32)
        got = _static(ds, shape, scores, seq, k)
        ref = _with_workspace(ds, shape, scores, seq, k)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu(), ref.cpu()), f"call with seed {seed}"
    assert ds.ds_device_errors() == 0


def test_static_scratch_topk_that_spills_into_the_array_matches_on_two_calls_in_a_row():
    # Nine keys in ten equal (0) and the rest 1, k about T/2: the threshold falls on the 0 keys, so every
    # CTA of the row's cluster keeps its whole slice (about 6250 pairs, more than its shared-memory list
    # holds) and spills the list into the scratch array; ties go to the lowest token indices.
    import top_sparse_decode_label_gb300 as ds
    B, H, T, k = 1, 4, 50000, 25000
    shape = _shape(ds, B, H, T)
    assert ds.ds_topk_workspace_bytes(shape, k) <= 16 << 20
    seq = torch.tensor([T], dtype=torch.int32, device=DEV)
    for seed in (3, 4):
        u = dsgen.uniform_int((B, H, T), 0, 9, seed, 6, device=DEV, dtype=torch.float32)
        scores = (u == 9).to(torch.float32)
        got = _static(ds, shape, scores, seq, k)
        ref = _with_workspace(ds, shape, scores, seq, k)
        torch.cuda.synchronize()
        assert torch.equal(got.cpu(), ref.cpu()), f"call with seed {seed}"
        assert (got >= 0).all()
    assert ds.ds_device_errors() == 0


def test_static_scratch_rejects_problems_larger_than_its_array():
    import top_sparse_decode_label_gb300 as ds
    shape = _shape(ds, 8, 4, 262144)           # needs about 67 MB of scratch
    assert ds.ds_topk_workspace_bytes(shape, 2048) > 16 << 20
    scores = torch.zeros((1,), device=DEV)
    seq = torch.zeros((8,), dtype=torch.int32, device=DEV)
    idx = torch.zeros((1,), dtype=torch.int32, device=DEV)
    with pytest.raises(ds.DsError) as e:
        ds.ds_topk_select_static(shape, scores, seq, 2048, idx)
    assert e.value.status == -4
