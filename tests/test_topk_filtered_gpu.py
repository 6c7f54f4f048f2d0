"""GPU parity of the exact top-k on long rows with a small k.

When a row's CTA slices span two passes or more and k is at most 1/64 of the
row, the selection first tries one filtered pass: a lower bound on the first
radix digit of the threshold, guessed from a sample of each slice, admits only
the keys at or above it. The guess is checked exactly and the row falls back
to the two full passes when it fails (a too-high guess, or a candidate list
that overflows). Whichever way a row goes, the indices must equal the
oracle's bit for bit; the cases below reach both ways: scores that are
stationary along the row (the guess holds), monotone rows (the first keys of
each slice are not typical), heavy ties, NaN and signed zeros, rows of mixed
lengths in one launch, and row lengths that leave the rows unaligned.
"""
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


def _topk_gpu(scores, seq, k):
    ds = _ds()
    B, H, Tm = scores.shape
    shape = ds.Shape(batch=B, num_q_heads=H, num_kv_heads=H, head_dim=128, page_size=64,
                     max_pages_per_req=max(1, -(-Tm // 64)), num_pages=1, max_seq_len=Tm)
    idx = torch.full((B, H, k), -7, dtype=torch.int32, device=DEV)
    ws = torch.empty(max(1, ds.ds_topk_workspace_bytes(shape, k)), dtype=torch.uint8, device=DEV)
    ds.ds_topk_select(shape, scores.to(DEV).contiguous(), seq.to(DEV), k, idx, ws)
    return idx.cpu()


def _scores(kind, B, H, T, seed):
    t = torch.arange(T, dtype=torch.float32)
    if kind == "normal":
        return dsgen.normal((B, H, T), seed, 5, dtype=torch.float32)
    if kind == "coarse":      # normal scores on a grid of 1/4: ties all along the tail
        return torch.round(dsgen.normal((B, H, T), seed, 5, dtype=torch.float32) * 4) / 4
    if kind == "decreasing":
        return (-t).expand(B, H, T).contiguous()
    if kind == "increasing":
        return t.expand(B, H, T).contiguous()
    if kind == "sink_recent":   # high first tokens, a shifted recent window, normal elsewhere
        s = dsgen.normal((B, H, T), seed, 5, dtype=torch.float32)
        s[..., :64] += 40.0
        s[..., -1024:] += 3.0
        return s
    if kind == "neg_inf":     # -inf everywhere but 5000 finite scores: the sample's maxima are -inf
        s = torch.full((B, H, T), float("-inf"))
        pos = dsgen.permutation(T, seed, 6)[:5000]
        s[..., pos] = dsgen.normal((B, H, 5000), seed, 7, dtype=torch.float32)
        return s
    if kind == "nan_zero":
        s = dsgen.normal((B, H, T), seed, 5, dtype=torch.float32)
        s[..., 1000:1500] = float("nan")
        s[..., 40000:41000] = 0.0
        s[..., 41000:42000] = -0.0
        return s
    raise ValueError(kind)


CASES = [
    # kind, B, H, T, seq_lens, k
    ("normal", 1, 4, 300000, [300000], 2048),
    ("normal", 3, 2, 262147, [262147, 250001, 16383], 1024),   # unaligned rows, one short row
    ("normal", 1, 1, 1 << 20, [1 << 20], 2048),
    ("normal", 1, 2, 400000, [399999], 64),
    ("coarse", 1, 4, 300000, [300000], 2048),
    ("decreasing", 1, 2, 300000, [300000], 2048),
    ("increasing", 1, 2, 300000, [300000], 2048),
    ("sink_recent", 2, 2, 300000, [300000, 200000], 1500),
    ("nan_zero", 1, 2, 300000, [300000], 4000),
    ("neg_inf", 1, 2, 300000, [300000], 2048),
]


@pytest.mark.parametrize("case", CASES, ids=[f"{c[0]}_{c[3]}_{c[5]}" for c in CASES])
def test_long_row_topk_bit_exact(case):
    kind, B, H, T, seq, k = case
    s = _scores(kind, B, H, T, T + k)
    seq_t = torch.tensor(seq, dtype=torch.int32)
    assert torch.equal(_topk_gpu(s, seq_t, k), oracle.topk(s, seq_t, k))


def test_long_row_threshold_inside_a_tie_class():
    # 3000 tokens share the k-th largest value, spread over every slice: the
    # lowest-index rule decides which of them are kept.
    T = 300000
    s = dsgen.normal((1, 1, T), 17, 5, dtype=torch.float32)
    tie = torch.arange(7, T, 100)
    s[0, 0, tie] = 3.25
    seq = torch.tensor([T], dtype=torch.int32)
    for k in (1000, 2000, 4000):
        assert torch.equal(_topk_gpu(s, seq, k), oracle.topk(s, seq, k)), k


def test_long_row_tie_class_inside_one_slice():
    # 2500 consecutive tokens share one value in the threshold's first-digit bin (scores 3 to 3.5), all
    # inside one CTA's slice: one CTA of the cluster holds nearly all of the keys that digits 2 and 3 and
    # the tie rule decide on. k = 1000 (the filtered variant) and k = 2500 (the two-pass variant) both put
    # the threshold inside the tie class.
    T = 300000
    s = dsgen.normal((1, 1, T), 19, 5, dtype=torch.float32)
    s[0, 0, 5000:7500] = 3.25
    seq = torch.tensor([T], dtype=torch.int32)
    for k in (1000, 2500):
        assert torch.equal(_topk_gpu(s, seq, k), oracle.topk(s, seq, k)), k
