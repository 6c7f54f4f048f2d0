"""Shared helpers of the GPU parity tests: run the library through its C ABI
and compare with the oracle under the stated tolerances."""
import math

import torch

import dsgen

# Attention output tolerance, elementwise |gpu - ref| <= ATOL + RTOL * |ref|:
# max-abs 2e-3 with relative 1e-2 for a bf16 KV cache, 2e-2 absolute for FP8.
RTOL = 1e-2
ATOL_BF16 = 2e-3
ATOL_FP8 = 2e-2
LSE_ATOL = 1e-3


def atol_for(w) -> float:
    return ATOL_FP8 if w.kv_dtype == "fp8_e4m3" else ATOL_BF16


def assert_close(gpu: torch.Tensor, ref: torch.Tensor, atol: float, what: str):
    g = gpu.detach().double().cpu()
    r = ref.detach().double().cpu()
    err = (g - r).abs()
    bad = ~(err <= atol + RTOL * r.abs())
    if bad.any():
        i = int(bad.flatten().nonzero()[0])
        raise AssertionError(f"{what}: {int(bad.sum())} elements outside tolerance; first at flat {i}: "
                             f"gpu {g.flatten()[i].item()} ref {r.flatten()[i].item()}; max err {err.max().item()}")


def assert_lse_close(gpu: torch.Tensor, ref: torch.Tensor, what: str):
    g = gpu.detach().double().cpu()
    r = ref.detach().double().cpu()
    ninf = torch.isinf(r) & (r < 0)
    assert torch.equal(torch.isinf(g) & (g < 0), ninf), f"{what}: -inf pattern differs"
    fin = ~ninf
    if fin.any():
        err = (g[fin] - r[fin]).abs().max().item()
        assert err <= LSE_ATOL, f"{what}: lse max err {err}"


def shape_of(inp):
    import top_sparse_decode_label_gb300 as ds
    return ds.Shape(**dsgen.shape_kwargs(inp))


def workload(name, B, Hq, Hkv, T, C, HL, k, kv="bf16", shuffle=True, seed=5, from_q=None, head_dim=128):
    return dsgen.Workload(name=name, batch=B, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=head_dim,
                          seq_lens=list(T), proxy_dim=C, label_heads=HL, top_k=k, kv_dtype=kv,
                          shuffle_pages=shuffle, seed=seed,
                          proxy_from_query=(HL != 1 or Hkv == 1) if from_q is None else from_q)


def run_decode(inp_gpu, shape, k):
    """The chained C entry point on device inputs: (idx, out, lse)."""
    import top_sparse_decode_label_gb300 as ds
    w = inp_gpu.w
    dev = inp_gpu.q.device
    idx = torch.full((w.batch, w.num_kv_heads, k), -7, dtype=torch.int32, device=dev)
    out = torch.full((w.batch, w.num_q_heads, w.head_dim), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((w.batch, w.num_q_heads), float("nan"), dtype=torch.float32, device=dev)
    # Stale bytes: the chained call needs no initialised workspace.
    ws = torch.full((ds.ds_decode_workspace_bytes(shape, w.proxy_dim, k),), 0xA5, dtype=torch.uint8, device=dev)
    ds.ds_sparse_decode(shape, inp_gpu.q, inp_gpu.qp, inp_gpu.label, inp_gpu.k_cache, inp_gpu.v_cache,
                        inp_gpu.k_scale, inp_gpu.v_scale, inp_gpu.page_table, inp_gpu.seq_lens, k, idx, out, lse,
                        ws)
    return idx, out, lse


def default_scale(w):
    return 1.0 / math.sqrt(w.head_dim)


def host_threads() -> int:
    import os
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_every_row(inp, k=None, num_splits: int = 1, split_mode: int = 0):
    """The oracle's (idx, out, lse) for every (request, KV head) row of a CPU ``dsgen.Inputs``.

    Each row is the oracle's four stages run on that row alone (its row mask); the rows are spread over
    the host cores (the C oracle releases the interpreter lock while it computes) and their results are
    assembled into full-size tensors: idx int32 [B, Hkv, k], out float64 [B, Hq, D], lse float64 [B, Hq].
    """
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    w = inp.w
    k = w.top_k if k is None else k
    B, Hkv, G = w.batch, w.num_kv_heads, w.group
    oracle.lib()
    idx = torch.full((B, Hkv, k), -1, dtype=torch.int32)
    out = torch.zeros((B, w.num_q_heads, w.head_dim), dtype=torch.float64)
    lse = torch.zeros((B, w.num_q_heads), dtype=torch.float64)

    def one(bg):
        b, g = bg
        m = torch.zeros((B, Hkv), dtype=torch.uint8)
        m[b, g] = 1
        _, ri, ro, rl = oracle.decode(inp, k=k, num_splits=num_splits, split_mode=split_mode, row_mask=m)
        hs = slice(g * G, (g + 1) * G)
        return b, g, ri[b, g].clone(), ro[b, hs].clone(), rl[b, hs].clone()

    rows = [(b, g) for b in range(B) for g in range(Hkv)]
    prev = torch.get_num_threads()
    torch.set_num_threads(1)
    try:
        with ThreadPoolExecutor(min(len(rows), host_threads())) as ex:
            for b, g, ri, ro, rl in ex.map(one, rows):
                idx[b, g] = ri
                out[b, g * G:(g + 1) * G] = ro
                lse[b, g * G:(g + 1) * G] = rl
    finally:
        torch.set_num_threads(prev)
    return idx, out, lse
