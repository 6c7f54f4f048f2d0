"""The pages' multi-rank decode step, on CPU with gloo ranks and the oracle.

sglang PR #43527 "QSA cache sharding", "QSA cache placement": every cache page
has one owner, placed page-interleaved; "Distributed QSA execution": each rank
scores only the tokens of the pages it owns and selects local candidates, the
candidates are merged into the exact global Top-K with deterministic global
token-ID tie-breaking, each owner computes the sparse attention partial over
the selected tokens it holds, and the partials are merged with FP32
log-sum-exp normalisation.

The library keeps that split on one GPU (the split-KV merge and the
shard-emulated top-k). This test runs it across processes: world ranks, rank r
owning logical page p of every request when p mod world == r; the local top-k
uses the oracle's selection rule on the rank's own tokens; an all_gather of
(score, token) candidates feeds the exact merge; an all_gather of (o, lse)
feeds the LSE merge. The result must equal the unsharded oracle step: the same
indices, and outputs equal up to double rounding.
"""
import os
import socket
import sys

import pytest
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
P = 64


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _workload():
    import dsgen
    # Two requests, one shorter with a partial last page; GQA groups of 4; integer proxy scores with ties.
    return dsgen.Workload(name="multirank", batch=2, num_q_heads=8, num_kv_heads=2, head_dim=128,
                          seq_lens=[64 * 23 + 17, 64 * 9], proxy_dim=16, label_heads=2, top_k=150,
                          kv_dtype="bf16", shuffle_pages=True, seed=77)


def _rank_step(rank: int, world: int, inp):
    """One decode step computed the pages' distributed way; returns (idx, out, lse) on every rank."""
    import torch.distributed as dist

    import oracle
    w = inp.w
    B, Hkv, G, k = w.batch, w.num_kv_heads, w.group, w.top_k
    T = inp.seq_lens.tolist()
    # ---- 1. scan: this rank's tokens only (the pages it owns), in global token order
    scores = oracle.index_score(inp.qp, inp.label, inp.page_table, inp.seq_lens, Hkv, w.max_seq_len)
    owned = [[t for t in range(T[b]) if (t // P) % world == rank] for b in range(B)]
    n_own = max(1, max(len(o) for o in owned))
    shard = torch.full((B, Hkv, n_own), float("nan"), dtype=torch.float32)
    for b in range(B):
        if owned[b]:
            shard[b, :, :len(owned[b])] = scores[b][:, owned[b]]
    # ---- 2. local top-k (the library's rule on the rank's own tokens), as (score, global token) candidates
    local = oracle.topk(shard, torch.tensor([len(o) for o in owned], dtype=torch.int32), k)
    cand_tok = torch.full((B, Hkv, k), -1, dtype=torch.int64)
    cand_score = torch.full((B, Hkv, k), float("nan"), dtype=torch.float32)
    for b in range(B):
        for g in range(Hkv):
            for j, pos in enumerate(local[b, g].tolist()):
                if pos >= 0:
                    cand_tok[b, g, j] = owned[b][pos]
                    cand_score[b, g, j] = shard[b, g, pos]
    toks = [torch.empty_like(cand_tok) for _ in range(world)]
    scs = [torch.empty_like(cand_score) for _ in range(world)]
    dist.all_gather(toks, cand_tok)
    dist.all_gather(scs, cand_score)
    # ---- 3. exact merge: the top-k of the union, equal scores to the lower global token
    idx = torch.full((B, Hkv, k), -1, dtype=torch.int32)
    for b in range(B):
        for g in range(Hkv):
            pairs = sorted((int(t), float(s)) for tt, ss in zip(toks, scs)
                           for t, s in zip(tt[b, g].tolist(), ss[b, g].tolist()) if t >= 0)
            row = torch.tensor([[[s for _, s in pairs]]], dtype=torch.float32)
            pick = oracle.topk(row, torch.tensor([len(pairs)], dtype=torch.int32), k)[0, 0].tolist()
            kept = [pairs[p][0] for p in pick if p >= 0]
            idx[b, g, :len(kept)] = torch.tensor(kept, dtype=torch.int32)
    # ---- 4. owner-side partials over the selected tokens this rank holds, then the LSE merge
    mine = torch.where((idx >= 0) & ((idx // P) % world == rank), idx, torch.full_like(idx, -1))
    mine = torch.stack([torch.stack([torch.cat([r[r >= 0], r[r < 0]]) for r in row]) for row in mine])
    o, l = oracle.sparse_attn(inp.q, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale, inp.page_table,
                              inp.seq_lens, mine)
    os_ = [torch.empty_like(o[0]) for _ in range(world)]
    ls_ = [torch.empty_like(l[0]) for _ in range(world)]
    dist.all_gather(os_, o[0].contiguous())
    dist.all_gather(ls_, l[0].contiguous())
    out, lse = oracle.lse_merge(torch.stack(os_), torch.stack(ls_))
    return idx, out, lse


def _rank_main(rank, world, port, results):
    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import dsgen
    torch.set_num_threads(1)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        inp = dsgen.make_inputs(_workload())
        idx, out, lse = _rank_step(rank, world, inp)
        results.put((rank, idx, out, lse))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 3])
def test_page_sharded_ranks_equal_the_unsharded_step(world):
    sys.path.insert(0, ROOT)
    import dsgen
    import oracle

    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, idx, out, lse = q.get(timeout=300)
        got[rank] = (idx, out, lse)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    inp = dsgen.make_inputs(_workload())
    _, ridx, rout, rlse = oracle.decode(inp)
    for rank, (idx, out, lse) in got.items():
        assert torch.equal(idx, ridx), f"rank {rank}: merged indices differ from the unsharded top-k"
        assert torch.allclose(out, rout, rtol=0, atol=1e-10), f"rank {rank}: merged output"
        assert torch.allclose(lse, rlse, rtol=0, atol=1e-10), f"rank {rank}: merged lse"
    # Every rank owned part of the selection: the merge really combined several owners.
    owners = {int(t) // P % world for t in ridx[ridx >= 0].tolist()}
    assert owners == set(range(world))
