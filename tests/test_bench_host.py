"""Host logic of the benchmark's multi-process path, on CPU: two gloo ranks join
the job, meet at the barrier, agree on the slowest rank's time, and only rank 0
prints the reference arm's line."""
import contextlib
import io
import json
import os
import socket
import sys

import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    os.environ.update(RANK=str(rank), LOCAL_RANK=str(rank), WORLD_SIZE=str(world), MASTER_ADDR="127.0.0.1",
                      MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist

    import bench
    w, r, _ = bench.dist_setup(world)
    assert (w, r) == (world, rank)
    assert dist.get_backend() == "gloo"
    bench.barrier(w)
    slowest = bench.max_over_ranks(1.5 + rank, w)
    # The reference arm under torchrun: rank 0 alone runs the oracle and prints.
    sys.argv = ["bench.py", "--impl", "reference", "--config", "0", "--steps", "1", "--warmup", "0"]
    out = io.StringIO()
    with contextlib.redirect_stdout(out):
        rc = bench.main()
    bench.barrier(w)
    dist.destroy_process_group()
    results.put((rank, slowest, rc, out.getvalue()))


def test_two_gloo_ranks_agree_on_the_slowest_time_and_only_rank0_prints():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = {}
    for _ in range(world):
        rank, slowest, rc, text = q.get(timeout=300)
        got[rank] = (slowest, rc, text)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == got[1][0] == 2.5
    assert got[0][1] == 0 and got[1][1] == 0
    assert got[1][2] == ""
    line = json.loads(got[0][2].strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["n_gpus"] == 2 and line["unit"] == "calls/s"
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["workload"] == "tiny_ds_b1_h4_t4096_c16_k256"


def test_oracle_rows_on_several_threads_match_one_thread():
    # The CPU baseline runs the oracle on (request, KV head) rows from several
    # host threads at once: each row's result must not depend on that.
    from concurrent.futures import ThreadPoolExecutor

    sys.path.insert(0, ROOT)
    import bench
    import dsgen
    import oracle

    w = dsgen.WORKLOADS[0].scaled(batch=2, num_q_heads=8, num_kv_heads=2, seq_lens=[700, 1500], top_k=64,
                                  name="threads")
    inp = dsgen.make_inputs(w, device="cpu")
    masks = bench.row_masks(w)
    assert len(masks) == 4 and all(int(m.sum()) == 1 for m in masks)
    one = [oracle.decode(inp, row_mask=m) for m in masks]
    with ThreadPoolExecutor(4) as ex:
        many = list(ex.map(lambda m: oracle.decode(inp, row_mask=m), masks * 3))
    for i, got in enumerate(many):
        want = one[i % 4]
        b, g = divmod(i % 4, 2)
        assert torch.equal(got[1][b, g], want[1][b, g])
        assert torch.equal(got[2][b, g * 4:(g + 1) * 4], want[2][b, g * 4:(g + 1) * 4])
    rate, n = bench.oracle_rows(inp, 60.0, 3, max_rows=7)
    assert n == 7 and rate > 0


def test_step_percentiles_nearest_rank():
    sys.path.insert(0, ROOT)
    import bench
    got = bench.step_percentiles([0.07, 0.05, 0.06, 0.052, 0.055])
    assert got == {"p10": 50.0, "p50": 55.0, "p90": 70.0}
    assert bench.step_percentiles([0.1]) == {"p10": 100.0, "p50": 100.0, "p90": 100.0}
    assert bench.step_percentiles([])["p50"] is None


def test_algorithmic_bytes_are_the_workloads_byte_counts():
    # Per call: the label / index rows scanned (B * T * label heads * C * 2) and the selected K and V rows
    # (B * Hkv * k * D * element size * 2), worked out by hand from each workload's shape.
    sys.path.insert(0, ROOT)
    import bench
    import dsgen
    want = {
        "llama8b_ds_b3_h32kv8_t60000_c32_k3000": (92_160_000, 36_864_000, 0),
        "longchat7b_ds_b3_h32kv32_t20000_c16_k1024": (61_440_000, 50_331_648, 0),
        "qsa_b8_h32kv4_t262144_idx64_k2048_fp8": (268_435_456, 16_777_216, 8 * 4 * 2048 * 8),
        "qsa_1m_b1_h32kv4_t1048576_idx64_k2048_fp8": (134_217_728, 2_097_152, 1 * 4 * 2048 * 8),
    }
    for w in dsgen.WORKLOADS[1:]:
        scan, kv, scales = want[w.name]
        ab = bench.alg_bytes(w)
        assert ab["scan"] == scan and ab["kv_rows"] == kv + scales, w.name
        assert ab["page_table"] == w.batch * -(-w.seq_lens[0] // 64) * 4
        assert ab["total"] == sum(v for key, v in ab.items() if key != "total")


def test_default_headline_is_the_largest_workload_and_the_others_ride_along():
    # The headline is the workload with the most algorithmic bytes per call (the QSA b8 x 262,144 decode);
    # the Llama-8B DS, longchat DS and 1M-token QSA workloads are measured in the same run.
    sys.path.insert(0, ROOT)
    import bench
    import dsgen
    old = sys.argv
    sys.argv = ["bench.py"]
    try:
        args = bench.parse_args()
    finally:
        sys.argv = old
    largest = max(range(len(dsgen.WORKLOADS)), key=lambda i: bench.alg_bytes(dsgen.WORKLOADS[i])["total"])
    assert args.config == largest == 3
    assert bench.workload_of(args).name == "qsa_b8_h32kv4_t262144_idx64_k2048_fp8"
    assert sorted(bench.also_configs(args)) == [1, 2, 4]
    assert bench.NOMINAL_HBM_GBS == 8000.0
