#!/usr/bin/env python
"""Benchmark of one decode step of top-k sparse attention on GB300.

A step is one call of the chained C entry point ds_sparse_decode (score every
cached token -> exact top-k -> sparse GQA attention over the selected tokens ->
log-sum-exp merge) over one batch of seeded synthetic inputs that are already
resident in HBM. The headline workload is the largest one, the QSA-shaped
decode (batch 8, 32 query / 4 KV heads, 262,144 tokens per request, 64-wide
index keys, top-k 2048, FP8 E4M3 paged KV); --config selects another one of
dsgen.WORKLOADS. The Llama-3.1-8B- and longchat-7b-shaped Double-Sparsity
workloads and the 1M-token QSA request (--also) are measured in the same run,
with the same steps and warm-up, into `per_config`.

Printed: one JSON line with calls/s (value), the achieved HBM bandwidth of the
step against the nominal 8 TB/s and against the measured copy bandwidth, the
dominant kernel's roofline, the end-to-end number through the C ABI with
host<->device copies, the oracle's CPU time on a bounded sample, clocks
sampled during the timed region, and the number of kernel launches; the same
fields for every workload of `per_config`.

Timing: W untimed warm-up steps, then exactly K timed steps; L2 is flushed
before every timed step (a 256 MiB device write, then a 256 MiB read so the
dirty lines are written back before the step starts), outside the CUDA events
that bracket each step on the launching stream. Under torchrun each rank runs
its own replica (weak scaling, no collective on the data path) and the
slowest rank's time is used.

`--impl reference` times the oracle (plain single-threaded C++, one
(request, KV head) row per host thread) on the same workload instead: each
step runs as many rows at once as the host has cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

import dsgen  # noqa: E402

METRIC = "sparse-decode attn calls/s + achieved HBM GB/s vs ~8 TB/s roofline, 1×GB300"
FALLBACK_HBM_GBS = 6800.0
# The nominal HBM3e bandwidth of one GB300 that the decode step's roofline
# fraction is stated against; the measured copy bandwidth is reported beside it.
NOMINAL_HBM_GBS = 8000.0


def parse_args():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=3,
                    help="headline workload, an index into dsgen.WORKLOADS (default: the QSA b8 x 262,144 "
                         "FP8 workload, the largest)")
    ap.add_argument("--also", default="1,2,4",
                    help="comma-separated further workloads measured in the same run into `per_config` "
                         "('none' for none)")
    ap.add_argument("--head-dim", type=int, default=None, help="override the workload's head dimension (128, 256)")
    ap.add_argument("--flush-mib", type=int, default=256)
    ap.add_argument("--cpu-budget-s", type=float, default=12.0, help="oracle time budget of the CPU baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--oracle-threads", type=int, default=0,
                    help="host threads of the oracle runs (default: every core this process may use)")
    return ap.parse_args()


# ----------------------------------------------------------------------------- accounting

def alg_bytes(w: dsgen.Workload) -> dict:
    """Algorithmic bytes of one call: what the method must move, per stage."""
    elt = 1 if w.kv_dtype == "fp8_e4m3" else 2
    scan = sum(T * w.label_heads * w.proxy_dim * 2 for T in w.seq_lens)
    pages = sum(-(-T // w.page_size) * 4 for T in w.seq_lens)
    keff = [min(w.top_k, T) for T in w.seq_lens]
    kv = sum(k * w.num_kv_heads * w.head_dim * elt * 2 for k in keff)
    scales = sum(k * w.num_kv_heads * 8 for k in keff) if elt == 1 else 0
    q = w.batch * w.num_q_heads * (w.head_dim + w.proxy_dim) * 2
    out = w.batch * w.num_q_heads * (w.head_dim * 2 + 4) + w.batch * w.num_kv_heads * w.top_k * 4
    return dict(scan=scan, page_table=pages, kv_rows=kv + scales, q=q, out=out,
                total=scan + pages + kv + scales + q + out)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured (MEASURED_PEAKS.json hbm_gbs: STREAM-style copy)"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback 6.8 TB/s (no MEASURED_PEAKS.json)"


def traffic_record(kernel_file: str, workload: str):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source is unchanged since."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    src = os.path.join(ROOT, "top_sparse_decode_label_gb300", "csrc", kernel_file)
    try:
        with open(path) as f:
            rec = json.load(f).get(workload, {}).get(kernel_file)
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        if rec and rec.get("source_sha") == sha:
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


def step_percentiles(step_ms) -> dict:
    """Median and 10th / 90th percentiles (nearest rank) of this rank's event-timed steps, in µs."""
    xs = sorted(step_ms)
    if not xs:
        return {"p10": None, "p50": None, "p90": None}
    at = lambda q: xs[min(len(xs) - 1, max(0, math.ceil(q * len(xs)) - 1))] * 1e3
    return {"p10": at(0.10), "p50": at(0.50), "p90": at(0.90)}


# ----------------------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons, timestamped on arrival."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.samples = []
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "50", "-i", gpu_id], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()

    def _read(self):
        for line in self.proc.stdout:
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 8:
                continue
            try:
                self.samples.append((time.time(), float(parts[0]), float(parts[1]),
                                     [n for n, v in zip(self.NAMES, parts[4:8]) if v.lower().startswith("active")]))
            except ValueError:
                continue

    def stop(self):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self, t0: float, t1: float):
        inside = [s for s in self.samples if t0 <= s[0] <= t1]
        window = "timed"
        use = inside
        if len(inside) < 3:
            use = [s for s in self.samples if s[0] <= t1]
            window = "soak+timed (timed region shorter than the sampling interval)"
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0, "window": window}
        reasons = sorted({r for s in use for r in s[3]})
        return {"sm_mhz": statistics.median(s[1] for s in use), "sm_max_mhz": max(s[2] for s in use),
                "reasons": reasons, "samples": len(use), "samples_in_timed_region": len(inside), "window": window}


# ----------------------------------------------------------------------------- distributed plumbing

def dist_setup(n_gpus: int):
    """Joins the torchrun job (one rank per GPU, NCCL; gloo on a host without CUDA)."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        if not dist.is_initialized():
            dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    """The largest x over all ranks (the slowest rank's time decides the job's)."""
    if world == 1:
        return x
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def workload_of(args, config: int = None) -> dsgen.Workload:
    """Workload `config` (default --config), with --head-dim applied (its name then says so)."""
    w = dsgen.WORKLOADS[args.config if config is None else config]
    if args.head_dim is not None and args.head_dim != w.head_dim:
        w = w.scaled(head_dim=args.head_dim, name=f"{w.name}_d{args.head_dim}")
    return w


def also_configs(args):
    """The workload indices of --also ('none' or '' for none)."""
    if args.also.strip().lower() == "none":
        return []
    return [int(x) for x in args.also.split(",") if x.strip() != ""]


def workload_config(w: dsgen.Workload, world: int, flush_mib: int) -> dict:
    """The `config` object of the JSON line; the same for both arms."""
    return {"workload": w.name, "batch": w.batch, "seq_len": w.max_seq_len, "num_q_heads": w.num_q_heads,
            "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim, "proxy_dim": w.proxy_dim,
            "label_heads": w.label_heads, "top_k": w.top_k, "kv_dtype": w.kv_dtype, "page_size": w.page_size,
            "l2": f"flushed before every timed step: {flush_mib} MiB device write, then a "
                  f"{flush_mib} MiB read so the write-back happens outside the timed region",
            "parallelism": f"replicas x{world}"}


# ----------------------------------------------------------------------------- CPU oracle

def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def row_masks(w: dsgen.Workload):
    """One row mask per (request, KV head) row of the call, in row order."""
    masks = []
    for b in range(w.batch):
        for g in range(w.num_kv_heads):
            m = torch.zeros((w.batch, w.num_kv_heads), dtype=torch.uint8)
            m[b, g] = 1
            masks.append(m)
    return masks


def oracle_rows(inp_cpu, budget_s: float, threads: int, max_rows: int = None):
    """Run the oracle on whole (request, KV head) rows until the budget is spent.

    `threads` worker threads each take the next row of the call (round robin) and run the four stages on it
    alone; the C oracle releases the interpreter lock while it computes, so the rows run in parallel on the
    host cores. Returns (rows per second, rows done).
    """
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    oracle.lib()                       # load once, before any worker thread
    masks = row_masks(inp_cpu.w)
    lock = threading.Lock()
    counter = [0]
    prev = torch.get_num_threads()
    torch.set_num_threads(1)

    def worker(deadline):
        done = 0
        while True:
            with lock:
                i = counter[0]
                counter[0] += 1
            if max_rows is not None and i >= max_rows:
                return done
            oracle.decode(inp_cpu, row_mask=masks[i % len(masks)])
            done += 1
            if time.perf_counter() >= deadline:
                return done

    try:
        with ThreadPoolExecutor(threads) as ex:
            t0 = time.perf_counter()
            futs = [ex.submit(worker, t0 + budget_s) for _ in range(threads)]
            n = sum(f.result() for f in futs)
            wall = time.perf_counter() - t0
    finally:
        torch.set_num_threads(prev)
    return n / wall, n


# ----------------------------------------------------------------------------- arms

def run_reference(args):
    world, rank, _ = int(os.environ.get("WORLD_SIZE", "1")), int(os.environ.get("RANK", "0")), 0
    if rank != 0:
        return 0
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    w = workload_of(args)
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    inp = dsgen.make_inputs(w, device=dev).to("cpu")
    rows_per_call = w.batch * w.num_kv_heads
    masks = row_masks(w)
    threads = args.oracle_threads or host_threads()
    oracle.lib()
    torch.set_num_threads(1)

    def step(pool, i):
        # `threads` rows of the call at once, one per host thread
        futs = [pool.submit(oracle.decode, inp, row_mask=masks[(i * threads + j) % len(masks)])
                for j in range(threads)]
        for f in futs:
            f.result()

    with ThreadPoolExecutor(threads) as pool:
        for i in range(args.warmup):
            step(pool, i)
        t0 = time.perf_counter()
        for i in range(args.steps):
            step(pool, args.warmup + i)
        dt = time.perf_counter() - t0
    calls_per_s = args.steps * threads / dt / rows_per_call
    sample = (f"{args.steps} steps, each {threads} (request, KV head) rows of the call ({rows_per_call} rows per "
              f"call) run at once on {threads} host threads: proxy scores of the row, its top-k, attention of its "
              f"{w.group} query heads, merge")
    line = {
        "impl": "reference", "metric": METRIC, "value": calls_per_s, "unit": "calls/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": workload_config(w, world, args.flush_mib),
        "cpu_baseline": {"value": calls_per_s, "unit": "calls/s", "cores": threads, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": calls_per_s, "unit": "calls/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


class _Device:
    """What every measured workload shares: the device, its stream, the L2 flush and the clock sampler."""

    def __init__(self, args):
        self.world, self.rank, local = dist_setup(args.gpus)
        self.dev = torch.device("cuda", local)
        torch.cuda.set_device(self.dev)
        self.stream = torch.cuda.current_stream(self.dev)
        self.flush_w = torch.empty(args.flush_mib << 20, dtype=torch.uint8, device=self.dev)
        self.flush_r = torch.zeros(args.flush_mib << 20, dtype=torch.uint8, device=self.dev)
        self.flush_sink = torch.empty((), dtype=torch.int64, device=self.dev)
        props = torch.cuda.get_device_properties(self.dev)
        gpu_id = "GPU-" + str(props.uuid) if getattr(props, "uuid", None) is not None else str(local)
        self.sampler = ClockSampler(gpu_id)

    def flush(self):
        # Evicts L2: a write of flush_w, then a read of flush_r so that the
        # dirty lines of the write are written back before the timed region.
        self.flush_w.zero_()
        torch.sum(self.flush_r, dim=0, dtype=torch.int64, out=self.flush_sink)


def measure(d: _Device, w: dsgen.Workload, args, extras: bool) -> dict:
    """Times the chained call on one workload; returns its fields of the JSON line."""
    import top_sparse_decode_label_gb300 as ds

    dev, stream, world = d.dev, d.stream, d.world
    inp = dsgen.make_inputs(w, device=dev)
    shape = ds.Shape(**dsgen.shape_kwargs(inp))
    k = w.top_k
    B, Hq, Hkv, D = w.batch, w.num_q_heads, w.num_kv_heads, w.head_dim

    idx = torch.empty((B, Hkv, k), dtype=torch.int32, device=dev)
    out = torch.empty((B, Hq, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, Hq), dtype=torch.float32, device=dev)
    ws = torch.zeros(ds.ds_decode_workspace_bytes(shape, w.proxy_dim, k), dtype=torch.uint8, device=dev)

    def step():
        ds.ds_sparse_decode(shape, inp.q, inp.qp, inp.label, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                            inp.page_table, inp.seq_lens, k, idx, out, lse, ws, stream=stream)

    for _ in range(args.warmup):
        d.flush()
        step()
    torch.cuda.synchronize()
    if ds.ds_device_errors() != 0:
        raise RuntimeError(f"{w.name}: device error word set during warm-up")

    # Untimed soak so that the clock record covers the timed region even when it is short.
    t_soak = time.time()
    while time.time() - t_soak < 1.0:
        for _ in range(50):
            d.flush()
            step()
        torch.cuda.synchronize()

    # ---- timed region: exactly K chained calls, L2 flushed before each.
    ev0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ev1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    t_wall0 = time.time()
    for i in range(args.steps):
        d.flush()
        ev0[i].record(stream)
        step()
        ev1[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    t_wall1 = time.time()
    step_ms = [a.elapsed_time(b) for a, b in zip(ev0, ev1)]
    total_s = max_over_ranks(sum(step_ms) / 1e3, world)
    calls_per_s = world * args.steps / total_s
    ms_per_step = total_s / args.steps * 1e3
    clocks = d.sampler.summary(t_wall0, t_wall1)
    if ds.ds_device_errors() != 0:
        raise RuntimeError(f"{w.name}: device error word set during the timed region")
    step_spread = step_percentiles(step_ms)

    # ---- per-stage breakdown: the same chained call, with events recorded between its stages.
    S = ds.ds_decode_num_splits(shape, k)
    nstage = min(args.steps, 500)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(nstage)]
    for e4 in evs:
        for e in e4:
            e.record(stream)  # creates the underlying event handles
    torch.cuda.synchronize()
    for i in range(nstage):
        d.flush()
        ds.ds_sparse_decode(shape, inp.q, inp.qp, inp.label, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                            inp.page_table, inp.seq_lens, k, idx, out, lse, ws, stream=stream, events=evs[i])
    torch.cuda.synchronize()
    stage_us = {name: statistics.mean(evs[i][j].elapsed_time(evs[i][j + 1]) for i in range(nstage)) * 1e3
                for j, name in enumerate(["index_score", "topk_select", "sparse_attn"])}

    # ---- end to end through the C ABI: per-step inputs from pinned host memory, results back.
    # A caller stages one step's inputs (q, qp, page table, sequence lengths)
    # in one pinned host buffer and the call's outputs (out, lse, idx) in one
    # device buffer, so each direction is a single copy; the library takes
    # views into them like any other device pointers. The read-back includes
    # the selected indices (B * Hkv * k int32) as well as out and lse: a caller
    # that needs only the attention output would copy less.
    def packed(tensors):
        nbytes = [t.numel() * t.element_size() for t in tensors]
        offs, o = [], 0
        for n in nbytes:
            offs.append(o)
            o += (n + 255) // 256 * 256
        return offs, o

    in_src = [inp.q, inp.qp, inp.page_table, inp.seq_lens]
    in_offs, in_bytes = packed(in_src)
    out_src = [out, lse, idx]
    out_offs, out_bytes = packed(out_src)
    d_in = torch.empty(in_bytes, dtype=torch.uint8, device=dev)
    d_out = torch.empty(out_bytes, dtype=torch.uint8, device=dev)
    h_in = torch.empty(in_bytes, dtype=torch.uint8).pin_memory()
    h_out = torch.empty(out_bytes, dtype=torch.uint8).pin_memory()

    def view(buf, off, like):
        n = like.numel() * like.element_size()
        return buf[off:off + n].view(like.dtype).view(like.shape)

    for t, o in zip(in_src, in_offs):
        view(h_in, o, t).copy_(t.cpu())
    e_q, e_qp, e_pt, e_sl = (view(d_in, o, t) for t, o in zip(in_src, in_offs))
    e_out, e_lse, e_idx = (view(d_out, o, t) for t, o in zip(out_src, out_offs))
    ee0 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ee1 = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    barrier(world)
    torch.cuda.synchronize()
    for i in range(args.steps):
        d.flush()
        ee0[i].record(stream)
        d_in.copy_(h_in, non_blocking=True)
        ds.ds_sparse_decode(shape, e_q, e_qp, inp.label, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                            e_pt, e_sl, k, e_idx, e_out, e_lse, ws, stream=stream)
        h_out.copy_(d_out, non_blocking=True)
        ee1[i].record(stream)
    torch.cuda.synchronize()
    barrier(world)
    e2e_s = max_over_ranks(sum(a.elapsed_time(b) for a, b in zip(ee0, ee1)) / 1e3, world)
    e2e_value = world * args.steps / e2e_s
    if not torch.equal(view(h_out, out_offs[2], idx), idx.cpu()):
        raise RuntimeError(f"{w.name}: the end-to-end call's indices differ from the device-resident call's")

    rec = {}
    if extras:
        rec.update(measure_extras(d, w, inp, shape, args))

    # ---- roofline: the step against HBM, and its dominant kernel
    peak, peak_src = measured_peak()
    ab = alg_bytes(w)
    step_gbs = ab["total"] / (ms_per_step * 1e-3) / 1e9
    dominant = max(stage_us, key=stage_us.get)
    dom_bytes, dom_file = stage_bytes(w, dominant)
    dom_gbs = dom_bytes / (stage_us[dominant] * 1e-6) / 1e9
    roofline = {"bound": "hbm", "kernel": dominant, "achieved": dom_gbs, "peak": peak, "unit": "GB/s",
                "frac": dom_gbs / peak, "frac_of_8000_gbs": dom_gbs / NOMINAL_HBM_GBS,
                "traffic": traffic_record(dom_file, w.name),
                "alg_bytes_per_launch": dom_bytes, "avg_launch_us": stage_us[dominant], "peak_source": peak_src}

    rec.update({
        "value": calls_per_s, "unit": "calls/s", "ms_per_step": ms_per_step, "step_us": step_spread,
        "config": workload_config(w, world, args.flush_mib),
        "tokens_per_s": calls_per_s * B, "scanned_tokens_per_s": calls_per_s * sum(w.seq_lens),
        "step_hbm": {"alg_bytes_per_call": ab["total"], "bytes_breakdown": ab, "achieved_gbs": step_gbs,
                     "frac_of_8000_gbs": step_gbs / NOMINAL_HBM_GBS,
                     "frac_of_measured_copy": step_gbs / peak, "measured_copy_gbs": peak},
        "stage_us": stage_us, "internal_splits": S,
        "roofline": roofline,
        "e2e": {"value": e2e_value, "unit": "calls/s", "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": out_bytes,
                "what": "one H2D copy of q, qp, page_table, seq_lens staged in one pinned buffer; the chained "
                        "call on views of it; one D2H copy of out, lse and the selected indices; KV and label "
                        "caches stay resident"},
        "clocks": clocks,
        "gpu_launches": args.steps * ds.ds_decode_kernel_launches(shape, k),
    })
    if d.rank == 0 and world == 1 and not args.no_cpu_baseline:
        budget = args.cpu_budget_s if extras else args.cpu_budget_s / 2
        rec["cpu_baseline"] = cpu_baseline(inp, args, budget)
    return rec


def stage_bytes(w: dsgen.Workload, stage: str):
    """Algorithmic bytes one launch of a stage's kernel moves, and its source file."""
    ab = alg_bytes(w)
    if stage == "index_score":
        return ab["scan"] + ab["page_table"] + w.batch * w.num_q_heads * w.proxy_dim * 2, "score.cu"
    if stage == "sparse_attn":
        return ab["kv_rows"] + ab["q"] + w.batch * w.num_kv_heads * w.top_k * 4, "attn.cu"
    # the top-k reads the row scores once and writes the indices
    return sum(T * 4 for T in w.seq_lens) * w.num_kv_heads + w.batch * w.num_kv_heads * w.top_k * 4, "topk.cu"


def cpu_baseline(inp, args, budget_s: float) -> dict:
    """The oracle on whole (request, KV head) rows of the call, on the host cores, scaled to calls/s."""
    w = inp.w
    rows_per_call = w.batch * w.num_kv_heads
    cpu = inp.to("cpu")
    threads = args.oracle_threads or host_threads()
    rate1, n1 = oracle_rows(cpu, budget_s / 3, 1)
    rate, n = oracle_rows(cpu, budget_s * 2 / 3, threads)
    what = (f"(request, KV head) rows of the {rows_per_call}-row call, each scored, top-k selected and "
            f"attended by the oracle")
    return {
        "value": rate / rows_per_call, "unit": "calls/s", "cores": threads, "kind": "oracle",
        "sample": f"{n} {what}, {threads} rows at a time on {threads} host threads",
        "single_thread": {"value": rate1 / rows_per_call, "unit": "calls/s", "cores": 1,
                          "sample": f"{n1} {what}, one at a time; {1e3 / rate1:.1f} ms per row"},
    }


def measure_extras(d: _Device, w: dsgen.Workload, inp, shape, args) -> dict:
    """Beside the headline, outside its timed region: the cache append, the shard-emulated top-k and
    (shared index keys only) the block-compressed selection."""
    import top_sparse_decode_label_gb300 as ds

    dev, stream = d.dev, d.stream
    k = w.top_k
    B, Hkv, D = w.batch, w.num_kv_heads, w.head_dim
    # ---- the step before the path: appending each request's new token (its
    # last position is rewritten with fresh rows; launch-latency-bound).
    append_us = None
    try:
        gen = torch.Generator(device="cpu").manual_seed(7)
        k_new = torch.randn((B, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
        v_new = torch.randn((B, Hkv, D), generator=gen).to(torch.bfloat16).to(dev)
        pos = (inp.seq_lens - 1).clamp(min=-1).to(torch.int32)
        if w.label_heads == Hkv:
            channels = torch.stack([torch.randperm(D, generator=gen)[:w.proxy_dim] for _ in range(Hkv)])
            channels, index_key = channels.to(torch.int32).to(dev), None
        else:
            channels = None
            index_key = torch.randn((B, w.proxy_dim), generator=gen).to(torch.bfloat16).to(dev)

        def append():
            ds.ds_cache_append(shape, k_new, v_new, inp.k_cache, inp.v_cache, inp.k_scale, inp.v_scale,
                               inp.page_table, pos, label=inp.label, channels=channels, index_key=index_key)

        # Device time per call: 200 calls captured in a CUDA graph (host launch cost excluded).
        reps = 200
        side = torch.cuda.Stream(dev)
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            for _ in range(3):
                append()
        torch.cuda.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            for _ in range(reps):
                append()
        graph.replay()
        torch.cuda.synchronize()
        ea = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
        ea[0].record(stream)
        graph.replay()
        ea[1].record(stream)
        torch.cuda.synchronize()
        append_us = ea[0].elapsed_time(ea[1]) * 1e3 / reps
        if ds.ds_device_errors() != 0:
            raise RuntimeError("device error word set by the cache append")
    except Exception as e:  # reported, never hides the main measurement
        append_us = f"failed: {e}"

    # ---- the shard-emulated top-k (4 page-interleaved shards, as the QSA
    # cache-sharding page runs it) beside the single-pass top-k, on this
    # workload's scores (no L2 flush: both read the scores from L2).
    sharded = None
    try:
        scores = torch.empty((B, Hkv, w.max_seq_len), dtype=torch.float32, device=dev)
        ds.ds_index_score(shape, inp.qp, inp.label, inp.page_table, inp.seq_lens, scores, stream=stream)
        idx1 = torch.empty((B, Hkv, k), dtype=torch.int32, device=dev)
        idx2 = torch.empty_like(idx1)
        ws1 = torch.empty(ds.ds_topk_workspace_bytes(shape, k), dtype=torch.uint8, device=dev)
        ws2 = torch.empty(ds.ds_topk_sharded_workspace_bytes(shape, k, 4), dtype=torch.uint8, device=dev)
        times = {}
        for name, fn in (("single_pass", lambda: ds.ds_topk_select(shape, scores, inp.seq_lens, k, idx1, ws1,
                                                                    stream=stream)),
                         ("sharded_4", lambda: ds.ds_topk_select_sharded(shape, scores, inp.seq_lens, k, 4, idx2,
                                                                          ws2, stream=stream))):
            for _ in range(5):
                fn()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(50):
                fn()
            e1.record(stream)
            torch.cuda.synchronize()
            times[name] = e0.elapsed_time(e1) * 1e3 / 50
        sharded = {"topk_us": times, "equal": bool(torch.equal(idx1, idx2))}
        del scores, ws1, ws2
    except Exception as e:
        sharded = f"failed: {e}"

    # ---- block-compressed selection (shared index keys only): the compressed
    # keys once, then the block-level decode step keeping top_k / 64 blocks of
    # 64 tokens, L2 flushed before each timed call like the main measurement.
    blocks_rec = None
    if w.label_heads == 1 and k >= 64:
        try:
            kb = k // 64
            bk = torch.empty((inp.num_pages, w.proxy_dim), dtype=torch.bfloat16, device=dev)
            ec = [torch.cuda.Event(enable_timing=True) for _ in range(2)]
            d.flush()
            ec[0].record(stream)
            ds.ds_block_compress(shape, inp.label, inp.page_table, inp.seq_lens, bk, stream=stream)
            ec[1].record(stream)
            blk = torch.empty((B, Hkv, kb), dtype=torch.int32, device=dev)
            bout = torch.empty((B, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device=dev)
            blse = torch.empty((B, w.num_q_heads), dtype=torch.float32, device=dev)
            bws = torch.empty(ds.ds_block_decode_workspace_bytes(shape, kb), dtype=torch.uint8, device=dev)
            bcall = lambda: ds.ds_sparse_decode_blocks(shape, inp.q, inp.qp, bk, inp.k_cache, inp.v_cache,
                                                       inp.k_scale, inp.v_scale, inp.page_table, inp.seq_lens, kb,
                                                       blk, bout, blse, bws, stream=stream)
            for _ in range(5):
                bcall()
            n_b = 50
            eb0 = [torch.cuda.Event(enable_timing=True) for _ in range(n_b)]
            eb1 = [torch.cuda.Event(enable_timing=True) for _ in range(n_b)]
            for i in range(n_b):
                d.flush()
                eb0[i].record(stream)
                bcall()
                eb1[i].record(stream)
            torch.cuda.synchronize()
            if ds.ds_device_errors() != 0:
                raise RuntimeError("device error word set by the block path")
            bt = sorted(a.elapsed_time(b) * 1e3 for a, b in zip(eb0, eb1))
            blocks_rec = {"kept_blocks": kb, "tokens_attended": kb * 64,
                          "us_per_call": sum(bt) / n_b, "calls_per_s": n_b / (sum(bt) * 1e-6),
                          "compress_us": ec[0].elapsed_time(ec[1]) * 1e3,
                          "what": "ds_sparse_decode_blocks: block scores over compressed page keys, exact top-k "
                                  "of blocks, attention over their tokens; compress_us is ds_block_compress of "
                                  "the whole cache, once (a cache-maintenance step, not part of the call)"}
        except Exception as e:  # reported, never hides the main measurement
            blocks_rec = f"failed: {e}"
    return {"cache_append_us": append_us, "sharded_topk": sharded, "block_select": blocks_rec}


# Keys of a workload's record that describe only that workload (the rest of the line is shared).
PER_CONFIG_KEYS = ("value", "unit", "ms_per_step", "step_us", "config", "tokens_per_s", "scanned_tokens_per_s",
                   "step_hbm", "stage_us", "internal_splits", "roofline", "e2e", "clocks", "gpu_launches",
                   "cpu_baseline")


def run_ours(args):
    import top_sparse_decode_label_gb300  # noqa: F401  (fails loudly when the library is missing)

    d = _Device(args)
    head = workload_of(args)
    others = [c for c in also_configs(args) if c != args.config]
    try:
        rec = measure(d, head, args, extras=True)
        torch.cuda.empty_cache()
        per_config = []
        for c in others:
            wc = workload_of(args, c)
            rc = measure(d, wc, args, extras=False)
            per_config.append({key: rc[key] for key in PER_CONFIG_KEYS if key in rc})
            torch.cuda.empty_cache()
    finally:
        d.sampler.stop()

    line = {"metric": METRIC, "value": rec["value"], "unit": "calls/s", "n_gpus": d.world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": rec["ms_per_step"], "step_us": rec["step_us"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic"}
    for key in PER_CONFIG_KEYS + ("block_select", "cache_append_us", "sharded_topk"):
        if key in rec and key not in line:
            line[key] = rec[key]
    line["per_config"] = per_config
    if d.rank == 0:
        print(json.dumps(line), flush=True)
    if d.world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse_args()
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
