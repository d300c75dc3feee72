#!/usr/bin/env python
"""Benchmark: FP8-KV decode attention, 32K context, batch 1, 48 layers, on one GB300.

One step = one decode step of a 48-layer model's attention over an FP8 KV cache: per layer one launch of
ftkv_decode_attn_store, which quantizes the new token's K/V into its slot and runs split-K decode attention
of the BF16 query over all 32,768 keys of that layer's 33,059-row pool (FTKV_DECODE_STABLE_HISTORY: the
history of a layer is not written by the launches before it, so each launch may start loading while the
previous one finishes).  The 48 layers' pools are distinct (1.67 GB, far beyond L2), so every step streams
from HBM.  The step is replayed as one CUDA graph.

Printed (rank 0): ONE JSON line on stdout, value = microseconds per step (lower is better), plus
  roofline     -- algorithmic bytes of the step / graph-timed step time (step level: the launches of a
                  step overlap, so a per-launch time is the step time / 48), against the measured HBM copy
                  bandwidth of MEASURED_PEAKS.json;
  cpu_baseline -- the FP64 C oracle on the host cores (all cores and one thread), timed on a stated
                  bounded sample and scaled to one step;
  e2e          -- the same step through the Python API with pinned host buffers: H2D of the queries
                  and new K/V, the step, D2H of the outputs, synchronized every step;
  clocks       -- nvidia-smi samples taken during the timed region.
Then one "detail" JSON line per other workload on stderr (configs 0, 1, 3, 4, the 40,000-key decode, cold
reconstruct, the BF16-KV comparison, 256-d heads and a sliding window), each with its own roofline and
cpu_baseline; --no-details skips them.  ``--impl reference`` times the oracle alone (the CPU reference arm).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time
from concurrent.futures import ThreadPoolExecutor

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "FP8-KV decode attn us/step and HBM GB/s (% of GB300 peak) at 32K ctx, batch 1"
HQ, HKV, D = 32, 4, 128


def parse_args():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=200)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--context", type=int, default=32768)
    p.add_argument("--pool-rows", type=int, default=33059)
    p.add_argument("--layers", type=int, default=48)
    p.add_argument("--num-splits", type=int, default=0)
    p.add_argument("--no-stable-history", action="store_true",
                   help="do not pass FTKV_DECODE_STABLE_HISTORY (every decode launch waits for the previous one)")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-details", action="store_true", help="headline line only")
    p.add_argument("--details-only", action="store_true", help="detail lines only (no headline)")
    p.add_argument("--no-cpu-baseline", action="store_true", help="skip the oracle timings (profiling runs)")
    p.add_argument("--detail", default="", help="comma-separated detail lines to run (default all): config0, "
                   "config1, config2_40k, bf16kv, d256, window, config3, reconstruct, config4")
    p.add_argument("--cpu-budget-s", type=float, default=20.0, help="bound on the oracle time of a sample")
    return p.parse_args()


# ------------------------------------------------------------------------------------------------
def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d.get("hbm_gbs", 6800.0), d.get("bf16_tflops", 1900.0), "measured"
    return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while the timed region runs."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.file = None

    def __enter__(self):
        self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=self.file, stderr=subprocess.DEVNULL)
        except (FileNotFoundError, OSError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        time.sleep(0.1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        self.file.flush()
        return False

    def summary(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        with open(self.file.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.file.name)
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip() == "Active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------------
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    on_gpu = dist.get_backend() == "nccl"
    t = torch.tensor([value], dtype=torch.float64, device="cuda" if on_gpu else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def decode_bytes_per_layer(n, head_dim=D):
    """Algorithmic bytes of one decode launch attending to n keys (batch 1): K and V codes and scales of every
    key, the slot table, the query and the output, plus the fused store of the new token (its BF16 K/V read,
    its codes and scales written)."""
    codes = n * HKV * head_dim * 2
    scales = n * HKV * 4 * 2
    slots = n * 4
    qo = HQ * head_dim * 2 * 2
    store = HKV * head_dim * 2 * 2 + (HKV * head_dim + HKV * 4) * 2
    return codes + scales + slots + qo + store


# ------------------------------------------------------------------------------------------------
# CPU oracle (the reported baseline and the reference arm): bounded samples, stated, scaled to the metric
def timed_min(fn, reps=2):
    best = None
    for _ in range(reps):
        t0 = time.perf_counter()
        fn()
        dt = time.perf_counter() - t0
        best = dt if best is None else min(best, dt)
    return best


def oracle_threads(n):
    import oracle
    oracle.set_threads(n)
    return oracle.get_threads()


def cpu_decode_layer_fn(context, pool_rows, layer=0):
    """One layer of the batch-1 decode step on the oracle: store of the new token + FP64 decode."""
    import oracle
    from fp8_kv_cache_ftkv_gb300 import inputs
    wl = inputs.decode_long(context, pool_rows, layers=48)
    L = wl.layer(layer)
    op = oracle.Pool(wl.num_rows, HKV, D)
    oracle.store_quant(op, L.k, L.v, L.slots)
    n = context

    def run():
        oracle.store_quant(op, L.k[n - 1:n], L.v[n - 1:n], L.slots[n - 1:n])
        oracle.decode_attn(op, L.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets, wl.sm_scale, HQ)
    return run


SKIP_CPU = False  # --no-cpu-baseline (profiling runs): cpu_baseline is null


def cpu_baseline_scaled(fn, units_in_sample, units_in_metric, unit, sample, budget_s, to_unit=1e6):
    """Time fn (one sample) on all host cores and on one thread (if that takes at most budget_s); scale the
    seconds to the metric's unit (to_unit: 1e6 for microseconds) and from the sample to the metric."""
    if SKIP_CPU:
        return None
    ncores = os.cpu_count() or 1
    cores = oracle_threads(ncores)
    t_all = timed_min(fn)
    single = None
    oracle_threads(1)
    t0 = time.perf_counter()
    fn()  # one single-thread sample only if it is cheap enough
    t1 = time.perf_counter() - t0
    if t1 <= budget_s:
        single = {"value": t1 * to_unit * units_in_metric / units_in_sample, "unit": unit, "cores": 1}
    oracle_threads(ncores)
    return {"value": t_all * to_unit * units_in_metric / units_in_sample, "unit": unit, "cores": cores,
            "kind": "oracle", "sample": sample, "single_thread": single}


def run_reference(args, world, rank):
    """The CPU reference arm: the FP64 oracle's decode step.  Each timed step runs L of the 48 layers in
    full (L = 48 when the whole run fits in ~150 s of oracle time) and is scaled to 48 layers."""
    if rank != 0:
        return
    cores = oracle_threads(os.cpu_count() or 1)
    fns = [cpu_decode_layer_fn(args.context, args.pool_rows, layer=l) for l in range(2)]
    t_layer = timed_min(fns[0], reps=1)
    L = int(max(1, min(args.layers, 150.0 / max(t_layer, 1e-6) / max(args.steps + args.warmup, 1))))
    fns += [cpu_decode_layer_fn(args.context, args.pool_rows, layer=l) for l in range(2, min(L, 48))]
    layer_fns = [fns[l % len(fns)] for l in range(L)]

    def one_step():
        t0 = time.perf_counter()
        for f in layer_fns:
            f()
        return time.perf_counter() - t0
    for _ in range(args.warmup):
        one_step()
    t0 = time.perf_counter()
    times = [one_step() for _ in range(args.steps)]
    wall = time.perf_counter() - t0
    us = statistics.median(times) * 1e6 * args.layers / L
    sample = (f"{L} of {args.layers} layers per timed step (store of the new token + FP64 decode over "
              f"{args.context} keys each, {min(L, 48)} distinct layers), scaled x{args.layers / L:g} to one step")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": us / 1e3, "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"decode_{args.context}_b1_{args.layers}layers", "context": args.context,
                   "batch": 1, "layers": args.layers, "Hq": HQ, "Hkv": HKV, "D": D, "pool_rows": args.pool_rows},
        "timed_region_s": wall,
        "cpu_baseline": {"value": us, "unit": "us/step", "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": us, "unit": "us/step", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


# ------------------------------------------------------------------------------------------------
def to_dev_fn(torch, device):
    return lambda b: torch.from_numpy(np.ascontiguousarray(b).view(np.int16)).view(torch.bfloat16).to(device)


def build_decode(args, torch, ops, inputs, device, context=None, pool_rows=None, head_dim=D, window=0):
    """The headline step (or a variant: head_dim 256, a sliding window) on the FP8 pool."""
    n = context or args.context
    wl = inputs.decode_long(n, pool_rows or args.pool_rows, layers=args.layers)
    wl.head_dim = head_dim
    wl.sm_scale = head_dim ** -0.5
    slots_d = torch.from_numpy(wl.req_to_slot).to(device)
    lens_d = torch.from_numpy(wl.seq_lens).to(device)
    to_dev = to_dev_fn(torch, device)
    # contiguous per-step inputs/outputs (views per layer), so a step's host<->device traffic is 3 copies
    q_all = torch.empty(args.layers, 1, HQ, head_dim, dtype=torch.bfloat16, device=device)
    kv_all = torch.empty(args.layers, 2, 1, HKV, head_dim, dtype=torch.bfloat16, device=device)
    out_all = torch.empty(args.layers, 1, HQ, head_dim, dtype=torch.bfloat16, device=device)
    pools = []
    all_slots = torch.from_numpy(wl.token_slots.astype(np.int32)).to(device)
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for l, L in enumerate(ex.map(wl.layer, range(args.layers))):
            pool = ops.KVPool.empty(wl.num_rows, HKV, device=device, head_dim=head_dim)
            ops.store_quant(pool, to_dev(L.k[:n - 1]), to_dev(L.v[:n - 1]), all_slots[:n - 1])
            pools.append(pool)
            q_all[l].copy_(to_dev(L.q))
            kv_all[l, 0].copy_(to_dev(L.k[n - 1:n]))
            kv_all[l, 1].copy_(to_dev(L.v[n - 1:n]))
    q = [q_all[l] for l in range(args.layers)]
    newk = [kv_all[l, 0] for l in range(args.layers)]
    newv = [kv_all[l, 1] for l in range(args.layers)]
    plan = ops.DecodePlan(HQ, HKV, 1, 1, 1, n, args.num_splits, device, window, head_dim)
    outs = [out_all[l] for l in range(args.layers)]
    torch.cuda.synchronize()

    def step():
        for l in range(args.layers):
            ops.decode_attn(pools[l], q[l], slots_d, lens_d, None, max_seq_len=n, max_q_rows=1, plan=plan,
                            out=outs[l], k_new=newk[l], v_new=newv[l], stable_history=not args.no_stable_history,
                            window=window, sm_scale=wl.sm_scale)

    return dict(step=step, q_all=q_all, kv_all=kv_all, out_all=out_all, plan=plan, pools=pools, n=n, wl=wl)


# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one decode_tok_kernel<4, 128> launch of the 32K
# batch-1 step, from an ncu capture of this kernel on the same launch geometry (4 distinct pools, cold L2); to be
# re-taken whenever the kernel changes.
TOK_TRAFFIC_PER_LAUNCH = 34_821_888


def bf16_bytes_per_layer(n):
    """Algorithmic bytes of one BF16-pool decode launch at n keys (batch 1): K and V rows of every key, the
    slot table, the query and the output, plus the copy of the new token's K/V rows into the pool."""
    return n * HKV * D * 2 * 2 + n * 4 + HQ * D * 2 * 2 + HKV * D * 2 * 2 * 2


def build_decode_bf16(args, torch, ops, inputs, device, context=None, pool_rows=None):
    """The headline step over BF16 pools (the unquantized comparison point): per layer one
    ftkv_decode_attn_bf16 launch that copies the new token into the pool and attends over all n keys."""
    n = context or args.context
    wl = inputs.decode_long(n, pool_rows or args.pool_rows, layers=args.layers)
    slots_d = torch.from_numpy(wl.req_to_slot).to(device)
    lens_d = torch.from_numpy(wl.seq_lens).to(device)
    to_dev = to_dev_fn(torch, device)
    idx = torch.from_numpy(wl.token_slots.astype(np.int64)).to(device)
    pools, q, newk, newv, outs = [], [], [], [], []
    with ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 4)) as ex:
        for L in ex.map(wl.layer, range(args.layers)):
            pool = ops.BF16Pool.empty(wl.num_rows, HKV, device=device)
            pool.k[idx[:n - 1]] = to_dev(L.k[:n - 1])
            pool.v[idx[:n - 1]] = to_dev(L.v[:n - 1])
            pools.append(pool)
            q.append(to_dev(L.q))
            newk.append(to_dev(L.k[n - 1:n]))
            newv.append(to_dev(L.v[n - 1:n]))
            outs.append(torch.empty(1, HQ, D, dtype=torch.bfloat16, device=device))
    plan = ops.DecodePlan(HQ, HKV, 1, 1, 1, n, args.num_splits, device)
    torch.cuda.synchronize()

    def step():
        for l in range(args.layers):
            ops.decode_attn_bf16(pools[l], q[l], slots_d, lens_d, None, max_seq_len=n, max_q_rows=1, plan=plan,
                                 out=outs[l], k_new=newk[l], v_new=newv[l],
                                 stable_history=not args.no_stable_history)

    return dict(step=step, plan=plan, pools=pools, n=n, wl=wl)


def graph_of(torch, stream, work):
    """Run `work` once eagerly (per-device set-up outside capture), then capture it as a CUDA graph."""
    with torch.cuda.stream(stream):
        work()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        work()
    return g


def time_graph(torch, stream, g, steps, warmup, clocks_gpu=None):
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clk = ClockSampler(clocks_gpu) if clocks_gpu is not None else None
    if clk:
        clk.__enter__()
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(steps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    if clk:
        clk.__exit__(None, None, None)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / steps, (clk.summary() if clk else None)


def run_ours(args, world, rank, local):
    import torch
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    from fp8_kv_cache_ftkv_gb300 import build as fbuild
    fbuild.build()
    from fp8_kv_cache_ftkv_gb300 import inputs, ops
    hbm_peak, bf16_peak, peak_src = peaks()
    stream = torch.cuda.Stream(device)

    fp8_ms = None
    if not args.details_only:
        fp8_ms = run_headline(args, world, rank, local, torch, ops, inputs, device, stream, hbm_peak, peak_src)
    if not args.no_details and rank == 0 and world == 1:
        run_details(args, torch, ops, inputs, device, stream, hbm_peak, bf16_peak, peak_src, fp8_ms)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_headline(args, world, rank, local, torch, ops, inputs, device, stream, hbm_peak, peak_src):
    st = build_decode(args, torch, ops, inputs, device)
    graph = graph_of(torch, stream, st["step"])
    barrier(world)
    ms_step, clocks = time_graph(torch, stream, graph, args.steps, args.warmup, clocks_gpu=local)
    ms_step = reduce_max(ms_step, world)
    n = args.context
    layer_bytes = decode_bytes_per_layer(n)
    step_bytes = args.layers * layer_bytes
    achieved = step_bytes / (ms_step * 1e-3) / 1e9

    # ---- e2e through the public API with pinned host buffers ----
    e2e = None
    h2d = args.layers * (HQ * D * 2 + 2 * HKV * D * 2)
    d2h = args.layers * HQ * D * 2
    if not args.no_e2e:
        q_host = st["q_all"].cpu().pin_memory()
        kv_host = st["kv_all"].cpu().pin_memory()
        out_host = torch.empty(st["out_all"].shape, dtype=torch.bfloat16).pin_memory()

        def e2e_step():
            with torch.cuda.stream(stream):
                st["q_all"].copy_(q_host, non_blocking=True)
                st["kv_all"].copy_(kv_host, non_blocking=True)
                graph.replay()
                out_host.copy_(st["out_all"], non_blocking=True)
            stream.synchronize()

        for _ in range(args.warmup):
            e2e_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            e2e_step()
        e2e_us = (time.perf_counter() - t0) / args.steps * 1e6
        e2e_us = reduce_max(e2e_us, world)
        e2e = {"value": e2e_us, "unit": "us/step", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and world == 1 and not SKIP_CPU:
        fn = cpu_decode_layer_fn(n, args.pool_rows)
        cpu = cpu_baseline_scaled(fn, 1, args.layers, "us/step",
                                  f"1 of {args.layers} layers (store of the new token + FP64 decode over {n} keys), "
                                  f"scaled x{args.layers} to one step", args.cpu_budget_s)

    errors = ops.device_errors()
    if rank == 0:
        us = ms_step * 1e3
        print(json.dumps({
            "metric": METRIC, "value": us, "unit": "us/step", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms_step, "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": "e4m3-kv/f16-mma/f32-acc", "data": "synthetic",
            "stable_history": not args.no_stable_history,
            "step": "per layer one launch: fused quantize-on-write of the new token + split-K decode + split merge",
            "config": {"workload": f"decode_{n}_b1_{args.layers}layers", "context": n, "batch": 1,
                       "layers": args.layers, "Hq": HQ, "Hkv": HKV, "D": D, "pool_rows": args.pool_rows,
                       "num_splits": st["plan"].num_splits, "graph": "one CUDA graph per step",
                       "l2": f"inputs larger than L2 ({step_bytes / 1e9:.2f} GB of distinct pools per step)",
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU"},
            "hbm_gbs": achieved, "hbm_frac": achieved / hbm_peak,
            "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm_peak, "unit": "GB/s",
                         "frac": achieved / hbm_peak, "traffic": TOK_TRAFFIC_PER_LAUNCH,
                         "kernel": "decode_tok_kernel<4, 128>",
                         "bytes_per_launch": layer_bytes, "per_launch_us": ms_step * 1e3 / args.layers,
                         "basis": "step level: algorithmic bytes of 48 launches / graph-timed step",
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"},
            "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps * args.layers,
            "clocks": clocks, "device_errors": errors,
        }), flush=True)
    del st, graph
    torch.cuda.empty_cache()
    return ms_step


# ------------------------------------------------------------------------------------------------
def detail_line(name, value, unit, roofline, cpu, extra=None):
    rec = {"detail": name, "value": value, "unit": unit, "higher_is_better": False, "roofline": roofline,
           "cpu_baseline": cpu}
    if extra:
        rec.update(extra)
    print(json.dumps(rec), file=sys.stderr, flush=True)


def hbm_roof(nbytes, ms, peak, src, kernel):
    a = nbytes / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": a, "peak": peak, "unit": "GB/s", "frac": a / peak, "traffic": None,
            "kernel": kernel, "bytes": nbytes, "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)"}


def run_details(args, torch, ops, inputs, device, stream, hbm_peak, bf16_peak, peak_src, fp8_ms=None):
    import oracle
    to_dev = to_dev_fn(torch, device)
    budget = args.cpu_budget_s
    chosen = set(args.detail.split(",")) if args.detail else None

    def want(key):
        return chosen is None or key in chosen
    steps, warm = max(20, args.steps // 4), 5

    # ---- config 0: one decode step, one layer, 512 keys in a 1,024-row pool (latency-dominated) ----
    if want("config0"):
        wl = inputs.decode_small()
        L = wl.layer(0)
        n = int(wl.seq_lens[0])
        pool = ops.KVPool.empty(wl.num_rows, wl.Hkv, device=device)
        ops.store_quant(pool, to_dev(L.k[:n - 1]), to_dev(L.v[:n - 1]), torch.from_numpy(L.slots[:n - 1]).to(device))
        qd, kn, vn = to_dev(L.q), to_dev(L.k[n - 1:n]), to_dev(L.v[n - 1:n])
        r2s, lens = torch.from_numpy(wl.req_to_slot).to(device), torch.from_numpy(wl.seq_lens).to(device)
        plan = ops.DecodePlan(HQ, HKV, 1, 1, 1, n, 0, device)
        out = torch.empty_like(qd)
        g = graph_of(torch, stream, lambda: ops.decode_attn(pool, qd, r2s, lens, None, max_seq_len=n, plan=plan, out=out,
                                                             k_new=kn, v_new=vn))
        ms, clk = time_graph(torch, stream, g, steps, warm)
        op = oracle.Pool(wl.num_rows, wl.Hkv, D)
        oracle.store_quant(op, L.k, L.v, L.slots)
        cpu = cpu_baseline_scaled(lambda: oracle.decode_attn(op, L.q, wl.req_to_slot, wl.seq_lens, wl.q_row_offsets,
                                                             wl.sm_scale, HQ), 1, 1, "us/call", "the whole call", budget)
        detail_line("config0_decode_512_b1", ms * 1e3, "us/call",
                    hbm_roof(decode_bytes_per_layer(n), ms, hbm_peak, peak_src, "decode_tok_kernel<4>"), cpu,
                    {"note": "one launch of 0.56 MB: latency-bound and L2-warm across replays"})
        del pool, g

    # ---- config 1: quantize-on-write, 8,192 tokens x 48 layers into 48 distinct 33,059-row pools ----
    if want("config1"):
        sw = inputs.store(layers=48)
        slots = torch.from_numpy(sw.slots).to(device)
        kv = []
        for l in range(sw.layers):
            k, v = sw.layer(l)
            kv.append((to_dev(k), to_dev(v)))
        pools = [ops.KVPool.empty(sw.num_rows, HKV, device=device) for _ in range(sw.layers)]

        def store_all():
            for (k, v), p in zip(kv, pools):
                ops.store_quant(p, k, v, slots)
        g = graph_of(torch, stream, store_all)
        ms, _ = time_graph(torch, stream, g, steps, warm)
        T = sw.slots.shape[0]
        nbytes = sw.layers * (T * HKV * D * 2 * 2 + T * (HKV * D + HKV * 4) * 2 + T * 4)
        k0, v0 = sw.layer(0)
        op = oracle.Pool(sw.num_rows, HKV, D)
        cpu = cpu_baseline_scaled(lambda: oracle.store_quant(op, k0, v0, sw.slots), 1, sw.layers, "us/step",
                                  f"1 of {sw.layers} layers (8,192 tokens), scaled x{sw.layers}", budget)
        detail_line("config1_store_8192x48", ms * 1e3, "us/step", hbm_roof(nbytes, ms, hbm_peak, peak_src, "store_quant_kernel"),
                    cpu, {"note": "48 distinct destination pools (1.67 GB): the written rows leave L2"})
        del kv, pools, g
        torch.cuda.empty_cache()

    # ---- config 2 at 40,000 keys in 40,290-row pools, 48 layers ----
    if want("config2_40k"):
        st = build_decode(args, torch, ops, inputs, device, context=40000, pool_rows=40290)
        g = graph_of(torch, stream, st["step"])
        ms, _ = time_graph(torch, stream, g, steps, warm)
        fn = cpu_decode_layer_fn(40000, 40290)
        cpu = cpu_baseline_scaled(fn, 1, args.layers, "us/step",
                                  f"1 of {args.layers} layers (store + FP64 decode over 40000 keys), scaled x{args.layers}",
                                  budget)
        detail_line("config2_decode_40000_b1_48layers", ms * 1e3, "us/step",
                    hbm_roof(args.layers * decode_bytes_per_layer(40000), ms, hbm_peak, peak_src, "decode_tok_kernel<4>"),
                    cpu, {"num_splits": st["plan"].num_splits})
        del st, g
        torch.cuda.empty_cache()

    # ---- the BF16-KV comparison point: the headline step (32K keys, batch 1, 48 layers, fused new-token write,
    if want("bf16kv"):
        # stable history) over BF16 pools ----
        st = build_decode_bf16(args, torch, ops, inputs, device)
        g = graph_of(torch, stream, st["step"])
        ms, _ = time_graph(torch, stream, g, steps, warm)
        n = args.context
        wlb = st["wl"]
        Lb = wlb.layer(0)
        hk = np.zeros((wlb.num_rows, HKV, D), np.uint16)
        hv = np.zeros_like(hk)
        hk[Lb.slots] = Lb.k
        hv[Lb.slots] = Lb.v
        cpu = cpu_baseline_scaled(lambda: oracle.decode_attn_bf16(hk, hv, Lb.q, wlb.req_to_slot, wlb.seq_lens,
                                                                  wlb.q_row_offsets, wlb.sm_scale, HQ),
                                  1, args.layers, "us/step",
                                  f"1 of {args.layers} layers (FP64 decode over {n} BF16 keys), scaled x{args.layers}",
                                  budget)
        extra = {"num_splits": st["plan"].num_splits, "kv_bytes_per_token_per_layer": HKV * D * 2 * 2,
                 "fp8_kv_bytes_per_token_per_layer": HKV * D * 2 + HKV * 4 * 2}
        if fp8_ms:
            extra["fp8_us_per_step"] = fp8_ms * 1e3
            extra["bf16_over_fp8_time"] = ms / fp8_ms
        detail_line(f"bf16kv_decode_{n}_b1_{args.layers}layers", ms * 1e3, "us/step",
                    hbm_roof(args.layers * bf16_bytes_per_layer(n), ms, hbm_peak, peak_src, "decode_bf16_kernel<4>"),
                    cpu, extra)
        del st, g, hk, hv, Lb
        torch.cuda.empty_cache()

    # ---- 256-d heads: the headline step with head_dim 256 (the Qwen3.6 full-attention case) ----
    if want("d256"):
        st = build_decode(args, torch, ops, inputs, device, head_dim=256)
        g = graph_of(torch, stream, st["step"])
        ms, _ = time_graph(torch, stream, g, steps, warm)
        n = args.context
        cpu = None
        if not SKIP_CPU:
            wl2 = st["wl"]
            L2 = wl2.layer(0)
            op = oracle.Pool(wl2.num_rows, HKV, 256)
            oracle.store_quant(op, L2.k, L2.v, L2.slots)
            cpu = cpu_baseline_scaled(lambda: oracle.decode_attn(op, L2.q, wl2.req_to_slot, wl2.seq_lens,
                                                                 wl2.q_row_offsets, wl2.sm_scale, HQ),
                                      1, args.layers, "us/step",
                                      f"1 of {args.layers} layers (FP64 decode over {n} 256-d keys), scaled x{args.layers}",
                                      budget)
            del op, L2
        detail_line(f"d256_decode_{n}_b1_{args.layers}layers", ms * 1e3, "us/step",
                    hbm_roof(args.layers * decode_bytes_per_layer(n, 256), ms, hbm_peak, peak_src,
                             "decode_tok_kernel<4,256>"), cpu, {"num_splits": st["plan"].num_splits, "head_dim": 256})
        del st, g
        torch.cuda.empty_cache()

    # ---- sliding window: the headline step attending to the last 4,095 keys (an odd window) ----
    if want("window"):
        W = 4095
        st = build_decode(args, torch, ops, inputs, device, window=W)
        g = graph_of(torch, stream, st["step"])
        ms, _ = time_graph(torch, stream, g, steps, warm)
        cpu = None
        if not SKIP_CPU:
            wl2 = st["wl"]
            L2 = wl2.layer(0)
            op = oracle.Pool(wl2.num_rows, HKV, D)
            oracle.store_quant(op, L2.k, L2.v, L2.slots)
            cpu = cpu_baseline_scaled(lambda: oracle.decode_attn(op, L2.q, wl2.req_to_slot, wl2.seq_lens,
                                                                 wl2.q_row_offsets, wl2.sm_scale, HQ, window=W),
                                      1, args.layers, "us/step",
                                      f"1 of {args.layers} layers (FP64 decode over the last {W} of {args.context} keys), "
                                      f"scaled x{args.layers}", budget)
            del op, L2
        detail_line(f"window{W}_decode_{args.context}_b1_{args.layers}layers", ms * 1e3, "us/step",
                    hbm_roof(args.layers * decode_bytes_per_layer(W), ms, hbm_peak, peak_src, "decode_tok_kernel<4>"),
                    cpu, {"num_splits": st["plan"].num_splits, "window": W,
                          "note": "bytes count the window's keys only: the slices cover nothing else"})
        del st, g
        torch.cuda.empty_cache()

    # ---- config 3: chunked prefill pipeline, one layer: for each of 4 chunks of 2,048 new tokens,
    if want("config3"):
        # reconstruct the FP8 prefix into the BF16 workspace, prefill the chunk, quantize-on-write the chunk ----
        pw = inputs.prefill()
        pool = ops.KVPool.empty(pw.num_rows, HKV, device=device)
        hist = torch.from_numpy(pw.hist_slots).to(device)
        ops.store_quant(pool, to_dev(pw.hist_k), to_dev(pw.hist_v), hist)
        slots_all = torch.from_numpy(np.concatenate([pw.hist_slots, pw.new_slots])).to(device)
        qd, kd, vd = to_dev(pw.q), to_dev(pw.k), to_dev(pw.v)
        H, C = pw.hist_slots.shape[0], pw.chunk
        ws_k = torch.empty(H + 3 * C, HKV, D, dtype=torch.bfloat16, device=device)
        ws_v = torch.empty_like(ws_k)
        outp = torch.empty_like(qd)
        pplan = ops.PrefillPlan(0, device)

        def pipeline():
            for c in range(pw.num_chunks):
                c0, c1 = c * C, (c + 1) * C
                P = H + c0
                ops.reconstruct_bf16(pool, slots_all[:P], ws_k[:P], ws_v[:P])
                ops.prefill_attn(qd[c0:c1], kd[c0:c1], vd[c0:c1], ws_k[:P], ws_v[:P], out=outp[c0:c1], plan=pplan)
                ops.store_quant(pool, kd[c0:c1], vd[c0:c1], slots_all[P:P + C])
        g = graph_of(torch, stream, pipeline)
        ms, _ = time_graph(torch, stream, g, max(10, steps // 4), 3)
        flops = sum((C * (H + c * C) + C * (C + 1) // 2) * HQ * D * 4 for c in range(pw.num_chunks))
        tf = flops / (ms * 1e-3) / 1e12
        # oracle: the same pipeline on every 16th query row of each chunk (attention), full reconstruct and store
        op = oracle.Pool(pw.num_rows, HKV, D)
        oracle.store_quant(op, pw.hist_k, pw.hist_v, pw.hist_slots)
        sall = np.concatenate([pw.hist_slots, pw.new_slots])

        def oracle_pipeline():
            for c in range(pw.num_chunks):
                c0, c1 = c * C, (c + 1) * C
                P = H + c0
                owk, owv = oracle.reconstruct(op, sall[:P])
                oracle.prefill_attn(pw.q[c0:c1], pw.k[c0:c1], pw.v[c0:c1], owk, owv, pw.sm_scale,
                                    np.arange(0, C, 16, dtype=np.int64))
                oracle.store_quant(op, pw.k[c0:c1], pw.v[c0:c1], sall[P:P + C])
        cpu = cpu_baseline_scaled(oracle_pipeline, 1, 1, "us/pipeline",
                                  "every 16th query row of each chunk (all heads), full reconstruct and store; not scaled",
                                  budget)
        detail_line("config3_chunked_prefill_4x2048_over_8192", ms * 1e3, "us/pipeline",
                    {"bound": "tensor", "achieved": tf, "peak": bf16_peak, "unit": "TFLOP/s", "frac": tf / bf16_peak,
                     "traffic": None, "kernel": "prefill_tc2_kernel (+ reconstruct, store)", "flops": flops,
                     "peak_source": f"{peak_src} (MEASURED_PEAKS.json bf16_tflops, burst)"}, cpu,
                    {"note": "4 x (reconstruct -> prefill -> store) in one graph; flops count causal pairs only"})
        del pool, g, ws_k, ws_v
        torch.cuda.empty_cache()

    # ---- reconstruct, cold: 8 distinct pools of 14,336 prefix rows into 8 distinct workspaces ----
    if want("reconstruct"):
        pw = inputs.prefill()
        P = pw.hist_slots.shape[0] + 3 * pw.chunk  # the last chunk's prefix: 14,336 rows
        rk, rv = inputs.kv_tokens(np.random.default_rng(5), P, 1.0)
        rslots = torch.from_numpy(np.random.default_rng(6).permutation(pw.num_rows)[:P].astype(np.int32)).to(device)
        rpools = []
        for _ in range(8):
            p = ops.KVPool.empty(pw.num_rows, HKV, device=device)
            ops.store_quant(p, to_dev(rk), to_dev(rv), rslots)
            rpools.append(p)
        wss = [(torch.empty(P, HKV, D, dtype=torch.bfloat16, device=device),
                torch.empty(P, HKV, D, dtype=torch.bfloat16, device=device)) for _ in range(8)]

        def recon_all():
            for p, (a, b) in zip(rpools, wss):
                ops.reconstruct_bf16(p, rslots, a, b)
        g = graph_of(torch, stream, recon_all)
        ms, _ = time_graph(torch, stream, g, steps, warm)
        nbytes = 8 * (P * (HKV * D + HKV * 4) * 2 + P * 4 + P * HKV * D * 2 * 2)
        op = oracle.Pool(pw.num_rows, HKV, D)
        oracle.store_quant(op, rk, rv, rslots.cpu().numpy())
        rs = rslots.cpu().numpy()
        cpu = cpu_baseline_scaled(lambda: oracle.reconstruct(op, rs), 1, 8, "us/iter", "1 of 8 pools, scaled x8", budget)
        detail_line("reconstruct_14336_rows_x8_cold", ms * 1e3, "us/iter",
                    hbm_roof(nbytes, ms, hbm_peak, peak_src, "reconstruct_kernel"), cpu,
                    {"note": "8 distinct pools and workspaces per iteration (0.5 GB): cold in L2"})
        del rpools, wss, g
        torch.cuda.empty_cache()

    # ---- config 4: batched multi-row decode, 64 requests, 1-8 rows, 2,000,000-row pool, one launch ----
    if want("config4"):
        bw = inputs.decode_batched()
        Lb = bw.layer(0)
        pool = ops.KVPool.empty(bw.num_rows, HKV, device=device)
        ops.store_quant(pool, to_dev(Lb.k), to_dev(Lb.v), torch.from_numpy(Lb.slots).to(device))
        qd = to_dev(Lb.q)
        r2s = torch.from_numpy(bw.req_to_slot).to(device)
        lens = torch.from_numpy(bw.seq_lens).to(device)
        offs = torch.from_numpy(bw.q_row_offsets).to(device)
        mq = int(np.diff(bw.q_row_offsets).max())
        stride = int(bw.req_to_slot.shape[1])
        plan = ops.DecodePlan(HQ, HKV, len(bw.seq_lens), int(bw.q_row_offsets[-1]), mq, stride, 0, device)
        out = torch.empty_like(qd)
        g = graph_of(torch, stream, lambda: ops.decode_attn(pool, qd, r2s, lens, offs, max_seq_len=stride,
                                                            max_q_rows=mq, plan=plan, out=out))
        ms, _ = time_graph(torch, stream, g, max(10, steps // 4), 3)
        keys = int(bw.seq_lens.sum())
        rows = int(bw.q_row_offsets[-1])
        nbytes = keys * (HKV * D * 2 + HKV * 4 * 2 + 4) + rows * HQ * D * 2 * 2
        op = oracle.Pool(bw.num_rows, HKV, D)
        sample_req = [0, 1, 2, 3]
        sub = np.concatenate([bw.req_to_slot[b, :bw.seq_lens[b]] for b in sample_req])
        starts = np.concatenate([[0], np.cumsum(bw.seq_lens)[:-1]])
        tok = np.concatenate([np.arange(starts[b], starts[b] + bw.seq_lens[b]) for b in sample_req])
        oracle.store_quant(op, Lb.k[tok], Lb.v[tok], sub)
        qrows = np.concatenate([np.arange(bw.q_row_offsets[b], bw.q_row_offsets[b + 1]) for b in sample_req])
        offs_s = np.concatenate([[0], np.cumsum(np.diff(bw.q_row_offsets)[sample_req])]).astype(np.int32)
        s_keys = int(bw.seq_lens[sample_req].sum())
        del Lb
        cpu = cpu_baseline_scaled(lambda: oracle.decode_attn(op, qd.view(torch.int16).cpu().numpy().view(np.uint16)[qrows],
                                                             bw.req_to_slot[sample_req], bw.seq_lens[sample_req], offs_s,
                                                             bw.sm_scale, HQ),
                                  s_keys, keys, "us/launch",
                                  f"requests {sample_req} ({s_keys} keys, all their rows), scaled by keys to all 64", budget)
        detail_line("config4_batched_multirow_64req", ms * 1e3, "us/launch",
                    hbm_roof(nbytes, ms, hbm_peak, peak_src, "decode_mr_kernel"), cpu,
                    {"keys": keys, "rows": rows, "num_splits": plan.num_splits})
        del pool, g
        torch.cuda.empty_cache()


def main():
    global SKIP_CPU
    args = parse_args()
    SKIP_CPU = args.no_cpu_baseline
    world, rank, local = dist_setup()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
