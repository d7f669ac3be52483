#!/usr/bin/env python
"""Mixed-step attention throughput on GB300: tokens/s and fraction of the step roofline.

One timed step is one pass of the whole hot path -- ms_mixed_step: the append
(ms_kv_append_rope) then the attention (ms_mixed_step_attention_ragged) in one
call -- over every batch of a workload.  By default all four
full-size workloads run one after another and print ONE JSON line: its top level
is the largest single-GPU step, the long-context bimodal batch (the last
4096-token chunk of a 32768-token prompt next to 512 decodes, 10 % of them at
64K-128K keys; 21 GB of KV read per step), and ``per_config`` carries the 7B MHA
(budget 512, nine batches per step), 13B MHA (budget 2048) and 8B GQA (budget
8192) steps with the same fields: value, ms_per_step, roofline (with the DRAM
traffic of a committed ncu capture of the current source), step_roofline, e2e
and cpu_baseline.  Inputs are seeded synthetic bf16 (N(0,1)); every KV pool is
larger than L2, so no flush is needed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config all|NAME] [--impl ours|reference]
  python bench.py --timeline | --split   (supplementary: step-latency timeline; decode/chunk split)

Under torchrun each rank runs its own replica (weak scaling); timing is the
max over ranks.  --impl reference times the fp64 CPU oracle on the bounded
sample of the top-level workload that cpu_baseline also times (same rule, same
--steps and --warmup), on one thread, and adds the same path over every host core.
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
import types

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
# the CPU oracle runs single-threaded (its reported core count is 1)
for _var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_var, "1")

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "mixed-step attention tokens/s on 1 GB300; % of step roofline (HBM GB/s | TFLOP/s)"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


# ---------------------------------------------------------------------------- distributed helpers

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def dist_init(backend: str):
    import torch.distributed as dist
    if not dist.is_initialized():
        dist.init_process_group(backend=backend)
    return dist


def reduce_max(value: float, dist=None, device=None) -> float:
    """Max of a float over ranks (identity without a process group)."""
    if dist is None or not dist.is_initialized():
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, dist=None, device=None) -> float:
    if dist is None or not dist.is_initialized():
        return value
    import torch
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


# ---------------------------------------------------------------------------- workload

def load_workload(name: str):
    wls = workloads.CONFIGS[name]()
    return wls if isinstance(wls, list) else [wls]


def describe(name: str, wls) -> str:
    wl = wls[0]
    n_dec = sum(1 for r in wl.requests if r.remaining == 0)
    return (f"{name}: H_q {wl.H_q}, H_kv {wl.H_kv}, D {wl.D}, page 16, budget {wl.token_budget}, "
            f"{n_dec} decodes + prefill chunk(s), {len(wls)} batch(es) per step")


def captured_traffic(config: str):
    """DRAM bytes of one captured batch (the append launch and the attention kernel), if every
    kernel source the capture lists still matches it."""
    import hashlib
    path = os.path.join(ROOT, "profiles", f"attention_kernel_{config}.traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f)
        for src, sha in rec["sources"].items():
            with open(os.path.join(ROOT, src), "rb") as f:
                if hashlib.sha256(f.read()).hexdigest() != sha:
                    return None  # a kernel changed since the counters were taken
    except (OSError, KeyError, ValueError, AttributeError):
        return None
    return rec


def read_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "bf16_tflops": float(d["bf16_tflops"]),
                "bf16_tflops_sustained": float(d.get("bf16_tflops_sustained", d["bf16_tflops"]))}, "measured"
    except (OSError, KeyError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


class ClockSampler:
    """nvidia-smi clock/throttle sampling in the background."""
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join(tempfile.gettempdir(), f"ms_bench_clocks_gpu{gpu_index}_{os.getpid()}.csv")

    def start(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"], stdout=self.fh,
                                         stderr=subprocess.DEVNULL)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.fh.close()
        sm, mx, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                    power.append(float(parts[3]))
                except ValueError:
                    continue
                for nm, val in zip(names, parts[5:9]):
                    if val.lower() == "active":
                        reasons.add(nm)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        load = [s for s, p in zip(sm, power) if p > 200.0] or sm
        return {"sm_mhz": statistics.median(load), "sm_max_mhz": max(mx), "samples": len(sm),
                "reasons": sorted(reasons)}


# ---------------------------------------------------------------------------- our arm

ALL_CONFIGS = ["long_bimodal_b4608", "mha7b_b512", "mha13b_b2048", "gqa8b_b8192"]


def config_block(name: str, wls, world: int) -> dict:
    """The ``config`` object of a line: the same for both arms (nothing in it is measured)."""
    wl0 = wls[0]
    pool_gb = 2 * wl0.num_pages * wl0.H_kv * wl0.page_size * wl0.D * 2 / 1e9
    tokens = 0
    for wl in wls:
        n_dec = sum(1 for r in wl.requests if r.remaining == 0)
        tokens += min(wl.token_budget, n_dec + sum(r.remaining for r in wl.requests if r.remaining > 0))
    return {"workload": describe(name, wls), "tokens_per_step": tokens, "batches_per_step": len(wls),
            "l2": f"inputs larger than L2 (KV pool {pool_gb:.2f} GB); no flush", "parallelism": f"replicas x{world}"}


def run_ours(args, world, rank, local):
    import torch

    import chunked_prefill_mixed_decode_gb300 as ms
    from chunked_prefill_mixed_decode_gb300 import build as msbuild

    msbuild.build()
    dist = None
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    if world > 1:
        dist = dist_init("nccl")
    names = ALL_CONFIGS if args.config == "all" else [args.config]
    results = {}
    for name in names:
        results[name] = measure_config(name, args, ms, world, rank, device, dist)
        torch.cuda.empty_cache()
    top = dict(results[names[0]])
    if len(names) > 1:
        top["per_config"] = {n: {k: v for k, v in results[n].items() if k not in ("metric", "n_gpus", "steps",
                                 "warmup", "higher_is_better", "scaling", "vs_baseline", "dtype", "data")}
                             for n in names[1:]}
    if rank == 0:
        print(json.dumps(top), flush=True)
    if dist is not None:
        dist.barrier()
        dist.destroy_process_group()


def measure_config(name, args, ms, world, rank, device, dist) -> dict:
    """Device time, roofline, end-to-end rate and CPU baseline of one workload."""
    import torch

    from chunked_prefill_mixed_decode_gb300 import roofline, step

    wls = load_workload(name)
    wl0 = wls[0]
    peaks, peak_src = read_peaks()

    # ---- setup (untimed): metadata, device buffers, one shared KV pool
    subs = []
    pool = workloads.kv_pool(wl0, 1000 + rank, device)
    max_pos = max(wl.max_pos for wl in wls) + 1
    cos, sin = step.rope_tables_device(max_pos, wl0.D, device)
    for i, wl in enumerate(wls):
        states = [(r.cached_len, r.remaining) for r in wl.requests]
        tables = [r.block_table for r in wl.requests]
        meta = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk, ragged=True)
        batch = step.to_device(meta, device)
        T = meta["num_tokens"]
        q, k, v = workloads.step_tensors(wl, T, 50 + i + 1000 * rank, device)
        rows = [(int(meta["q_start_pos"][s]), int(meta["cu_seqlens_q"][s + 1] - meta["cu_seqlens_q"][s]))
                for s in range(meta["num_rows"])]
        counts = roofline.step_counts(rows, wl.H_q, wl.H_kv, wl.D)
        subs.append(dict(wl=wl, states=states, tables=tables, meta=meta, batch=batch, q=q, k=k, v=v,
                         q_rot=torch.empty_like(q), out=torch.empty_like(q), counts=counts))
    ws_bytes = max(ms.attention_workspace_size(max(s["meta"]["num_rows"], 1), max(s["meta"]["num_tokens"], 1),
                                               s["batch"].context_total, wl0.H_q, wl0.H_kv, wl0.D) for s in subs)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=device)
    status = torch.zeros(1, dtype=torch.int32, device=device)
    stream = torch.cuda.current_stream(device)
    k_cache, v_cache = pool

    def one_step(events=None):
        # a batch's events bracket its step call (append, then attention, whose kernels
        # launch as programmatic dependents of the append's)
        for j, s in enumerate(subs):
            b = s["batch"]
            if events is not None:
                events[j][0].record(stream)
            step.run_step(s["q"], s["k"], s["v"], b, cos, sin, k_cache, v_cache, s["out"], ws, q_rot=s["q_rot"],
                          dev_status=status, stream=stream)
            if events is not None:
                events[j][1].record(stream)

    for _ in range(args.warmup):
        one_step()
    torch.cuda.synchronize()
    if ms.read_status(status) or ms.read_status(ws):
        raise RuntimeError(f"{name}: device status set during warm-up")

    # ---- timed device region
    n_sub = len(subs)
    attn_events = [[(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                    for _ in range(n_sub)] for _ in range(args.steps)]
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    sampler = ClockSampler(device.index if "CUDA_VISIBLE_DEVICES" not in os.environ else device.index)
    sampler.start()
    if dist is not None:
        dist.barrier()
    torch.cuda.synchronize()
    t0.record(stream)
    for it in range(args.steps):
        one_step(attn_events[it])
    t1.record(stream)
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    clocks = sampler.stop()
    elapsed_ms = t0.elapsed_time(t1)
    if ms.read_status(status) or ms.read_status(ws):
        raise RuntimeError(f"{name}: device status set during the timed region")
    attn_ms = [[attn_events[it][j][0].elapsed_time(attn_events[it][j][1]) for it in range(args.steps)]
               for j in range(n_sub)]
    tokens_per_step = sum(s["meta"]["num_tokens"] for s in subs)
    max_ms = reduce_max(elapsed_ms, dist, device)
    total_tokens = reduce_sum(tokens_per_step * args.steps, dist, device)
    value = total_tokens / (max_ms / 1e3)
    ms_per_step = max_ms / args.steps

    # ---- roofline of one batch of the path (append + attention call: the dominant, and only,
    # launch group; 4 launches) and of the whole step
    grp_bytes = sum(s["counts"]["step_bytes"] for s in subs)
    attn_flops = sum(s["counts"]["flops"] for s in subs)
    grp_avg_ms = sum(statistics.mean(a) for a in attn_ms) / n_sub  # mean over batches of the mean duration
    grp_bytes_avg = grp_bytes / n_sub
    flops_avg = attn_flops / n_sub
    t_mem = grp_bytes_avg / (peaks["hbm_gbs"] * 1e9)
    t_flop = flops_avg / (peaks["bf16_tflops_sustained"] * 1e12)
    if t_mem >= t_flop:
        achieved = grp_bytes_avg / (grp_avg_ms / 1e3) / 1e9
        roof = {"bound": "hbm", "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(achieved / peaks["hbm_gbs"], 4), "traffic": None}
    else:
        achieved = flops_avg / (grp_avg_ms / 1e3) / 1e12
        roof = {"bound": "tensor", "achieved": round(achieved, 1), "peak": peaks["bf16_tflops_sustained"],
                "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_tflops_sustained"], 4), "traffic": None}
    cap = captured_traffic(name)
    if cap is not None and "append_dram_bytes" in cap:
        # scale the captured batch's DRAM bytes (append + attention) to the average batch
        b = int(cap.get("batch", 0))
        scale = grp_bytes_avg / subs[b]["counts"]["step_bytes"]
        roof["traffic"] = int((cap["dram_bytes_read"] + cap["dram_bytes_write"] + cap["append_dram_bytes"]) * scale)
        roof["traffic_source"] = (f"ncu capture of batch {b} (append + attention kernels)"
                                  + (", scaled by algorithmic bytes" if n_sub > 1 else ""))
        roof["traffic_vs_alg_bytes"] = round(roof["traffic"] / grp_bytes_avg, 4)
    roof["kernel"] = ("one batch of the path: ms_mixed_step (the append with the prologue in its launch, "
                      "then the persistent attention_kernel)")
    roof["peak_source"] = (f"{peak_src} ({'MEASURED_PEAKS.json' if peak_src == 'measured' else 'recipe fallback'})"
                           + ("; sustained bf16 (kernel timed inside a step)" if roof["bound"] == "tensor" else ""))
    all_ms = [t for a in attn_ms for t in a]
    roof["per_launch"] = {"alg_bytes": int(grp_bytes_avg), "alg_flops": int(flops_avg),
                          "avg_ms": round(grp_avg_ms, 4), "median_ms": round(statistics.median(all_ms), 4),
                          "min_ms": round(min(all_ms), 4)}
    step_bytes = sum(s["counts"]["step_bytes"] for s in subs)
    step_flops = attn_flops
    t_roof = max(step_bytes / (peaks["hbm_gbs"] * 1e9), step_flops / (peaks["bf16_tflops_sustained"] * 1e12))
    step_roof = {"alg_bytes": int(step_bytes), "alg_flops": int(step_flops),
                 "t_roof_ms": round(t_roof * 1e3, 4), "t_meas_ms": round(ms_per_step, 4),
                 "frac_of_roofline": round(t_roof * 1e3 / ms_per_step, 4),
                 "bound": "hbm" if step_bytes / (peaks["hbm_gbs"] * 1e9) >= step_flops / (
                     peaks["bf16_tflops_sustained"] * 1e12) else "tensor",
                 "vs_nominal_8TBps": round(step_bytes / (8000e9) * 1e3 / ms_per_step, 4)}

    # ---- end to end through the public API with host buffers
    e2e = run_e2e(args, ms, step, subs, cos, sin, k_cache, v_cache, ws, status, device, stream, dist)

    line = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms_per_step, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded N(0,1) bf16; KV pool larger than L2)",
        "config": config_block(name, wls, world),
        "roofline": roof, "step_roofline": step_roof, "e2e": e2e,
        # per batch: the append with the prologue in its launch (one kernel on steps of at most
        # FUSED_STEP_MAX_ROWS rows, else two), then the persistent attention kernel
        "gpu_launches": sum(2 if s["meta"]["num_rows"] <= ms.FUSED_STEP_MAX_ROWS else 3 for s in subs) * args.steps,
        "clocks": clocks,
    }
    del subs, ws, pool, k_cache, v_cache
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(name, args)
    return line


def run_e2e(args, ms, step, subs, cos, sin, k_cache, v_cache, ws, status, device, stream, dist):
    """Same metric through the public API from host buffers, pipelined as a serving loop would be:
    every step, per batch, the C++ scheduler builds the metadata on the host, which goes H2D in one
    packed copy with q/k/v from pinned memory; the output comes back D2H.  Uploads, compute and
    downloads run on three streams ordered by events, with two device slots per batch, so step s + 1
    uploads while step s computes and step s - 1 downloads; the timed region ends with a full sync
    after the last step's download."""
    import torch
    host = []
    for s in subs:
        host.append(dict(q=s["q"].cpu().pin_memory(), k=s["k"].cpu().pin_memory(), v=s["v"].cpu().pin_memory(),
                         out=torch.empty_like(s["out"], device="cpu").pin_memory()))
    # two device slots per batch: its inputs, q_rot and output
    slots = [[dict(q=s["q"], k=s["k"], v=s["v"], q_rot=s["q_rot"], out=s["out"]),
              dict(q=torch.empty_like(s["q"]), k=torch.empty_like(s["k"]), v=torch.empty_like(s["v"]),
                   q_rot=torch.empty_like(s["q_rot"]), out=torch.empty_like(s["out"]))] for s in subs]
    n = max(1, min(args.steps, args.e2e_steps))
    up, down = torch.cuda.Stream(device), torch.cuda.Stream(device)
    stagers = [step.MetaStager(s["meta"]["num_rows"], s["meta"]["num_tokens"],
                               s["meta"]["num_rows"] + 1 + int(s["meta"]["bt_offsets"][-1]), device) for s in subs]
    computed = [[None, None] for _ in subs]  # compute of the slot's last step: its inputs are free after it
    fetched = [[None, None] for _ in subs]   # download of the slot's last output: the slot's out is free after it
    counter = {"step": 0, "h2d": 0, "d2h": 0}

    def e2e_step():
        h2d = d2h = 0
        par = counter["step"] & 1
        for i, (s, hb) in enumerate(zip(subs, host)):
            wl = s["wl"]
            sl = slots[i][par]
            meta = ms.build_batch_metadata(s["states"], s["tables"], wl.token_budget, wl.max_chunk, ragged=True)
            if computed[i][par] is not None:
                up.wait_event(computed[i][par])
            b = stagers[i].stage(meta, up)
            with torch.cuda.stream(up):
                sl["q"].copy_(hb["q"], non_blocking=True)
                sl["k"].copy_(hb["k"], non_blocking=True)
                sl["v"].copy_(hb["v"], non_blocking=True)
                ready = torch.cuda.Event()
                ready.record(up)
            stream.wait_event(ready)
            if fetched[i][par] is not None:
                stream.wait_event(fetched[i][par])
            step.run_step(sl["q"], sl["k"], sl["v"], b, cos, sin, k_cache, v_cache, sl["out"], ws, q_rot=sl["q_rot"],
                          dev_status=status, stream=stream)
            fin = torch.cuda.Event()
            fin.record(stream)
            computed[i][par] = fin
            down.wait_event(fin)
            with torch.cuda.stream(down):
                hb["out"].copy_(sl["out"], non_blocking=True)
                got = torch.cuda.Event()
                got.record(down)
            fetched[i][par] = got
            h2d += b.h2d_bytes + (sl["q"].numel() + sl["k"].numel() + sl["v"].numel()) * 2
            d2h += sl["out"].numel() * 2
        counter["step"] += 1
        counter["h2d"], counter["d2h"] = h2d, d2h

    for _ in range(2):
        e2e_step()
    torch.cuda.synchronize()
    if dist is not None:
        dist.barrier()
    t = time.perf_counter()
    for _ in range(n):
        e2e_step()
    torch.cuda.synchronize()
    el = time.perf_counter() - t
    el = reduce_max(el, dist, device)
    tokens = reduce_sum(sum(s["meta"]["num_tokens"] for s in subs) * n, dist, device)
    return {"value": round(tokens / el, 1), "unit": "tokens/s", "h2d_bytes_per_step": int(counter["h2d"]),
            "d2h_bytes_per_step": int(counter["d2h"]), "steps": n,
            "pipeline": "3 streams, 2 device slots per batch; full sync after the last step"}


# ---------------------------------------------------------------------------- oracle (CPU) timing
#
# Both arms time the oracle on the same sample of a workload: its first batch, with its decodes taken
# evenly spaced in input order (so a bimodal mix keeps its shape) and each chunk row cut to its first
# tokens, scaled by one fraction f.  f is the largest value whose estimated oracle time fits the
# per-step budget, from a fixed cost model (seconds per gathered key per KV head, and per key per
# (token, head) pair) -- no timing probe -- so both arms pick the same sample for the same --steps and
# --warmup.  The budget is about two minutes over the reference arm's warm-up and timed steps.

ORACLE_S_PER_GATHERED_KEY = 1.5e-6   # one KV head, D = 128: page gather + fp64 conversion of K and V
ORACLE_S_PER_ATTENDED_KEY = 2.0e-7   # one (token, head) pair, D = 128: scores, exponentials, weighted sum


def _oracle_sample_states(wl, f_dec: float, f_chunk: float):
    dec = [r for r in wl.requests if r.remaining == 0]
    prm = [r for r in wl.requests if r.remaining > 0]
    n_dec = min(len(dec), max(1, int(round(len(dec) * f_dec)))) if dec else 0
    picked = [dec[(i * len(dec)) // n_dec] for i in range(n_dec)] if n_dec else []
    left = wl.token_budget - len(dec)
    chunks = []
    for r in prm:  # the chunk rows the full step schedules, each cut to its first tokens
        take = min(r.remaining, left)
        if take <= 0:
            break
        left -= take
        chunks.append((r, min(take, max(2, int(round(take * f_chunk))))))
    return picked, chunks


def _oracle_cost(wl, picked, chunks) -> float:
    scale = wl.D / 128.0
    t = 0.0
    for r in picked:
        keys = r.cached_len + 1
        t += keys * (wl.H_kv * ORACLE_S_PER_GATHERED_KEY + wl.H_q * ORACLE_S_PER_ATTENDED_KEY) * scale
    for r, n in chunks:
        t += (r.cached_len + n) * wl.H_kv * ORACLE_S_PER_GATHERED_KEY * scale
        t += n * wl.H_q * (r.cached_len + (n + 1) / 2) * ORACLE_S_PER_ATTENDED_KEY * scale
    return t


def _largest_fraction(cost, budget: float) -> float:
    """Largest f in (0, 1] with cost(f) <= budget (bisection; the smallest sample if none fits)."""
    if cost(1.0) <= budget:
        return 1.0
    lo, hi = 0.0, 1.0
    for _ in range(30):
        mid = (lo + hi) / 2
        if cost(mid) <= budget:
            lo = mid
        else:
            hi = mid
    return max(lo, 1e-9)


def oracle_sample(config: str, steps: int, warmup: int, step_seconds: float = 0.0):
    """(sample workload, description) of the bounded oracle step for this workload and run length.
    Decodes and chunk tokens each get half of the per-step budget (all of it when the step has
    only one kind).  step_seconds > 0 overrides the budget derived from steps + warmup."""
    wl = load_workload(config)[0]
    budget = step_seconds if step_seconds > 0 else min(8.0, max(0.5, 120.0 / max(steps + warmup, 1)))
    has_dec = any(r.remaining == 0 for r in wl.requests)
    has_chunk = any(r.remaining > 0 for r in wl.requests)
    share = budget / 2 if has_dec and has_chunk else budget
    f_dec = _largest_fraction(lambda f: _oracle_cost(wl, _oracle_sample_states(wl, f, 0.0)[0], []), share)
    f_chk = _largest_fraction(lambda f: _oracle_cost(wl, [], _oracle_sample_states(wl, 0.0, f)[1]), share)
    picked, chunks = _oracle_sample_states(wl, f_dec, f_chk)
    states = [(r.cached_len, 0) for r in picked] + [(r.cached_len, n) for r, n in chunks]
    rng = np.random.default_rng(8)
    reqs, total = workloads.assign_pages(states, rng)
    n_tok = len(picked) + sum(n for _, n in chunks)
    sub = workloads.Workload(wl.name + "_sample", wl.H_q, wl.H_kv, wl.D, n_tok, reqs, total, seed=8)
    long_dec = sum(1 for r in picked if r.cached_len >= 65536)
    desc = (f"{len(picked)} decodes taken evenly from the first batch's {sum(1 for r in wl.requests if r.remaining == 0)}"
            + (f" ({long_dec} of them 64K+)" if long_dec else "")
            + f" + {', '.join(f'{n} tokens of the chunk at c = {r.cached_len}' for r, n in chunks) or 'no chunk'}"
            + f", all {wl.H_q} heads (estimated {_oracle_cost(wl, picked, chunks):.2f} s per step)")
    return sub, desc


def _oracle_prepare(sub, seed):
    """Seeded inputs of one sampled step, as the oracle takes them (bf16 bit arrays)."""
    states = [(r.cached_len, r.remaining) for r in sub.requests]
    tables = [r.block_table for r in sub.requests]
    q, k, v = workloads.step_tensors(sub, sub.token_budget, seed, "cpu")
    kc, vc = workloads.kv_pool(sub, seed, "cpu")
    return dict(sub=sub, states=states, tables=tables, q=workloads.bf16_bits(q), k=workloads.bf16_bits(k),
                v=workloads.bf16_bits(v), kp=workloads.bf16_bits(kc), vp=workloads.bf16_bits(vc))


def _oracle_front(prep):
    """Schedule, metadata and the RoPE append of the sampled step (the oracle's own order)."""
    import oracle
    sub = prep["sub"]
    rows, _ = oracle.schedule(prep["states"], sub.token_budget)
    meta = oracle.batch_metadata(rows, prep["tables"], len(prep["states"]))
    T = meta["num_tokens"]
    q_rot, kp2, vp2 = oracle.kv_append(prep["q"][:T], prep["k"][:T], prep["v"][:T], meta["positions"],
                                       meta["slot_mapping"], prep["kp"], prep["vp"])
    return meta, T, q_rot, kp2, vp2


def _oracle_run(prep):
    """Time the oracle's whole path (schedule, metadata, append, attention) on one sampled step."""
    import oracle
    t = time.perf_counter()
    meta, T, q_rot, kp2, vp2 = _oracle_front(prep)
    oracle.attention_all(q_rot, kp2, vp2, meta, prep["sub"].H_kv)
    return T, time.perf_counter() - t


# all-cores leg: the same oracle functions over (row, KV head) blocks in worker processes (spawned:
# never forked from a process that holds a CUDA context).  The step's inputs -- q, k, v and the
# cached pools, resident like the GPU's HBM copy -- are written once, untimed, to .npy files the
# workers memory-map.  Per run the parent schedules and builds the metadata; each block appends its
# row's new tokens for one KV head into a copy of that row's pages (oracle.kv_append) and attends a
# share of the row's (token, head) pairs (oracle.attention_rows).
_W = {}


def _worker_attend(args):
    import oracle
    path, t0, t1, c0, table, positions, kvh, G, tokens = args
    if _W.get("path") != path:
        _W.clear()
        _W["path"] = path
        _W.update({k: np.load(os.path.join(path, k + ".npy"), mmap_mode="r") for k in ("q", "k", "v", "kp", "vp")})
    n = len(table)
    mk = np.ascontiguousarray(_W["kp"][table, kvh:kvh + 1])
    mv = np.ascontiguousarray(_W["vp"][table, kvh:kvh + 1])
    # in the copy, logical page i of the row is page i, so a token's slot is its position
    q_rot, mk, mv = oracle.kv_append(np.asarray(_W["q"][t0:t1, kvh * G:(kvh + 1) * G]),
                                     np.asarray(_W["k"][t0:t1, kvh:kvh + 1]), np.asarray(_W["v"][t0:t1, kvh:kvh + 1]),
                                     positions, positions, mk, mv)
    meta = {"cu_seqlens_q": np.array([0, t1 - t0]), "q_start_pos": np.array([c0]),
            "block_tables": np.arange(n)[None, :]}
    res = oracle.attention_rows(q_rot, mk, mv, meta, 1, select=[(t - t0, h) for t in tokens for h in range(G)])
    return len(res)


def _oracle_run_parallel(prep, pool, n_workers, tmpdir):
    """The oracle's path with its append and attention spread over worker processes."""
    import oracle
    t = time.perf_counter()
    sub = prep["sub"]
    rows, _ = oracle.schedule(prep["states"], sub.token_budget)
    meta = oracle.batch_metadata(rows, prep["tables"], len(prep["states"]))
    T = meta["num_tokens"]
    H_q, H_kv = prep["q"].shape[1], sub.H_kv
    G = H_q // H_kv
    cu, c0, bt = meta["cu_seqlens_q"], meta["q_start_pos"], meta["block_tables"]
    tasks = []
    per_block = max(1, -(-T * H_kv // (4 * n_workers)))  # about four blocks of (token, KV head) per worker
    for s in range(meta["num_rows"]):
        a, b = int(cu[s]), int(cu[s + 1])
        table = bt[s][: -(-(int(c0[s]) + b - a) // 16)].astype(np.int64)
        pos = meta["positions"][a:b]
        for kvh in range(H_kv):
            for x in range(a, b, per_block):
                tasks.append((tmpdir, a, b, int(c0[s]), table, pos, kvh, G, list(range(x, min(b, x + per_block)))))
    tasks.sort(key=lambda tk: -(tk[3] + tk[2] - tk[1]) * len(tk[8]))  # longest first
    n = sum(pool.map(_worker_attend, tasks, chunksize=1))
    assert n == T * H_q
    return T, time.perf_counter() - t


def cpu_baseline(config: str, args) -> dict:
    """The oracle on the bounded sample the reference arm times (same rule, same --steps/--warmup):
    one thread, repeated for about args.cpu_seconds; then the same path with its attention over
    every host core (worker processes), repeated likewise."""
    sub, desc = oracle_sample(config, args.steps, args.warmup, args.oracle_step_seconds)
    prep = _oracle_prepare(sub, 8)
    tok = sec = 0.0
    reps = 0
    while sec < args.cpu_seconds or reps == 0:
        t, s_ = _oracle_run(prep)
        tok += t
        sec += s_
        reps += 1
    out = {"value": round(tok / sec, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{desc}; fp64 numpy, one thread, {reps} runs, {sec:.1f} s"}
    if not args.no_parallel_oracle:
        out["all_cores"] = parallel_oracle(prep, args.cpu_seconds / 2)
    return out


def parallel_oracle(prep, seconds: float) -> dict:
    import multiprocessing as mp
    n_workers = os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory(prefix="ms_oracle_") as tmpdir, ctx.Pool(n_workers) as pool:
        for k in ("q", "k", "v", "kp", "vp"):  # the step's inputs, resident before the clock starts
            np.save(os.path.join(tmpdir, k + ".npy"), np.ascontiguousarray(prep[k]))
        _oracle_run_parallel(prep, pool, n_workers, tmpdir)  # untimed: workers import numpy and the oracle
        tok = sec = 0.0
        reps = 0
        while sec < seconds or reps == 0:
            t, s_ = _oracle_run_parallel(prep, pool, n_workers, tmpdir)
            tok += t
            sec += s_
            reps += 1
    return {"value": round(tok / sec, 2), "unit": "tokens/s", "cores": n_workers, "kind": "oracle",
            "how": f"append and attention over {n_workers} spawned worker processes by (row, KV head, token "
                   f"block); schedule and metadata in the parent; {reps} runs, {sec:.1f} s"}


def run_reference(args, world, rank):
    """The oracle as the reference arm: each step the bounded sample that cpu_baseline also times."""
    if rank != 0:
        return
    name = ALL_CONFIGS[0] if args.config == "all" else args.config
    wls = load_workload(name)
    sub, desc = oracle_sample(name, args.steps, args.warmup, args.oracle_step_seconds)
    prep = _oracle_prepare(sub, 8)
    for _ in range(args.warmup):
        _oracle_run(prep)
    tot_tok = tot_s = 0.0
    for _ in range(args.steps):
        tk, s = _oracle_run(prep)
        tot_tok += tk
        tot_s += s
    value = tot_tok / tot_s
    cpu = {"value": round(value, 2), "unit": "tokens/s", "cores": 1, "kind": "oracle",
           "sample": f"{desc}; fp64 numpy, one thread, {args.steps} runs"}
    if not args.no_parallel_oracle:
        cpu["all_cores"] = parallel_oracle(prep, min(args.cpu_seconds / 2, 8.0))
    line = {"metric": METRIC, "value": round(value, 2), "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_block(name, wls, world), "impl": "reference", "cpu_baseline": cpu,
            "e2e": {"value": round(value, 2), "unit": "tokens/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- step-latency timeline

GRAPH_BUCKETS_512 = [16, 32, 64, 96, 128, 192, 256, 384, 512]

TIMELINE_SCENARIOS = [
    ("decode-first, budget 512", dict(token_budget=512)),
    ("decode-first, budget 512, CUDA graph per token bucket", dict(token_budget=512, graph=GRAPH_BUCKETS_512)),
    ("decode-first, budget 2048", dict(token_budget=2048)),
    ("no chunking (budget holds the whole prompt)", dict(token_budget=None)),
    ("prefill-first, budget 512", dict(token_budget=512, policy=1)),
    ("fair share, decode share 10 %, budget 512", dict(token_budget=512, policy=2, decode_share_permille=100)),
]


def _percentile(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q)) if len(xs) else 0.0


def run_timeline(args, local):
    """Rounds of the engine around a long prompt's arrival, one scenario per scheduling setting:
    per-step prefill tokens, decode tokens and device step latency, the decodes' inter-token
    gaps and the prompt's time to first token (one attention layer)."""
    import torch

    import chunked_prefill_mixed_decode_gb300 as ms
    from chunked_prefill_mixed_decode_gb300 import build as msbuild
    from chunked_prefill_mixed_decode_gb300 import step
    from chunked_prefill_mixed_decode_gb300.driver import RoundDriver

    msbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    sc = workloads.long_prompt_arrival()
    n_dec = len(sc.decode_ctx)
    pages = sum(-(-(c + sc.decode_new) // 16) for c in sc.decode_ctx) + -(-(sc.prompt_len + sc.prompt_new) // 16)
    shape = types.SimpleNamespace(num_pages=pages, H_q=sc.H_q, H_kv=sc.H_kv, page_size=16, D=sc.D)
    k_cache, v_cache = workloads.kv_pool(shape, 77, device)
    max_pos = max(max(sc.decode_ctx) + sc.decode_new, sc.prompt_len + sc.prompt_new) + 1
    cos, sin = step.rope_tables_device(max_pos, sc.D, device)
    big = n_dec + sc.prompt_len
    q, k, v = workloads.step_tensors(shape, big, 78, device)
    results = []
    for label, kw in TIMELINE_SCENARIOS:
        kw = dict(kw)
        budget = kw.pop("token_budget") or big
        buckets = kw.pop("graph", None)
        eng = ms.Engine(pages, budget, **kw)
        dec_ids = [eng.add_request(c, sc.decode_new, c) for c in sc.decode_ctx]
        row_pages = -(-max(max(sc.decode_ctx) + sc.decode_new, sc.prompt_len + sc.prompt_new) // 16)
        drv = RoundDriver(eng, k_cache, v_cache, cos, sin, sc.H_q, sc.H_kv, sc.D, graph_buckets=buckets,
                          max_row_pages=row_pages)
        sq, sk, sv = q, k, v
        if drv.graph is not None:  # the step's inputs live in the graph's fixed buffers
            B = buckets[-1]
            drv.graph.q.copy_(q[:B])
            drv.graph.k.copy_(k[:B])
            drv.graph.v.copy_(v[:B])
            sq, sk, sv = drv.graph.q, drv.graph.k, drv.graph.v
        recs, pid, prompt_done_round, prefilled = [], None, None, 0
        rnd = 0
        while True:
            if rnd == sc.arrival_round:
                pid = eng.add_request(sc.prompt_len, sc.prompt_new)
            rec = drv.step(sq, sk, sv)
            d = np.diff(rec["cu_seqlens_q"])
            if pid is not None:
                for rid, n in zip(rec["row_request_id"].tolist(), d.tolist()):
                    if rid == pid and prompt_done_round is None:
                        prefilled += n
                        if prefilled == sc.prompt_len:
                            prompt_done_round = rnd
            recs.append(rec)
            rnd += 1
            if prompt_done_round is not None and rnd > prompt_done_round + sc.tail_rounds:
                break
            if rnd > 4000:
                raise RuntimeError("timeline did not finish")
        t_end = np.cumsum([r["device_ms"] for r in recs])
        last_tok = {}
        gaps = []
        dec_set = set(dec_ids)
        for s_, r in enumerate(recs):
            for rid in r["row_request_id"][: r["decode_tokens"]].tolist():
                if rid in dec_set:
                    if rid in last_tok and s_ >= sc.arrival_round:
                        gaps.append(t_end[s_] - t_end[last_tok[rid]])
                    last_tok[rid] = s_
        a = sc.arrival_round
        steady = [r["device_ms"] for r in recs[4:a]]
        window = [r["device_ms"] for r in recs[a:prompt_done_round + 1]]
        ttft = float(t_end[prompt_done_round] - (t_end[a - 1] if a > 0 else 0.0))
        executed = sum(r.get("bucket", r["prefill_tokens"] + r["decode_tokens"]) for r in recs)
        scheduled = sum(r["prefill_tokens"] + r["decode_tokens"] for r in recs)
        results.append({
            "scenario": label, "token_budget": budget, "graph_buckets": buckets,
            "pad_tokens": executed - scheduled, "pad_fraction": round((executed - scheduled) / executed, 4),
            "steady_step_ms": round(statistics.median(steady), 4),
            "steady_wall_ms": round(statistics.median(r["wall_ms"] for r in recs[4:a]), 4),
            "prefill_steps": prompt_done_round - a + 1,
            "max_step_ms_during_prefill": round(max(window), 4),
            "median_step_ms_during_prefill": round(statistics.median(window), 4),
            "decode_gap_ms": {"p50": round(_percentile(gaps, 50), 4), "p99": round(_percentile(gaps, 99), 4),
                              "max": round(max(gaps), 4) if gaps else 0.0},
            "prompt_ttft_ms": round(ttft, 4),
            "host_ms_median": round(statistics.median(r["host_ms"] for r in recs), 3),
            "steps": [[r["round"], r["decode_tokens"], r["prefill_tokens"], round(r["device_ms"], 4)]
                      for r in recs],
        })
        del drv, eng
    line = {"timeline": sc.name, "layer": f"H_q {sc.H_q}, H_kv {sc.H_kv}, D {sc.D}, page 16",
            "decodes": n_dec, "decode_ctx": "U[512, 4096]", "prompt_len": sc.prompt_len,
            "arrival_round": sc.arrival_round, "latency": "device time of append + attention per step",
            "scenarios": results}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------- decode / chunk split

SPLIT_CONFIGS = ["mha7b_b512", "mha13b_b2048", "gqa8b_b8192", "long_bimodal_b4608"]


def _call_times(fn, reps: int, stream, flush) -> list:
    """Device milliseconds of each of reps launches of fn(), each timed alone with CUDA events on
    the launching stream after flush() has overwritten L2 (outside the events); 3 warm-ups first."""
    import torch
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    pairs = []
    for _ in range(reps):
        flush()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        pairs.append((e0, e1))
    torch.cuda.synchronize()
    return [a.elapsed_time(b) for a, b in pairs]


def run_split(args, local):
    """Attribute each workload's step to its two bounds: the attention call on the mixed batch, on
    its decode rows alone (HBM GB/s of their KV reads) and on its prefill chunks alone (TFLOP/s
    of their causal pairs), plus the append on the mixed batch.  Every variant reads the same KV
    pool; each call is timed alone with CUDA events after a write of twice the L2 size has evicted
    what the previous call left there, summed over the workload's batches."""
    import torch

    import chunked_prefill_mixed_decode_gb300 as ms
    from chunked_prefill_mixed_decode_gb300 import build as msbuild
    from chunked_prefill_mixed_decode_gb300 import roofline, step

    msbuild.build()
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    stream = torch.cuda.current_stream(device)
    peaks, peak_src = read_peaks()
    reps = max(5, args.split_reps)
    l2 = int(getattr(torch.cuda.get_device_properties(device), "L2_cache_size", 0) or (129 << 20))
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device=device)
    n_flush = [0]

    def flush():
        n_flush[0] += 1
        flush_buf.fill_(n_flush[0] & 0xFF)

    out = []
    for name in args.split_configs:
        wls = load_workload(name)
        wl0 = wls[0]
        k_cache, v_cache = workloads.kv_pool(wl0, 1000, device)
        cos, sin = step.rope_tables_device(max(wl.max_pos for wl in wls) + 1, wl0.D, device)
        status = torch.zeros(1, dtype=torch.int32, device=device)
        acc = {"mixed_ms": 0.0, "append_ms": 0.0, "decode_only_ms": 0.0, "chunk_only_ms": 0.0,
               "decode_bytes": 0, "decode_kv_bytes": 0, "chunk_flops": 0, "append_bytes": 0, "mixed_bytes": 0,
               "mixed_flops": 0}
        for i, wl in enumerate(wls):
            parts = {"mixed": wl.requests,
                     "decode_only": [r for r in wl.requests if r.remaining == 0],
                     "chunk_only": [r for r in wl.requests if r.remaining > 0]}
            for label, reqs in parts.items():
                states = [(r.cached_len, r.remaining) for r in reqs]
                tables = [r.block_table for r in reqs]
                meta = ms.build_batch_metadata(states, tables, wl.token_budget, wl.max_chunk)
                T = meta["num_tokens"]
                if T == 0:
                    continue
                b = step.to_device(meta, device)
                q, k, v = workloads.step_tensors(wl, T, 50 + i, device)
                q_rot, o = torch.empty_like(q), torch.empty_like(q)
                ws = step.workspace_for(b, wl.H_q, wl.H_kv, wl.D, device)
                rows = [(int(meta["q_start_pos"][s_]), int(meta["cu_seqlens_q"][s_ + 1] - meta["cu_seqlens_q"][s_]))
                        for s_ in range(meta["num_rows"])]
                cnt = roofline.step_counts(rows, wl.H_q, wl.H_kv, wl.D)

                def append():
                    ms.kv_append_rope(q, k, v, b.positions, b.slot_mapping, cos, sin, k_cache, v_cache,
                                      q_rot=q_rot, dev_status=status, stream=stream)

                def attend():
                    ms.mixed_step_attention(q_rot, k_cache, v_cache, b.cu_seqlens_q, b.q_start_pos,
                                            b.context_lens, b.block_tables, b.context_total, o, ws, stream=stream)

                append()
                times = _call_times(attend, reps, stream, flush)
                t_attn = sum(times) / len(times)
                acc[label + "_median"] = acc.get(label + "_median", 0.0) + statistics.median(times)
                acc[label + "_min"] = acc.get(label + "_min", 0.0) + min(times)
                if ms.read_status(status) or ms.read_status(ws):
                    raise RuntimeError(f"device status set in {name} {label}")
                acc[label + "_ms"] += t_attn
                if label == "mixed":
                    times = _call_times(append, reps, stream, flush)
                    acc["append_ms"] += sum(times) / len(times)
                    acc["append_bytes"] += cnt["append_bytes"]
                    acc["mixed_bytes"] += cnt["attn_bytes"]
                    acc["mixed_flops"] += cnt["flops"]
                elif label == "decode_only":
                    acc["decode_bytes"] += cnt["attn_bytes"]
                    acc["decode_kv_bytes"] += cnt["decode_kv_bytes"]
                else:
                    acc["chunk_flops"] += cnt["flops"]
                del b, q, k, v, q_rot, o, ws
        del k_cache, v_cache
        torch.cuda.empty_cache()
        hbm, tf = peaks["hbm_gbs"], peaks["bf16_tflops"]
        dec_gbs = acc["decode_bytes"] / (acc["decode_only_ms"] / 1e3) / 1e9 if acc["decode_only_ms"] else None
        chk_tf = acc["chunk_flops"] / (acc["chunk_only_ms"] / 1e3) / 1e12 if acc["chunk_only_ms"] else None
        t_roof_mixed = max(acc["mixed_bytes"] / (hbm * 1e9), acc["mixed_flops"] / (tf * 1e12)) * 1e3
        out.append({
            "config": name, "batches": len(wls),
            "attention_mixed_ms": round(acc["mixed_ms"], 4),
            "attention_mixed_frac_of_roofline": round(t_roof_mixed / acc["mixed_ms"], 4),
            "append_ms": round(acc["append_ms"], 4),
            "append_gbs": round(acc["append_bytes"] / (acc["append_ms"] / 1e3) / 1e9, 1),
            "decode_only_ms": round(acc["decode_only_ms"], 4),
            "decode_only_gbs": round(dec_gbs, 1) if dec_gbs else None,
            "decode_only_hbm_frac": round(dec_gbs / hbm, 4) if dec_gbs else None,
            "chunk_only_ms": round(acc["chunk_only_ms"], 4),
            "chunk_only_tflops": round(chk_tf, 1) if chk_tf else None,
            "chunk_only_tensor_frac": round(chk_tf / tf, 4) if chk_tf else None,
            "mixed_vs_sum_of_parts": round(acc["mixed_ms"] / (acc["decode_only_ms"] + acc["chunk_only_ms"]), 4),
            # per call: median and minimum of the timed calls, summed over the workload's batches
            "median_ms": {lab: round(acc[lab + "_median"], 4) for lab in ("mixed", "decode_only", "chunk_only")
                          if lab + "_median" in acc},
            "min_ms": {lab: round(acc[lab + "_min"], 4) for lab in ("mixed", "decode_only", "chunk_only")
                       if lab + "_min" in acc},
        })
    line = {"split": "attention call per workload: mixed, decode rows only, prefill chunks only",
            "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"], "source": peak_src,
                      "note": "each call timed alone: the burst tensor peak applies"},
            "reps": reps, "l2_flush_bytes": int(flush_buf.numel()), "configs": out}
    print(json.dumps(line), flush=True)


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="all", choices=["all"] + sorted(workloads.CONFIGS),
                    help="one workload, or all four (the default): the line's top level is the long bimodal "
                         "step, the others go under per_config")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--no-parallel-oracle", action="store_true", help="skip the all-cores oracle leg")
    ap.add_argument("--oracle-step-seconds", type=float, default=0.0,
                    help="estimated oracle seconds of one sampled step (default: about two minutes over "
                         "--steps + --warmup, at most 8 s)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--timeline", action="store_true",
                    help="step-latency timeline around a long prompt's arrival (one JSON line)")
    ap.add_argument("--split", action="store_true",
                    help="decode-only / chunk-only / mixed attention timings per workload (one JSON line)")
    ap.add_argument("--split-configs", nargs="+", default=SPLIT_CONFIGS, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--split-reps", type=int, default=20)
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)  # at least three untimed warm-up steps
    world, rank, local = dist_env()
    if args.impl == "reference":
        run_reference(args, world, rank)
        return
    if args.timeline:
        if rank == 0:
            run_timeline(args, local)
        return
    if args.split:
        if rank == 0:
            run_split(args, local)
        return
    run_ours(args, world, rank, local)


if __name__ == "__main__":
    main()
