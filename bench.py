#!/usr/bin/env python
"""Decode benchmark of the persistent megakernel on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME] [--impl reference]

One step = one mk_decode_step (the whole decoder forward pass for the
workload's batch, one kernel launch) over seeded synthetic weights and KV
cache resident in HBM.  Prints ONE JSON line on rank 0.  With N > 1 (torchrun)
every rank runs an independent replica on its own GPU (the path does not
shard); value = all ranks' passes / the slowest rank's time.

The reference arm (--impl reference) is the CPU oracle run on the host cores
on a bounded number of steps of the same workload.
"""
import argparse
import csv
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

from synth.workloads import (WORKLOADS, contexts, first_tokens, make_kv, make_model,  # noqa: E402
                             max_ctx, step_tokens)

METRIC = "decode forward passes/s (batch 1, Llama-1B shape); % of GB300 HBM roofline"
DEFAULT = "llama1b_ctx1024"


def args_():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=128)
    p.add_argument("--warmup", type=int, default=10)
    p.add_argument("--impl", default="mine", choices=["mine", "reference"])
    p.add_argument("--config", default=DEFAULT, choices=sorted(WORKLOADS))
    p.add_argument("--seed", type=int, default=0)
    p.add_argument("--sched", default="static", choices=["dynamic", "static", "hybrid"])
    p.add_argument("--attn-chunk", type=int, default=0,
                   help="mk_config.attn_chunk (0: the planner's choice)")
    p.add_argument("--l2kb", type=int, default=0,
                   help="mk_config.l2_prefetch_kb: KB per block prefetched into L2 ahead of the ring")
    p.add_argument("--stream", action="store_true",
                   help="batch 1: per-warp streams of async copies instead of the shared page ring")
    p.add_argument("--no-baselines", action="store_true", help="skip multi-kernel and CPU legs")
    p.add_argument("--no-workloads", action="store_true",
                   help="skip the other workloads' lines (ctx 8192, ragged batch 8, Llama-8B)")
    p.add_argument("--trace", default="", help="write a per-instruction trace (npz) here")
    p.add_argument("--layers", type=int, default=0,
                   help="profiling only: override the workload's layer count (a smaller case)")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_sha256():
    """Hash of the kernel sources (names and bytes), to tell whether a
    recorded ncu traffic figure still describes the kernel being timed."""
    import glob
    import hashlib
    pat = os.path.join(ROOT, "persistent_megakernel_decode_block_gb300", "csrc", "*")
    fs = sorted([f for f in glob.glob(pat) if f.endswith((".cu", ".cuh", ".cpp", ".h"))] +
                [os.path.join(ROOT, "include", "mk.h")], key=os.path.basename)
    h = hashlib.sha256()
    for f in fs:
        h.update(os.path.basename(f).encode())
        with open(f, "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()


def recorded_traffic(workload):
    """dram bytes read + written per launch from the committed ncu summary of
    this workload, or None when the kernel changed since that capture."""
    kernel = "mk_megakernel_tc" if WORKLOADS[workload]["batch"] > 1 else "mk_megakernel"
    path = os.path.join(ROOT, "profiles", "%s_%s_sections.md" % (kernel, workload))
    try:
        kv = {}
        for line in open(path):
            if ":" in line and not line.startswith(("|", "#", " ", "`")):
                k, v = line.split(":", 1)
                kv[k.strip()] = v.strip()
        if kv.get("kernel_source_sha256") != kernel_sha256():
            return None
        return float(kv["traffic_bytes_per_launch"])
    except Exception:
        return None


def algorithmic_bytes(m, weight_bytes, positions):
    """weights once + KV rows below each position read + one K/V row written"""
    row = m["n_kv_heads"] * m["head_dim"] * 2  # bytes of one position, one layer, K or V
    kv_read = 2 * m["n_layers"] * row * int(np.sum(positions))
    kv_write = 2 * m["n_layers"] * row * len(positions)
    return weight_bytes + kv_read + kv_write


class Clocks:
    """nvidia-smi sampling during the timed region."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu):
        self.gpu, self.proc = gpu, None
        self.path = tempfile.mktemp(suffix=".csv")

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "200"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.25)
            self.proc.terminate()
            self.proc.wait()
            self.f.close()

    def summary(self):
        rows = []
        try:
            for r in csv.reader(open(self.path)):
                if len(r) >= 9:
                    rows.append([x.strip() for x in r])
        except Exception:
            return None
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for n, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": float(rows[0][2]) if rows[0][2].replace(".", "").isdigit() else None,
                "reasons": sorted(reasons), "samples": len(rows)}


def dist():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws == 1:
        return 0, 1, None
    import torch.distributed as td
    td.init_process_group("nccl" if os.environ.get("MK_BENCH_BACKEND") != "gloo" else "gloo")
    return td.get_rank(), ws, td


def max_over_ranks(x, td, device=None):
    """Largest value over ranks (the slowest replica's time)."""
    if td is None:
        return x
    import torch
    t = torch.tensor([x], dtype=torch.float64, device=device)
    td.all_reduce(t, op=td.ReduceOp.MAX)
    return float(t.item())


def barrier(td, device=None):
    if td is not None:
        if device is not None:
            td.barrier(device_ids=[device.index])
        else:
            td.barrier()


def cpu_facts():
    """Threads the host offers and its CPU model (lscpu, else /proc/cpuinfo)."""
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.strip().startswith("Model name:"):
                model = line.split(":", 1)[1].strip()
                break
    except Exception:
        pass
    if not model:
        try:
            for line in open("/proc/cpuinfo"):
                if line.lower().startswith(("model name", "cpu part")):
                    model = line.split(":", 1)[1].strip()
                    break
        except Exception:
            pass
    import platform
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.machine()}


def time_workload(mk, torch, dev, name, a, fp8=False):
    """Another workload, timed as the headline one (same steps and warm-up,
    static lists, device-resident inputs, CUDA events on the launching
    stream, clocks sampled): ms/step, passes/s and roofline fraction.  fp8:
    the same workload with FP8 weights (MK_FLAG_FP8_WEIGHTS); its roofline
    bytes are the FP8 codes and row scales."""
    w = WORKLOADS[name]
    m, B = w["model"], w["batch"]
    ctx, mctx = contexts(name, a.seed), max_ctx(name, a.seed)
    span = w["steps"]
    weights = make_model(m, a.seed)
    k0, v0 = make_kv(m, B, mctx, ctx, a.seed)

    def up(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev)

    plan = mk.mk_plan(mk.make_config(m, B, mctx, sched_mode=mk.MK_SCHED_STATIC,
                                     flags=mk.MK_FLAG_FP8_WEIGHTS if fp8 else 0))
    try:
        info = mk.mk_plan_info(plan)
        mk.mk_load_weights(plan, {"embed": up(weights["embed"]),
                                  "final_norm": up(weights["final_norm"]),
                                  "lm_head": None if m["tie_embeddings"] else up(weights["lm_head"]),
                                  "layers": [{k: up(v) for k, v in lw.items()}
                                             for lw in weights["layers"]]})
        del weights
        torch.cuda.empty_cache()
        kc, vc = up(k0), up(v0)
        total = a.warmup + a.steps
        toks = torch.from_numpy(step_tokens(m, B, total, a.seed)).to(dev)
        pos_host = np.stack([ctx + (s % span) for s in range(total)]).astype(np.int32)
        poss = torch.from_numpy(pos_host).to(dev)
        logits = torch.zeros(B, m["vocab"], dtype=torch.float32, device=dev)
        stream = torch.cuda.Stream(device=dev)
        for s in range(a.warmup):
            mk.mk_decode_step(plan, toks[s], poss[s], (kc, vc), logits, stream)
        stream.synchronize()
        assert mk.mk_status(plan, stream) == 0
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize(dev)
        clocks = Clocks(dev.index)
        with clocks:
            with torch.cuda.stream(stream):
                e0.record(stream)
                for s in range(a.steps):
                    mk.mk_decode_step(plan, toks[a.warmup + s], poss[a.warmup + s], (kc, vc),
                                      logits, stream)
                e1.record(stream)
            stream.synchronize()
        code = mk.mk_status(plan, stream)
        assert code == 0, mk.mk_error_string(code)
        ms = e0.elapsed_time(e1) / a.steps
        bytes_step = float(np.mean([algorithmic_bytes(m, info["weight_bytes"], p)
                                    for p in pos_host[a.warmup:]]))
        peak, peak_kind = peaks()
        achieved = bytes_step / (ms * 1e-3) / 1e9
        return {"ms_per_step": ms, "passes_per_s": 1000.0 / ms, "batch": B,
                "tokens_per_s": 1000.0 * B / ms,
                "roofline": {"achieved": achieved, "peak": peak, "unit": "GB/s",
                             "frac": achieved / peak, "bytes_per_step": bytes_step,
                             "traffic": None if fp8 else recorded_traffic(name),
                             "peak_kind": peak_kind + " hbm_gbs"},
                "kernel": "mk_megakernel_tc" if B > 1 else "mk_megakernel_q8" if fp8
                          else "mk_megakernel",
                "weights": "fp8 e4m3, one scale per row" if fp8 else "bf16",
                "clocks": clocks.summary()}
    finally:
        mk.mk_destroy(plan)
        torch.cuda.empty_cache()


def cpu_oracle(name, seed, weights, budget_s, max_steps=None):
    """The oracle as it stands on the host cores: one untimed step, then
    steps until ~budget_s of work.  Returns (passes/s, steps timed)."""
    import oracle
    w = WORKLOADS[name]
    m, B = w["model"], w["batch"]
    ctx, mctx = contexts(name, seed), max_ctx(name, seed)
    k0, v0 = make_kv(m, B, mctx, ctx, seed)
    ref = oracle.Model(m, weights, B, mctx, k0, v0)
    toks = first_tokens(m, B, seed)
    ref.step(toks, ctx)
    n, t0 = 0, time.perf_counter()
    while True:
        ref.step(toks, ctx + 1 + n % max(1, w["steps"] - 1))
        n += 1
        dt = time.perf_counter() - t0
        if dt >= budget_s or (max_steps and n >= max_steps):
            return n / dt, n, dt


def run_reference(a):
    rank, ws, td = dist()
    if rank != 0:
        return
    w = WORKLOADS[a.config]
    m = w["model"]
    weights = make_model(m, a.seed)
    # bounded: every timed step is one full oracle decode step; the number of
    # steps is capped so the run stays within a few minutes
    per = cpu_oracle(a.config, a.seed, weights, 0.0, max_steps=1)[2]
    k = max(1, min(a.steps, int(120.0 / max(per, 1e-3))))
    rate, n, dt = cpu_oracle(a.config, a.seed, weights, 1e9, max_steps=k)
    line = {"impl": "reference", "metric": METRIC, "value": rate, "unit": "passes/s",
            "n_gpus": a.gpus, "steps": n, "warmup": 1, "ms_per_step": 1000 * dt / n,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "config": {"workload": a.config, "batch": w["batch"]},
            "cpu_baseline": dict({"value": rate, "unit": "passes/s", "cores": 1, "kind": "oracle",
                                  "sample": "%d full oracle decode steps of %s (of %d requested)"
                                            % (n, a.config, a.steps)}, **cpu_facts()),
            "e2e": {"value": rate, "unit": "passes/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_mine(a):
    import torch

    from persistent_megakernel_decode_block_gb300 import mk

    rank, ws, td = dist()
    local = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = WORKLOADS[a.config]
    m, B, name = dict(w["model"]), w["batch"], a.config
    if a.layers:
        m["n_layers"] = a.layers
    ctx, mctx = contexts(name, a.seed), max_ctx(name, a.seed)
    span = w["steps"]  # positions ctx .. ctx+span-1 exist in the cache
    weights = make_model(m, a.seed)
    k0, v0 = make_kv(m, B, mctx, ctx, a.seed)

    def up(x):
        return torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).to(dev)

    cfg = mk.make_config(m, B, mctx, sched_mode={"static": mk.MK_SCHED_STATIC,
                                                 "hybrid": mk.MK_SCHED_HYBRID,
                                                 "dynamic": mk.MK_SCHED_DYNAMIC}[a.sched],
                         flags=(mk.MK_FLAG_TRACE if a.trace else 0) | (mk.MK_FLAG_STREAM_B1 if a.stream else 0),
                         l2_prefetch_kb=a.l2kb, attn_chunk=a.attn_chunk)
    plan = mk.mk_plan(cfg)
    info = mk.mk_plan_info(plan)
    mk.mk_load_weights(plan, {"embed": up(weights["embed"]), "final_norm": up(weights["final_norm"]),
                              "lm_head": None if m["tie_embeddings"] else up(weights["lm_head"]),
                              "layers": [{k: up(v) for k, v in lw.items()}
                                         for lw in weights["layers"]]})
    torch.cuda.empty_cache()
    kc, vc = up(k0), up(v0)
    total = a.warmup + a.steps
    toks = torch.from_numpy(step_tokens(m, B, total, a.seed)).to(dev)
    pos_host = np.stack([ctx + (s % span) for s in range(total)]).astype(np.int32)
    poss = torch.from_numpy(pos_host).to(dev)
    logits = torch.zeros(B, m["vocab"], dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream(device=dev)

    def step(s, kind="mega", graph=False):
        if kind == "mega":
            mk.mk_decode_step(plan, toks[s], poss[s], (kc, vc), logits, stream)
        else:
            mk.mk_multikernel_step(plan, toks[s], poss[s], (kc, vc), logits, graph, stream)

    def timed(kind="mega", graph=False, per_step=True):
        for s in range(a.warmup):
            step(s, kind, graph)
        stream.synchronize()
        code = mk.mk_status(plan, stream)
        assert code == 0, mk.mk_error_string(code)
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(a.steps + 1)]
        barrier(td, dev)
        torch.cuda.synchronize(dev)
        with torch.cuda.stream(stream):
            ev[0].record(stream)
            for s in range(a.steps):
                step(a.warmup + s, kind, graph)
                if per_step or s == a.steps - 1:
                    ev[s + 1].record(stream)
        stream.synchronize()
        torch.cuda.synchronize(dev)
        barrier(td, dev)
        code = mk.mk_status(plan, stream)
        assert code == 0, mk.mk_error_string(code)
        tot = ev[0].elapsed_time(ev[a.steps])
        per = [ev[s].elapsed_time(ev[s + 1]) for s in range(a.steps)] if per_step else []
        return tot, per

    clocks = Clocks(local)
    with clocks:
        total_ms, per = timed("mega")
    total_ms = max_over_ranks(total_ms, td, dev)
    ms = total_ms / a.steps
    per_sorted = sorted(per)
    ms_med = per_sorted[len(per) // 2]
    value = ws * a.steps / (total_ms / 1000.0)

    timed_pos = pos_host[a.warmup:]
    bytes_step = float(np.mean([algorithmic_bytes(m, info["weight_bytes"], p) for p in timed_pos]))
    peak, peak_kind = peaks()
    achieved = bytes_step / (ms * 1e-3) / 1e9

    extra = {}
    if a.trace:
        tr = mk.mk_read_trace(plan)
        rec, _, _ = mk.mk_plan_tables(plan)
        np.savez_compressed(a.trace, trace=tr, op=rec["op"], layer=rec["layer"], b=rec["b"],
                            g=rec["g"], chunk=rec["chunk"], positions=pos_host[-1])

    # end to end through the host-buffer entry point: tokens/positions in,
    # logits out, every step, pinned host memory
    h_tok = torch.from_numpy(step_tokens(m, B, total, a.seed)).pin_memory()
    h_pos = torch.from_numpy(pos_host).pin_memory()
    h_log = torch.zeros(B, m["vocab"], dtype=torch.float32).pin_memory()
    for s in range(a.warmup):
        mk.mk_decode_step_host(plan, h_tok[s], h_pos[s], (kc, vc), h_log, stream)
    barrier(td, dev)
    t0 = time.perf_counter()
    for s in range(a.steps):
        mk.mk_decode_step_host(plan, h_tok[a.warmup + s], h_pos[a.warmup + s], (kc, vc), h_log,
                               stream)
    e2e_s = max_over_ranks(time.perf_counter() - t0, td, dev)
    code = mk.mk_status(plan, stream)
    assert code == 0, mk.mk_error_string(code)
    e2e = {"value": ws * a.steps / e2e_s, "unit": "passes/s", "h2d_bytes_per_step": 8 * B,
           "d2h_bytes_per_step": 4 * B * m["vocab"]}

    if not a.no_baselines:
        mk_ms, _ = timed("multi", False, per_step=False)
        mg_ms, _ = timed("multi", True, per_step=False)
        nph = info["n_phases"]
        extra["multikernel"] = {
            "launches_per_step": nph + 1,
            "ms_per_step": mk_ms / a.steps, "passes_per_s": 1000.0 * a.steps / mk_ms,
            "graph_ms_per_step": mg_ms / a.steps, "graph_passes_per_s": 1000.0 * a.steps / mg_ms}

    cpu = None
    if rank == 0 and not a.no_baselines:
        rate, n, dt = cpu_oracle(name, a.seed, weights, 12.0)
        cpu = {"value": rate, "unit": "passes/s", "cores": 1, "kind": "oracle",
               "sample": "%d full oracle decode steps of %s (%.1f s, single thread)" % (n, name, dt)}
        cpu.update(cpu_facts())
    mk.mk_destroy(plan)
    del weights, kc, vc
    torch.cuda.empty_cache()
    if rank == 0 and not a.no_workloads and name == DEFAULT and not a.layers and not a.trace:
        extra["workloads"] = {o: time_workload(mk, torch, dev, o, a) for o in
                              ("llama1b_ctx8192", "llama1b_b8_ragged", "llama1b_b32_ragged",
                               "llama8b_ctx2048")}
        # the same headline workload with FP8 weights (a lower-precision mode,
        # not the headline: its bytes per step are about half)
        extra["workloads"]["llama1b_ctx1024_fp8"] = time_workload(mk, torch, dev, DEFAULT, a,
                                                                  fp8=True)
    if rank != 0:
        return
    line = {
        "metric": METRIC, "value": value, "unit": "passes/s", "n_gpus": ws, "steps": a.steps,
        "warmup": a.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": name, "batch": B, "ctx": [int(c) for c in ctx][:8],
                   "max_ctx": mctx, "sched": a.sched,
                   "l2": "inputs larger than L2 (%.2f GB of weights streamed per step)"
                         % (info["weight_bytes"] / 1e9),
                   "weights": "bf16", "kv_cache": "bf16"},
        "us_per_token": {"median": 1000 * ms_med, "p10": 1000 * per_sorted[len(per) // 10],
                         "p90": 1000 * per_sorted[(9 * len(per)) // 10]},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": recorded_traffic(name),
                     "bytes_per_step": bytes_step, "peak_kind": peak_kind + " hbm_gbs"},
        "gpu_launches": a.steps,
        "e2e": e2e,
        "clocks": clocks.summary(),
        "cpu_baseline": cpu,
        "plan": {k: info[k] for k in ("n_instr", "n_blocks", "ring_pages", "page_bytes",
                                       "smem_bytes", "attn_nchunk")},
    }
    line.update(extra)
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    a = args_()
    if a.impl == "reference":
        run_reference(a)
    else:
        run_mine(a)
