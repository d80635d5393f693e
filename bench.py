#!/usr/bin/env python3
"""Benchmark of the DSpark ragged-verification hot path on GB300.

One step = the whole hot path on one batch: schedule, pack, verify (compact, greedy) and the
compact scatter, issued as the two fused calls dspark_schedule_pack and dspark_verify_scatter,
on the large-vocab mixed-traffic workload (B=256
requests, block gamma=8, V=151936 bf16 logits, three acceptance classes a = 0.9/0.65/0.35,
theta(M) = 0.004 M, alpha(bs) = 0.01 bs, bias 2, tiers every 32 up to 2048). The packed
target logits of the scheduled windows are produced off the clock (they stand in for the
target model's forward) and stay resident; three seeded batches rotate so every step reads
more than L2 holds.

Prints one JSON line. `value` is packed verify rows per second over the whole step with
inputs resident in HBM; `e2e` repeats the measurement with the step's inputs copied from
pinned host memory and the results read back inside the timed region; `roofline` reports the
streaming kernel's algorithmic bytes (M * V * 2 per launch) over its CUDA-event time against
the measured HBM copy bandwidth (and the whole verify call beside it); `latency_b1` times the
batch-1 decode step; `verify_legs` the verify call on the other workloads; `cpu_baseline`
times the CPU oracle on a bounded sample.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "packed verify rows/s & logits HBM GB/s vs GB300 peak; sched+pack µs/step"
NOMINAL_HBM_GBS = 8000.0     # the GB300's nominal HBM3e bandwidth, for context beside the measured peak
UNIT = "rows/s"
WORKLOAD = "large_vocab_mixed"
FALLBACK_HBM_GBS = 6800.0
PROFILE = os.path.join(ROOT, "profiles", "verify_large_vocab_mixed.md")
N_BATCHES = 3


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batches", type=int, default=N_BATCHES)
    ap.add_argument("--latency-steps", type=int, default=10000)
    ap.add_argument("--stream-kernel", default="auto", choices=["auto", "register", "bulk"],
                    help="which logit-streaming kernel verify uses (results are identical)")
    ap.add_argument("--config-reps", type=int, default=30,
                    help="timed verify calls per extra workload leg (0: skip the legs)")
    ap.add_argument("--event-every", type=int, default=100,
                    help="record the per-kernel events on every n-th timed step only: an event "
                         "between two kernels stops the second from launching early, so a "
                         "sampled step runs about 10-15 us slower")
    return ap.parse_args()


def dist_setup(n):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def sum_over_ranks(x, world):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64,
                     device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def profile_traffic():
    """DRAM bytes over algorithmic bytes of the captured verify-stream launch recorded in
    profiles/, if the source files the record names still hash to the value recorded with it."""
    try:
        with open(PROFILE) as f:
            text = f.read()
    except OSError:
        return None
    rec = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith("- "):
            k, v = line.strip()[2:].split(":", 1)
            rec[k.strip()] = v.strip().strip("`")
    h = hashlib.sha256()
    try:
        for name in rec.get("sources", "").split():
            with open(os.path.join(ROOT, "speculative_decoding_ragged_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    if not rec.get("sources") or rec.get("sources_sha256_16") != h.hexdigest()[:16]:
        return None
    try:
        return float(rec["traffic_over_algorithmic"])
    except (KeyError, ValueError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region."""
    FIELDS = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            pass

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.strip()]
        if self.uuid:
            mine = [r for r in rows if len(r) > 1 and self.uuid.replace("GPU-", "") in r[1]]
            rows = mine or rows
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


def make_inputs(wl, seeds, dev, st):
    """Per batch: device conf/tokens, device packed logits of the scheduled windows (the
    library's own dspark_schedule decides them, off the clock: the packed rows stand in for the
    target forward over the packed batch), and pinned host copies for the end-to-end leg."""
    from speculative_decoding_ragged_gb300 import synth
    batches = []
    for seed in seeds:
        bt = synth.make_batch(wl, seed=seed)
        conf = torch.as_tensor(bt.conf, device=dev)
        st.schedule(conf)
        w = st.windows.cpu().numpy()
        M = int(w.sum())
        tier = min([t for t in wl.tiers if t >= M] or [M])
        packed = synth.gather_packed(bt.target, bt.B, bt.gamma, w, rows_cap=tier)
        batches.append(dict(
            bt=bt, windows=w, M=M, conf=conf,
            tokens=torch.as_tensor(bt.tokens, device=dev),
            packed=packed.to(dev),
            conf_h=torch.as_tensor(bt.conf).pin_memory(),
            tokens_h=torch.as_tensor(bt.tokens).pin_memory(),
            packed_h=packed.pin_memory()))
        bt.target = None          # the full block is not needed any more
    st.status.zero_()
    return batches


def run_native(args, rank, world, local):
    from speculative_decoding_ragged_gb300 import build, synth
    from speculative_decoding_ragged_gb300.step import DSparkStep
    build.build()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    from speculative_decoding_ragged_gb300 import _binding as bd
    bd.set_stream_kernel({"auto": bd.STREAM_AUTO, "register": bd.STREAM_REGISTER,
                          "bulk": bd.STREAM_BULK}[args.stream_kernel])
    wl = synth.WORKLOADS[args.workload]
    seeds = [1000 * rank + i for i in range(args.batches)]
    st = DSparkStep(wl.B, wl.gamma, wl.V, wl.tiers, wl.bias,
                    wl.alpha_slope * np.arange(wl.B + 1),
                    wl.theta_slope * np.arange(wl.B * wl.gamma + 1), mode="compact",
                    out_cap=1 << 16, device=dev)
    batches = make_inputs(wl, seeds, dev, st)
    stream = torch.cuda.current_stream()
    nb = len(batches)
    calls = [st.prepare(b["conf"], b["tokens"], b["packed"]) for b in batches]

    def step(i, ev=None):
        # fused calls: dspark_schedule_pack, then dspark_verify_scatter (whose compact scatter
        # runs inside the finaliser); on sampled steps the library also records ev[3], ev[4]
        # around its streaming kernel
        sched_pack, verify_scatter = calls[i % nb]
        if ev is not None:
            ev[0].record(stream)
        sched_pack()
        if ev is not None:
            ev[1].record(stream)
            bd.set_stream_events(ev[3], ev[4])
        verify_scatter()
        if ev is not None:
            bd.set_stream_events(None, None)
            ev[2].record(stream)

    for i in range(args.warmup):
        step(i)
        st.out_len.zero_()
    torch.cuda.synchronize()

    # device-resident timed region: K steps, events around sched+pack and verify each step
    K = args.steps
    sampled = [i for i in range(K) if i % max(1, args.event_every) == 0]
    evs = {i: [torch.cuda.Event(enable_timing=True) for _ in range(5)] for i in sampled}
    for ev in evs.values():           # torch creates events lazily: make them exist
        for e in ev:
            e.record(stream)
    torch.cuda.synchronize()
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    clocks.start()
    t_start.record(stream)
    for i in range(K):
        step(i, evs.get(i))
    t_end.record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    barrier(world)
    ms = t_start.elapsed_time(t_end)
    ms = max_over_ranks(ms, world)
    rows = sum(batches[i % nb]["M"] for i in range(K))
    rows = sum_over_ranks(rows, world)
    sched_us = [evs[i][0].elapsed_time(evs[i][1]) * 1e3 for i in sampled]
    verify_us = [evs[i][1].elapsed_time(evs[i][2]) * 1e3 for i in sampled]
    stream_us = [evs[i][3].elapsed_time(evs[i][4]) * 1e3 for i in sampled]
    verify_bytes = [batches[i % nb]["M"] * wl.V * 2 for i in sampled]
    ach_gbs = sum(verify_bytes) / (sum(verify_us) * 1e-6) / 1e9          # the whole verify call
    kern_gbs = sum(verify_bytes) / (sum(stream_us) * 1e-6) / 1e9         # its streaming kernel
    peak, peak_kind = measured_peak()
    ratio = profile_traffic()     # DRAM bytes / algorithmic bytes of a captured launch
    traffic = None if ratio is None else ratio * statistics.mean(verify_bytes)
    value = rows / (ms * 1e-3)

    # end to end through the C ABI with host buffers: every step copies its confidences,
    # tokens and packed logits from pinned host memory and reads its results back, inside the
    # timed region. The copies run on a stream of their own into two alternating input sets,
    # so the next step's copy overlaps this step's compute (the copy link is the bound).
    E = min(args.e2e_steps, K)
    acc_h = torch.empty(wl.B, dtype=torch.int32).pin_memory()
    com_h = torch.empty((wl.B, wl.gamma), dtype=torch.int32).pin_memory()
    pk_rows = max(b["packed"].shape[0] for b in batches)
    inbuf = [dict(conf=torch.empty_like(batches[0]["conf"]),
                  tok=torch.empty_like(batches[0]["tokens"]),
                  pk=torch.empty((pk_rows, wl.V), dtype=batches[0]["packed"].dtype, device=dev))
             for _ in range(2)]
    copy_stream = torch.cuda.Stream(device=dev)
    copied = [torch.cuda.Event() for _ in range(2)]
    consumed = [torch.cuda.Event() for _ in range(2)]
    h2d = d2h = 0
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    barrier(world)
    e0.record(stream)
    copy_stream.wait_event(e0)
    e2e_rows = 0
    for i in range(E):
        b = batches[i % nb]
        k = i % 2
        buf = inbuf[k]
        with torch.cuda.stream(copy_stream):
            if i >= 2:
                copy_stream.wait_event(consumed[k])      # the step that last read this set
            buf["conf"].copy_(b["conf_h"], non_blocking=True)
            buf["tok"].copy_(b["tokens_h"], non_blocking=True)
            buf["pk"][: b["M"]].copy_(b["packed_h"][: b["M"]], non_blocking=True)
            copied[k].record(copy_stream)
        stream.wait_event(copied[k])
        st.run(buf["conf"], buf["tok"], buf["pk"])
        acc_h.copy_(st.accept_len, non_blocking=True)
        com_h.copy_(st.committed, non_blocking=True)
        consumed[k].record(stream)
        h2d += b["conf_h"].numel() * 4 + b["tokens_h"].numel() * 4 + b["M"] * wl.V * 2
        d2h += (acc_h.numel() + com_h.numel()) * 4
        e2e_rows += b["M"]
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(e0.elapsed_time(e1), world)
    e2e_rows = sum_over_ranks(e2e_rows, world)

    latency = latency_leg(dev, args.latency_steps) if args.latency_steps > 0 else None
    legs = config_legs(dev, args.config_reps) if args.config_reps > 0 and rank == 0 else None

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(batches, wl, args.cpu_seconds)
    if rank != 0:
        return None
    verify_mean_us = statistics.mean(verify_us)
    return {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": wl.B, "gamma": wl.gamma, "V": wl.V,
                   "mode": "compact", "verify": "greedy", "logits": "bf16",
                   "stream_kernel": args.stream_kernel,
                   "batches_rotating": nb, "rows_per_step_mean": rows / K / world,
                   "l2": "inputs larger than L2: each step reads >=300 MB of packed logits, "
                         f"{nb} batches rotate",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "logits_gbs": ach_gbs,
        "sched_pack_us": statistics.median(sched_us),
        "verify_us": statistics.median(verify_us),
        "step_us": ms / K * 1e3,
        "events_sampled_steps": len(sampled),
        "roofline": {"bound": "hbm",
                     "kernel": f"verify streaming kernel ({stream_kernel_name(wl, args)})",
                     "achieved": kern_gbs, "peak": peak, "peak_source": peak_kind,
                     "unit": "GB/s", "frac": kern_gbs / peak, "traffic": traffic,
                     "frac_of_nominal_8tbs": kern_gbs / NOMINAL_HBM_GBS,
                     "algorithmic_bytes_per_launch": statistics.mean(verify_bytes),
                     "launch_us_mean": statistics.mean(stream_us),
                     "launch_us_p10_p90": [percentile(stream_us, 10), percentile(stream_us, 90)],
                     "verify_call": {"what": "dspark_verify_scatter: streaming kernel, then "
                                             "finaliser with the fused scatter",
                                     "achieved": ach_gbs, "frac": ach_gbs / peak,
                                     "us_mean": verify_mean_us,
                                     "us_p10_p90": [percentile(verify_us, 10),
                                                    percentile(verify_us, 90)]}},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_rows / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d // max(E, 1), "d2h_bytes_per_step": d2h // max(E, 1),
                "steps": E, "h2d_gbs": h2d / (e2e_ms * 1e-3) / 1e9,
                "overlap": "next step's copy on its own stream during this step's compute"},
        "gpu_launches": K * st.launches_per_step,
        "clocks": clk,
        "latency_b1": latency,
        "verify_legs": legs,
    }


def latency_leg(dev, steps, pool=64):
    """Per-step time of the batch-1 workload (B=1, gamma=16, V=129280 bf16, compact), greedy
    and stochastic (T = 0.7): `steps` consecutive steps cycling through `pool` seeded inputs
    (the pool's logits exceed L2), launched eagerly (the fused calls: three kernels per greedy
    step, four per stochastic step), as one CUDA graph replay per step, and as one graph
    holding a whole pool cycle (the GPU-side step time)."""
    from speculative_decoding_ragged_gb300 import synth
    from speculative_decoding_ragged_gb300.step import DSparkGraph, DSparkStep
    wl = synth.WORKLOADS["latency_b1"]
    out = {"steps": steps, "pool_blocks": pool}
    for stochastic in (False, True):
        st = DSparkStep(wl.B, wl.gamma, wl.V, wl.tiers, wl.bias, wl.alpha_slope * np.arange(2),
                        wl.theta_slope * np.arange(wl.gamma + 1), out_cap=16,
                        stochastic=stochastic, device=dev)
        entries = []
        for k in range(pool):
            target, draft = synth.make_logits(wl, seed=0, pool_index=k)
            bt = synth.make_batch(wl, seed=0, step=k, stochastic=stochastic,
                                  logits=(target, draft))
            # B = 1: the packed rows of any window are the block's leading rows
            entries.append((torch.as_tensor(bt.conf, device=dev),
                            torch.as_tensor(bt.tokens, device=dev), bt.target.to(dev),
                            bt.draft.to(dev) if stochastic else None))
        kw = dict(temperature=wl.temperature, seed=7)
        calls = [st.prepare(*e, step=k, **kw) for k, e in enumerate(entries)]
        graphs = [DSparkGraph(st, *e, step_index=k, **kw) for k, e in enumerate(entries)]
        cycle = torch.cuda.CUDAGraph()
        with torch.cuda.graph(cycle):
            for k, e in enumerate(entries):
                for c in st.prepare(*e, step=k, **kw):
                    c()
        stream = torch.cuda.current_stream()
        name = "stochastic" if stochastic else "greedy"
        out[f"{name}_launches_per_step"] = st.launches_per_step
        for mode in ("eager", "graph", "graph_cycle"):
            def one(i):
                if mode == "eager":
                    for c in calls[i % pool]:
                        c()
                elif mode == "graph":
                    graphs[i % pool].replay()
                elif i % pool == 0:
                    cycle.replay()
            n = steps - steps % pool
            for i in range(2 * pool):
                one(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n):
                one(i)
            e1.record(stream)
            torch.cuda.synchronize()
            out[f"{name}_step_us_{mode}"] = e0.elapsed_time(e1) * 1e3 / n
        out["pool_mb"] = round(sum(sum(t.numel() * t.element_size() for t in e[2:] if t is not None)
                                   for e in entries) / 1e6, 1)
        del graphs, cycle, calls, entries
    return out


def stream_kernel_name(wl, args):
    """The streaming kernel this run used: the one asked for, else the library's default for
    the workload's full size (B*gamma rows of V logits; the bulk kernel from 64 MB)."""
    if args.stream_kernel == "bulk":
        return "TMA bulk-copy kernel"
    if args.stream_kernel == "register":
        return "register-streaming kernel"
    full = wl.B * wl.gamma * wl.V * (2 if wl.dtype == "bf16" else 4)
    return "TMA bulk-copy kernel" if full >= (64 << 20) else "register-streaming kernel"


def percentile(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


# (workload, mode, stochastic): the other workloads' verify launches, timed alone
CONFIG_LEGS = [("stochastic", "compact", True), ("stochastic", "cap_accept", True),
               ("high_load", "compact", False), ("high_load", "cap_accept", False)]


def config_legs(dev, reps):
    """Roofline of dspark_verify_scatter (stream + finalize with the fused scatter, + the bonus
    kernel when stochastic) on the other workloads, each launch timed alone with CUDA events on
    its stream after an L2 flush (a 256 MB buffer read between launches). Windows come from
    the library's own schedule. Algorithmic bytes: the target rows the mode verifies (M
    compact, B*gamma cap-accept), the draft rows of the tested drafts (stochastic: M - B
    compact, B*(gamma-1) cap-accept) and the bonus pass (two rows per request that rejected,
    one per request that accepted its whole window), each V*e bytes."""
    from speculative_decoding_ragged_gb300 import synth
    from speculative_decoding_ragged_gb300.step import DSparkStep
    peak, _ = measured_peak()
    flush = torch.ones(64 << 20, dtype=torch.int32, device=dev)     # 256 MB, read to evict L2
    stream = torch.cuda.current_stream()
    out = {}
    cache = {}
    for name, mode, stochastic in CONFIG_LEGS:
        wl = synth.WORKLOADS[name]
        if name not in cache:
            cache.clear()
            cache[name] = synth.make_batch(wl, seed=77, stochastic=stochastic)
        bt = cache[name]
        B, g, V = wl.B, wl.gamma, wl.V
        e = 2 if wl.dtype == "bf16" else 4
        st = DSparkStep(B, g, V, wl.tiers, bt.bias, bt.alpha, bt.theta, mode=mode,
                        stochastic=stochastic, out_cap=g * (reps + 8), device=dev)
        conf = torch.as_tensor(bt.conf, device=dev)
        tokens = torch.as_tensor(bt.tokens, device=dev)
        st.schedule_pack(conf, tokens)
        torch.cuda.synchronize()
        w = st.windows.cpu().numpy()
        M = int(w.sum())
        if mode == "compact":
            tier = int(st.meta[1].item())
            target = synth.gather_packed(bt.target, B, g, w, rows_cap=tier).to(dev)
        else:
            target = bt.target.to(dev)
        draft = bt.draft.to(dev) if stochastic else None
        call = st.verify_scatter(target, tokens, draft, temperature=wl.temperature, seed=5,
                                 prepare=True)
        for _ in range(3):
            call()
        torch.cuda.synchronize()
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(reps)]
        for e0, e1 in evs:
            torch.max(flush)      # a read: evicts the logits from L2 without leaving dirty lines
            e0.record(stream)
            call()
            e1.record(stream)
        torch.cuda.synchronize()
        us = [e0.elapsed_time(e1) * 1e3 for e0, e1 in evs]
        rows_t = M if mode == "compact" else B * g
        rows_d = 0
        bonus = 0
        if stochastic:
            rows_d = (M - B) if mode == "compact" else B * (g - 1)
            acc = st.accept_len.cpu().numpy()
            bonus = int(np.sum(np.where(acc < w, 2, 1)))
        algo = (rows_t + rows_d + bonus) * V * e
        med = statistics.median(us)
        out[f"{name}/{mode}"] = {
            "B": B, "gamma": g, "V": V, "verify": "stochastic" if stochastic else "greedy",
            "M": M, "algorithmic_bytes": algo, "us_median": med,
            "us_p10_p90": [percentile(us, 10), percentile(us, 90)],
            "gbs": algo / (med * 1e-6) / 1e9, "frac": algo / (med * 1e-6) / 1e9 / peak,
            "frac_of_nominal_8tbs": algo / (med * 1e-6) / 1e9 / NOMINAL_HBM_GBS,
            "launches": 3 if stochastic else 2, "reps": reps, "l2": "flushed between launches"}
        del st, target, draft, call
    del flush
    return out


def oracle_inputs(bt, n_req, packed_bits=None):
    """Host inputs of the oracle's step on the first n_req requests as a batch of their own:
    its confidences, tokens and cost tables, and the packed rows of its own schedule (the
    stand-in for the target forward, prepared off the clock)."""
    import oracle
    from speculative_decoding_ragged_gb300 import synth
    B, g = n_req, bt.gamma
    inp = dict(conf=bt.conf[:B], tokens=bt.tokens[:B], alpha=bt.alpha[:B + 1],
               theta=bt.theta[:B * g + 1], bias=bt.bias, tiers=bt.tiers,
               cap=int(max(int(bt.tiers.max()), B * g)))
    if packed_bits is None:
        w = oracle.schedule(inp["conf"], bt.bias, inp["alpha"], inp["theta"])["windows"]
        packed = synth.gather_packed(bt.target, B, g, w)
        packed_bits = packed.view(torch.int16).numpy().view(np.uint16)
    inp["packed_bits"] = packed_bits
    return inp


def oracle_step(inp):
    """The CPU oracle's whole step; returns the packed rows it verified."""
    import oracle
    s = oracle.schedule(inp["conf"], inp["bias"], inp["alpha"], inp["theta"])
    w = s["windows"]
    p = oracle.pack(w, inp["tokens"], inp["tiers"], inp["cap"])
    v = oracle.verify(oracle.COMPACT, False, inp["packed_bits"], inp["tokens"], cu=p["cu"],
                      windows=w)
    B = w.shape[0]
    oracle.scatter(v["committed"], v["accept_len"], np.full((B, 64), -1, np.int32),
                   np.zeros(B, np.int32))
    return p["M"]


def cpu_baseline(batches, wl, seconds):
    """The oracle as it stands, single-threaded, on whole steps of the same batches until
    `seconds` of CPU work have run (at least one step)."""
    inputs = [oracle_inputs(b["bt"], b["bt"].B,
                            b["packed_h"].view(torch.int16).numpy().view(np.uint16))
              for b in batches]
    rows, n, t0 = 0, 0, time.perf_counter()
    while True:
        rows += oracle_step(inputs[n % len(inputs)])
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    dt = time.perf_counter() - t0
    return {"value": rows / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} whole steps (schedule, pack, compact greedy verify, scatter) of the "
                      f"{wl.name} workload, {rows} packed rows, single thread",
            "cpu": cpu_model(), "host_cores": os.cpu_count()}


ARM_PARTS = {"0xd4f": "Arm Neoverse V2", "0xd40": "Arm Neoverse V1", "0xd0c": "Arm Neoverse N1",
             "0xd49": "Arm Neoverse N2", "0xd8e": "Arm Neoverse N3", "0xd84": "Arm Neoverse V3"}


def cpu_model():
    """The host CPU's model name (x86), or its Arm part number with the core's name."""
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                key = line.lower()
                if key.startswith("model name"):
                    return line.split(":", 1)[1].strip()
                if key.startswith("cpu part"):
                    part = line.split(":", 1)[1].strip().lower()
                    return f"{ARM_PARTS.get(part, 'Arm core')} (CPU part {part})"
    except OSError:
        pass
    return None


def run_reference(args, rank, world):
    """The reference arm: the CPU oracle (the method restated plainly) on this arm's workload,
    each step a bounded sample so the whole run ends within minutes."""
    if rank != 0:
        return None
    import oracle
    from speculative_decoding_ragged_gb300 import synth
    oracle.build()
    wl = synth.WORKLOADS[args.workload]
    bt = synth.make_batch(wl, seed=0)
    full = oracle_inputs(bt, bt.B)
    t0 = time.perf_counter()
    oracle_step(full)
    t_full = time.perf_counter() - t0
    budget = 150.0
    n_req = bt.B
    if (args.steps + args.warmup) * t_full > budget:
        n_req = max(1, int(bt.B * budget / ((args.steps + args.warmup) * t_full)))
    inp = full if n_req == bt.B else oracle_inputs(bt, n_req)
    for _ in range(args.warmup):
        oracle_step(inp)
    rows, t0 = 0, time.perf_counter()
    for _ in range(args.steps):
        rows += oracle_step(inp)
    dt = time.perf_counter() - t0
    value = rows / dt
    sample = (f"each step: the whole oracle step on the first {n_req} of {bt.B} requests of the "
              f"{wl.name} workload, single thread")
    return {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": args.workload, "B": wl.B, "gamma": wl.gamma, "V": wl.V,
                       "mode": "compact", "verify": "greedy", "logits": "bf16",
                       "parallelism": "single CPU thread"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def main():
    args = parse()
    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        out = run_reference(args, rank, world)
    else:
        out = run_native(args, rank, world, local)
    if rank == 0 and out is not None:
        print(json.dumps(out))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
