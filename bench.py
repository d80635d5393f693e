#!/usr/bin/env python3
"""Benchmark of the DSpark ragged-verification hot path on GB300.

One step = the whole hot path on one batch: schedule, pack, verify (compact, greedy) and the
compact scatter, issued as the two fused calls dspark_schedule_pack and dspark_verify_scatter,
on the large-vocab mixed-traffic workload (B=256 requests, block gamma=8, V=151936 bf16
logits, three acceptance classes a = 0.9/0.65/0.35, theta(M) = 0.004 M, alpha(bs) = 0.01 bs,
bias 2, tiers every 32 up to 2048). The packed target logits of the scheduled windows are
produced off the clock (they stand in for the target model's forward) and stay resident; three
seeded batches rotate so every step reads more than L2 holds.

Prints one JSON line.
  value        packed verify rows per second over whole steps, inputs resident in HBM (events
               around the K timed steps only, nothing recorded between a step's kernels; a
               sleep kernel holds the GPU while the host enqueues them, so host speed does not
               enter; the host's cost per step is reported under `timing`);
  e2e          the same rows/s with the step's inputs copied from pinned host memory and the
               results read back inside the timed region;
  legs         every workload timed alone: each of >= 30 launches after an L2 flush, events
               around the whole verify call and (recorded by the library) around its streaming
               kernel, plus the schedule-and-pack call; rows/s, GB/s and the fraction of the
               measured and nominal HBM peaks, with p10/p90; the high-load workload at each
               theta of its sweep in compact and cap-accept mode; the oracle timed per workload;
  roofline     the large-vocab leg's streaming kernel: algorithmic bytes (M * V * 2 per launch)
               over its mean event time, against the measured HBM copy bandwidth;
  latency_b1   per-step time of the batch-1 workload over consecutive steps;
  cpu_baseline the CPU oracle on a bounded sample of the headline workload;
  clocks       nvidia-smi samples over the whole measured region (headline, e2e, legs).

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
TRAFFIC_RECORD = os.path.join(ROOT, "profiles", "verify_stream_traffic.json")
N_BATCHES = 3
CHAINED_CALLS = 256      # back-to-back calls per chained timing in each workload leg


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="oracle time on the headline workload")
    ap.add_argument("--cpu-seconds-leg", type=float, default=3.0,
                    help="oracle time on each other workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--batches", type=int, default=N_BATCHES)
    ap.add_argument("--latency-steps", type=int, default=10000)
    ap.add_argument("--stream-kernel", default="auto", choices=["auto", "register", "bulk"],
                    help="which logit-streaming kernel verify uses (results are identical)")
    ap.add_argument("--config-reps", type=int, default=40,
                    help="timed launches per workload leg (0: skip the legs)")
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


def whole_job(ms_local, rows_local, world):
    """The job's time (the slowest rank's), rows (every rank's) and rows/s over all ranks."""
    ms = max_over_ranks(ms_local, world)
    rows = sum_over_ranks(rows_local, world)
    return ms, rows, rows / (ms * 1e-3)


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def traffic_ratio():
    """DRAM bytes over algorithmic bytes of the captured full-size streaming launch (the JSON
    record under profiles/), while the source files it names still hash to the value recorded
    with it; None once the kernel has changed since the counters were taken."""
    try:
        with open(TRAFFIC_RECORD) as f:
            rec = json.load(f)
        h = hashlib.sha256()
        for name in rec["sources"]:
            with open(os.path.join(ROOT, "speculative_decoding_ragged_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
        if h.hexdigest()[:16] != rec["sources_sha256_16"]:
            return None
        return float(rec["traffic_over_algorithmic"])
    except (OSError, KeyError, ValueError, TypeError):
        return None


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the GPU is measured."""
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
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"],
                    "samples": 0}
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
        sm, mx, pw, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 10:
                continue
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
                pw.append(float(r[4]))
            except ValueError:
                continue
            for name, val in zip(names, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm), "sm_mhz_min": min(sm) if sm else None,
                "power_w_max": max(pw) if pw else None,
                "region": "headline steps, e2e steps, workload legs and the batch-1 leg"}


def percentile(xs, q):
    return float(np.percentile(np.asarray(xs, dtype=np.float64), q))


def spread(xs):
    return {"median": statistics.median(xs), "mean": statistics.mean(xs),
            "p10": percentile(xs, 10), "p90": percentile(xs, 90), "n": len(xs)}


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
        target = bt.target.to(dev)
        packed = synth.gather_packed(target, bt.B, bt.gamma, w, rows_cap=tier)
        del target
        batches.append(dict(
            bt=bt, windows=w, M=M, conf=conf,
            tokens=torch.as_tensor(bt.tokens, device=dev), packed=packed,
            conf_h=torch.as_tensor(bt.conf).pin_memory(),
            tokens_h=torch.as_tensor(bt.tokens).pin_memory(),
            packed_h=packed.cpu().pin_memory()))
    st.status.zero_()
    return batches


class LegTimer:
    """Times calls one at a time: before each, `pre` (history reset) and an L2 flush (a 256 MB
    read, long enough that the host has queued the call before the GPU reaches it); events
    around the call, or (recorded by the library) around its logit-streaming kernel alone (an
    event between two kernels costs the second its early launch, so the two are timed in
    separate passes)."""

    def __init__(self, dev):
        from speculative_decoding_ragged_gb300 import _binding as bd
        self.bd = bd
        self.flush = torch.ones(64 << 20, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream()

    def run(self, call, reps, pre=None, stream_events=True):
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(reps)]
        for e in ev:                      # torch creates events lazily: make them exist
            for x in e:
                x.record(self.stream)
        torch.cuda.synchronize()
        for e in ev:
            if pre is not None:
                pre()
            torch.max(self.flush)         # a read: evicts the inputs without dirtying L2
            e[0].record(self.stream)
            if stream_events:
                self.bd.set_stream_events(e[1], e[2])
            call()
            if stream_events:
                self.bd.set_stream_events(None, None)
            e[3].record(self.stream)
        torch.cuda.synchronize()
        call_us = [e[0].elapsed_time(e[3]) * 1e3 for e in ev]
        stream_us = [e[1].elapsed_time(e[2]) * 1e3 for e in ev] if stream_events else None
        return call_us, stream_us


def leg_record(name, wl, mode, stochastic, M, rows_t, rows_d, bonus_rows, call_us, stream_us,
               sp_us, step_us, peak, extra=None):
    """One workload leg: algorithmic bytes (target rows the mode verifies, draft rows of the
    tested drafts, bonus rows) per call, rows/s over the whole call, GB/s and fractions."""
    e = 2 if wl.dtype == "bf16" else 4
    algo = (rows_t + rows_d + bonus_rows) * wl.V * e
    stream_bytes = (rows_t + rows_d) * wl.V * e
    call = spread(call_us)
    rec = {"workload": name, "B": wl.B, "gamma": wl.gamma, "V": wl.V, "dtype": wl.dtype,
           "verify": "stochastic" if stochastic else "greedy", "mode": mode, "M": M,
           "rows_streamed": rows_t + rows_d, "bonus_rows": bonus_rows,
           "algorithmic_bytes": algo,
           "call_us": call, "rows_per_s": M / (call["median"] * 1e-6),
           "call_gbs": algo / (call["mean"] * 1e-6) / 1e9,
           "call_frac": algo / (call["mean"] * 1e-6) / 1e9 / peak,
           "call_frac_of_nominal_8tbs": algo / (call["mean"] * 1e-6) / 1e9 / NOMINAL_HBM_GBS}
    if stream_us is not None:
        s = spread(stream_us)
        rec.update({"stream_us": s, "stream_bytes": stream_bytes,
                    "stream_gbs": stream_bytes / (s["mean"] * 1e-6) / 1e9,
                    "stream_frac": stream_bytes / (s["mean"] * 1e-6) / 1e9 / peak})
    if sp_us is not None:
        rec["sched_pack_us"] = spread(sp_us)
    if step_us is not None:
        rec["step_us"] = spread(step_us)
    rec["l2"] = "flushed (256 MB read) before every timed call"
    if extra:
        rec.update(extra)
    return rec


def step_for(wl, bt, mode, stochastic, dev, out_cap):
    from speculative_decoding_ragged_gb300.step import DSparkStep
    return DSparkStep(wl.B, wl.gamma, wl.V, wl.tiers, bt.bias, bt.alpha, bt.theta, mode=mode,
                      stochastic=stochastic, out_cap=out_cap, device=dev)


def run_leg(timer, name, wl, bt, mode, stochastic, dev, reps, target_full, draft, peak,
            extra=None, batches=None):
    """One workload leg: windows from the library's own schedule (off the clock), packed rows
    gathered on the device, then `reps` timed verify calls, schedule-and-pack calls and whole
    steps. `batches` (the headline's) rotate instead of one batch when given."""
    from speculative_decoding_ragged_gb300 import synth
    B, g = wl.B, wl.gamma
    # histories deep enough for every call of a chained timing (64 + 2 * CHAINED_CALLS)
    st = step_for(wl, bt, mode, stochastic, dev, out_cap=g * 3 * CHAINED_CALLS)
    kw = dict(temperature=wl.temperature, seed=5, step=0)
    entries = []
    for b in (batches or [None]):
        conf = b["conf"] if b else torch.as_tensor(bt.conf, device=dev)
        tokens = b["tokens"] if b else torch.as_tensor(bt.tokens, device=dev)
        st.schedule_pack(conf, tokens)
        torch.cuda.synchronize()
        w = st.windows.cpu().numpy()
        M = int(w.sum())
        if b is not None:
            target = b["packed"]
        elif mode == "compact":
            target = synth.gather_packed(target_full, B, g, w, rows_cap=int(st.meta[1].item()))
        else:
            target = target_full
        entries.append(dict(conf=conf, tokens=tokens, target=target, M=M, w=w))
    verify = [st.verify_scatter(e["target"], e["tokens"], draft, prepare=True, **kw)
              for e in entries]
    sched = [st.schedule_pack(e["conf"], e["tokens"], prepare=True) for e in entries]
    steps = [st.prepare(e["conf"], e["tokens"], e["target"], draft, **kw) for e in entries]
    n = len(entries)
    reset = st.out_len.zero_
    for k in range(3):
        sched[k % n]()
        verify[k % n]()
        reset()
    torch.cuda.synchronize()
    # verify alone needs the windows and cu_seqlens of its own batch: one batch at a time;
    # the whole call without events inside it, then the streaming kernel alone
    call_us, stream_us = [], []
    for k in range(n):
        sched[k]()
        r = (reps + n - 1 - k) // n
        c, _ = timer.run(verify[k], r, pre=reset, stream_events=False)
        _, s = timer.run(verify[k], r, pre=reset)
        call_us += c
        stream_us += s
    st.out_len.zero_()
    sp_us, _ = timer.run(lambda: sched[0](), reps, stream_events=False)
    it = iter(range(10 ** 9))

    def whole():
        k = next(it) % n
        for c in steps[k]:
            c()
    step_us, _ = timer.run(whole, reps, pre=reset, stream_events=False)
    torch.cuda.synchronize()
    # the same calls back to back, as a serving loop issues them (host held ahead of the GPU):
    # device time per call of schedule-and-pack, of verify on the first batch's windows, and of
    # whole steps with the batches rotating; inputs stay in L2 when they fit (below 129 MB)
    stream = torch.cuda.current_stream()
    chained = {}
    st.out_len.zero_()
    chained["sched_pack_us"] = host_and_device_us(lambda i: sched[i % n](), CHAINED_CALLS,
                                                  stream)[1]
    sched[0]()
    st.out_len.zero_()
    chained["verify_us"] = host_and_device_us(lambda i: verify[0](), CHAINED_CALLS, stream)[1]
    st.out_len.zero_()
    chained["step_us"] = host_and_device_us(lambda i: whole(), CHAINED_CALLS // 2, stream)[1]
    st.out_len.zero_()
    torch.cuda.synchronize()
    Ms = [e["M"] for e in entries]
    M = statistics.mean(Ms)
    rows_t = M if mode == "compact" else B * g
    rows_d = 0
    bonus = 0
    if stochastic:
        rows_d = (M - B) if mode == "compact" else B * (g - 1)
        # the bonus pass of the last batch: two rows per request that rejected a draft
        # (residual of target and draft rows), one per request that accepted its whole window
        sched[-1]()
        verify[-1]()
        torch.cuda.synchronize()
        acc = st.accept_len.cpu().numpy()
        bonus = int(np.sum(np.where(acc < entries[-1]["w"], 2, 1)))
    ex = {"launches_per_call": st.launches_per_step - (1 if g > 1 else 2),
          "launches_per_step": st.launches_per_step, "reps": len(call_us),
          "batches_rotating": n, "status": int(st.status.item()), "chained": chained}
    if extra:
        ex.update(extra)
    return leg_record(name, wl, mode, stochastic, M, rows_t, rows_d, bonus, call_us, stream_us,
                      sp_us, step_us, peak, ex)


def workload_legs(dev, reps, headline_batches, args):
    """Every workload of the benchmark, each verify call timed alone (see LegTimer)."""
    from speculative_decoding_ragged_gb300 import synth
    peak, _ = measured_peak()
    timer = LegTimer(dev)
    legs = {}
    # large-vocab mixed (the headline workload): its own rotating batches
    wl = synth.WORKLOADS["large_vocab_mixed"]
    legs["large_vocab_mixed/compact"] = run_leg(
        timer, "large_vocab_mixed", wl, headline_batches[0]["bt"], "compact", False, dev, reps,
        None, None, peak, batches=headline_batches)
    # tiny greedy, stochastic, batch-1 (greedy and stochastic T = 0.7)
    for name, modes, samplers in (("tiny_greedy", ("compact",), (False,)),
                                  ("stochastic", ("compact", "cap_accept"), (True,)),
                                  ("latency_b1", ("compact",), (False, True))):
        wl = synth.WORKLOADS[name]
        for stochastic in samplers:
            bt = synth.make_batch(wl, seed=77, stochastic=stochastic)
            target = bt.target.to(dev)
            draft = bt.draft.to(dev) if stochastic else None
            for mode in modes:
                key = f"{name}/{mode}" + ("/stochastic" if name == "latency_b1" and stochastic else "")
                legs[key] = run_leg(timer, name, wl, bt, mode, stochastic, dev, reps, target,
                                    draft, peak)
            del target, draft
    # high load: the theta sweep, compact and cap-accept, one logits block shared
    wl = synth.WORKLOADS["high_load"]
    bt = synth.make_batch(wl, seed=77)
    target = bt.target.to(dev)
    for theta in synth.HIGH_LOAD_THETAS:
        bt.theta = theta * np.arange(wl.B * wl.gamma + 1, dtype=np.float64)
        for mode in ("compact", "cap_accept"):
            legs[f"high_load/theta{theta}/{mode}"] = run_leg(
                timer, "high_load", wl, bt, mode, False, dev, reps, target, None, peak,
                extra={"theta_slope": theta})
    del target, timer
    torch.cuda.empty_cache()
    return legs


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

    def step(i):
        # fused calls: dspark_schedule_pack, then dspark_verify_scatter (whose compact scatter
        # runs inside the kernel that decides each request's tokens)
        for c in calls[i % nb]:
            c()

    for i in range(args.warmup):
        step(i)
        st.out_len.zero_()
    torch.cuda.synchronize()
    # the host's time to enqueue one step (a few more untimed steps)
    t0 = time.perf_counter()
    for i in range(8):
        step(i)
    host_step_s = (time.perf_counter() - t0) / 8
    torch.cuda.synchronize()
    st.out_len.zero_()

    # device-resident timed region: K whole steps, events around the loop only. A sleep kernel
    # holds the GPU while the host enqueues the steps, so the events time the GPU running them
    # back to back (with their programmatic-dependent-launch overlap) whatever the host's speed:
    # a slow or contended host would otherwise leave the GPU idle between launches and count
    # the gaps. The host's own cost per step is reported beside it, and the end-to-end leg
    # below includes it.
    K = args.steps
    t_start, t_end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world)
    torch.cuda.synchronize()
    held = hold_gpu(host_step_s * K)
    t_start.record(stream)
    for i in range(K):
        step(i)
    t_end.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    ms, rows, value = whole_job(t_start.elapsed_time(t_end),
                                sum(batches[i % nb]["M"] for i in range(K)), world)

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
    # untimed: one copy of every batch's host inputs, so that the first transfers from each
    # pinned buffer (measured at 75-180 GB/s against about 210 GB/s after) are not timed
    with torch.cuda.stream(copy_stream):
        for j, b in enumerate(batches):
            inbuf[j % 2]["pk"][: b["M"]].copy_(b["packed_h"][: b["M"]], non_blocking=True)
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
    del inbuf

    legs = None
    if args.config_reps > 0 and rank == 0:
        legs = workload_legs(dev, max(args.config_reps, 1), batches, args)
    latency = latency_leg(dev, args.latency_steps) if args.latency_steps > 0 else None
    clk = clocks.stop()

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(batches, wl, args.cpu_seconds)
        if legs is not None:
            oracle_legs(legs, args.cpu_seconds_leg)
    if rank != 0:
        return None
    peak, peak_kind = measured_peak()
    out = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": args.workload, "B": wl.B, "gamma": wl.gamma, "V": wl.V,
                   "mode": "compact", "verify": "greedy", "logits": "bf16",
                   "stream_kernel": args.stream_kernel,
                   "batches_rotating": nb, "rows_per_step_mean": rows / K / world,
                   "l2": "inputs larger than L2: each step reads >=300 MB of packed logits, "
                         f"{nb} batches rotate; legs flush L2 before every timed call",
                   "parallelism": f"replicas{world}" if world > 1 else "single GPU"},
        "step_us": ms / K * 1e3,
        "timing": {"what": "CUDA events around the K timed steps on the launching stream",
                   "host_held": held,
                   "how": "a sleep kernel held the GPU while the host enqueued the steps, so "
                          "the events time the GPU running them back to back" if held else
                          "steps enqueued as the GPU ran them",
                   "host_us_per_step": host_step_s * 1e6},
        "cpu_baseline": cpu,
        "e2e": {"value": e2e_rows / (e2e_ms * 1e-3), "unit": UNIT,
                "h2d_bytes_per_step": h2d // max(E, 1), "d2h_bytes_per_step": d2h // max(E, 1),
                "steps": E, "h2d_gbs": h2d / (e2e_ms * 1e-3) / 1e9,
                "overlap": "next step's copy on its own stream during this step's compute"},
        "gpu_launches": K * st.launches_per_step,
        "clocks": clk,
        "latency_b1": latency,
        "legs": legs,
    }
    if legs is not None:
        lv = legs["large_vocab_mixed/compact"]
        ratio = traffic_ratio()
        per_launch = lv["stream_bytes"]
        s_mean = lv["stream_us"]["mean"]
        achieved = per_launch / (s_mean * 1e-6) / 1e9
        out["sched_pack_us"] = lv["sched_pack_us"]["median"]
        out["verify_us"] = lv["call_us"]["median"]
        out["logits_gbs"] = lv["call_gbs"]
        out["roofline"] = {
            "bound": "hbm", "kernel": f"verify streaming kernel ({stream_kernel_name(wl, args)})",
            "achieved": achieved, "peak": peak, "peak_source": peak_kind, "unit": "GB/s",
            "frac": achieved / peak,
            "traffic": None if ratio is None else ratio * per_launch,
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS,
            "algorithmic_bytes_per_launch": per_launch,
            "launch_us_mean": s_mean, "launch_us_p10_p90": [lv["stream_us"]["p10"],
                                                            lv["stream_us"]["p90"]],
            "samples": lv["stream_us"]["n"],
            "timing": "CUDA events on the launching stream around each launch, one launch "
                      "at a time after an L2 flush; the 3 headline batches rotate",
            "verify_call": {"what": "dspark_verify_scatter, the whole call",
                            "achieved": lv["call_gbs"], "frac": lv["call_frac"],
                            "us_mean": lv["call_us"]["mean"],
                            "us_p10_p90": [lv["call_us"]["p10"], lv["call_us"]["p90"]]}}
    return out


def hold_gpu(host_seconds):
    """Enqueues a sleep kernel long enough for the host to enqueue work that takes it about
    host_seconds (capped at 0.25 s); False where this torch has no sleep kernel."""
    if not hasattr(torch.cuda, "_sleep"):
        return False
    torch.cuda._sleep(int(2.07e9 * min(host_seconds * 1.5 + 2e-3, 0.25)))   # cycles at max clock
    return True


def host_and_device_us(fn, n, stream):
    """(host submission us, device us) per call of fn: the host's time to enqueue n calls while
    a sleep kernel holds the GPU (so no launch waits on the GPU), and the GPU's time for the n
    calls back to back once the sleep ends (events after it). (None, None) where this torch
    has no sleep kernel."""
    if not hasattr(torch.cuda, "_sleep"):
        return None, None
    for i in range(64):
        fn(i)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for i in range(n):
        fn(i)
    rough = (time.perf_counter() - t0) / n
    torch.cuda.synchronize()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda._sleep(int(2.07e9 * (rough * n * 1.5 + 2e-3)))    # cycles at the maximum clock
    t0 = time.perf_counter()
    e0.record(stream)
    for i in range(n):
        fn(i)
    e1.record(stream)
    host = (time.perf_counter() - t0) / n * 1e6
    torch.cuda.synchronize()
    return host, e0.elapsed_time(e1) * 1e3 / n


def latency_leg(dev, steps, pool=64):
    """Per-step time of the batch-1 workload (B=1, gamma=16, V=129280 bf16, compact), greedy
    and stochastic (T = 0.7), `steps` consecutive steps cycling through `pool` seeded inputs
    (the pool's logits exceed L2): launched eagerly (the fused calls through ctypes) and as one
    graph holding a whole pool cycle (the GPU-side step time). Beside them, host submission
    and device time per step of each way to issue a step (host_and_device_us): eager, one
    graph per pool entry (rotating), and one graph on fixed buffers replayed every step (how a
    serving loop replays: new inputs land in the captured buffers; its logits stay in L2 at
    this size, as do those of the eager step on the same buffers beside it)."""
    from speculative_decoding_ragged_gb300 import _binding as bd
    from speculative_decoding_ragged_gb300 import synth
    from speculative_decoding_ragged_gb300.step import DSparkGraph, DSparkStep
    wl = synth.WORKLOADS["latency_b1"]
    out = {"steps": steps, "pool_blocks": pool}
    stream = torch.cuda.current_stream()
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
        # one graph holding a whole pool cycle, captured through the library's C ABI
        capture = torch.cuda.Stream(device=dev)
        with torch.cuda.stream(capture):
            cycle_calls = [st.prepare(*e, step=k, **kw) for k, e in enumerate(entries)]
            cycle = bd.StepGraph(capture)
            for cc in cycle_calls:
                for c in cc:
                    c()
            cycle.end()
        cycle_launch = cycle.prepare_launch()
        name = "stochastic" if stochastic else "greedy"
        out[f"{name}_launches_per_step"] = st.launches_per_step

        def eager(i):
            for c in calls[i % pool]:
                c()

        def eager_static(i):
            for c in calls[0]:
                c()

        def cycle_step(i):
            if i % pool == 0:
                cycle_launch()

        # the consecutive-step timings of the workload: wall time per step on the device
        n = steps - steps % pool
        for mode, fn in (("eager", eager), ("graph_cycle", cycle_step)):
            for i in range(2 * pool):
                fn(i)
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for i in range(n):
                fn(i)
            e1.record(stream)
            torch.cuda.synchronize()
            out[f"{name}_step_us_{mode}"] = e0.elapsed_time(e1) * 1e3 / n
        # host submission against device time, each way of issuing a step
        # (eager: 128 steps, 384 launches, stay under the launch queue's depth while the GPU
        # is held; more would block the host and count the GPU's time as the host's)
        for mode, fn, reps in (("eager", eager, 128), ("eager_static", eager_static, 128),
                               ("graph_rotating", lambda i: graphs[i % pool].replay(), 384),
                               ("graph_static", lambda i: graphs[0].replay(), 384),
                               ("graph_cycle", lambda i: cycle_launch(), 16)):
            host, devus = host_and_device_us(fn, reps, stream)
            per = pool if mode == "graph_cycle" else 1
            out[f"{name}_{mode}"] = {"host_us": None if host is None else host / per,
                                     "device_us": None if devus is None else devus / per}
        out["pool_mb"] = round(sum(sum(t.numel() * t.element_size() for t in e[2:] if t is not None)
                                   for e in entries) / 1e6, 1)
        del graphs, cycle, cycle_launch, cycle_calls, calls, entries
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


def _bits(t):
    t = t.contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def oracle_inputs(bt, n_req, mode="compact", stochastic=False):
    """Host inputs of the oracle's step on the first n_req requests as a batch of their own:
    its confidences, tokens, cost tables, and the target rows its mode verifies (compact: the
    packed rows of the oracle's own schedule), prepared off the clock as the stand-in for the
    target forward."""
    import oracle
    from speculative_decoding_ragged_gb300 import synth
    B, g = n_req, bt.gamma
    inp = dict(conf=bt.conf[:B], tokens=bt.tokens[:B], alpha=bt.alpha[:B + 1],
               theta=bt.theta[:B * g + 1], bias=bt.bias, tiers=bt.tiers,
               cap=int(max(int(bt.tiers.max()), B * g)), mode=mode, stochastic=stochastic,
               temperature=bt.wl.temperature)
    if mode == "compact":
        w = oracle.schedule(inp["conf"], bt.bias, inp["alpha"], inp["theta"])["windows"]
        inp["target_bits"] = _bits(synth.gather_packed(bt.target, B, g, w))
    else:
        inp["target_bits"] = _bits(bt.target[:B * g])
    inp["draft_bits"] = _bits(bt.draft[:B * (g - 1)]) if stochastic else None
    return inp


def oracle_step(inp):
    """The CPU oracle's whole step; returns the packed rows it verified."""
    import oracle
    s = oracle.schedule(inp["conf"], inp["bias"], inp["alpha"], inp["theta"])
    w = s["windows"]
    p = oracle.pack(w, inp["tokens"], inp["tiers"], inp["cap"])
    mode = oracle.COMPACT if inp["mode"] == "compact" else oracle.CAP_ACCEPT
    v = oracle.verify(mode, inp["stochastic"], inp["target_bits"], inp["tokens"], cu=p["cu"],
                      windows=w, draft=inp["draft_bits"], temperature=inp["temperature"],
                      seed=5, step=0)
    B = w.shape[0]
    oracle.scatter(v["committed"], v["accept_len"], np.full((B, 64), -1, np.int32),
                   np.zeros(B, np.int32))
    return p["M"]


def time_oracle(inputs, seconds):
    rows, n, t0 = 0, 0, time.perf_counter()
    while True:
        rows += oracle_step(inputs[n % len(inputs)])
        n += 1
        if time.perf_counter() - t0 >= seconds:
            break
    return rows, n, time.perf_counter() - t0


def cpu_baseline(batches, wl, seconds):
    """The oracle as it stands, single-threaded, on whole steps of the same batches until
    `seconds` of CPU work have run (at least one step)."""
    inputs = [oracle_inputs(b["bt"], b["bt"].B) for b in batches]
    rows, n, dt = time_oracle(inputs, seconds)
    return {"value": rows / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} whole steps (schedule, pack, compact greedy verify, scatter) of the "
                      f"{wl.name} workload, {rows} packed rows, single thread",
            "cpu": cpu_model(), "host_cores": os.cpu_count()}


def oracle_legs(legs, seconds):
    """The oracle's rows/s beside each workload leg (single thread, bounded sample; the
    high-load sweep at its middle theta in both modes)."""
    from speculative_decoding_ragged_gb300 import synth
    done = {}
    for key, leg in legs.items():
        name = leg["workload"]
        if name == "large_vocab_mixed":
            continue
        theta = leg.get("theta_slope")
        if theta is not None and theta != 0.004:
            continue
        wl = synth.WORKLOADS[name]
        stochastic = leg["verify"] == "stochastic"
        tag = (name, stochastic)
        if tag not in done:
            done[tag] = synth.make_batch(wl, seed=77, stochastic=stochastic)
        bt = done[tag]
        inp = oracle_inputs(bt, bt.B, leg["mode"], stochastic)
        rows, n, dt = time_oracle([inp], seconds)
        leg["oracle"] = {"rows_per_s": rows / dt, "cores": 1, "kind": "oracle",
                         "sample": f"{n} whole steps of this workload and mode, single thread",
                         "gpu_over_oracle": leg["rows_per_s"] / (rows / dt)}


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
