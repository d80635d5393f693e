"""Step-cost recorder and additive-model check on one GPU.

"DSpark in SGLang" (LMSYS blog summary), A2 method details, cost-table profiling and modelling
(Fig. 6): step times are recorded over batch sizes and verified-token counts, the additive model
T(bs, K) = bias + alpha(bs) + theta(bs + K) is fitted to them, and the fit's predictions are set
against measured steps. The serving engine that produced the pages' records is not part of this
library, so each recorded step here is this library's decode step around a synthetic forward
stand-in with the two cost terms the model separates:

* per-request floor (alpha): a read of a per-request cache slice (`ctx_bytes` per request),
  standing in for the draft pass and the attention reads that grow with the batch size;
* verified-token cost (theta): an LM-head GEMM [tier, H] x [H, V] in bf16 (a cuBLAS call through
  torch) that produces the target logits the step verifies, over the capture tier the packed
  rows are padded to.

Windows are forced (the extra tokens K spread evenly over the requests) so that every (bs, M)
cell of the grid is recorded; the scheduler still runs inside every step. The recorded samples
are split in two: the fit uses one part, the other is predicted and compared.

    python -m speculative_decoding_ragged_gb300.sps_profile [--out FILE.json]
"""
from __future__ import annotations

import argparse
import json
import sys
from typing import Optional, Sequence

import numpy as np
import torch

from . import synth
from .costfit import compare, fit_additive, tier_key
from .step import DSparkStep


def forced_windows(bs: int, gamma: int, M: int) -> np.ndarray:
    """Windows summing to M: 1 + (M - bs) extra tokens spread as evenly as possible."""
    extra = M - bs
    if not 0 <= extra <= (gamma - 1) * bs:
        raise ValueError("M out of range for this batch")
    w = np.full(bs, 1 + extra // bs, np.int32)
    w[: extra % bs] += 1
    return w


class StandIn:
    """The synthetic forward: per-request cache reads plus an LM-head GEMM over tier rows."""

    def __init__(self, max_bs: int, max_rows: int, H: int, V: int, ctx_bytes: int, device):
        g = torch.Generator(device=device).manual_seed(0)
        self.kv = torch.randn(max_bs, ctx_bytes // 2, generator=g, device=device,
                              dtype=torch.bfloat16)
        self.kv_out = torch.empty(max_bs, device=device, dtype=torch.float32)
        self.hidden = (torch.randn(max_rows, H, generator=g, device=device) / H ** 0.5).to(
            torch.bfloat16)
        self.w = torch.randn(H, V, generator=g, device=device, dtype=torch.bfloat16)
        self.logits = torch.empty(max_rows, V, device=device, dtype=torch.bfloat16)

    def __call__(self, bs: int, rows: int) -> torch.Tensor:
        torch.sum(self.kv[:bs], dim=1, dtype=torch.float32, out=self.kv_out[:bs])
        out = self.logits[:rows]
        torch.mm(self.hidden[:rows], self.w, out=out)
        return out


def grid_M(bs: int, gamma: int, tiers: Sequence[int], points: int) -> list:
    """Up to `points` values of M for batch size bs, both ends included: bs, the capture tiers
    between bs and gamma*bs (so that batch sizes share theta entries and the fit is
    over-determined), and gamma*bs, evenly thinned."""
    cand = sorted(set([bs, gamma * bs] + [int(t) for t in tiers if bs < t < gamma * bs]))
    if len(cand) <= points:
        return cand
    idx = np.unique(np.round(np.linspace(0, len(cand) - 1, points)).astype(int))
    return [cand[i] for i in idx]


def record(batch_sizes: Sequence[int], gamma: int = 8, V: int = 151936, H: int = 4096,
           tiers: Optional[Sequence[int]] = None, points: int = 12, ctx_bytes: int = 2 << 20,
           warmup: int = 3, reps: int = 10, device="cuda") -> list:
    """Median step time (us) of every (bs, M) grid cell (grid_M per batch size)."""
    device = torch.device(device)
    tiers = list(tiers) if tiers is not None else list(range(32, 2049, 32))
    max_bs = max(batch_sizes)
    max_rows = int(max(max(tiers), max_bs * gamma))
    fwd = StandIn(max_bs, max_rows, H, V, ctx_bytes, device)
    wl = synth.WORKLOADS["large_vocab_mixed"].with_(V=64)
    samples = []
    for bs in batch_sizes:
        alpha = np.zeros(bs + 1)
        theta = 0.004 * np.arange(bs * gamma + 1)
        st = DSparkStep(bs, gamma, V, tiers, 1.0, alpha, theta, device=device)
        bt = synth.make_batch(wl.with_(B=bs, gamma=gamma), seed=bs)
        conf = torch.as_tensor(bt.conf, device=device)
        tokens = torch.as_tensor(bt.tokens, device=device)
        for M in grid_M(bs, gamma, tiers, points):
            w = torch.as_tensor(forced_windows(bs, gamma, M), device=device)
            rows = int(tier_key([M], tiers)[0])

            def step():
                st.schedule(conf)
                st.windows.copy_(w)
                st.pack(tokens)
                logits = fwd(bs, rows)
                st.verify(logits, tokens)
                st.scatter()
                st.out_len.zero_()

            for _ in range(warmup):
                step()
            times = []
            for _ in range(reps):
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                torch.cuda.synchronize()
                e0.record()
                step()
                e1.record()
                torch.cuda.synchronize()
                times.append(e0.elapsed_time(e1) * 1e3)
            if int(st.meta[0].item()) != M or int(st.meta[1].item()) != rows:
                raise RuntimeError("packed rows differ from the forced windows")
            samples.append(dict(bs=bs, M=M, tier=rows, us=float(np.median(times))))
        del st
    return samples


def evaluate(samples: list, tiers: Optional[Sequence[int]]) -> dict:
    """Fit on two of every three cells of each batch size (the ends always in) and predict the
    third; a held-out cell whose key no training cell shares is predicted by interpolation."""
    bs = np.array([s["bs"] for s in samples])
    M = np.array([s["M"] for s in samples])
    T = np.array([s["us"] for s in samples])
    train = np.ones(bs.size, bool)
    for b in np.unique(bs):
        idx = np.flatnonzero(bs == b)
        train[idx[1:-1][1::3]] = False
    fit = fit_additive(bs[train], M[train], T[train], tiers=tiers)
    held = ~train
    return dict(
        fit=dict(bias_us=fit.bias, bs_knots=fit.bs_knots.tolist(),
                 alpha_us=fit.alpha_knots.tolist(), tier_knots=fit.key_knots.tolist(),
                 theta_us=fit.theta_knots.tolist(), residual_rms_us=fit.residual_rms,
                 n_train=int(train.sum())),
        train=compare(fit, bs[train], M[train], T[train]),
        held_out=compare(fit, bs[held], M[held], T[held]) if held.any() else None,
        rows=[dict(s, predicted_us=float(p), held_out=bool(h))
              for s, p, h in zip(samples, fit.predict(bs, M), held)],
    )


def main(argv=None) -> int:
    ap = argparse.ArgumentParser(description=__doc__.splitlines()[0])
    ap.add_argument("--batch-sizes", default="1,2,4,8,16,24,32,48,64,96,128,192,256")
    ap.add_argument("--gamma", type=int, default=8)
    ap.add_argument("--V", type=int, default=151936)
    ap.add_argument("--H", type=int, default=4096)
    ap.add_argument("--points", type=int, default=12)
    ap.add_argument("--reps", type=int, default=10)
    ap.add_argument("--out", default=None)
    a = ap.parse_args(argv)
    if not torch.cuda.is_available():
        print("a CUDA device is required", file=sys.stderr)
        return 2
    tiers = list(range(32, 2049, 32))
    bss = [int(x) for x in a.batch_sizes.split(",")]
    samples = record(bss, gamma=a.gamma, V=a.V, H=a.H, tiers=tiers, points=a.points,
                     reps=a.reps)
    res = evaluate(samples, tiers)
    res["config"] = dict(gamma=a.gamma, V=a.V, H=a.H, tiers="32..2048 step 32",
                         batch_sizes=bss, points=a.points, reps=a.reps,
                         device=torch.cuda.get_device_name())
    text = json.dumps(res)
    if a.out:
        with open(a.out, "w") as f:
            f.write(text + "\n")
    print(json.dumps(dict(train=res["train"], held_out=res["held_out"],
                          bias_us=res["fit"]["bias_us"])))
    return 0


if __name__ == "__main__":
    sys.exit(main())
