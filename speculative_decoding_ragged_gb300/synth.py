"""Seeded synthetic workloads for the DSpark ragged-verification hot path.

This module only generates inputs: confidences, block tokens, target and draft logits, cost
tables and capture tiers, shaped like the five workloads below. It contains none of the
method's arithmetic (no survivals, no scheduling, no verify) and is the one module both the CUDA
path's tests/benchmark and the CPU oracle's tests draw inputs from.

The pages measure on real serving traffic (gsm8k / arena-hard / poetry mixed requests and a
fixed GSM8K prompt sweep on DeepSeek-V4 models); those datasets and models are not used. These
synthetic recipes stand in for them: acceptance classes stand in for easy / medium / hard
traffic ("DSpark in SGLang", A3 mixed traffic, figure 4), logits are Gaussian with a planted
peak, confidences are Beta-distributed around each request's acceptance rate.

Recipes (all from ``numpy.random.default_rng`` seeded with ``(seed, step, tag)``):
  * target logits ~ N(0, sigma^2) per entry (+ ``spike`` at one uniform id per row), rounded to
    the workload dtype (bf16 rounds to nearest even);
  * greedy drafts: d_j equals the argmax of target row j-1 with probability a_b, else a uniform
    other id;
  * stochastic drafts: draft logits = target logits + N(0, draft_sigma^2), rounded to the dtype;
    d_j is sampled from softmax(draft row j-1 / temperature) (Gumbel-max);
  * confidences c[b, j] ~ Beta(conc * a_b, conc * (1 - a_b));
  * cost tables alpha[bs] = alpha_slope * bs (bs = 0..B), theta[M] = theta_slope * M
    (M = 0..B*gamma), scalar bias.
"""
from __future__ import annotations

import dataclasses
from dataclasses import dataclass, field
from typing import Callable, Optional, Sequence

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    gamma: int
    V: int
    dtype: str                      # "bf16" | "f32"
    stochastic: bool
    modes: tuple                    # verify modes the workload runs: "compact", "cap_accept", ...
    temperature: float
    bias: float
    alpha_slope: float
    theta_slope: float
    tiers: tuple
    sigma: float
    spike: Optional[float]
    draft_sigma: Optional[float]
    conc: float                     # Beta concentration of the confidences
    accept: Callable[[np.random.Generator, int], np.ndarray]  # a_b for B requests
    steps: int = 1
    logit_pool: int = 0             # >0: logits cycle through this many pre-generated blocks
    note: str = ""

    def with_(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


def _fixed(values):
    values = np.asarray(values, np.float64)

    def f(rng, B):
        return np.resize(values, B)
    return f


def _uniform(lo, hi):
    def f(rng, B):
        return rng.uniform(lo, hi, size=B)
    return f


def _classes(levels):
    """Equal thirds (remainder to the first classes), e.g. 86/85/85 for B = 256."""
    def f(rng, B):
        k = len(levels)
        sizes = [B // k + (1 if i < B % k else 0) for i in range(k)]
        return np.concatenate([np.full(s, lv) for s, lv in zip(sizes, levels)])
    return f


WORKLOADS = {
    "tiny_greedy": Workload(
        name="tiny_greedy", B=4, gamma=4, V=1024, dtype="f32", stochastic=False,
        modes=("compact", "cap_accept", "static"), temperature=1.0, bias=1.0, alpha_slope=0.05,
        theta_slope=0.02, tiers=(8, 16, 32), sigma=3.0, spike=None, draft_sigma=None, conc=8.0,
        accept=_fixed([0.9, 0.7, 0.5, 0.3]),
        note="B=4, gamma=4, V=1024 fp32 N(0,3^2); a_b = 0.9/0.7/0.5/0.3; greedy"),
    "stochastic": Workload(
        name="stochastic", B=32, gamma=8, V=32000, dtype="bf16", stochastic=True,
        modes=("compact", "cap_accept"), temperature=1.0, bias=1.0, alpha_slope=0.05,
        theta_slope=0.02, tiers=tuple(range(16, 257, 16)), sigma=2.0, spike=6.0,
        draft_sigma=0.5, conc=10.0, accept=_uniform(0.4, 0.95),
        note="B=32, gamma=8, V=32000 bf16 N(0,2^2)+6 spike; draft = target + N(0,0.5^2); T=1"),
    "large_vocab_mixed": Workload(
        name="large_vocab_mixed", B=256, gamma=8, V=151936, dtype="bf16", stochastic=False,
        modes=("compact",), temperature=1.0, bias=2.0, alpha_slope=0.01, theta_slope=0.004,
        tiers=tuple(range(32, 2049, 32)), sigma=2.0, spike=6.0, draft_sigma=None, conc=12.0,
        accept=_classes([0.9, 0.65, 0.35]),
        note="B=256, gamma=8, V=151936 bf16 N(0,2^2)+6 spike; classes a=0.9/0.65/0.35; greedy"),
    "latency_b1": Workload(
        name="latency_b1", B=1, gamma=16, V=129280, dtype="bf16", stochastic=False,
        modes=("compact",), temperature=0.7, bias=1.0, alpha_slope=0.05, theta_slope=0.02,
        tiers=(1, 2, 4, 8, 16, 32), sigma=2.0, spike=6.0, draft_sigma=0.5, conc=20.0,
        accept=_fixed([0.85]), steps=10000, logit_pool=16,
        note="B=1, gamma=16, V=129280 bf16; a=0.85, c~Beta(17,3); greedy and stochastic T=0.7"),
    "high_load": Workload(
        name="high_load", B=512, gamma=8, V=151936, dtype="bf16", stochastic=False,
        modes=("compact", "cap_accept"), temperature=1.0, bias=2.0, alpha_slope=0.01,
        theta_slope=0.004, tiers=tuple(range(64, 4097, 64)), sigma=2.0, spike=6.0,
        draft_sigma=None, conc=10.0, accept=_uniform(0.2, 0.95),
        note="B=512, gamma=8, V=151936 bf16; a~U(0.2,0.95); theta in {0.001,0.004,0.016}*M"),
}
HIGH_LOAD_THETAS = (0.001, 0.004, 0.016)


@dataclass
class Batch:
    """One decode step's inputs, on the host."""
    wl: Workload
    seed: int
    step: int
    a: np.ndarray            # [B] acceptance rate per request
    conf: np.ndarray         # [B, gamma-1] float32
    tokens: np.ndarray       # [B, gamma] int32; column 0 = anchor, 1.. = drafts
    target: torch.Tensor     # [B*gamma, V] block-order target logits (bf16 or f32, CPU)
    draft: Optional[torch.Tensor]  # [B*(gamma-1), V] draft logits (stochastic) or None
    alpha: np.ndarray        # [B+1] float64
    theta: np.ndarray        # [B*gamma+1] float64
    tiers: np.ndarray        # int32

    @property
    def B(self):
        return self.wl.B

    @property
    def gamma(self):
        return self.wl.gamma

    @property
    def V(self):
        return self.wl.V

    @property
    def bias(self):
        return self.wl.bias

    def logits_bits(self, t: torch.Tensor) -> np.ndarray:
        """numpy view the CPU oracle takes: uint16 bit patterns for bf16, float32 for f32."""
        t = t.contiguous()
        if t.dtype == torch.bfloat16:
            return t.view(torch.int16).numpy().view(np.uint16)
        return t.numpy()


def _torch_dtype(name):
    return {"bf16": torch.bfloat16, "f32": torch.float32}[name]


def _rng(seed, step, tag):
    return np.random.default_rng([int(seed), int(step), int(tag)])


def _gaussian_rows(rng, rows, V, sigma, spike, dtype, block_rows=256):
    """[rows, V] logits ~ N(0, sigma^2) (+ spike at one uniform id per row) in `dtype`."""
    out = torch.empty((rows, V), dtype=dtype)
    for r0 in range(0, rows, block_rows):
        r1 = min(rows, r0 + block_rows)
        x = rng.standard_normal((r1 - r0, V), dtype=np.float32)
        x *= np.float32(sigma)
        if spike is not None:
            ids = rng.integers(0, V, size=r1 - r0)
            x[np.arange(r1 - r0), ids] += np.float32(spike)
        out[r0:r1] = torch.from_numpy(x).to(dtype)
    return out


def _first_argmax(rows: torch.Tensor, block_rows=256) -> np.ndarray:
    # first index among equal maxima, on the values the verify sees (after dtype rounding)
    out = np.empty(rows.shape[0], np.int64)
    for r0 in range(0, rows.shape[0], block_rows):
        out[r0:r0 + block_rows] = torch.argmax(rows[r0:r0 + block_rows].float(), dim=-1).numpy()
    return out


def _gumbel_sample(rng, logits: torch.Tensor, temperature: float, block_rows=256) -> np.ndarray:
    out = np.empty(logits.shape[0], np.int64)
    for r0 in range(0, logits.shape[0], block_rows):
        x = logits[r0:r0 + block_rows].float().numpy().astype(np.float64) / temperature
        g = -np.log(-np.log(rng.uniform(np.finfo(np.float64).tiny, 1.0, size=x.shape)))
        out[r0:r0 + block_rows] = np.argmax(x + g, axis=-1)
    return out


def make_logits(wl: Workload, seed: int, pool_index: int = 0):
    """(target [B*gamma, V], draft [B*(gamma-1), V] or None) for one block (or pool entry)."""
    dt = _torch_dtype(wl.dtype)
    rng = _rng(seed, pool_index, 1)
    target = _gaussian_rows(rng, wl.B * wl.gamma, wl.V, wl.sigma, wl.spike, dt)
    draft = None
    if wl.draft_sigma is not None:
        L = wl.gamma - 1
        rng_d = _rng(seed, pool_index, 2)
        t3 = target.view(wl.B, wl.gamma, wl.V)[:, :L, :]
        draft = torch.empty((wl.B * L, wl.V), dtype=dt)
        d3 = draft.view(wl.B, L, wl.V)
        for b0 in range(0, wl.B, 32):
            b1 = min(wl.B, b0 + 32)
            noise = rng_d.standard_normal((b1 - b0, L, wl.V), dtype=np.float32)
            noise *= np.float32(wl.draft_sigma)
            d3[b0:b1] = (t3[b0:b1].float() + torch.from_numpy(noise)).to(dt)
    return target, draft


def make_batch(wl: Workload, seed: int = 0, step: int = 0, *, stochastic: Optional[bool] = None,
               theta_slope: Optional[float] = None, logits=None) -> Batch:
    """One step's inputs. `logits` = (target, draft) reuses pre-generated blocks (pools)."""
    stochastic = wl.stochastic if stochastic is None else stochastic
    if theta_slope is not None:
        wl = wl.with_(theta_slope=theta_slope)
    B, gamma, V = wl.B, wl.gamma, wl.V
    L = gamma - 1
    if logits is None:
        pool_index = (step % wl.logit_pool) if wl.logit_pool else 0
        logits = make_logits(wl, seed, pool_index)
    target, draft = logits
    if stochastic and draft is None:
        raise ValueError(f"workload {wl.name} has no draft logits recipe")

    rng_a = _rng(seed, 0, 3)                   # acceptance classes are fixed across steps
    a = wl.accept(rng_a, B).astype(np.float64)
    rng = _rng(seed, step, 4)
    conf = rng.beta(wl.conc * a[:, None], wl.conc * (1.0 - a[:, None]), size=(B, L))
    conf = conf.astype(np.float32)

    tokens = np.empty((B, gamma), np.int64)
    tokens[:, 0] = rng.integers(0, V, size=B)  # anchor: last committed token
    if L > 0:
        if stochastic:
            tokens[:, 1:] = _gumbel_sample(rng, draft, wl.temperature).reshape(B, L)
        else:
            t3 = target.view(B, gamma, V)[:, :L, :].reshape(B * L, V)
            best = _first_argmax(t3).reshape(B, L)
            other = rng.integers(0, V - 1, size=(B, L)) if V > 1 else np.zeros((B, L), np.int64)
            other = other + (other >= best)
            hit = rng.uniform(size=(B, L)) < a[:, None]
            tokens[:, 1:] = np.where(hit, best, other if V > 1 else best)
    alpha = wl.alpha_slope * np.arange(B + 1, dtype=np.float64)
    theta = wl.theta_slope * np.arange(B * gamma + 1, dtype=np.float64)
    return Batch(wl=wl, seed=seed, step=step, a=a, conf=conf, tokens=tokens.astype(np.int32),
                 target=target, draft=draft, alpha=alpha, theta=theta,
                 tiers=np.asarray(wl.tiers, np.int32))


def custom(name="custom", **kw) -> Workload:
    """A workload with explicit sizes for edge-case tests (defaults: tiny greedy recipe)."""
    base = WORKLOADS["tiny_greedy"]
    if "accept" in kw and not callable(kw["accept"]):
        kw["accept"] = _fixed(kw["accept"])
    return base.with_(name=name, **kw)


def gather_packed(target_block: torch.Tensor, B: int, gamma: int, windows,
                  rows_cap: Optional[int] = None) -> torch.Tensor:
    """Stand-in for the target forward over the packed batch: the block-order rows
    (b, i < w_b) front-packed into [rows_cap >= M, V] (pad rows zero). Works on CPU or GPU."""
    w = np.asarray(windows, np.int64)
    idx = np.concatenate([b * gamma + np.arange(w[b]) for b in range(B)]) if B else \
        np.zeros(0, np.int64)
    M = idx.size
    rows_cap = max(M, 1) if rows_cap is None else rows_cap
    out = torch.zeros((rows_cap, target_block.shape[1]), dtype=target_block.dtype,
                      device=target_block.device)
    if M:
        out[:M] = target_block.index_select(0, torch.as_tensor(idx, device=target_block.device))
    return out
