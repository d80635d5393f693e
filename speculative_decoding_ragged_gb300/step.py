"""A buffer-owning runner of one DSpark decode step: schedule -> pack -> verify -> scatter.

All buffers are allocated once, on the device, at construction; `run` only enqueues the
library calls on the current stream and never synchronises, so it can be timed with CUDA
events or captured into a CUDA graph. By default the step uses the two fused calls
(dspark_schedule_pack, dspark_verify_scatter: three kernels); with fused=False it issues the
four single calls (five kernels). Both give identical
results.
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

from . import _binding as bd


def launches_per_step(gamma: int, stochastic: bool, fused: bool) -> int:
    """Kernel launches of one step: schedule (+ pack), verify (the streaming kernel, then the
    greedy finaliser or the stochastic bonus kernel), scatter unless fused."""
    verify = 2
    if fused:
        return (1 if gamma > 1 else 2) + verify
    return 2 + verify + 1


class DSparkStep:
    def __init__(self, B: int, gamma: int, V: int, tiers: Sequence[int], bias: float,
                 alpha, theta, *, mode: str = "compact", stochastic: bool = False,
                 out_cap: int = 4096, fused: bool = True, device="cuda"):
        self.B, self.gamma, self.V = B, gamma, V
        self.mode = mode
        self.stochastic = stochastic
        self.fused = fused
        self.launches_per_step = launches_per_step(gamma, stochastic, fused)
        self.device = torch.device(device)
        dev = dict(device=self.device)
        i32 = dict(dtype=torch.int32, **dev)
        self.cost = bd.CostTable(bias, torch.as_tensor(np.asarray(alpha, np.float64), **dev),
                                 torch.as_tensor(np.asarray(theta, np.float64), **dev))
        self.tiers = torch.as_tensor(np.asarray(tiers, np.int32), **dev)
        self.packed_cap = int(max(max(tiers), B * gamma))
        self.windows = torch.zeros(B, **i32)
        self.k_star = torch.zeros(1, **i32)
        self.cu = torch.zeros(B + 1, **i32)
        self.packed_ids = torch.zeros(self.packed_cap, **i32)
        self.row_req = torch.zeros(self.packed_cap, **i32)
        self.row_pos = torch.zeros(self.packed_cap, **i32)
        self.meta = torch.zeros(2, **i32)
        self.status = torch.zeros(1, **i32)
        self.accept_len = torch.zeros(B, **i32)
        self.committed = torch.zeros(B, gamma, **i32)
        self.ceiling = torch.zeros(B, **i32)
        ws = bd.dspark_verify_workspace_bytes(B, gamma, V, stochastic)
        self.workspace = torch.empty(max(ws, 16), dtype=torch.uint8, **dev)
        self.out_tokens = torch.full((B, out_cap), -1, **i32)
        self.out_len = torch.zeros(B, **i32)

    def schedule(self, conf: torch.Tensor):
        bd.dspark_schedule(conf, self.cost, self.windows, self.k_star, self.status)

    def pack(self, block_tokens: torch.Tensor):
        bd.dspark_pack(self.windows, block_tokens, self.tiers, self.cu, self.packed_ids,
                       self.meta, self.row_req, self.row_pos, self.status)

    def verify(self, target: torch.Tensor, block_tokens: torch.Tensor,
               draft: Optional[torch.Tensor] = None, *, temperature: float = 1.0, seed: int = 0,
               step: int = 0, row_prob: Optional[torch.Tensor] = None):
        bd.dspark_verify(self.mode, target, block_tokens, self.accept_len, self.committed,
                         self.workspace, stochastic=self.stochastic, draft=draft,
                         cu_seqlens=self.cu, windows=self.windows, ceiling_len=self.ceiling,
                         row_prob=row_prob, temperature=temperature, seed=seed, step=step,
                         status=self.status)

    def scatter(self):
        bd.dspark_scatter(self.committed, self.accept_len, self.out_tokens, self.out_len,
                          self.status)

    def schedule_pack(self, conf: torch.Tensor, block_tokens: torch.Tensor, prepare=False):
        return bd.dspark_schedule_pack(conf, self.cost, block_tokens, self.tiers, self.windows,
                                       self.k_star, self.cu, self.packed_ids, self.meta,
                                       self.row_req, self.row_pos, self.status, prepare=prepare)

    def verify_scatter(self, target: torch.Tensor, block_tokens: torch.Tensor,
                       draft: Optional[torch.Tensor] = None, *, temperature: float = 1.0,
                       seed: int = 0, step: int = 0, row_prob: Optional[torch.Tensor] = None,
                       prepare=False):
        return bd.dspark_verify_scatter(
            self.mode, target, block_tokens, self.accept_len, self.committed, self.workspace,
            self.out_tokens, self.out_len, stochastic=self.stochastic, draft=draft,
            cu_seqlens=self.cu, windows=self.windows, ceiling_len=self.ceiling,
            row_prob=row_prob, temperature=temperature, seed=seed, step=step,
            status=self.status, prepare=prepare)

    def prepare(self, conf, block_tokens, target, draft=None, *, temperature=1.0, seed=0,
                step=0, row_prob=None):
        """The step's calls, checked and marshalled once for these input tensors (which must
        stay alive and in place): [schedule_pack, verify_scatter] when fused, else [schedule,
        pack, verify, scatter]; each a callable that re-issues its C call on the current stream
        without Python-side checks."""
        if self.fused:
            return [self.schedule_pack(conf, block_tokens, prepare=True),
                    self.verify_scatter(target, block_tokens, draft, temperature=temperature,
                                        seed=seed, step=step, row_prob=row_prob, prepare=True)]
        return [
            bd.dspark_schedule(conf, self.cost, self.windows, self.k_star, self.status,
                               prepare=True),
            bd.dspark_pack(self.windows, block_tokens, self.tiers, self.cu, self.packed_ids,
                           self.meta, self.row_req, self.row_pos, self.status, prepare=True),
            bd.dspark_verify(self.mode, target, block_tokens, self.accept_len, self.committed,
                             self.workspace, stochastic=self.stochastic, draft=draft,
                             cu_seqlens=self.cu, windows=self.windows, ceiling_len=self.ceiling,
                             row_prob=row_prob, temperature=temperature, seed=seed, step=step,
                             status=self.status, prepare=True),
            bd.dspark_scatter(self.committed, self.accept_len, self.out_tokens, self.out_len,
                              self.status, prepare=True),
        ]

    def run(self, conf, block_tokens, target, draft=None, *, temperature=1.0, seed=0, step=0,
            row_prob=None):
        """One whole step. `target` holds the rows this mode verifies: the packed [>=M, V]
        rows of the scheduled windows (compact) or the full block [B*gamma, V]."""
        if self.fused:
            self.schedule_pack(conf, block_tokens)
            self.verify_scatter(target, block_tokens, draft, temperature=temperature, seed=seed,
                                step=step, row_prob=row_prob)
            return
        self.schedule(conf)
        self.pack(block_tokens)
        self.verify(target, block_tokens, draft, temperature=temperature, seed=seed, step=step,
                    row_prob=row_prob)
        self.scatter()


class DSparkGraph:
    """One decode step captured as a CUDA graph over fixed input buffers, through the
    library's own capture entry points (dspark_graph_begin / dspark_graph_end): replay() is one
    dspark_graph_launch, a single cudaGraphLaunch from C.

    Every kernel sizes itself on the device (verify reads M from cu_seqlens), so a single
    graph serves every window allocation and every tier: replay() launches the whole step —
    schedule, pack, verify, scatter — with one call. New inputs are written into the same
    tensors (conf, block_tokens, target, draft) before a replay. The step's status word keeps
    accumulating across replays until the caller zeroes it. `steps` > 1 captures that many
    consecutive steps (Philox step counters step_index, step_index + 1, ...) in one graph.
    """

    def __init__(self, step: DSparkStep, conf, block_tokens, target, draft=None, *,
                 temperature=1.0, seed=0, step_index=0, row_prob=None, steps=1):
        self.step = step
        kw = dict(temperature=temperature, seed=seed, row_prob=row_prob)
        # one eager run first: per-device set-up of the library happens outside the capture
        for call in step.prepare(conf, block_tokens, target, draft, step=step_index, **kw):
            call()
        torch.cuda.synchronize()
        # capture on a side stream (the legacy default stream cannot be captured); the calls
        # are prepared while it is current, so they are issued on it
        capture = torch.cuda.Stream(device=step.device)
        with torch.cuda.stream(capture):
            self._calls = [step.prepare(conf, block_tokens, target, draft, step=step_index + k,
                                        **kw) for k in range(steps)]
            self.graph = bd.StepGraph(capture)
            try:
                for calls in self._calls:
                    for call in calls:
                        call()
            finally:
                self.graph.end()
        self._replay = self.graph.prepare_launch()     # replays on the caller's stream

    def replay(self):
        self._replay()
