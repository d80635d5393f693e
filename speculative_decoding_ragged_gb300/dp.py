"""Data-parallel tier agreement for the ragged verify.

"DSpark in SGLang" (LMSYS blog summary), A2, ragged verify over full CUDA graphs: under
data-parallel attention the ranks share one capture tier — the largest tier any rank needs —
and shrink together when every rank's packed total falls. Each rank schedules and packs its
own requests (dspark_schedule, dspark_pack); the only exchange is one all-reduce(MAX) of an
int32 tier per step. After the agreement a rank re-packs with the agreed tier as its only tier
(dspark_pack pads rows M..tier), so every rank replays the same graph shape.

Every call of this build runs on one GPU, so the collective runs over whatever process group
the caller provides: gloo on CPU in the tests, NCCL on device tensors in a multi-GPU job.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch
import torch.distributed as dist


def tier_for(M: int, tiers: Sequence[int]) -> int:
    """The smallest tier holding M rows (M itself when none does), as dspark_pack rounds."""
    fitting = [t for t in tiers if t >= M]
    return min(fitting) if fitting else M


def agree_tier(local_tier: torch.Tensor, group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """All-reduce(MAX) of each rank's tier, in place: every rank ends with the largest tier any
    rank needs. `local_tier` is a one-element int32 tensor (for instance meta[1:2] written by
    dspark_pack), on the device the group's backend serves."""
    if local_tier.numel() != 1:
        raise ValueError("local_tier must hold exactly one value")
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(local_tier, op=dist.ReduceOp.MAX, group=group)
    return local_tier


class TierSync:
    """Per-step tier agreement of one DP rank, with the history of agreed tiers.

    step(local_M) returns the tier this rank must replay: max over ranks of tier_for(M)."""

    def __init__(self, tiers: Sequence[int], group: Optional[dist.ProcessGroup] = None,
                 device: Optional[torch.device] = None):
        self.tiers = sorted(int(t) for t in tiers)
        self.group = group
        self.device = device or torch.device("cpu")
        self.history = []

    def step(self, local_M: int) -> int:
        t = torch.tensor([tier_for(int(local_M), self.tiers)], dtype=torch.int32,
                         device=self.device)
        agreed = int(agree_tier(t, self.group).item())
        self.history.append(agreed)
        return agreed
