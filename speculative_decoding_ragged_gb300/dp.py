"""Data-parallel tier agreement for the ragged verify.

"DSpark in SGLang" (LMSYS blog summary), A2, ragged verify over full CUDA graphs: under
data-parallel attention the ranks share one capture tier — the largest tier any rank needs —
and shrink together when every rank's packed total falls. Each rank schedules and packs its
own requests (dspark_schedule_pack writes meta = {M, tier}); the only exchange is one
all-reduce(MAX) of that int32 tier per step, done in place on meta[1] where the pack wrote it,
so the host never reads M or the tier. The rank then re-packs with the agreed tier as its only
tier (dspark_pack pads rows M..tier), so every rank replays the same graph shape.

The collective runs over whatever process group the caller provides: gloo on CPU tensors in
the multi-rank tests, NCCL on device tensors in a multi-GPU job.
"""
from __future__ import annotations

from typing import Optional

import torch
import torch.distributed as dist


def agree_tier(local_tier: torch.Tensor, group: Optional[dist.ProcessGroup] = None) -> torch.Tensor:
    """All-reduce(MAX) of each rank's tier, in place: every rank ends with the largest tier any
    rank needs. `local_tier` is a one-element int32 tensor (meta[1:2] as dspark_pack wrote it),
    on the device the group's backend serves. Without an initialised process group this is the
    identity (a single rank agrees with itself)."""
    if local_tier.numel() != 1 or local_tier.dtype != torch.int32:
        raise ValueError("local_tier must be a one-element int32 tensor")
    if dist.is_available() and dist.is_initialized():
        dist.all_reduce(local_tier, op=dist.ReduceOp.MAX, group=group)
    return local_tier


class TierSync:
    """Per-step tier agreement of one DP rank, driven from the pack's own output.

    step(meta) all-reduces meta[1] (the tier dspark_pack or dspark_schedule_pack wrote) in
    place and copies the agreed value into `self.tiers`, a one-element device tensor that is
    the tiers argument of the rank's re-pack: dspark_pack(..., tiers=sync.tiers, ...). Nothing
    is read back to the host; the collective is enqueued on the current stream (NCCL) or runs
    on the CPU tensors it is given (gloo)."""

    def __init__(self, group: Optional[dist.ProcessGroup] = None,
                 device: Optional[torch.device] = None):
        self.group = group
        self.tiers = torch.zeros(1, dtype=torch.int32, device=device or "cpu")

    def step(self, meta: torch.Tensor) -> torch.Tensor:
        if meta.numel() < 2 or meta.dtype != torch.int32:
            raise ValueError("meta must be the int32 {M, tier} pair dspark_pack writes")
        if meta.device != self.tiers.device:
            raise ValueError("meta and the agreed-tier buffer must share a device")
        agree_tier(meta[1:2], self.group)
        self.tiers.copy_(meta[1:2])          # a separate buffer: the re-pack writes meta again
        return self.tiers
