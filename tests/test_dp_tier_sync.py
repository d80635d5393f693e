"""DP tier agreement across ranks ("DSpark in SGLang", A2: under DP attention every rank replays
the largest tier any rank needs and the ranks shrink together), on two gloo ranks on CPU.

Each rank schedules its own requests with the oracle, packs, and agrees on the tier; the agreed
tier must be the maximum of the ranks' own tiers at every step, identical on both ranks, and
fall only when every rank's load falls."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


LOADS = {  # per rank and step: theta slope (a higher slope shrinks the windows)
    0: [0.001, 0.004, 0.016, 0.016, 0.001],
    1: [0.016, 0.004, 0.004, 0.016, 0.016],
}


def _rank(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import oracle
        from speculative_decoding_ragged_gb300 import synth
        from speculative_decoding_ragged_gb300.dp import TierSync, tier_for
        wl = synth.WORKLOADS["high_load"].with_(B=64, V=64)
        sync = TierSync(wl.tiers)
        local = []
        for step, slope in enumerate(LOADS[rank]):
            bt = synth.make_batch(wl, seed=100 + rank, step=step, theta_slope=slope)
            w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
            M = int(w.sum())
            local.append(tier_for(M, wl.tiers))
            agreed = sync.step(M)
            # re-pack with the agreed tier as the only tier: rows M..agreed are padding
            pk = oracle.pack(w, bt.tokens, np.array([agreed], np.int32), agreed)
            assert pk["tier"] == agreed and pk["status"] == 0
            assert (pk["row_req"][M:agreed] == -1).all()
        out[rank] = (local, sync.history)
    finally:
        dist.destroy_process_group()


def test_two_ranks_agree_on_the_max_tier_and_shrink_together():
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    out = manager.dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    local0, agreed0 = out[0]
    local1, agreed1 = out[1]
    assert agreed0 == agreed1
    assert agreed0 == [max(a, b) for a, b in zip(local0, local1)]
    assert len(set(agreed0)) > 1          # the shared tier moves with the ranks' loads
    for s in range(1, len(agreed0)):      # it falls only when no rank still needs the old one
        if agreed0[s] < agreed0[s - 1]:
            assert local0[s] < agreed0[s - 1] and local1[s] < agreed0[s - 1]


def test_tier_for_matches_pack_rounding():
    from speculative_decoding_ragged_gb300.dp import tier_for
    assert tier_for(8, [4, 8, 16]) == 8
    assert tier_for(9, [16, 4, 12]) == 12
    assert tier_for(40, [8, 16]) == 40


def test_agree_tier_without_a_group_is_identity():
    from speculative_decoding_ragged_gb300.dp import agree_tier
    t = torch.tensor([96], dtype=torch.int32)
    assert int(agree_tier(t).item()) == 96
    with pytest.raises(ValueError):
        agree_tier(torch.tensor([1, 2], dtype=torch.int32))
