"""DP tier agreement across ranks ("DSpark in SGLang", A2: under DP attention every rank replays
the largest tier any rank needs and the ranks shrink together), on two gloo ranks on CPU.

Each rank schedules its own requests with the oracle and packs them; the ranks agree on the
tier by an all-reduce(MAX) of meta[1] as the pack wrote it. The agreed tier must be the maximum
of the ranks' own tiers at every step, identical on both ranks, fall only when every rank's load
falls, and serve as the only tier of each rank's re-pack."""
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
        from speculative_decoding_ragged_gb300.dp import TierSync
        wl = synth.WORKLOADS["high_load"].with_(B=64, V=64)
        sync = TierSync()
        local, agreed_hist = [], []
        for step, slope in enumerate(LOADS[rank]):
            bt = synth.make_batch(wl, seed=100 + rank, step=step, theta_slope=slope)
            w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
            pk = oracle.pack(w, bt.tokens, bt.tiers, int(max(bt.tiers)))
            # meta = {M, tier} as the pack wrote it: the all-reduce runs on meta[1] in place
            meta = torch.tensor([pk["M"], pk["tier"]], dtype=torch.int32)
            local.append(pk["tier"])
            tiers = sync.step(meta)
            agreed = int(tiers.item())           # read by the test only
            assert int(meta[1]) == agreed and int(meta[0]) == pk["M"]
            agreed_hist.append(agreed)
            # re-pack with the agreed tier as the only tier: rows M..agreed are padding
            re = oracle.pack(w, bt.tokens, tiers.numpy(), agreed)
            assert re["tier"] == agreed and re["status"] == 0
            assert (re["row_req"][pk["M"]:agreed] == -1).all()
        out[rank] = (local, agreed_hist)
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


def test_agree_tier_without_a_group_is_identity():
    from speculative_decoding_ragged_gb300.dp import agree_tier
    t = torch.tensor([96], dtype=torch.int32)
    assert int(agree_tier(t).item()) == 96
    with pytest.raises(ValueError):
        agree_tier(torch.tensor([1, 2], dtype=torch.int32))
    with pytest.raises(ValueError):
        agree_tier(torch.tensor([1], dtype=torch.int64))


def test_tier_sync_writes_the_repack_tiers_without_a_group():
    from speculative_decoding_ragged_gb300.dp import TierSync
    sync = TierSync()
    meta = torch.tensor([37, 64], dtype=torch.int32)
    tiers = sync.step(meta)
    assert tiers.dtype == torch.int32 and tiers.numel() == 1 and int(tiers) == 64
    meta[1] = 0                              # the re-pack writes meta again: tiers stay put
    assert int(tiers) == 64
    with pytest.raises(ValueError):
        sync.step(torch.tensor([1], dtype=torch.int32))
