"""A decode step captured as one CUDA graph replays to exactly the eager results, for new
inputs written into the captured buffers and for windows (hence M and the tier) that change
from step to step: the kernels size themselves on the device."""
import numpy as np
import pytest
import torch

from speculative_decoding_ragged_gb300 import synth
from speculative_decoding_ragged_gb300.step import DSparkGraph, DSparkStep

from gpu_util import device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


@pytest.mark.parametrize("stochastic", [False, True])
def test_graph_replay_matches_eager(dev, stochastic):
    wl = synth.WORKLOADS["stochastic"].with_(B=24, V=4096) if stochastic else \
        synth.WORKLOADS["large_vocab_mixed"].with_(B=48, V=8192)
    args = (wl.B, wl.gamma, wl.V, wl.tiers, wl.bias, wl.alpha_slope * np.arange(wl.B + 1),
            wl.theta_slope * np.arange(wl.B * wl.gamma + 1))
    eager = DSparkStep(*args, mode="cap_accept", stochastic=stochastic, out_cap=64, device=dev)
    graphed = DSparkStep(*args, mode="cap_accept", stochastic=stochastic, out_cap=64, device=dev)
    dt = torch.bfloat16
    conf = torch.zeros((wl.B, wl.gamma - 1), dtype=torch.float32, device=dev)
    tokens = torch.zeros((wl.B, wl.gamma), dtype=torch.int32, device=dev)
    target = torch.zeros((wl.B * wl.gamma, wl.V), dtype=dt, device=dev)
    draft = torch.zeros((wl.B * (wl.gamma - 1), wl.V), dtype=dt, device=dev) if stochastic else None
    g = DSparkGraph(graphed, conf, tokens, target, draft, seed=3)
    graphed.out_len.zero_()
    graphed.out_tokens.fill_(-1)
    graphed.status.zero_()
    Ms = set()
    for step in range(6):
        bt = synth.make_batch(wl, seed=10 + step, stochastic=stochastic)
        conf.copy_(torch.as_tensor(bt.conf))
        tokens.copy_(torch.as_tensor(bt.tokens))
        target.copy_(bt.target)
        if stochastic:
            draft.copy_(bt.draft)
        g.replay()
        eager.run(conf, tokens, target, draft, seed=3)
        torch.cuda.synchronize()
        for name in ("windows", "k_star", "accept_len", "committed", "ceiling", "out_tokens",
                     "out_len"):
            np.testing.assert_array_equal(getattr(graphed, name).cpu().numpy(),
                                          getattr(eager, name).cpu().numpy(), err_msg=name)
        Ms.add(int(graphed.windows.sum().item()))
    assert len(Ms) > 1          # the replays saw different packed totals
    assert int(graphed.status.item()) == int(eager.status.item())
