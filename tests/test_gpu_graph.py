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


@pytest.mark.parametrize("mode", ["compact", "cap_accept"])
@pytest.mark.parametrize("stochastic", [False, True])
def test_graph_replay_matches_oracle_across_tiers(dev, mode, stochastic):
    """The replayed step against the CPU oracle, step by step: windows, cu_seqlens, M and the
    tier, accept lengths, committed tokens and the appended histories. The cost table's theta
    changes between replays (the graph reads it from the same device buffer), so the packed
    total and the tier change too; in compact mode the packed rows of the oracle's windows are
    written into the captured logits buffer before each replay (the target forward's stand-in)."""
    import oracle
    from gpu_util import bits, compare_stochastic
    wl = synth.WORKLOADS["stochastic"].with_(B=24, V=4096) if stochastic else \
        synth.WORKLOADS["large_vocab_mixed"].with_(B=48, V=8192, tiers=tuple(range(48, 385, 48)))
    B, g, V = wl.B, wl.gamma, wl.V
    slopes = (0.001, 0.05, 0.004, 0.3, 0.0)
    st = DSparkStep(B, g, V, wl.tiers, wl.bias, wl.alpha_slope * np.arange(B + 1),
                    slopes[0] * np.arange(B * g + 1), mode=mode, stochastic=stochastic,
                    out_cap=64, device=dev)
    rows = st.packed_cap if mode == "compact" else B * g
    conf = torch.zeros((B, g - 1), dtype=torch.float32, device=dev)
    tokens = torch.zeros((B, g), dtype=torch.int32, device=dev)
    target = torch.zeros((rows, V), dtype=torch.bfloat16, device=dev)
    draft = torch.zeros((B * (g - 1), V), dtype=torch.bfloat16, device=dev) if stochastic else None
    graph = DSparkGraph(st, conf, tokens, target, draft, seed=9, temperature=wl.temperature)
    st.out_len.zero_()
    st.out_tokens.fill_(-1)
    st.status.zero_()
    hist = np.full((B, 64), -1, np.int32)
    hlen = np.zeros(B, np.int32)
    tiers_seen, near = set(), 0
    for k, slope in enumerate(slopes):
        bt = synth.make_batch(wl, seed=40 + k, stochastic=stochastic, theta_slope=slope)
        st.cost.theta.copy_(torch.as_tensor(bt.theta))
        rs = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
        w = rs["windows"]
        rp = oracle.pack(w, bt.tokens, bt.tiers, st.packed_cap)
        if mode == "compact":
            tgt_host = synth.gather_packed(bt.target, B, g, w, rows_cap=rows)
        else:
            tgt_host = bt.target
        conf.copy_(torch.as_tensor(bt.conf))
        tokens.copy_(torch.as_tensor(bt.tokens))
        target.copy_(tgt_host)
        if stochastic:
            draft.copy_(bt.draft)
        graph.replay()
        torch.cuda.synchronize()
        rv = oracle.verify(oracle.COMPACT if mode == "compact" else oracle.CAP_ACCEPT,
                           stochastic, bits(tgt_host), bt.tokens, cu=rp["cu"], windows=w,
                           draft=bits(bt.draft) if stochastic else None,
                           temperature=wl.temperature, seed=9, step=0)
        np.testing.assert_array_equal(st.windows.cpu().numpy(), w)
        assert int(st.k_star.item()) == rs["k_star"]
        np.testing.assert_array_equal(st.cu.cpu().numpy(), rp["cu"])
        np.testing.assert_array_equal(st.meta.cpu().numpy(), [rp["M"], rp["tier"]])
        tiers_seen.add(rp["tier"])
        got = dict(accept_len=st.accept_len.cpu().numpy(), committed=st.committed.cpu().numpy(),
                   ceiling_len=st.ceiling.cpu().numpy(), status=rv["status"])
        if stochastic:
            got["row_prob"] = rv["row_prob"]          # the graph's step records none
            n, _ = compare_stochastic(got, rv, rows_used=0)
            near += n
        else:
            np.testing.assert_array_equal(got["accept_len"], rv["accept_len"])
            np.testing.assert_array_equal(got["committed"], rv["committed"])
        if mode == "cap_accept":
            np.testing.assert_array_equal(got["ceiling_len"], rv["ceiling_len"])
        sc = oracle.scatter(rv["committed"], rv["accept_len"], hist, hlen)
        hist, hlen = sc["out_tokens"], sc["out_len"]
    assert len(tiers_seen) >= 2, tiers_seen      # one captured graph served several tiers
    if near == 0:
        np.testing.assert_array_equal(st.out_len.cpu().numpy(), hlen)
        np.testing.assert_array_equal(st.out_tokens.cpu().numpy(), hist)
    assert int(st.status.item()) == 0
