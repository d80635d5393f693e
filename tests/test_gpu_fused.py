"""The fused entry points against the single calls and the oracle: dspark_schedule_pack must
equal dspark_schedule then dspark_pack, and dspark_verify_scatter must equal dspark_verify then
dspark_scatter, output by output and bit for bit ("DSpark in SGLang", A2 method details,
performance: the step's small operations fused into fewer kernels)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth

from gpu_util import device, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def _cost(dev, bias, alpha, theta):
    return bd.CostTable(bias, torch.as_tensor(np.asarray(alpha, np.float64), device=dev),
                        torch.as_tensor(np.asarray(theta, np.float64), device=dev))


def _sched_pack_outputs(dev, B, cap):
    def full(n):
        return torch.full((max(n, 1),), -7, dtype=torch.int32, device=dev)[:n]
    return dict(windows=full(B), k_star=full(1), cu=full(B + 1), packed=full(cap),
                row_req=full(cap), row_pos=full(cap), meta=full(2),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _host(o):
    torch.cuda.synchronize()
    return {k: v.cpu().numpy() for k, v in o.items()}


@pytest.mark.parametrize("B,gamma", [(1, 2), (1, 16), (4, 4), (33, 8), (256, 8), (600, 8),
                                     (1000, 17), (8192, 2), (2048, 9), (32, 2), (2, 17), (1, 32),
                                     (33, 2)])
def test_schedule_pack_equals_the_two_calls(dev, B, gamma):
    rng = np.random.default_rng(B * 31 + gamma)
    for trial in range(3):
        a = rng.uniform(0.1, 0.95, size=B)
        conf = rng.beta(8 * a[:, None], 8 * (1 - a[:, None]), size=(B, gamma - 1))
        if trial == 1:
            conf = np.round(conf * 8) / 8          # many equal survivals: tie rule
        conf = conf.astype(np.float32)
        tokens = rng.integers(0, 150000, size=(B, gamma))
        bias = float(rng.uniform(0.5, 3))
        alpha = rng.uniform(0, 0.1) * np.arange(B + 1)
        theta = rng.uniform(0, 0.05) * np.arange(B * gamma + 1)
        tiers = np.arange(1, 65) * max(1, B * gamma // 48)
        if trial == 2:
            tiers = tiers[:3]                       # tier overflow for most budgets
        cap = [B * gamma + 8, int(tiers.max()) + 3, max(1, B * gamma // 3)][trial]
        cost = _cost(dev, bias, alpha, theta)
        c, t, tr = (torch.as_tensor(conf, device=dev), i32(tokens, dev), i32(tiers, dev))
        f = _sched_pack_outputs(dev, B, cap)
        bd.dspark_schedule_pack(c, cost, t, tr, f["windows"], f["k_star"], f["cu"], f["packed"],
                                f["meta"], f["row_req"], f["row_pos"], f["status"])
        s = _sched_pack_outputs(dev, B, cap)
        bd.dspark_schedule(c, cost, s["windows"], s["k_star"], s["status"])
        bd.dspark_pack(s["windows"], t, tr, s["cu"], s["packed"], s["meta"], s["row_req"],
                       s["row_pos"], s["status"])
        f, s = _host(f), _host(s)
        for k in f:
            np.testing.assert_array_equal(f[k], s[k], err_msg=k)
        r = oracle.schedule(conf, bias, alpha, theta)
        np.testing.assert_array_equal(f["windows"], r["windows"])
        pk = oracle.pack(r["windows"], tokens, tiers, cap)
        np.testing.assert_array_equal(f["packed"], pk["packed_ids"])
        assert (int(f["meta"][0]), int(f["meta"][1])) == (pk["M"], pk["tier"])
        assert int(f["status"][0]) == r["status"] | pk["status"]


def test_schedule_pack_degenerate_sizes(dev):
    cost = _cost(dev, 1.0, np.zeros(8), np.full(40, 0.1))
    for B, gamma in [(0, 4), (5, 1)]:
        f = _sched_pack_outputs(dev, B, 16)
        conf = torch.zeros((B, gamma - 1), dtype=torch.float32, device=dev)
        tokens = i32(np.arange(B * gamma).reshape(B, gamma), dev)
        bd.dspark_schedule_pack(conf, cost, tokens, i32([4, 8], dev), f["windows"], f["k_star"],
                                f["cu"], f["packed"], f["meta"], f["row_req"], f["row_pos"],
                                f["status"])
        f = _host(f)
        assert int(f["k_star"][0]) == 0
        if B:
            assert (f["windows"] == 1).all() and f["meta"].tolist() == [B, 8]


def _verify_outputs(dev, B, gamma, rows, cap, out_len0):
    return dict(acc=torch.full((B,), -7, dtype=torch.int32, device=dev),
                com=torch.full((B, gamma), -7, dtype=torch.int32, device=dev),
                ceil=torch.full((B,), -7, dtype=torch.int32, device=dev),
                prob=torch.full((max(rows, 1), 2), -7.0, dtype=torch.float32, device=dev),
                out=torch.full((B, cap), -5, dtype=torch.int32, device=dev),
                out_len=i32(out_len0, dev),
                status=torch.zeros(1, dtype=torch.int32, device=dev))


def _run_pair(dev, mode, tgt, drf, tokens, cu, windows, stochastic, cap, out_len0, **kw):
    B, gamma = tokens.shape
    rows, V = tgt.shape
    ws = torch.empty(max(bd.dspark_verify_workspace_bytes(B, gamma, V, stochastic), 16),
                     dtype=torch.uint8, device=dev)
    t = i32(tokens, dev)
    cu_d = None if cu is None else i32(cu, dev)
    w_d = None if windows is None else i32(windows, dev)
    f = _verify_outputs(dev, B, gamma, rows, cap, out_len0)
    bd.dspark_verify_scatter(mode, tgt, t, f["acc"], f["com"], ws, f["out"], f["out_len"],
                             stochastic=stochastic, draft=drf, cu_seqlens=cu_d, windows=w_d,
                             ceiling_len=f["ceil"], row_prob=f["prob"], status=f["status"], **kw)
    s = _verify_outputs(dev, B, gamma, rows, cap, out_len0)
    bd.dspark_verify(mode, tgt, t, s["acc"], s["com"], ws, stochastic=stochastic, draft=drf,
                     cu_seqlens=cu_d, windows=w_d, ceiling_len=s["ceil"], row_prob=s["prob"],
                     status=s["status"], **kw)
    bd.dspark_scatter(s["com"], s["acc"], s["out"], s["out_len"], s["status"])
    return _host(f), _host(s)


@pytest.mark.parametrize("name", ["tiny_greedy", "stochastic", "large_vocab_mixed", "latency_b1"])
@pytest.mark.parametrize("mode", ["compact", "cap_accept", "static"])
def test_verify_scatter_equals_the_two_calls(dev, name, mode):
    wl = synth.WORKLOADS[name]
    if name == "large_vocab_mixed":
        wl = wl.with_(B=64)
    for stochastic in ((False, True) if wl.draft_sigma is not None else (False,)):
        bt = synth.make_batch(wl, seed=5, stochastic=stochastic)
        B, gamma = bt.tokens.shape
        rng = np.random.default_rng(B + gamma)
        cap = 3 * gamma
        out_len0 = rng.integers(0, cap + 1, size=B)       # some histories overflow
        w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
        if mode == "compact":
            tgt = synth.gather_packed(bt.target, B, gamma, w).to(dev)
            cu = np.concatenate([[0], np.cumsum(w)])
        else:
            tgt = bt.target.to(dev)
            cu = None
        drf = bt.draft.to(dev) if stochastic else None
        f, s = _run_pair(dev, mode, tgt, drf, bt.tokens, cu,
                         None if mode == "static" else w, stochastic, cap, out_len0,
                         temperature=wl.temperature, seed=11, step=3)
        for k in f:
            np.testing.assert_array_equal(f[k], s[k], err_msg=f"{k} stochastic={stochastic}")


def test_verify_scatter_bad_rows_and_lengths(dev):
    # a compact buffer one row short: the last request flags BAD_ROWS and commits nothing, its
    # history only has its length checked; negative and oversized lengths flag BAD_LENGTH
    wl = synth.WORKLOADS["stochastic"].with_(B=4, V=1024)
    for stochastic in (False, True):
        bt = synth.make_batch(wl, seed=2, stochastic=stochastic)
        B, gamma = bt.tokens.shape
        w = np.full(B, gamma, np.int32)
        cu = np.concatenate([[0], np.cumsum(w)])
        tgt = synth.gather_packed(bt.target, B, gamma, w)[: B * gamma - 1].to(dev)
        drf = bt.draft.to(dev) if stochastic else None
        out_len0 = np.array([-3, 2, 100, 5])[:B]
        f, s = _run_pair(dev, "compact", tgt, drf, bt.tokens, cu, w, stochastic, 8, out_len0,
                         temperature=1.0, seed=1, step=0)
        for k in f:
            np.testing.assert_array_equal(f[k], s[k], err_msg=k)
        st = int(f["status"][0])
        assert st & bd.STATUS_BAD_ROWS and st & bd.STATUS_BAD_LENGTH
        assert f["acc"][B - 1] == 0


def test_fused_step_equals_single_calls_over_steps(dev):
    from speculative_decoding_ragged_gb300.step import DSparkStep
    wl = synth.WORKLOADS["stochastic"]
    bts = [synth.make_batch(wl, seed=9, step=k, stochastic=True) for k in range(4)]
    steps = []
    for fused in (True, False):
        st = DSparkStep(wl.B, wl.gamma, wl.V, wl.tiers, bts[0].bias, bts[0].alpha, bts[0].theta,
                        stochastic=True, out_cap=64, fused=fused, device=dev)
        hist = []
        for k, bt in enumerate(bts):
            w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
            M = int(w.sum())
            tier = int(min([t for t in wl.tiers if t >= M] or [M]))
            packed = synth.gather_packed(bt.target, wl.B, wl.gamma, w, rows_cap=tier).to(dev)
            st.run(torch.as_tensor(bt.conf, device=dev), torch.as_tensor(bt.tokens, device=dev),
                   packed, bt.draft.to(dev), temperature=wl.temperature, seed=4, step=k)
            torch.cuda.synchronize()
            hist.append((st.windows.cpu().numpy().copy(), st.accept_len.cpu().numpy().copy(),
                         st.committed.cpu().numpy().copy()))
        steps.append((hist, st.out_tokens.cpu().numpy(), st.out_len.cpu().numpy(),
                      int(st.status.item())))
    (h1, o1, l1, s1), (h2, o2, l2, s2) = steps
    for a, b in zip(h1, h2):
        for x, y in zip(a, b):
            np.testing.assert_array_equal(x, y)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(l1, l2)
    assert s1 == s2
