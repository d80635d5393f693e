"""GPU parity of dspark_scatter (histories, overflow truncation, bad lengths) and of a
multi-step run of the whole path through DSparkStep against the oracle's chained calls."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth
from speculative_decoding_ragged_gb300.step import DSparkStep

from gpu_util import device, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


@pytest.mark.parametrize("B,gamma,cap", [(0, 4, 8), (1, 1, 1), (5, 8, 20), (700, 16, 64),
                                         (33, 32, 40), (9000, 8, 9)])
def test_scatter_parity(dev, B, gamma, cap):
    rng = np.random.default_rng(B + cap)
    committed = rng.integers(0, 1000, size=(B, gamma)).astype(np.int32)
    L = rng.integers(0, gamma + 1, size=B).astype(np.int32)
    n0 = rng.integers(0, cap + 1, size=B).astype(np.int32)
    if B > 3:
        L[0], n0[1], L[2] = gamma + 2, -3, -1
    hist = rng.integers(-9, 0, size=(B, cap)).astype(np.int32)
    out_t, out_l = i32(hist, dev), i32(n0, dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    bd.dspark_scatter(i32(committed, dev), i32(L, dev), out_t, out_l, st)
    torch.cuda.synchronize()
    r = oracle.scatter(committed, L, hist, n0)
    np.testing.assert_array_equal(out_t.cpu().numpy(), r["out_tokens"])
    np.testing.assert_array_equal(out_l.cpu().numpy(), r["out_len"])
    assert int(st.item()) == r["status"]


def test_multi_step_histories(dev):
    """Ten chained steps of the whole path (new confidences and drafts every step): the
    device histories equal the oracle's chained schedule/pack/verify/scatter."""
    wl = synth.custom(B=12, gamma=6, V=2048, dtype="bf16", sigma=2.0, spike=6.0,
                      accept=np.linspace(0.9, 0.3, 12), tiers=(16, 32, 48, 64, 72))
    st = DSparkStep(wl.B, wl.gamma, wl.V, wl.tiers, wl.bias,
                    wl.alpha_slope * np.arange(wl.B + 1),
                    wl.theta_slope * np.arange(wl.B * wl.gamma + 1), out_cap=40, device=dev)
    hist = np.full((wl.B, 40), -1, np.int32)
    hlen = np.zeros(wl.B, np.int32)
    status = 0
    for step in range(10):
        bt = synth.make_batch(wl, seed=5, step=step)
        s = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
        p = oracle.pack(s["windows"], bt.tokens, bt.tiers, st.packed_cap)
        packed = synth.gather_packed(bt.target, bt.B, bt.gamma, s["windows"], rows_cap=p["tier"])
        v = oracle.verify(oracle.COMPACT, False, packed.view(torch.int16).numpy().view(np.uint16),
                          bt.tokens, cu=p["cu"], windows=s["windows"])
        sc = oracle.scatter(v["committed"], v["accept_len"], hist, hlen)
        hist, hlen = sc["out_tokens"], sc["out_len"]
        status |= s["status"] | p["status"] | v["status"] | sc["status"]
        st.run(torch.as_tensor(bt.conf, device=dev), torch.as_tensor(bt.tokens, device=dev),
               packed.to(dev))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(st.out_tokens.cpu().numpy(), hist)
    np.testing.assert_array_equal(st.out_len.cpu().numpy(), hlen)
    assert int(st.status.item()) == status
