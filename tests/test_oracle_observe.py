"""Pins of the oracle's observability counters ("DSpark in SGLang", A2 observability:
calibration metrics such as ECE, and the acceptance ceiling that cap-accept recovers).

A hand-worked example (outcomes observed up to the first rejection of the full block, later
drafts censored), the totals the definition fixes (observed drafts = sum min(c_b, gamma-1),
accepted = sum (c_b - 1)), bin edges, clamping, and a perfectly calibrated synthetic source
whose calibration error vanishes while a miscalibrated one's does not."""
import numpy as np

from speculative_decoding_ragged_gb300._binding import ece, utilisation

TWO32 = 1 << 32


def test_hand_worked_example(oracle_mod):
    conf = np.array([[0.9, 0.8, 0.1], [0.5, 0.5, 0.5]], np.float32)
    ceiling = np.array([3, 1], np.int32)      # request 0: d1, d2 accepted, d3 rejected
    accept = np.array([2, 1], np.int32)       # request 1: d1 rejected, d2, d3 censored
    out = oracle_mod.observe(conf, accept, ceiling, 10)
    h = out["hist"].astype(np.int64)
    expect = np.zeros((10, 3), np.int64)
    for x, k, acc in [(0.9, 9, 1), (0.8, 8, 1), (0.1, 1, 0), (0.5, 5, 0)]:
        expect[k, 0] += 1
        expect[k, 1] += int(np.rint(np.float64(np.float32(x)) * TWO32))
        expect[k, 2] += acc
    np.testing.assert_array_equal(h, expect)
    assert out["util"].tolist() == [3, 4] and out["status"] == 0
    # ECE by hand: bins 9, 8 accepted at conf .9/.8; bins 1, 5 rejected at .1/.5
    e = ece(h)
    assert abs(e - (0.1 + 0.2 + 0.1 + 0.5) / 4) < 1e-7
    assert utilisation(out["util"]) == 0.75


def test_totals_follow_the_definition(oracle_mod):
    rng = np.random.default_rng(5)
    for _ in range(30):
        B, gamma, nb = int(rng.integers(1, 50)), int(rng.integers(1, 17)), int(rng.integers(1, 40))
        conf = rng.uniform(-0.2, 1.2, size=(B, gamma - 1)).astype(np.float32)
        ceiling = rng.integers(1, gamma + 1, size=B).astype(np.int32)
        accept = np.minimum(ceiling, rng.integers(1, gamma + 1, size=B)).astype(np.int32)
        out = oracle_mod.observe(conf, accept, ceiling, nb)
        h = out["hist"].astype(np.int64)
        assert h[:, 0].sum() == np.minimum(ceiling, gamma - 1).sum()
        assert h[:, 2].sum() == (ceiling - 1).sum()
        assert (h[:, 2] <= h[:, 0]).all()
        assert out["util"].tolist() == [int(accept.sum()), int(ceiling.sum())]


def test_bin_edges_clamping_and_flags(oracle_mod):
    conf = np.array([[0.0, 1.0, 0.25, np.nan, 2.0, -1.0]], np.float32)
    out = oracle_mod.observe(conf, np.array([9], np.int32), np.array([7], np.int32), 4)
    h = out["hist"].astype(np.int64)
    # bins: 0.0 -> 0, 1.0 -> 3 (top bin), 0.25 -> 1, NaN -> 0, 2.0 -> 3, -1.0 -> 0
    assert h[:, 0].tolist() == [3, 1, 0, 2]
    assert h[3, 1] == 2 * TWO32 and h[0, 1] == 0
    assert h[:, 2].sum() == 6                 # ceiling 7 = gamma: every draft accepted
    assert out["status"] == 0x80 and out["util"].tolist() == [7, 7]


def test_calibrated_source_has_small_ece(oracle_mod):
    rng = np.random.default_rng(0)
    B, gamma = 20000, 6
    conf = rng.uniform(0.05, 0.95, size=(B, gamma - 1)).astype(np.float32)
    acc = rng.uniform(size=conf.shape) < conf          # each draft accepted with prob = conf
    lead = np.where((~acc).any(axis=1), (~acc).argmax(axis=1), gamma - 1)
    ceiling = (lead + 1).astype(np.int32)
    out = oracle_mod.observe(conf, ceiling, ceiling, 20)
    assert ece(out["hist"]) < 0.01
    over = oracle_mod.observe(np.clip(conf * 1.3, 0, 1), ceiling, ceiling, 20)
    assert ece(over["hist"]) > 0.05
