"""GPU parity of dspark_schedule and dspark_pack against the oracle: bit-exact windows, K*,
status bits, cu_seqlens, tiers and packed rows, from tiny to the maximum sizes."""
import numpy as np
import pytest
import torch

from speculative_decoding_ragged_gb300 import synth
import oracle

from gpu_util import device, gpu_pack, gpu_schedule

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


def tables(rng, B, gamma, kind):
    M = np.arange(B * gamma + 1, dtype=np.float64)
    alpha = rng.uniform(0, 0.1) * np.arange(B + 1, dtype=np.float64)
    bias = float(rng.uniform(0.5, 3))
    if kind == 0:
        theta = rng.uniform(0, 0.05) * M
    elif kind == 1:
        theta = np.ceil(M / 64) * rng.uniform(0, 0.2)
    elif kind == 2:
        theta = rng.uniform(0, 1.0, size=M.size)
    elif kind == 3:     # negative bias and an offset theta: T > 0 only through cancellation
        bias = -5.0
        theta = 6.0 + rng.uniform(0, 0.05) * M
    else:               # a mix of negative, zero, tiny and huge entries
        theta = rng.choice([-1.0, 0.0, 1e-30, 1e25, 0.5], size=M.size) * rng.uniform(0.5, 1.5, M.size)
    return bias, alpha, theta


SIZES = [(1, 1), (1, 2), (4, 4), (3, 32), (7, 8), (100, 5), (256, 8), (512, 8), (1000, 17),
         (2048, 9), (8192, 2), (8192, 3), (5, 1), (1023, 2), (1025, 3),
         # the one-warp kernel's range (n <= 32) and just past it
         (32, 2), (16, 3), (2, 17), (11, 3), (1, 32), (1, 16), (33, 2), (3, 12),
         # the 256-thread block (n <= 256) at its edge and the 1024-thread block just past it
         (128, 3), (8, 32), (257, 2), (52, 6)]


@pytest.mark.parametrize("B,gamma", SIZES)
def test_schedule_parity_random(dev, B, gamma):
    rng = np.random.default_rng(B * 100 + gamma)
    for trial in range(6):
        a = rng.uniform(0.1, 0.95, size=B)
        conf = rng.beta(8 * a[:, None], 8 * (1 - a[:, None]), size=(B, gamma - 1))
        if trial == 1:
            conf = np.round(conf * 8) / 8          # many equal survivals: tie rule
        if trial == 2:
            conf[rng.uniform(size=conf.shape) < 0.05] = np.nan
            conf[rng.uniform(size=conf.shape) < 0.05] = 1.5
        conf = conf.astype(np.float32)
        bias, alpha, theta = tables(rng, B, gamma, trial % 5)
        g = gpu_schedule(dev, conf, bias, alpha, theta)
        r = oracle.schedule(conf, bias, alpha, theta)
        np.testing.assert_array_equal(g["windows"], r["windows"])
        assert g["k_star"] == r["k_star"] and g["status"] == r["status"]


@pytest.mark.parametrize("name", list(synth.WORKLOADS))
def test_schedule_parity_workloads(dev, name):
    wl = synth.WORKLOADS[name]
    thetas = synth.HIGH_LOAD_THETAS if name == "high_load" else (wl.theta_slope,)
    small = wl.with_(V=64)                      # the schedule never reads logits
    for seed in range(3):
        for th in thetas:
            bt = synth.make_batch(small, seed=seed, theta_slope=th)
            g = gpu_schedule(dev, bt.conf, bt.bias, bt.alpha, bt.theta)
            r = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
            np.testing.assert_array_equal(g["windows"], r["windows"])
            assert g["k_star"] == r["k_star"] and g["status"] == r["status"] == 0


def test_schedule_invalid_cost_and_empty(dev):
    conf = np.full((3, 4), 0.5, np.float32)
    g = gpu_schedule(dev, conf, 1.0, np.zeros(4), np.full(16, -5.0))
    assert g["status"] == 0x10 and g["k_star"] == 0 and (g["windows"] == 1).all()
    g = gpu_schedule(dev, np.zeros((0, 4), np.float32), 1.0, np.zeros(1), np.zeros(1))
    assert g["k_star"] == 0
    g = gpu_schedule(dev, np.zeros((6, 0), np.float32), 1.0, np.zeros(7), np.full(7, -1.0))
    assert g["status"] == 0x10 and (g["windows"] == 1).all()


def tie_table(B, near=()):
    """Every objective exactly B 2^31 (gamma = 2, confidences 0.5, bias 2, theta[B + K] = K / B,
    B a power of two); each K in `near` one ulp above the rest (its theta lowered by 2^-51)."""
    conf = np.full((B, 1), 0.5, np.float32)
    theta = np.zeros(2 * B + 1)
    theta[B:] = np.arange(B + 1) / B
    for k in near:
        theta[B + k] -= 2.0 ** -51
    return conf, 2.0, np.zeros(B + 1), theta


@pytest.mark.parametrize("B", [1, 16, 32, 64, 256, 4096, 8192])
def test_schedule_exact_and_one_ulp_ties(dev, B):
    """Objectives that tie exactly or differ by one ulp, which no screen can order: both
    kernels (one warp up to 32 candidates, the block kernel's bucket and bitonic sorts) must
    fall back to the exact objectives and agree with the oracle."""
    rng = np.random.default_rng(B)
    cases = [()] + [tuple(int(k) for k in rng.choice(np.arange(1, B + 1), size=m, replace=False))
                    for m in (1, 2, 5) if m <= B]
    for near in cases:
        conf, bias, alpha, theta = tie_table(B, near)
        g = gpu_schedule(dev, conf, bias, alpha, theta)
        r = oracle.schedule(conf, bias, alpha, theta)
        assert r["k_star"] == (min(near) if near else 0)
        np.testing.assert_array_equal(g["windows"], r["windows"])
        assert g["k_star"] == r["k_star"] and g["status"] == r["status"] == 0


@pytest.mark.parametrize("B,gamma", [(64, 8), (256, 8), (600, 6), (2048, 9)])
def test_schedule_k_star_at_and_near_zero(dev, B, gamma):
    """Steep cost tables put the argmax at K = 0 or among the first few K, where the block
    kernel's exact pass holds K = 0 in its first slot (with or without other candidates)."""
    from speculative_decoding_ragged_gb300.step import DSparkStep
    rng = np.random.default_rng(7 * B + gamma)
    M = np.arange(B * gamma + 1, dtype=np.float64)
    seen = set()
    for trial in range(10):
        conf = rng.uniform(0.05, 0.99, size=(B, gamma - 1)).astype(np.float32)
        alpha = np.zeros(B + 1)
        bias = float(rng.uniform(0.001, 0.1))
        if trial == 0:
            theta = np.where(M <= B, 0.0, 1e6)              # any candidate is ruinous: K* = 0
        else:
            # the first candidate's gain against its cost near break-even
            step = float(np.exp(rng.uniform(np.log(0.5), np.log(2.0)))) * (bias + 1.0) / B
            theta = np.where(M <= B, M / B, 1.0 + (M - B) * step)
        g = gpu_schedule(dev, conf, bias, alpha, theta)
        r = oracle.schedule(conf, bias, alpha, theta)
        np.testing.assert_array_equal(g["windows"], r["windows"])
        assert g["k_star"] == r["k_star"] and g["status"] == r["status"] == 0
        st = DSparkStep(B, gamma, 64, [B * gamma], bias, alpha, theta, device=dev)
        st.schedule_pack(torch.as_tensor(conf, device=dev),
                         torch.zeros((B, gamma), dtype=torch.int32, device=dev))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(st.windows.cpu().numpy(), r["windows"])
        assert int(st.k_star.item()) == r["k_star"]
        seen.add(min(r["k_star"], 10))
    assert 0 in seen and len(seen - {0}) > 0, seen


@pytest.mark.parametrize("B,gamma", [(0, 4), (1, 1), (2, 6), (33, 8), (1025, 4), (8192, 8),
                                     (300, 32)])
def test_pack_parity(dev, B, gamma):
    rng = np.random.default_rng(B + gamma)
    for trial in range(4):
        windows = rng.integers(1, gamma + 1, size=B)
        if trial == 3 and B:
            windows[rng.uniform(size=B) < 0.1] = gamma + 3      # clamped, flagged
            windows[rng.uniform(size=B) < 0.1] = 0
        tokens = rng.integers(0, 150000, size=(B, gamma))
        tiers = rng.permutation(np.arange(1, B * gamma + 9))[:int(rng.integers(1, 20))]
        if trial == 0:
            tiers = np.arange(1, 64) * max(1, B * gamma // 32)
        cap = [B * gamma + 8, int(tiers.max()) + 3, max(1, B * gamma // 2), 0][trial]
        g = gpu_pack(dev, windows, tokens, tiers, cap)
        r = oracle.pack(windows, tokens, tiers, cap)
        for key in ("cu", "packed_ids", "row_req", "row_pos"):
            np.testing.assert_array_equal(g[key], r[key], err_msg=key)
        assert (g["M"], g["tier"], g["status"]) == (r["M"], r["tier"], r["status"])


def test_pack_page_example(dev):
    tokens = np.array([[10, 11, 12, 13, 14, 15], [20, 21, 22, 23, 24, 25]])
    g = gpu_pack(dev, np.array([2, 6]), tokens, np.array([16, 4, 8]), 16)
    assert g["cu"].tolist() == [0, 2, 8] and g["M"] == 8 and g["tier"] == 8
    assert g["packed_ids"][:8].tolist() == [10, 11, 20, 21, 22, 23, 24, 25]
    assert (g["packed_ids"][8:] == -7).all()
