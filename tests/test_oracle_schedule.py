"""Pins of the oracle's confidence scheduler ("DSpark in SGLang", A2: survival = product of
confidences along the block; T(bs,K) = bias + alpha(bs) + theta(bs+K); argmax of expected
committed tokens over step cost).

* survival keys against numpy's float32 running product and rint (an independent computation);
* the argmax against brute-force enumeration of every window allocation (B <= 3, gamma <= 4);
* closed forms: theta = 0 keeps every positive survival, a huge theta keeps none, equal
  survivals fill requests in (b, j) order, an all-invalid cost table;
* the budget-shrink invariant: K* never grows when theta's slope grows.
"""
import itertools

import numpy as np
import pytest

TWO32 = 1 << 32


def np_keys(conf):
    c = np.clip(np.nan_to_num(np.asarray(conf, np.float32), nan=0.0), 0.0, 1.0)
    s = np.multiply.accumulate(c, axis=1, dtype=np.float32)  # sequential fp32 products
    return np.rint(s.astype(np.float64) * TWO32).astype(np.uint64)


def test_survival_keys_match_numpy(oracle_mod):
    rng = np.random.default_rng(0)
    for _ in range(20):
        B, L = rng.integers(1, 40), rng.integers(1, 16)
        conf = rng.beta(2, 1, size=(B, L)).astype(np.float32)
        conf[rng.uniform(size=conf.shape) < 0.05] = 1.0
        conf[rng.uniform(size=conf.shape) < 0.02] = 0.0
        np.testing.assert_array_equal(oracle_mod.survival_keys(conf), np_keys(conf))


def test_survival_keys_clamp_and_nan(oracle_mod):
    conf = np.array([[1.5, 0.5, np.nan, 0.5], [-0.25, 0.9, 0.9, 0.9]], np.float32)
    keys = oracle_mod.survival_keys(conf)
    np.testing.assert_array_equal(keys[0], [TWO32, TWO32 // 2, 0, 0])
    np.testing.assert_array_equal(keys[1], [0, 0, 0, 0])


def brute_force(conf, bias, alpha, theta):
    """Best objective over every allocation w in [1..gamma]^B, and the smallest K reaching it."""
    keys = np_keys(conf)
    B, L = keys.shape
    t0 = bias + alpha[B]
    best, best_k, best_ws = None, None, []
    for w in itertools.product(range(1, L + 2), repeat=B):
        K = sum(x - 1 for x in w)
        T = t0 + theta[B + K]
        if not (T > 0 and np.isfinite(T)):
            continue
        E = B * TWO32 + sum(int(keys[b, :w[b] - 1].sum()) for b in range(B))
        obj = float(E) / T
        if best is None or obj > best or (obj == best and K < best_k):
            best, best_k = obj, K
    if best is not None:
        for w in itertools.product(range(1, L + 2), repeat=B):
            K = sum(x - 1 for x in w)
            T = t0 + theta[B + K]
            if K != best_k:
                continue
            E = B * TWO32 + sum(int(keys[b, :w[b] - 1].sum()) for b in range(B))
            if float(E) / T == best:
                best_ws.append(w)
    return best, best_k, best_ws


def random_tables(rng, B, gamma, kind):
    n_m = B * gamma + 1
    bias = float(rng.uniform(0.1, 3.0))
    alpha = rng.uniform(0.0, 0.2) * np.arange(B + 1, dtype=np.float64)
    M = np.arange(n_m, dtype=np.float64)
    if kind == 0:
        theta = rng.uniform(0.0, 0.5) * M
    elif kind == 1:   # convex, like a compute-bound regime beyond a knee
        knee = rng.integers(1, n_m)
        theta = rng.uniform(0.0, 0.05) * M + rng.uniform(0.0, 1.0) * np.maximum(0, M - knee)
    elif kind == 2:   # stepwise, like graph tiers
        theta = rng.uniform(0.0, 0.6) * np.ceil(M / rng.integers(1, 4))
    else:             # arbitrary non-negative table
        theta = rng.uniform(0.0, 2.0, size=n_m)
    return bias, alpha, theta


@pytest.mark.parametrize("B,gamma", [(1, 2), (1, 4), (2, 3), (2, 4), (3, 3), (3, 4)])
def test_schedule_equals_brute_force(oracle_mod, B, gamma):
    rng = np.random.default_rng(100 * B + gamma)
    for trial in range(300 if B < 3 else 120):
        conf = rng.beta(rng.uniform(0.5, 8), rng.uniform(0.5, 4), size=(B, gamma - 1))
        if trial % 7 == 0:   # force equal survivals across requests (tie rule)
            conf[:] = conf[0:1, :]
        if trial % 11 == 0:
            conf = np.round(conf * 4) / 4
        conf = conf.astype(np.float32)
        bias, alpha, theta = random_tables(rng, B, gamma, trial % 4)
        out = oracle_mod.schedule(conf, bias, alpha, theta)
        best, best_k, best_ws = brute_force(conf, bias, alpha, theta)
        assert out["status"] == 0
        assert out["k_star"] == best_k
        assert out["obj"][best_k] == best
        assert tuple(int(x) for x in out["windows"]) in best_ws
        assert int(out["windows"].sum()) == B + best_k


def test_tie_rule_fills_lower_request_then_lower_position(oracle_mod):
    """Equal survivals: the first K* candidates in (b, j) order are taken."""
    B, gamma = 3, 4
    conf = np.ones((B, gamma - 1), np.float32)
    theta = np.zeros(B * gamma + 1)
    theta[B + 6:] = 1e9        # any K > 5 is hopeless, K = 5 is the best
    out = oracle_mod.schedule(conf, 1.0, np.zeros(B + 1), theta)
    assert out["k_star"] == 5
    np.testing.assert_array_equal(out["windows"], [4, 3, 1])


def tie_table(B, near=()):
    """gamma = 2, every confidence 0.5 (key 2^31), bias 2, alpha 0, theta[B + K] = K / B with
    B a power of two: E(K) = (2B + K) 2^31 and T(K) = (2B + K) / B are exact doubles, so every
    objective is exactly B 2^31. Each K in `near` gets theta lowered by 2^-51 (one ulp of T),
    which lifts its objective one ulp above the others."""
    conf = np.full((B, 1), 0.5, np.float32)
    theta = np.zeros(2 * B + 1)
    K = np.arange(B + 1)
    theta[B:] = K / B
    for k in near:
        theta[B + k] -= 2.0 ** -51
    return conf, 2.0, np.zeros(B + 1), theta


@pytest.mark.parametrize("B", [1, 16, 64])
def test_equal_objectives_take_the_smallest_k(oracle_mod, B):
    """Exact ties: every K has the same objective, so K* = 0 (the smallest K)."""
    conf, bias, alpha, theta = tie_table(B)
    out = oracle_mod.schedule(conf, bias, alpha, theta)
    assert all(o == B * 2.0 ** 31 for o in out["obj"])
    assert out["k_star"] == 0
    np.testing.assert_array_equal(out["windows"], 1)


def test_one_ulp_apart_objectives(oracle_mod):
    """Near ties: a K whose step time is one ulp shorter wins by one ulp of the objective;
    among two such K the smaller wins; the windows fill requests in order (equal keys)."""
    B = 64
    conf, bias, alpha, theta = tie_table(B, near=(37,))
    out = oracle_mod.schedule(conf, bias, alpha, theta)
    assert out["obj"][37] == np.nextafter(B * 2.0 ** 31, np.inf)
    assert out["k_star"] == 37
    np.testing.assert_array_equal(out["windows"], [2] * 37 + [1] * (B - 37))
    conf, bias, alpha, theta = tie_table(B, near=(50, 21))
    out = oracle_mod.schedule(conf, bias, alpha, theta)
    assert out["k_star"] == 21


def test_theta_zero_keeps_every_positive_survival(oracle_mod):
    rng = np.random.default_rng(5)
    B, gamma = 17, 8
    conf = rng.uniform(0.2, 1.0, size=(B, gamma - 1)).astype(np.float32)
    out = oracle_mod.schedule(conf, 1.0, 0.05 * np.arange(B + 1), np.zeros(B * gamma + 1))
    np.testing.assert_array_equal(out["windows"], gamma)
    assert out["k_star"] == B * (gamma - 1)


def test_huge_theta_keeps_nothing(oracle_mod):
    rng = np.random.default_rng(6)
    B, gamma = 9, 6
    conf = rng.uniform(0.0, 1.0, size=(B, gamma - 1)).astype(np.float32)
    out = oracle_mod.schedule(conf, 1.0, np.zeros(B + 1), 1e6 * np.arange(B * gamma + 1))
    np.testing.assert_array_equal(out["windows"], 1)
    assert out["k_star"] == 0


def test_zero_survivals_are_never_taken(oracle_mod):
    B, gamma = 4, 5
    conf = np.full((B, gamma - 1), 0.9, np.float32)
    conf[1, 1] = 0.0        # request 1 survives one draft only
    conf[3, :] = 0.0        # request 3 none
    out = oracle_mod.schedule(conf, 1.0, np.zeros(B + 1), np.zeros(B * gamma + 1))
    np.testing.assert_array_equal(out["windows"], [5, 2, 5, 1])


def test_invalid_cost_table(oracle_mod):
    B, gamma = 2, 3
    conf = np.full((B, gamma - 1), 0.5, np.float32)
    theta = np.full(B * gamma + 1, -10.0)
    out = oracle_mod.schedule(conf, 1.0, np.zeros(B + 1), theta)
    assert out["status"] == 0x10 and out["k_star"] == 0
    np.testing.assert_array_equal(out["windows"], 1)
    # only K = 3 has a positive finite T
    theta = np.full(B * gamma + 1, np.inf)
    theta[B + 3] = 1.0
    out = oracle_mod.schedule(conf, 0.0, np.zeros(B + 1), theta)
    assert out["status"] == 0 and out["k_star"] == 3


def test_degenerate_sizes(oracle_mod):
    out = oracle_mod.schedule(np.zeros((0, 3), np.float32), 1.0, np.zeros(1), np.zeros(1))
    assert out["k_star"] == 0 and out["windows"].size == 0
    out = oracle_mod.schedule(np.zeros((5, 0), np.float32), 1.0, np.zeros(6), np.zeros(6))
    assert out["k_star"] == 0
    np.testing.assert_array_equal(out["windows"], 1)


def test_budget_shrinks_as_theta_grows(oracle_mod):
    """With linear alpha, theta and a positive bias, the mean of (B ones, then sorted
    survivals <= 1) never rises with K, so a steeper theta never favours a larger K."""
    rng = np.random.default_rng(11)
    for trial in range(40):
        B, gamma = int(rng.integers(1, 64)), int(rng.integers(2, 10))
        a = rng.uniform(0.2, 0.95, size=B)
        conf = rng.beta(10 * a[:, None], 10 * (1 - a[:, None]), size=(B, gamma - 1))
        conf = conf.astype(np.float32)
        alpha = 0.01 * np.arange(B + 1)
        prev = None
        for slope in [0.0, 0.0005, 0.001, 0.002, 0.004, 0.008, 0.016, 0.05, 0.2, 1.0]:
            out = oracle_mod.schedule(conf, 2.0, alpha, slope * np.arange(B * gamma + 1))
            if prev is not None:
                assert out["k_star"] <= prev
            prev = out["k_star"]
