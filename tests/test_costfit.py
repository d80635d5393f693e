"""The additive cost-table fit ("DSpark in SGLang", A2 method details, cost-table profiling and
modelling): T(bs, K) = bias + alpha(bs) + theta(bs + K), fitted by least squares.

Pins that do not re-run the fit's own routine: the two-way-layout closed form of least squares
(row mean + column mean - grand mean), exact recovery of an additive table up to the gauge,
the tier key, the linear interpolation of the full tables, and the scheduler's decisions on
fitted against true tables."""
import numpy as np
import pytest

from speculative_decoding_ragged_gb300.costfit import compare, fit_additive, tier_key


def test_complete_two_way_layout_matches_the_anova_closed_form():
    # one sample per (bs, M) cell of a complete grid: the least-squares additive fit of a
    # two-way table without interaction is y_i. + y_.j - y_.. (textbook closed form)
    rng = np.random.default_rng(0)
    bss = np.array([1, 3, 4, 9])
    Ms = np.array([10, 12, 20, 31, 40])
    Y = rng.uniform(1, 5, size=(bss.size, Ms.size))           # not additive
    bs, M = np.meshgrid(bss, Ms, indexing="ij")
    fit = fit_additive(bs.ravel(), M.ravel(), Y.ravel())
    closed = Y.mean(axis=1, keepdims=True) + Y.mean(axis=0, keepdims=True) - Y.mean()
    np.testing.assert_allclose(fit.predict(bs, M), closed, rtol=1e-12, atol=1e-12)
    assert fit.alpha_knots[0] == 0 and fit.theta_knots[0] == 0
    # the gauge-fixed tables are the closed form's row and column effects, re-based
    np.testing.assert_allclose(fit.alpha_knots, Y.mean(axis=1) - Y.mean(axis=1)[0], atol=1e-12)
    np.testing.assert_allclose(fit.theta_knots, Y.mean(axis=0) - Y.mean(axis=0)[0], atol=1e-12)


def test_exact_additive_tables_are_recovered_on_an_incomplete_design():
    rng = np.random.default_rng(1)
    bss = np.array([1, 2, 4, 8, 16])
    alpha = {b: rng.uniform(0, 3) for b in bss}
    theta = {m: rng.uniform(0, 9) for m in range(1, 129)}
    bias = 2.5
    bs, M = [], []
    for b in bss:                                  # each bs sees M in [b, 8b]: a staircase
        for m in rng.choice(np.arange(b, 8 * b + 1), size=min(6, 7 * b + 1), replace=False):
            bs.append(b)
            M.append(int(m))
    bs, M = np.array(bs), np.array(M)
    T = np.array([bias + alpha[b] + theta[m] for b, m in zip(bs, M)])
    fit = fit_additive(bs, M, T)
    np.testing.assert_allclose(fit.predict(bs, M), T, rtol=1e-12)
    assert fit.residual_rms < 1e-10
    b0, m0 = fit.bs_knots[0], fit.key_knots[0]
    np.testing.assert_allclose(fit.alpha_knots, [alpha[b] - alpha[b0] for b in fit.bs_knots],
                               atol=1e-10)
    np.testing.assert_allclose(fit.theta_knots, [theta[m] - theta[m0] for m in fit.key_knots],
                               atol=1e-10)
    assert abs(fit.bias - (bias + alpha[b0] + theta[m0])) < 1e-10


def test_noise_fit_stays_within_the_noise():
    rng = np.random.default_rng(2)
    tiers = list(range(8, 257, 8))
    bs = rng.choice([1, 2, 4, 8, 16, 32], size=600)
    M = bs + rng.integers(0, 7 * bs + 1)
    true = 3.0 + 0.05 * bs + 0.01 * tier_key(M, tiers)
    sigma = 0.02
    T = true + rng.normal(0, sigma, size=bs.size)
    fit = fit_additive(bs, M, T, tiers=tiers)
    assert fit.residual_rms <= sigma * 1.05
    err = fit.predict(bs, M) - true
    assert np.sqrt(np.mean(err ** 2)) < 0.6 * sigma     # far more samples than parameters
    r = compare(fit, bs, M, T)
    assert r["n"] == 600 and r["r2"] > 0.99 and r["mean_abs_rel"] < 0.01


def test_tier_key_is_the_padded_row_count():
    tiers = [32, 64, 96]
    assert tier_key([1, 32, 33, 96, 97, 0], tiers).tolist() == [32, 32, 64, 96, 97, 32]
    assert tier_key([5, 7], None).tolist() == [5, 7]
    # samples in one tier share a theta entry: a per-tier step function is fitted exactly
    bs = np.array([1, 1, 2, 2, 4, 4, 4])
    M = np.array([1, 40, 2, 33, 4, 64, 70])
    theta = {32: 0.0, 64: 1.5, 96: 4.0}
    alpha = {1: 0.0, 2: 0.25, 4: 0.75}
    T = np.array([1.0 + alpha[b] + theta[int(k)] for b, k in zip(bs, tier_key(M, tiers))])
    fit = fit_additive(bs, M, T, tiers=tiers)
    assert fit.key_knots.tolist() == [32, 64, 96]
    np.testing.assert_allclose(fit.theta_knots, [0.0, 1.5, 4.0], atol=1e-12)
    np.testing.assert_allclose(fit.predict([1, 2], [63, 90]), [2.5, 5.25], atol=1e-12)


def test_full_tables_interpolate_between_knots_and_hold_the_ends():
    bs = np.array([2, 2, 6, 6])
    M = np.array([10, 20, 10, 20])
    T = np.array([1.0, 3.0, 2.0, 4.0])           # alpha(6) - alpha(2) = 1, theta(20) - theta(10) = 2
    fit = fit_additive(bs, M, T)
    bias, alpha, theta = fit.tables(B=8, gamma=3)
    assert alpha.shape == (9,) and theta.shape == (25,)
    np.testing.assert_allclose(alpha, [0, 0, 0, 0.25, 0.5, 0.75, 1, 1, 1], atol=1e-12)
    np.testing.assert_allclose(theta[:10], 0, atol=1e-12)
    np.testing.assert_allclose(theta[15], 1.0, atol=1e-12)
    np.testing.assert_allclose(theta[20:], 2.0, atol=1e-12)
    assert abs(bias - 1.0) < 1e-12


def test_disconnected_samples_are_refused():
    # bs 1 only ever with M 1..2 and bs 8 only with M 50..51: the offset between the two
    # groups is not determined
    with pytest.raises(ValueError):
        fit_additive([1, 1, 8, 8], [1, 2, 50, 51], [1.0, 2.0, 3.0, 4.0])
    with pytest.raises(ValueError):
        fit_additive([], [], [])
    with pytest.raises(ValueError):
        fit_additive([4], [3], [1.0])             # M < bs


def test_fitted_tables_drive_the_scheduler_like_the_true_ones():
    import oracle
    from speculative_decoding_ragged_gb300 import synth
    rng = np.random.default_rng(3)
    wl = synth.WORKLOADS["stochastic"].with_(V=64)
    B, gamma = wl.B, wl.gamma
    bt = synth.make_batch(wl, seed=4)
    # the true tables: a convex theta and a mild alpha
    Ms = np.arange(B * gamma + 1)
    theta_true = 0.002 * Ms + 1e-6 * Ms ** 2
    alpha_true = 0.01 * np.arange(B + 1)
    bias = 1.0
    bs = rng.integers(1, B + 1, size=3000)
    bs[:B] = np.arange(1, B + 1)
    M = bs + rng.integers(0, (gamma - 1) * bs + 1)
    M[-(B * gamma - B + 1):] = np.arange(B, B * gamma + 1)     # every M the scheduler reads
    bs[-(B * gamma - B + 1):] = B
    T = bias + alpha_true[bs] + theta_true[M]
    fit = fit_additive(bs, M, T)
    fb, fa, ft = fit.tables(B, gamma)
    r_true = oracle.schedule(bt.conf, bias, alpha_true, theta_true)
    r_fit = oracle.schedule(bt.conf, fb, fa, ft)
    np.testing.assert_array_equal(r_fit["windows"], r_true["windows"])
    assert r_fit["k_star"] == r_true["k_star"]


def test_forced_windows_sum_to_M_and_stay_in_range():
    from speculative_decoding_ragged_gb300.sps_profile import forced_windows
    for bs, gamma in [(1, 8), (5, 3), (256, 8)]:
        for M in range(bs, gamma * bs + 1, max(1, bs // 3)):
            w = forced_windows(bs, gamma, M)
            assert w.sum() == M and w.min() >= 1 and w.max() <= gamma
            assert w.max() - w.min() <= 1
    with pytest.raises(ValueError):
        forced_windows(4, 2, 9)


def test_recorder_grid_includes_both_ends_and_shares_tiers():
    from speculative_decoding_ragged_gb300.sps_profile import grid_M
    tiers = list(range(32, 2049, 32))
    grids = {bs: grid_M(bs, 8, tiers, 12) for bs in (1, 16, 48, 256)}
    for bs, g in grids.items():
        assert g[0] == bs and g[-1] == 8 * bs and len(g) <= 12 and g == sorted(set(g))
    assert set(grids[16]) & set(grids[48])          # batch sizes meet on common tiers
