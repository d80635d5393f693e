"""Pins of the oracle's counter-based generator and of how verify keys and maps its uniforms.

The oracle's Philox4x64-10 is hand-written C; numpy ships an independent implementation of the
same published generator (``numpy.random.Philox``, Salmon et al., SC'11), which pins it word
for word. numpy advances its counter by one before producing a block, so block ``c`` is read
from a generator started at ``c - 1``.
"""
import numpy as np
import pytest


def numpy_philox(ctr, key):
    c = sum(int(x) << (64 * i) for i, x in enumerate(ctr))
    k = sum(int(x) << (64 * i) for i, x in enumerate(key))
    bg = np.random.Philox(key=k, counter=(c - 1) % (1 << 256))
    return bg.random_raw(4).astype(np.uint64)


def test_philox_matches_numpy_random_counters(oracle_mod):
    rng = np.random.default_rng(1234)
    cases = [((0, 0, 0, 0), (0, 0)), ((2**64 - 1,) * 4, (2**64 - 1,) * 2),
             ((1, 0, 0, 0), (0, 0)), ((0, 0, 0, 1), (0, 1))]
    for _ in range(200):
        ctr = tuple(int(x) for x in rng.integers(0, 2**64, size=4, dtype=np.uint64))
        key = tuple(int(x) for x in rng.integers(0, 2**64, size=2, dtype=np.uint64))
        cases.append((ctr, key))
    for ctr, key in cases:
        mine = oracle_mod.philox4x64_10(np.array(ctr, np.uint64), np.array(key, np.uint64))
        np.testing.assert_array_equal(mine, numpy_philox(ctr, key), err_msg=f"{ctr} {key}")


def test_verify_uniforms_are_keyed_by_seed_request_position_step(oracle_mod):
    """diag_u[b, i] must be word 0 of Philox(key=(seed,0), ctr=(b,i,step,0)) >> 40, * 2^-24."""
    B, gamma, V = 3, 5, 8
    rng = np.random.default_rng(7)
    target = rng.standard_normal((B * gamma, V)).astype(np.float32)
    draft = rng.standard_normal((B * (gamma - 1), V)).astype(np.float32)
    tokens = rng.integers(0, V, size=(B, gamma)).astype(np.int32)
    for seed, step in [(0, 0), (99, 5), (2**40 + 3, 2**33 + 1)]:
        out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft,
                                temperature=1.0, seed=seed, step=step)
        for b in range(B):
            for i in range(gamma - 1):
                w0 = int(numpy_philox((b, i, step, 0), (seed, 0))[0])
                u = np.float32((w0 >> 40) * 2.0**-24)
                assert out["u"][b, i] == u


def test_uniforms_are_uniform(oracle_mod):
    """Kolmogorov-Smirnov on the 24-bit accept uniforms of 20000 counters."""
    stats = pytest.importorskip("scipy.stats")
    us = []
    for b in range(20000):
        w = oracle_mod.philox4x64_10(np.array([b, 3, 11, 0], np.uint64),
                                     np.array([5, 0], np.uint64))
        us.append((int(w[0]) >> 40) * 2.0**-24)
    assert stats.kstest(us, "uniform").pvalue > 1e-3
