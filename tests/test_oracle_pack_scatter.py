"""Pins of the oracle's front-pack and compact scatter.

Front-pack ("DSpark in SGLang", A2, ragged verify over full CUDA graphs): cu_seqlens against
numpy's cumulative sum, the tier against a sorted search, every packed row mapped back to its
(request, position), the page's own two-request example (one request verifies 2 tokens,
another 6). Compact scatter ("DSpark in SGLang", A2, performance: fused compact scatter): each
history grows by its accept length and holds the committed prefix.
"""
import json
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def check_pack(out, windows, tokens, tiers, cap):
    B, gamma = tokens.shape
    w = np.clip(windows, 1, gamma)
    np.testing.assert_array_equal(out["cu"], np.concatenate([[0], np.cumsum(w)]))
    M = int(w.sum())
    assert out["M"] == M
    st = np.sort(tiers)
    k = np.searchsorted(st, M, side="left")
    tier = int(st[k]) if k < st.size else M
    assert out["tier"] == tier
    seen = set()
    for r in range(min(M, cap)):
        b, i = int(out["row_req"][r]), int(out["row_pos"][r])
        assert 0 <= i < w[b]
        assert out["packed_ids"][r] == tokens[b, i]
        seen.add((b, i))
    if M <= cap:
        assert seen == {(b, i) for b in range(B) for i in range(w[b])}
    for r in range(M, min(tier, cap)):
        assert out["packed_ids"][r] == 0 and out["row_req"][r] == -1 and out["row_pos"][r] == -1
    for r in range(max(tier, M), cap):     # never written
        assert out["packed_ids"][r] == -7
    return M, tier


def test_pack_random(oracle_mod):
    rng = np.random.default_rng(3)
    for _ in range(200):
        B, gamma = int(rng.integers(0, 40)), int(rng.integers(1, 17))
        windows = rng.integers(1, gamma + 1, size=B).astype(np.int32)
        tokens = rng.integers(0, 50000, size=(B, gamma)).astype(np.int32)
        tiers = rng.choice(np.arange(1, B * gamma + 40), size=int(rng.integers(1, 6)),
                           replace=False).astype(np.int32)
        cap = int(max(tiers.max(), B * gamma))
        out = oracle_mod.pack(windows, tokens, tiers, cap)
        M, tier = check_pack(out, windows, tokens, tiers, cap)
        expect = 0 if tiers.max() >= M else 0x01
        assert out["status"] == expect


def test_pack_page_example():
    """The page's ragged example: two requests verifying 2 and 6 tokens pack into 8 rows."""
    with open(os.path.join(GOLDEN, "ragged_pack_example.json")) as f:
        ex = json.load(f)
    import oracle
    tokens = np.array(ex["tokens"], np.int32)
    for case in ex["tier_sets"]:
        out = oracle.pack(np.array(ex["windows"], np.int32), tokens,
                          np.array(case["tiers"], np.int32), 32)
        assert out["cu"].tolist() == ex["cu_seqlens"]
        assert out["M"] == ex["M"]
        assert out["tier"] == case["tier"]
        assert out["packed_ids"][:ex["M"]].tolist() == ex["packed_ids"]


def test_pack_flags(oracle_mod):
    tokens = np.arange(12, dtype=np.int32).reshape(3, 4)
    out = oracle_mod.pack(np.array([0, 9, 2], np.int32), tokens, np.array([4], np.int32), 16)
    assert out["status"] == 0x04 | 0x01          # bad windows clamped; M = 7 above tier 4
    assert out["cu"].tolist() == [0, 1, 5, 7] and out["tier"] == 7
    out = oracle_mod.pack(np.array([4, 4, 4], np.int32), tokens, np.array([16], np.int32), 10)
    assert out["status"] == 0x02                 # tier 16 above capacity 10
    assert out["packed_ids"].tolist() == list(range(10))


def test_scatter(oracle_mod):
    rng = np.random.default_rng(9)
    for _ in range(100):
        B, gamma, cap = int(rng.integers(0, 30)), int(rng.integers(1, 17)), int(rng.integers(1, 64))
        committed = rng.integers(0, 1000, size=(B, gamma)).astype(np.int32)
        L = rng.integers(0, gamma + 1, size=B).astype(np.int32)
        n0 = rng.integers(0, cap + 1, size=B).astype(np.int32)
        hist = rng.integers(-5, 0, size=(B, cap)).astype(np.int32)
        out = oracle_mod.scatter(committed, L, hist, n0)
        overflow = False
        for b in range(B):
            n1 = min(cap, int(n0[b]) + int(L[b]))
            assert out["out_len"][b] == n1
            assert out["out_tokens"][b, n0[b]:n1].tolist() == committed[b, :n1 - n0[b]].tolist()
            assert out["out_tokens"][b, :n0[b]].tolist() == hist[b, :n0[b]].tolist()
            assert out["out_tokens"][b, n1:].tolist() == hist[b, n1:].tolist()
            overflow |= int(n0[b]) + int(L[b]) > cap
        assert out["status"] == (0x08 if overflow else 0)


def test_scatter_bad_lengths(oracle_mod):
    out = oracle_mod.scatter(np.array([[1, 2, 3]], np.int32), np.array([7], np.int32),
                             np.zeros((1, 8), np.int32), np.array([-2], np.int32))
    assert out["status"] == 0x80
    assert out["out_len"].tolist() == [3] and out["out_tokens"][0, :3].tolist() == [1, 2, 3]


def test_oracle_reproduces_its_golden_fixture():
    """Regression fixture: the oracle still writes what tests/golden/make_golden.py stored."""
    import importlib.util
    spec = importlib.util.spec_from_file_location("make_golden",
                                                  os.path.join(GOLDEN, "make_golden.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    with open(os.path.join(GOLDEN, "tiny_greedy_oracle.json")) as f:
        stored = json.load(f)
    assert json.loads(json.dumps(mod.compute())) == stored
