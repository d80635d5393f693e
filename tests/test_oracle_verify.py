"""Pins of the oracle's verify.

Greedy (the draft survives iff it equals the target's argmax; the accept length ends at the
first divergence — lshu.cn DSpark article, 1.2): row argmax against numpy.argmax on the widened
rows, accept lengths against a numpy first-mismatch search.
Stochastic (accept with probability min(1, p/q) — lshu.cn article, 2.3 and 3.3): softmax
statistics and p(d), q(d) against numpy float64; the law of the emitted tokens against p by a
chi-square test (speculative sampling reproduces the target distribution); special cases that
reduce to closed forms (q == p accepts everything; a vanishing temperature reduces to greedy;
q(d) = 0 accepts).
Modes ("DSpark in SGLang", A2, verify-mode design): compact == cap-accept committed tokens,
ceiling >= accept length, accept length <= window, static == compact at full windows.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_ragged_gb300 import synth


def bf16_bits(x):
    return torch.from_numpy(np.ascontiguousarray(x, np.float32)).to(torch.bfloat16) \
        .view(torch.int16).numpy().view(np.uint16)


def widen(bits):
    return (bits.astype(np.uint32) << 16).view(np.float32)


def np_softmax64(row, T):
    x = row.astype(np.float64) / T
    x -= x.max()
    e = np.exp(x)
    return e / e.sum()


def test_row_argmax_matches_numpy(oracle_mod):
    rng = np.random.default_rng(2)
    for V in [1, 2, 7, 1000, 4099]:
        x = rng.standard_normal((6, V)).astype(np.float32) * 3
        x[0, :] = 1.0                                      # all equal: index 0
        if V > 3:
            x[1, [1, 3]] = 50.0                            # planted tie: first wins
            x[2, :] = -np.inf
            x[2, V - 1] = -1e30
        bits = bf16_bits(x)
        for r in range(6):
            assert oracle_mod.row_argmax(x, r) == int(np.argmax(x[r]))
            assert oracle_mod.row_argmax(bits, r) == int(np.argmax(widen(bits[r])))


def test_softmax_stats_match_numpy(oracle_mod):
    rng = np.random.default_rng(4)
    for V, T in [(1, 1.0), (16, 0.7), (3000, 1.0), (3000, 2.5)]:
        x = (rng.standard_normal((3, V)) * 4).astype(np.float32)
        for r in range(3):
            m, z = oracle_mod.row_softmax_stats(x, r, T)
            assert m == float(x[r].max())
            zz = np.sum(np.exp((x[r].astype(np.float64) - x[r].max()) / T))
            assert abs(z - zz) <= 1e-12 * zz


def greedy_reference(target_rows_of, tokens, w, gamma, V):
    """numpy accept length and committed row for one request."""
    g = np.array([int(np.argmax(target_rows_of(i))) for i in range(w)])
    d = tokens[1:w]
    mism = np.nonzero(d != g[:w - 1])[0]
    L = (int(mism[0]) + 1) if mism.size else w
    return L, g[:L]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_greedy_modes_against_numpy(oracle_mod, dtype):
    wl = synth.custom(B=6, gamma=5, V=301, dtype=dtype, accept=[0.95, 0.8, 0.6, 0.4, 0.2, 0.05],
                      sigma=3.0)
    for seed in range(8):
        bt = synth.make_batch(wl, seed=seed)
        full = bt.logits_bits(bt.target)
        widened = widen(full) if dtype == "bf16" else full
        sch = oracle_mod.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
        w = sch["windows"]
        pk = oracle_mod.pack(w, bt.tokens, bt.tiers, 64)
        packed = bt.logits_bits(synth.gather_packed(bt.target, bt.B, bt.gamma, w))
        comp = oracle_mod.verify(oracle_mod.COMPACT, False, packed, bt.tokens, cu=pk["cu"],
                                 windows=w)
        cap = oracle_mod.verify(oracle_mod.CAP_ACCEPT, False, full, bt.tokens, windows=w)
        stat = oracle_mod.verify(oracle_mod.STATIC, False, full, bt.tokens)
        for b in range(bt.B):
            rows = lambda i: widened[b * bt.gamma + i]
            L, g = greedy_reference(rows, bt.tokens[b], int(w[b]), bt.gamma, bt.V)
            assert comp["accept_len"][b] == L
            assert comp["committed"][b, :L].tolist() == g.tolist()
            assert (comp["committed"][b, L:] == -1).all()
            Lf, gf = greedy_reference(rows, bt.tokens[b], bt.gamma, bt.gamma, bt.V)
            assert cap["ceiling_len"][b] == Lf and stat["accept_len"][b] == Lf
            assert stat["committed"][b, :Lf].tolist() == gf.tolist()
        np.testing.assert_array_equal(comp["committed"], cap["committed"])
        np.testing.assert_array_equal(comp["accept_len"], cap["accept_len"])
        assert (cap["ceiling_len"] >= cap["accept_len"]).all()
        assert (comp["accept_len"] <= w).all() and (comp["accept_len"] >= 1).all()
        assert (comp["ceiling_len"] == -1).all()
        np.testing.assert_array_equal(stat["ceiling_len"], stat["accept_len"])


def test_static_equals_compact_at_full_windows(oracle_mod):
    wl = synth.custom(B=5, gamma=4, V=97)
    bt = synth.make_batch(wl, seed=1)
    full = bt.logits_bits(bt.target)
    w = np.full(bt.B, bt.gamma, np.int32)
    cu = np.arange(bt.B + 1, dtype=np.int32) * bt.gamma
    comp = oracle_mod.verify(oracle_mod.COMPACT, False, full, bt.tokens, cu=cu, windows=w)
    stat = oracle_mod.verify(oracle_mod.STATIC, False, full, bt.tokens)
    np.testing.assert_array_equal(comp["committed"], stat["committed"])
    np.testing.assert_array_equal(comp["accept_len"], stat["accept_len"])


def test_verify_flags_and_bad_rows(oracle_mod):
    x = np.zeros((6, 8), np.float32)
    x[:, 3] = 1.0
    tokens = np.array([[0, 3, 9, 3], [0, -1, 3, 3]], np.int32)
    out = oracle_mod.verify(oracle_mod.CAP_ACCEPT, False, x, tokens, windows=np.array([4, 4]))
    # request 0: rows 0..3 fit in 6 rows -> d1 = 3 accepted, d2 = 9 bad token (rejected)
    # request 1: rows 4..7 exceed the 6-row buffer -> nothing committed
    assert out["status"] == 0x40 | 0x20
    assert out["accept_len"].tolist() == [2, 0]
    assert out["committed"][0].tolist() == [3, 3, -1, -1]
    assert out["committed"][1].tolist() == [-1, -1, -1, -1]


def test_compact_rows_end_at_the_packed_total(oracle_mod):
    # compact verifies the packed rows [0, cu[B]) only: a request whose window reaches past
    # cu[B] commits nothing, although the buffer holds the row (the rows of the others are
    # verified as usual); the same request with cu[B] covering its rows is verified
    x = np.zeros((8, 8), np.float32)
    x[:, 3] = 1.0
    tokens = np.array([[0, 3, 3], [0, 3, 3], [0, 3, 3]], np.int32)
    w = np.array([2, 2, 2], np.int32)
    short = oracle_mod.verify(oracle_mod.COMPACT, False, x, tokens, cu=np.array([0, 2, 4, 5]),
                              windows=w)
    assert short["status"] == 0x20
    assert short["accept_len"].tolist() == [2, 2, 0]
    assert short["committed"][2].tolist() == [-1, -1, -1]
    full = oracle_mod.verify(oracle_mod.COMPACT, False, x, tokens, cu=np.array([0, 2, 4, 6]),
                             windows=w)
    assert full["status"] == 0
    assert full["accept_len"].tolist() == [2, 2, 2]
    assert full["committed"][2].tolist() == [3, 3, -1]


def test_compact_tested_rows_belong_to_one_request(oracle_mod):
    # each packed row is one request's: request 0's tested row 0 is also request 1's first row
    # (cu[1] = 0) -> nothing committed; sharing only a last row (cu = 0, 1, 3) is fine
    x = np.zeros((8, 8), np.float32)
    x[:, 3] = 1.0
    tokens = np.array([[0, 3, 3], [0, 3, 3], [0, 3, 3]], np.int32)
    w = np.array([2, 2, 2], np.int32)
    out = oracle_mod.verify(oracle_mod.COMPACT, False, x, tokens, cu=np.array([0, 0, 2, 4]),
                            windows=w)
    assert out["status"] == 0x20
    assert out["accept_len"].tolist() == [0, 2, 2]
    ok = oracle_mod.verify(oracle_mod.COMPACT, False, x, tokens, cu=np.array([0, 1, 3, 5]),
                           windows=w)
    assert ok["status"] == 0
    assert ok["accept_len"].tolist() == [2, 2, 2]


def make_stochastic(oracle_mod, B, gamma, V, rng, T=1.0, same=False):
    target = (rng.standard_normal((B * gamma, V)) * 2).astype(np.float32)
    draft = target[np.arange(B * (gamma - 1)) // (gamma - 1) * gamma
                   + np.arange(B * (gamma - 1)) % (gamma - 1)].copy()
    if not same:
        draft += (rng.standard_normal(draft.shape) * 0.7).astype(np.float32)
    tokens = np.zeros((B, gamma), np.int32)
    for b in range(B):
        for i in range(gamma - 1):
            q = np_softmax64(draft[b * (gamma - 1) + i], T)
            tokens[b, i + 1] = rng.choice(V, p=q)
    return target, draft, tokens


def test_stochastic_probabilities_match_numpy(oracle_mod):
    rng = np.random.default_rng(12)
    B, gamma, V, T = 4, 5, 333, 0.7
    target, draft, tokens = make_stochastic(oracle_mod, B, gamma, V, rng, T)
    out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft,
                            temperature=T, seed=3, step=1)
    for b in range(B):
        for i in range(gamma - 1):
            d = tokens[b, i + 1]
            p = np_softmax64(target[b * gamma + i], T)[d]
            q = np_softmax64(draft[b * (gamma - 1) + i], T)[d]
            pr = out["row_prob"][b * gamma + i]
            assert abs(pr[0] - p) <= 1e-6 * p and abs(pr[1] - q) <= 1e-6 * q
            assert out["ratio"][b, i] == np.float32(p / q) or \
                abs(out["ratio"][b, i] - p / q) <= 1e-12 * (p / q) + np.spacing(np.float32(p / q))
        assert (out["row_prob"][b * gamma + gamma - 1] == -1).all()


def test_identical_draft_accepts_everything(oracle_mod):
    rng = np.random.default_rng(13)
    B, gamma, V = 50, 6, 40
    target, draft, tokens = make_stochastic(oracle_mod, B, gamma, V, rng, same=True)
    out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft, seed=1)
    np.testing.assert_array_equal(out["accept_len"], gamma)
    np.testing.assert_array_equal(out["committed"][:, :gamma - 1], tokens[:, 1:])


def test_zero_draft_probability_accepts(oracle_mod):
    V = 6
    target = np.zeros((2, V), np.float32)
    draft = np.zeros((1, V), np.float32)
    draft[0, 2] = -np.inf                       # q(2) = 0
    tokens = np.array([[0, 2]], np.int32)
    out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft, seed=5)
    assert out["accept_len"][0] == 2 and out["committed"][0, 0] == 2
    assert out["ratio"][0, 0] == np.inf


def test_vanishing_temperature_reduces_to_greedy(oracle_mod):
    """T -> 0: p and q become one-hot at their argmaxes, the draft d = argmax q is accepted iff
    it is the target argmax, and the residual bonus is the target argmax: greedy verify."""
    rng = np.random.default_rng(14)
    B, gamma, V = 40, 5, 64
    target = (rng.permuted(np.tile(np.arange(V), (B * gamma, 1)), axis=1) * 1.0).astype(np.float32)
    draft = (rng.permuted(np.tile(np.arange(V), (B * (gamma - 1), 1)), axis=1) * 1.0) \
        .astype(np.float32)
    tokens = np.zeros((B, gamma), np.int32)
    tokens[:, 1:] = np.argmax(draft, axis=1).reshape(B, gamma - 1)
    for b in range(B):                          # make about half the drafts agree
        for i in range(gamma - 1):
            if rng.uniform() < 0.6:
                r = b * (gamma - 1) + i
                t = target[b * gamma + i].copy()
                draft[r] = t
                tokens[b, i + 1] = int(np.argmax(t))
    sto = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft,
                            temperature=1e-3, seed=9)
    gre = oracle_mod.verify(oracle_mod.STATIC, False, target, tokens)
    np.testing.assert_array_equal(sto["accept_len"], gre["accept_len"])
    np.testing.assert_array_equal(sto["committed"], gre["committed"])


def chi2_pvalue(counts, probs):
    stats = pytest.importorskip("scipy.stats")
    n = counts.sum()
    exp = n * probs
    return float(stats.chi2.sf(((counts - exp) ** 2 / exp).sum(), probs.size - 1))


def laws_setup(V=16):
    p_logits = np.log(np.linspace(1.0, 3.0, V) * np.r_[np.ones(V // 2), 2 * np.ones(V - V // 2)])
    q_logits = np.log(np.linspace(3.0, 1.0, V) ** 2)
    return p_logits.astype(np.float32), q_logits.astype(np.float32)


@pytest.mark.parametrize("seed", [0, 1])
def test_first_token_law_is_p(oracle_mod, seed):
    """Rejection plus residual sampling emits its first token with law p (V = 16)."""
    V, N = 16, 150_000
    pl, ql = laws_setup(V)
    p, q = np_softmax64(pl, 1.0), np_softmax64(ql, 1.0)
    rng = np.random.default_rng(seed)
    gamma = 2
    target = np.tile(pl, (N * gamma, 1))
    draft = np.tile(ql, (N, 1))
    tokens = np.zeros((N, gamma), np.int32)
    tokens[:, 1] = rng.choice(V, size=N, p=q)
    out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft,
                            seed=1000 + seed, step=seed)
    first = out["committed"][:, 0]
    assert chi2_pvalue(np.bincount(first, minlength=V), p) > 1e-3
    # the accept rate of the draft is sum_v min(p_v, q_v)
    acc = (out["accept_len"] == 2).mean()
    assert abs(acc - np.minimum(p, q).sum()) < 4 * np.sqrt(acc * (1 - acc) / N)


def test_second_token_law_given_first_accepted(oracle_mod):
    V, N = 16, 150_000
    pl, ql = laws_setup(V)
    p2l = pl[::-1].copy()
    p2 = np_softmax64(p2l, 1.0)
    q2l = np.log(np.linspace(1.0, 2.0, V)).astype(np.float32)
    q, q2 = np_softmax64(ql, 1.0), np_softmax64(q2l, 1.0)
    rng = np.random.default_rng(21)
    gamma = 3
    target = np.tile(np.stack([pl, p2l, pl]), (N, 1))
    draft = np.tile(np.stack([ql, q2l]), (N, 1))
    tokens = np.zeros((N, gamma), np.int32)
    tokens[:, 1] = rng.choice(V, size=N, p=q)
    tokens[:, 2] = rng.choice(V, size=N, p=q2)
    out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft, seed=77)
    sel = out["accept_len"] >= 2
    second = out["committed"][sel, 1]
    assert chi2_pvalue(np.bincount(second, minlength=V), p2) > 1e-3


def test_bonus_after_full_acceptance_has_law_p(oracle_mod):
    V, N = 16, 120_000
    pl, _ = laws_setup(V)
    pb = np.log(np.arange(1, V + 1, dtype=np.float64)).astype(np.float32)
    rng = np.random.default_rng(31)
    gamma = 2
    target = np.tile(np.stack([pl, pb]), (N, 1))
    draft = np.tile(pl, (N, 1))                 # q == p: the draft is always accepted
    tokens = np.zeros((N, gamma), np.int32)
    tokens[:, 1] = rng.choice(V, size=N, p=np_softmax64(pl, 1.0))
    out = oracle_mod.verify(oracle_mod.STATIC, True, target, tokens, draft=draft, seed=4)
    assert (out["accept_len"] == 2).all()
    assert chi2_pvalue(np.bincount(out["committed"][:, 1], minlength=V),
                       np_softmax64(pb, 1.0)) > 1e-3


def test_stochastic_compact_equals_cap_accept(oracle_mod):
    wl = synth.WORKLOADS["stochastic"].with_(B=6, V=500)
    bt = synth.make_batch(wl, seed=2)
    sch = oracle_mod.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
    w = sch["windows"]
    pk = oracle_mod.pack(w, bt.tokens, bt.tiers, 256)
    packed = bt.logits_bits(synth.gather_packed(bt.target, bt.B, bt.gamma, w))
    full = bt.logits_bits(bt.target)
    draft = bt.logits_bits(bt.draft)
    for step in range(4):
        comp = oracle_mod.verify(oracle_mod.COMPACT, True, packed, bt.tokens, cu=pk["cu"],
                                 windows=w, draft=draft, seed=11, step=step)
        cap = oracle_mod.verify(oracle_mod.CAP_ACCEPT, True, full, bt.tokens, windows=w,
                                draft=draft, seed=11, step=step)
        np.testing.assert_array_equal(comp["committed"], cap["committed"])
        np.testing.assert_array_equal(comp["accept_len"], cap["accept_len"])
        assert (cap["ceiling_len"] >= cap["accept_len"]).all()
        assert (comp["accept_len"] <= w).all()
