"""The oracle's pins catch plausible mistakes: each case plants one mistake in a temporary copy
of the oracle's C source (a wrong constant, a dropped term, a flipped comparison, an index off
by one), builds that copy on the CPU, runs the pins named for it against the copy and requires
at least one of them to fail. The oracle itself is never modified; the regular pin tests show
that the unmodified oracle passes the same pins.

Sources of the pinned behaviour: Philox4x64-10 (Salmon et al., SC'11, via numpy.random.Philox);
"DSpark in SGLang" (LMSYS blog summary), A2 method details (survival product, cost model,
ragged pack, verify modes, compact scatter, observability); lshu.cn DSpark article, 1.2 and
2.3/3.3 (greedy first divergence, min(1, p/q) with the residual bonus)."""
import importlib.util
import os

import pytest

import test_oracle_observe as t_obs
import test_oracle_pack_scatter as t_pack
import test_oracle_philox as t_phi
import test_oracle_schedule as t_sch
import test_oracle_verify as t_ver

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
ORACLE = os.path.join(ROOT, "oracle")

# name: (text in dspark_oracle.c, its planted replacement, [(pin, kwargs), ...])
MUTANTS = {
    "philox multiplier": (
        "M0 = 0xD2E7470EE14C6C93ULL", "M0 = 0xD2E7470EE14C6C95ULL",
        [(t_phi.test_philox_matches_numpy_random_counters, {})]),
    "philox key schedule": (
        "W0 = 0x9E3779B97F4A7C15ULL", "W0 = 0x9E3779B97F4A7C17ULL",
        [(t_phi.test_philox_matches_numpy_random_counters, {})]),
    "accept uniform drops a bit": (
        "(float)(w[0] >> 40) * 0x1p-24f", "(float)(w[0] >> 41) * 0x1p-24f",
        [(t_phi.test_uniforms_are_uniform, {}),
         (t_ver.test_first_token_law_is_p, {"seed": 0})]),
    "confidence not clamped above 1": (
        "    if (x > 1.0f) return 1.0f;\n", "",
        [(t_sch.test_survival_keys_clamp_and_nan, {})]),
    "survival not a product": (
        "s = s * clamp_conf(conf[(size_t)b * L + j]);", "s = clamp_conf(conf[(size_t)b * L + j]);",
        [(t_sch.test_survival_keys_match_numpy, {})]),
    "objective drops the batch term": (
        "(double)((uint64_t)B * 4294967296ULL + S)", "(double)(S + 1)",
        [(t_sch.test_schedule_equals_brute_force, {"B": 2, "gamma": 3})]),
    "ties go to the larger K": (
        "if (best_k < 0 || value > best)", "if (best_k < 0 || value >= best)",
        [(t_sch.test_zero_survivals_are_never_taken, {})]),
    "equal survivals: higher request first": (
        "if (a->b != c->b) return a->b < c->b ? -1 : 1;",
        "if (a->b != c->b) return a->b > c->b ? -1 : 1;",
        [(t_sch.test_tie_rule_fills_lower_request_then_lower_position, {})]),
    "theta read at M + 1": (
        "T = T + theta[B + K];", "T = T + theta[B + K + (K < n ? 1 : 0)];",
        [(t_sch.test_schedule_equals_brute_force, {"B": 2, "gamma": 3})]),
    "tier must exceed M": (
        "if (tiers[t] >= M && (tier < 0 || tiers[t] < tier))",
        "if (tiers[t] > M && (tier < 0 || tiers[t] < tier))",
        [(t_pack.test_pack_random, {})]),
    "padding rows keep a request": (
        "        if (row_req) row_req[r] = -1;\n", "        if (row_req) row_req[r] = 0;\n",
        [(t_pack.test_pack_random, {})]),
    "argmax keeps the last maximum": (
        "if (x > best) { best = x; best_v = v; }", "if (x >= best) { best = x; best_v = v; }",
        [(t_ver.test_row_argmax_matches_numpy, {})]),
    "softmax ignores the temperature": (
        "return exp((logit_at(base, dtype, V, row, v) - m) / T) / z;",
        "return exp(logit_at(base, dtype, V, row, v) - m) / z;",
        [(t_ver.test_stochastic_probabilities_match_numpy, {})]),
    "residual not clamped at zero": (
        "r = p - q > 0.0 ? p - q : 0.0;", "r = p - q > -0.02 ? p - q + 0.02 : 0.0;",
        [(t_ver.test_first_token_law_is_p, {"seed": 0})]),
    "accept ratio inverted": (
        "ratio = (float)(p / q);", "ratio = (float)(q / p);",
        [(t_ver.test_first_token_law_is_p, {"seed": 0})]),
    "walk runs past the window": (
        "while (Lc - 1 < w - 1 && acc[Lc - 1]) ++Lc;", "while (Lc - 1 < w && acc[Lc - 1]) ++Lc;",
        [(t_ver.test_greedy_modes_against_numpy, {"dtype": "f32"}),
         (t_ver.test_stochastic_compact_equals_cap_accept, {})]),
    "full-acceptance bonus from the row before": (
        "const int bonus = draw_bonus(target, draft, dtype, V, base + pos,",
        "const int bonus = draw_bonus(target, draft, dtype, V, base + (rejected ? pos : pos - 1),",
        [(t_ver.test_bonus_after_full_acceptance_has_law_p, {})]),
    "history length not capped": (
        "out_len[b] = (n + L < out_cap) ? n + L : out_cap;", "out_len[b] = n + L;",
        [(t_pack.test_scatter, {}), (t_pack.test_scatter_bad_lengths, {})]),
    "calibration outcomes not censored": (
        "for (int j = 0; j < L && j <= c - 1; ++j) {", "for (int j = 0; j < L; ++j) {",
        [(t_obs.test_hand_worked_example, {}), (t_obs.test_totals_follow_the_definition, {})]),
    "rejected draft counted as accepted": (
        "if (j < c - 1) hist[3 * k + 2] += 1;", "if (j <= c - 1) hist[3 * k + 2] += 1;",
        [(t_obs.test_hand_worked_example, {})]),
}


def _mutant(name, old, new, tmp_path):
    with open(os.path.join(ORACLE, "dspark_oracle.c")) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation site of '{name}' not found exactly once"
    d = tmp_path / "mutant"
    d.mkdir()
    (d / "dspark_oracle.c").write_text(src.replace(old, new))
    spec = importlib.util.spec_from_file_location("oracle_mutant", os.path.join(ORACLE, "__init__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod._SRC = str(d / "dspark_oracle.c")
    mod._SO = str(d / "libdspark_oracle.so")
    mod._LIB = None
    mod.build(force=True)
    return mod


@pytest.mark.parametrize("name", list(MUTANTS))
def test_pins_catch_the_planted_mistake(name, tmp_path):
    old, new, pins = MUTANTS[name]
    mod = _mutant(name, old, new, tmp_path)
    caught = []
    for pin, kw in pins:
        try:
            pin(oracle_mod=mod, **kw)
        except Exception as e:      # an assertion, or the mutant breaking an invariant outright
            caught.append(f"{pin.__name__}: {type(e).__name__}")
    assert caught, f"no pin caught '{name}'"
