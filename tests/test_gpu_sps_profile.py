"""The step-cost recorder on the GPU: forced windows pack to the intended M and tier, step
times are recorded for every grid cell, and the additive fit of them predicts the held-out
cells ("DSpark in SGLang", A2 method details, cost-table profiling and modelling)."""
import math

import pytest

pytestmark = pytest.mark.gpu


def test_record_and_fit_small_grid():
    from speculative_decoding_ragged_gb300 import sps_profile
    tiers = [8, 16, 32, 64]
    samples = sps_profile.record([1, 2, 4, 8], gamma=4, V=4096, H=256, tiers=tiers, points=4,
                                 ctx_bytes=1 << 16, warmup=2, reps=3)
    assert len(samples) == sum(len(sps_profile.grid_M(b, 4, tiers, 4)) for b in [1, 2, 4, 8])
    for s in samples:
        assert s["bs"] <= s["M"] <= 4 * s["bs"] and s["tier"] >= s["M"]
        assert math.isfinite(s["us"]) and s["us"] > 0
    res = sps_profile.evaluate(samples, tiers)
    assert res["train"]["n"] + (res["held_out"]["n"] if res["held_out"] else 0) == len(samples)
    assert all(math.isfinite(r["predicted_us"]) for r in res["rows"])
