"""Seeded random configurations through the fused step against the oracle: batch sizes from
1 to 300 (the one-warp and the block scheduler), block widths up to 32, vocabularies with and
without V % 8 == 0 (vector and scalar loads), bf16 and fp32, compact / cap-accept / static,
greedy and stochastic at several temperatures, small and large tier sets, histories that fill
up; the larger vocabularies reach the TMA bulk-copy streaming kernel. Every output is
compared: windows, K*, cu_seqlens, packed rows, tier, accept lengths, committed tokens,
ceilings, p(d) and q(d), histories and status bits (bit-exact, stochastic decisions and draws
exact except counted near-ties). Sources as in the other parity tests:
"DSpark in SGLang" (LMSYS blog summary), A2 method details; lshu.cn DSpark article."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth
from speculative_decoding_ragged_gb300.step import DSparkStep

from gpu_util import MODE, bits, compare_stochastic, device

pytestmark = pytest.mark.gpu

N_CASES = 200


@pytest.fixture(scope="module")
def dev():
    return device()


def draw_case(rng):
    B = int(rng.choice([1, 2, 3, 5, 8, 16, 31, 32, 33, 64, 65, 127, 300]))
    gamma = int(rng.integers(1, 33 if B <= 64 else 9))
    V = int(rng.choice([64, 257, 1000, 1024, 3001, 4096, 9000, 32000, 65536],
                       p=[0.12, 0.12, 0.12, 0.12, 0.12, 0.12, 0.12, 0.08, 0.08]))
    dtype = str(rng.choice(["bf16", "f32"]))
    stochastic = bool(rng.uniform() < 0.5)
    mode = str(rng.choice(["compact", "cap_accept", "static"]))
    T = float(rng.choice([0.3, 0.7, 1.0, 1.7]))
    n_tiers = int(rng.integers(1, 9))
    tiers = sorted(set(int(t) for t in rng.integers(1, B * gamma + 16, size=n_tiers)))
    out_cap = int(rng.integers(gamma, 4 * gamma + 1))
    return B, gamma, V, dtype, stochastic, mode, T, tiers, out_cap


@pytest.mark.parametrize("case", range(N_CASES))
def test_fused_step_matches_the_oracle(dev, case):
    rng = np.random.default_rng(9000 + case)
    _check_fused_step(dev, case, rng, *draw_case(rng))


@pytest.mark.parametrize("B,gamma,stochastic", [(1024, 5, False), (2049, 3, True),
                                                (4096, 4, False), (8192, 2, True),
                                                (4000, 5, False),
                                                # greedy finaliser CTAs of two or four
                                                # requests with idle slots in the last one
                                                (201, 4, False), (299, 3, False),
                                                (513, 2, False)])
def test_fused_step_large_batches(dev, B, gamma, stochastic):
    """Batches up to the limit (more requests than threads in the scheduler and the pack, the
    bitonic scheduler past 4096 candidates), and greedy batches whose size the finaliser's
    requests per CTA do not divide, with a small vocabulary so that the oracle stays quick."""
    rng = np.random.default_rng(B + gamma)
    tiers = sorted(set(int(t) for t in rng.integers(B, B * gamma + 1, size=6)))
    _check_fused_step(dev, B, rng, B, gamma, 512, "bf16", stochastic, "compact", 1.0, tiers,
                      2 * gamma)


def _check_fused_step(dev, case, rng, B, gamma, V, dtype, stochastic, mode, T, tiers, out_cap):
    wl = synth.WORKLOADS["stochastic"].with_(B=B, gamma=gamma, V=V, dtype=dtype, temperature=T,
                                             tiers=tuple(tiers),
                                             theta_slope=float(rng.uniform(0.001, 0.05)))
    bt = synth.make_batch(wl, seed=case, stochastic=stochastic)
    st = DSparkStep(B, gamma, V, tiers, bt.bias, bt.alpha, bt.theta, mode=mode,
                    stochastic=stochastic, out_cap=out_cap, device=dev)
    st.out_len.copy_(torch.as_tensor(rng.integers(0, out_cap + 1, size=B).astype(np.int32)))
    out_len0 = st.out_len.cpu().numpy().copy()
    conf = torch.as_tensor(bt.conf, device=dev)
    tokens = torch.as_tensor(bt.tokens, device=dev)

    # schedule and pack against the oracle
    st.schedule_pack(conf, tokens)
    torch.cuda.synchronize()
    rs = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
    np.testing.assert_array_equal(st.windows.cpu().numpy(), rs["windows"])
    assert int(st.k_star.item()) == rs["k_star"]
    w = rs["windows"]
    rp = oracle.pack(w, bt.tokens, np.asarray(tiers, np.int32), st.packed_cap)
    np.testing.assert_array_equal(st.cu.cpu().numpy(), rp["cu"])
    for key, t in (("packed_ids", st.packed_ids), ("row_req", st.row_req), ("row_pos", st.row_pos)):
        np.testing.assert_array_equal(t.cpu().numpy()[: rp["tier"]], rp[key][: rp["tier"]],
                                      err_msg=key)
    assert st.meta.cpu().tolist() == [rp["M"], rp["tier"]]
    assert int(st.status.item()) == rs["status"] | rp["status"]

    # verify and scatter against the oracle
    if mode == "compact":
        target = synth.gather_packed(bt.target, B, gamma, w, rows_cap=max(rp["tier"], rp["M"]))
    else:
        target = bt.target
    rows = target.shape[0]
    prob = torch.full((max(rows, 1), 2), -7.0, dtype=torch.float32, device=dev)
    st.status.zero_()
    draft = bt.draft if stochastic else None
    st.verify_scatter(target.to(dev), tokens, None if draft is None else draft.to(dev),
                      temperature=T, seed=case, step=3, row_prob=prob)
    torch.cuda.synchronize()
    kw = dict(cu=rp["cu"] if mode == "compact" else None, windows=None if mode == "static" else w)
    r = oracle.verify(MODE[mode], stochastic, bits(target), bt.tokens, draft=None if draft is None
                      else bits(draft), temperature=T, seed=case, step=3, **kw)
    g = dict(accept_len=st.accept_len.cpu().numpy(), committed=st.committed.cpu().numpy(),
             ceiling_len=st.ceiling.cpu().numpy(), row_prob=prob.cpu().numpy()[:rows],
             status=int(st.status.item()) & ~(bd.STATUS_OUT_OVERFLOW | bd.STATUS_BAD_LENGTH))
    if stochastic:
        near, _ = compare_stochastic(g, r, rp["M"] if mode == "compact" else B * gamma)
        assert near <= max(1, B // 8)
    else:
        np.testing.assert_array_equal(g["accept_len"], r["accept_len"])
        np.testing.assert_array_equal(g["committed"], r["committed"])
        np.testing.assert_array_equal(g["ceiling_len"], r["ceiling_len"])
        assert g["status"] == r["status"]
    # the fused scatter against the oracle's scatter of the device's own commits
    sc = oracle.scatter(g["committed"], g["accept_len"], np.full((B, out_cap), -1, np.int32),
                        out_len0)
    np.testing.assert_array_equal(st.out_len.cpu().numpy(), sc["out_len"])
    ot = st.out_tokens.cpu().numpy()
    for b in range(B):
        n0, n1 = int(out_len0[b]), int(sc["out_len"][b])
        np.testing.assert_array_equal(ot[b, n0:n1], sc["out_tokens"][b, n0:n1])
