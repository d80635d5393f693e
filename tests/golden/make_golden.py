"""Writes tests/golden/tiny_greedy_oracle.json from the CPU oracle alone.

The fixture records the oracle's schedule, pack, verify (compact, cap-accept, static) and
scatter outputs on the tiny greedy workload (B=4, gamma=4, V=1024 fp32 logits, seed 0), so a
later change to the oracle's arithmetic shows up as a diff against it. Run from the repo root:
    python tests/golden/make_golden.py
"""
import json
import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
from speculative_decoding_ragged_gb300 import synth  # noqa: E402

OUT = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_greedy_oracle.json")


def compute(seed=0):
    wl = synth.WORKLOADS["tiny_greedy"]
    bt = synth.make_batch(wl, seed=seed)
    sch = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)
    w = sch["windows"]
    cap = int(max(wl.tiers))
    pk = oracle.pack(w, bt.tokens, bt.tiers, cap)
    full = bt.logits_bits(bt.target)
    packed = bt.logits_bits(synth.gather_packed(bt.target, bt.B, bt.gamma, w))
    res = {}
    res["compact"] = oracle.verify(oracle.COMPACT, False, packed, bt.tokens, cu=pk["cu"],
                                   windows=w)
    res["cap_accept"] = oracle.verify(oracle.CAP_ACCEPT, False, full, bt.tokens, windows=w)
    res["static"] = oracle.verify(oracle.STATIC, False, full, bt.tokens)
    hist = np.full((bt.B, 16), -1, np.int32)
    sc = oracle.scatter(res["compact"]["committed"], res["compact"]["accept_len"], hist,
                        np.zeros(bt.B, np.int32))
    return {
        "source": "CPU oracle (oracle/dspark_oracle.c) on the tiny greedy workload, seed 0; "
                  "written by tests/golden/make_golden.py",
        "windows": w.tolist(), "k_star": sch["k_star"],
        "cu_seqlens": pk["cu"].tolist(), "M": pk["M"], "tier": pk["tier"],
        "packed_ids": pk["packed_ids"][:pk["tier"]].tolist(),
        "verify": {m: {"accept_len": r["accept_len"].tolist(),
                       "committed": r["committed"].tolist(),
                       "ceiling_len": r["ceiling_len"].tolist()} for m, r in res.items()},
        "out_len": sc["out_len"].tolist(), "out_tokens": sc["out_tokens"].tolist(),
    }


if __name__ == "__main__":
    with open(OUT, "w") as f:
        json.dump(compute(), f, indent=1)
    print("wrote", OUT)
