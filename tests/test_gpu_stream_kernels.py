"""The two logit-streaming kernels of verify (register streaming, and TMA bulk copies into a
shared-memory ring) must give bit-identical results: every output of dspark_verify_scatter,
for every workload, mode and sampler. The register kernel is pinned to the oracle by the other
GPU tests, so equality here carries that parity over to the bulk-copy kernel."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth

from gpu_util import device, i32, ref_verify, assert_greedy_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    d = device()
    yield d
    bd.set_stream_kernel(bd.STREAM_AUTO)


def _run(dev, kernel, mode, tgt, drf, tokens, cu, windows, stochastic, **kw):
    bd.set_stream_kernel(kernel)
    try:
        B, gamma = tokens.shape
        rows, V = tgt.shape
        ws = torch.empty(max(bd.dspark_verify_workspace_bytes(B, gamma, V, stochastic), 16),
                         dtype=torch.uint8, device=dev)
        o = dict(acc=torch.full((B,), -7, dtype=torch.int32, device=dev),
                 com=torch.full((B, gamma), -7, dtype=torch.int32, device=dev),
                 ceil=torch.full((B,), -7, dtype=torch.int32, device=dev),
                 prob=torch.full((max(rows, 1), 2), -7.0, dtype=torch.float32, device=dev),
                 out=torch.full((B, 4 * gamma), -5, dtype=torch.int32, device=dev),
                 out_len=torch.zeros(B, dtype=torch.int32, device=dev),
                 status=torch.zeros(1, dtype=torch.int32, device=dev))
        bd.dspark_verify_scatter(mode, tgt, i32(tokens, dev), o["acc"], o["com"], ws, o["out"],
                                 o["out_len"], stochastic=stochastic, draft=drf,
                                 cu_seqlens=None if cu is None else i32(cu, dev),
                                 windows=None if windows is None else i32(windows, dev),
                                 ceiling_len=o["ceil"], row_prob=o["prob"], status=o["status"],
                                 **kw)
        torch.cuda.synchronize()
        return {k: v.cpu().numpy() for k, v in o.items()}
    finally:
        bd.set_stream_kernel(bd.STREAM_AUTO)


CASES = [("tiny_greedy", False), ("stochastic", True), ("stochastic", False),
         ("large_vocab_mixed", False), ("latency_b1", False), ("latency_b1", True),
         ("high_load", False)]


@pytest.mark.parametrize("name,stochastic", CASES)
@pytest.mark.parametrize("mode", ["compact", "cap_accept", "static"])
def test_bulk_equals_register(dev, name, stochastic, mode):
    wl = synth.WORKLOADS[name]
    if name == "high_load" and mode != "compact":
        wl = wl.with_(B=128)                  # the full block of every request: keep it small
    bt = synth.make_batch(wl, seed=21, stochastic=stochastic)
    B, gamma = bt.tokens.shape
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
    if mode == "compact":
        tgt = synth.gather_packed(bt.target, B, gamma, w).to(dev)
        cu = np.concatenate([[0], np.cumsum(w)])
    else:
        tgt = bt.target.to(dev)
        cu = None
    drf = bt.draft.to(dev) if stochastic else None
    args = (mode, tgt, drf, bt.tokens, cu, None if mode == "static" else w, stochastic)
    kw = dict(temperature=wl.temperature, seed=3, step=1)
    r = _run(dev, bd.STREAM_REGISTER, *args, **kw)
    k = _run(dev, bd.STREAM_BULK, *args, **kw)
    for key in r:
        np.testing.assert_array_equal(k[key], r[key], err_msg=key)
    assert (k["status"][0] & bd.STATUS_STALL) == 0


def test_bulk_greedy_matches_the_oracle(dev):
    wl = synth.WORKLOADS["large_vocab_mixed"].with_(B=48)
    bt = synth.make_batch(wl, seed=8)
    B, gamma = bt.tokens.shape
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
    packed = synth.gather_packed(bt.target, B, gamma, w)
    cu = np.concatenate([[0], np.cumsum(w)])
    g = _run(dev, bd.STREAM_BULK, "compact", packed.to(dev), None, bt.tokens, cu, w, False)
    r = ref_verify("compact", packed, bt.tokens, cu=cu, windows=w)
    assert_greedy_equal(dict(accept_len=g["acc"], committed=g["com"], ceiling_len=g["ceil"],
                             status=int(g["status"][0])), r)


def test_misaligned_rows_fall_back_to_the_register_kernel(dev):
    # rows that start 4 bytes off a 16-byte boundary: the bulk request must still be served
    wl = synth.WORKLOADS["tiny_greedy"]
    bt = synth.make_batch(wl, seed=4)
    B, gamma = bt.tokens.shape
    base = torch.zeros(bt.target.numel() + 1, dtype=torch.float32, device=dev)
    tgt = base[1:].view(B * gamma, wl.V)
    tgt.copy_(bt.target.to(dev))
    r = _run(dev, bd.STREAM_REGISTER, "static", tgt, None, bt.tokens, None, None, False)
    k = _run(dev, bd.STREAM_BULK, "static", tgt, None, bt.tokens, None, None, False)
    for key in r:
        np.testing.assert_array_equal(k[key], r[key], err_msg=key)


def test_stream_events_time_the_streaming_kernel_alone(dev):
    wl = synth.WORKLOADS["large_vocab_mixed"].with_(B=64)
    bt = synth.make_batch(wl, seed=2)
    B, gamma = bt.tokens.shape
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
    tgt = synth.gather_packed(bt.target, B, gamma, w).to(dev)
    cu = np.concatenate([[0], np.cumsum(w)])
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    bd.set_stream_events(ev[1], ev[2])
    try:
        ev[0].record()
        r = _run(dev, bd.STREAM_AUTO, "compact", tgt, None, bt.tokens, cu, w, False)
        ev[3].record()
    finally:
        bd.set_stream_events(None, None)
    torch.cuda.synchronize()
    kernel_ms, call_ms = ev[1].elapsed_time(ev[2]), ev[0].elapsed_time(ev[3])
    assert 0.0 < kernel_ms < call_ms
    assert r["status"][0] == 0
