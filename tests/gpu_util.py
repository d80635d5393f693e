"""Helpers of the GPU parity tests: run each C-ABI call on cuda:0 with sentinel-filled outputs,
run the oracle on the same host inputs, and compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth

MODE = {"static": oracle.STATIC, "compact": oracle.COMPACT, "cap_accept": oracle.CAP_ACCEPT}
NEAR_TIE = 1e-6      # accept decisions / bonus draws closer than this to their threshold
PROB_RTOL = 1e-5     # p(d), q(d) relative tolerance (fp32 device vs fp64 oracle)


def device() -> torch.device:
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_ragged_gb300 import build
    build.build()
    bd.lib()
    oracle.build()
    return torch.device("cuda:0")


def i32(x, dev):
    return torch.as_tensor(np.ascontiguousarray(x, np.int32), device=dev)


def bits(t: torch.Tensor) -> np.ndarray:
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16)
    return t.numpy()


def gpu_schedule(dev, conf, bias, alpha, theta):
    conf = np.ascontiguousarray(conf, np.float32)
    B = conf.shape[0]
    w = torch.full((B,), -7, dtype=torch.int32, device=dev)
    k = torch.full((1,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    cost = bd.CostTable(bias, torch.as_tensor(np.asarray(alpha, np.float64), device=dev),
                        torch.as_tensor(np.asarray(theta, np.float64), device=dev))
    bd.dspark_schedule(torch.as_tensor(conf, device=dev), cost, w, k, st)
    torch.cuda.synchronize()
    return dict(windows=w.cpu().numpy(), k_star=int(k.item()), status=int(st.item()))


def gpu_pack(dev, windows, tokens, tiers, cap):
    B = tokens.shape[0]
    cu = torch.full((B + 1,), -7, dtype=torch.int32, device=dev)
    packed = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)[:cap]
    rr = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)[:cap]
    rp = torch.full((max(cap, 1),), -7, dtype=torch.int32, device=dev)[:cap]
    meta = torch.full((2,), -7, dtype=torch.int32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    bd.dspark_pack(i32(windows, dev), i32(tokens, dev), i32(tiers, dev), cu, packed, meta, rr, rp,
                   st)
    torch.cuda.synchronize()
    m = meta.cpu().numpy()
    return dict(cu=cu.cpu().numpy(), packed_ids=packed.cpu().numpy(), row_req=rr.cpu().numpy(),
                row_pos=rp.cpu().numpy(), M=int(m[0]), tier=int(m[1]), status=int(st.item()))


def gpu_verify(dev, mode, target, tokens, *, stochastic=False, draft=None, cu=None, windows=None,
               temperature=1.0, seed=0, step=0, target_dev=None, draft_dev=None):
    """target / draft: torch logits (CPU or CUDA). Returns host numpy outputs."""
    B, gamma = tokens.shape
    tgt = target_dev if target_dev is not None else target.to(dev)
    drf = draft_dev if draft_dev is not None else (draft.to(dev) if draft is not None else None)
    rows, V = tgt.shape
    acc = torch.full((B,), -7, dtype=torch.int32, device=dev)
    com = torch.full((B, gamma), -7, dtype=torch.int32, device=dev)
    ceil = torch.full((B,), -7, dtype=torch.int32, device=dev)
    prob = torch.full((max(rows, 1), 2), -7.0, dtype=torch.float32, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ws = torch.empty(max(bd.dspark_verify_workspace_bytes(B, gamma, V, stochastic), 16),
                     dtype=torch.uint8, device=dev)
    bd.dspark_verify(mode, tgt, i32(tokens, dev), acc, com, ws, stochastic=stochastic, draft=drf,
                     cu_seqlens=None if cu is None else i32(cu, dev),
                     windows=None if windows is None else i32(windows, dev), ceiling_len=ceil,
                     row_prob=prob, temperature=temperature, seed=seed, step=step, status=st)
    torch.cuda.synchronize()
    return dict(accept_len=acc.cpu().numpy(), committed=com.cpu().numpy(),
                ceiling_len=ceil.cpu().numpy(), row_prob=prob.cpu().numpy()[:rows],
                status=int(st.item()))


def ref_verify(mode, target, tokens, *, stochastic=False, draft=None, cu=None, windows=None,
               temperature=1.0, seed=0, step=0):
    return oracle.verify(MODE[mode], stochastic, bits(target), tokens, cu=cu, windows=windows,
                         draft=None if draft is None else bits(draft), temperature=temperature,
                         seed=seed, step=step)


def assert_greedy_equal(g, r, used_rows=None):
    np.testing.assert_array_equal(g["accept_len"], r["accept_len"])
    np.testing.assert_array_equal(g["committed"], r["committed"])
    np.testing.assert_array_equal(g["ceiling_len"], r["ceiling_len"])
    assert g["status"] == r["status"]


def compare_stochastic(g, r, rows_used: int):
    """Accept decisions and bonus draws must match except at counted near-ties; p(d), q(d)
    within PROB_RTOL. Returns (number of near-tie requests, max relative p/q error)."""
    gp, rp = g["row_prob"][:rows_used], r["row_prob"][:rows_used]
    tested = rp[:, 0] >= 0
    np.testing.assert_array_equal(gp[~tested], rp[~tested])
    rel = np.abs(gp[tested] - rp[tested]) / np.maximum(np.abs(rp[tested]), 1e-30)
    worst = float(rel.max()) if rel.size else 0.0
    assert worst <= PROB_RTOL, f"p/q relative error {worst}"
    near = 0
    B = g["accept_len"].shape[0]
    for b in range(B):
        gL, rL = int(g["accept_len"][b]), int(r["accept_len"][b])
        if gL == rL and (g["committed"][b] == r["committed"][b]).all():
            continue
        if gL != rL:
            i = min(gL, rL) - 1
            gap = abs(float(r["ratio"][b, i]) - float(r["u"][b, i]))
            assert gap < NEAR_TIE, f"request {b}: accept lengths {gL} vs {rL}, gap {gap}"
            near += 1
            continue
        np.testing.assert_array_equal(g["committed"][b, :gL - 1], r["committed"][b, :rL - 1])
        assert r["margin"][b] < NEAR_TIE, f"request {b}: bonus differs, margin {r['margin'][b]}"
        near += 1
    assert g["status"] == r["status"]
    return near, worst
