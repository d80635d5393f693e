"""Edge cases of verify against the oracle, with both streaming kernels: one workspace serving
calls of every size and mode, the workspace head in each of its states (garbage, left by a
call, zeroed, its first bytes overwritten), requests whose rows the buffer does not hold (a short buffer, or
none at all: bad rows, nothing committed, (-1, -1) on the rows the buffer does hold), rows before
cu_seqlens[0], requests whose windows reach into the next request's rows, fewer rows than
requests, random non-decreasing cu_seqlens, and batches of more than 4096 requests."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth

from gpu_util import MODE, bits, compare_stochastic, device, i32

pytestmark = pytest.mark.gpu

KERNELS = {"register": bd.STREAM_REGISTER, "bulk": bd.STREAM_BULK}


@pytest.fixture(scope="module")
def dev():
    d = device()
    yield d
    bd.set_stream_kernel(bd.STREAM_AUTO)


def run(dev, ws, mode, tgt, tokens, cu, windows, stochastic, draft=None, kernel="register",
        **kw):
    bd.set_stream_kernel(KERNELS[kernel])
    try:
        B, gamma = tokens.shape
        rows = tgt.shape[0]
        o = dict(accept_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
                 committed=torch.full((B, gamma), -7, dtype=torch.int32, device=dev),
                 ceiling_len=torch.full((B,), -7, dtype=torch.int32, device=dev),
                 row_prob=torch.full((max(rows, 1), 2), -7.0, dtype=torch.float32, device=dev),
                 status=torch.zeros(1, dtype=torch.int32, device=dev))
        # an empty buffer still needs a valid pointer: a one-row allocation passed with
        # target_rows = 0 through the C ABI directly
        tgt_d = tgt.to(dev) if rows else torch.zeros((1, tgt.shape[1]), dtype=tgt.dtype,
                                                      device=dev)
        args = list(bd._verify_args(
            mode, tgt_d, i32(tokens, dev), o["accept_len"], o["committed"], ws, stochastic,
            None if draft is None else draft.to(dev), None if cu is None else i32(cu, dev),
            None if windows is None else i32(windows, dev), o["ceiling_len"], o["row_prob"],
            kw.get("temperature", 1.0), kw.get("seed", 0), kw.get("step", 0)))
        args[3] = rows
        args += [bd._ptr(o["status"], "status"), bd._stream(None)]
        bd._check("dspark_verify", bd.lib().dspark_verify(*args))
        torch.cuda.synchronize()
        out = {k: v.cpu().numpy() for k, v in o.items()}
        out["status"] = int(out["status"][0])
        out["row_prob"] = out["row_prob"][:rows]
        return out
    finally:
        bd.set_stream_kernel(bd.STREAM_AUTO)


def ref(mode, tgt, tokens, cu, windows, stochastic, draft=None, **kw):
    return oracle.verify(MODE[mode], stochastic, bits(tgt), tokens, cu=cu, windows=windows,
                         draft=None if draft is None else bits(draft), **kw)


def check(g, r, stochastic, rows_used):
    if stochastic:
        near, _ = compare_stochastic(g, r, rows_used)
        assert near == 0
    else:
        np.testing.assert_array_equal(g["accept_len"], r["accept_len"])
        np.testing.assert_array_equal(g["committed"], r["committed"])
        assert g["status"] == r["status"]
    np.testing.assert_array_equal(g["ceiling_len"], r["ceiling_len"])


@pytest.mark.parametrize("kernel", ["register", "bulk"])
@pytest.mark.parametrize("stochastic", [False, True])
def test_one_workspace_serves_calls_of_every_size_and_mode(dev, kernel, stochastic):
    # the largest size's workspace, filled with garbage once, then calls of shrinking and
    # growing sizes in every mode: each call rewrites what it reads (the first call finds no
    # valid head and splits the bulk kernel's units evenly; the later ones hand out tickets)
    sizes = [(48, 8, 4096), (5, 6, 2056), (64, 4, 8192), (17, 8, 1024), (48, 8, 4096)]
    need = max(bd.dspark_verify_workspace_bytes(B, g, V, stochastic) for B, g, V in sizes)
    ws = torch.full((need,), 0xA5, dtype=torch.uint8, device=dev)
    wl0 = synth.WORKLOADS["stochastic"] if stochastic else synth.WORKLOADS["large_vocab_mixed"]
    for k, (B, g, V) in enumerate(sizes):
        wl = wl0.with_(B=B, gamma=g, V=V, tiers=(B * g,))
        bt = synth.make_batch(wl, seed=300 + k, stochastic=stochastic)
        w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
        cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
        for mode in ("compact", "cap_accept", "static"):
            tgt = synth.gather_packed(bt.target, B, g, w) if mode == "compact" else bt.target
            win = None if mode == "static" else w
            kw = dict(temperature=wl.temperature, seed=k, step=1) if stochastic else {}
            gres = run(dev, ws, mode, tgt, bt.tokens, cu if mode == "compact" else None, win,
                       stochastic, bt.draft if stochastic else None, kernel, **kw)
            rres = ref(mode, tgt, bt.tokens, cu if mode == "compact" else None, win, stochastic,
                       bt.draft if stochastic else None, **kw)
            check(gres, rres, stochastic, tgt.shape[0])


def head_words(ws):
    """(unit counter, tags) of the workspace head: its bytes 4..8, and bytes 0..4 and 8..16."""
    h = ws[:16].cpu().numpy()
    return int(h[4:8].view(np.uint32)[0]), (int(h[:4].view(np.uint32)[0]),
                                             int(h[8:16].view(np.uint64)[0]))


@pytest.mark.parametrize("stochastic", [False, True])
def test_workspace_head_in_every_state(dev, stochastic):
    # the bulk kernel hands out half of its units by ticket from the workspace head when the
    # previous call left it valid, else splits them evenly: the results must not depend on it
    wl0 = synth.WORKLOADS["stochastic"] if stochastic else synth.WORKLOADS["large_vocab_mixed"]
    sizes = [(40, 8, 16384), (7, 5, 30000)]
    need = max(bd.dspark_verify_workspace_bytes(B, g, V, stochastic) for B, g, V in sizes)
    gen = torch.Generator(device="cpu").manual_seed(5)
    ws = torch.randint(0, 256, (need,), dtype=torch.uint8, generator=gen).to(dev)
    tags = set()
    states = ["garbage", "left", "left", "zeroed", "left", "overwritten", "left"]
    for k, state in enumerate(states):
        if state == "zeroed":
            ws[:256].zero_()
        if state == "overwritten":
            # another tensor's write over the first bytes (a caching allocator reuses freed
            # blocks): the low tag and the counter garbage, the 64-bit tag intact
            ws[:8].copy_(torch.tensor([7, 0, 0, 0, 9, 9, 9, 9], dtype=torch.uint8))
        B, g, V = sizes[k % 2]
        wl = wl0.with_(B=B, gamma=g, V=V, tiers=(B * g,))
        bt = synth.make_batch(wl, seed=500 + k, stochastic=stochastic)
        w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
        cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
        tgt = synth.gather_packed(bt.target, B, g, w)
        kw = dict(temperature=wl.temperature, seed=k, step=2) if stochastic else {}
        drf = bt.draft if stochastic else None
        gres = run(dev, ws, "compact", tgt, bt.tokens, cu, w, stochastic, drf, "bulk", **kw)
        rres = ref("compact", tgt, bt.tokens, cu, w, stochastic, drf, **kw)
        check(gres, rres, stochastic, tgt.shape[0])
        counter, tag = head_words(ws)
        assert counter == 0            # left ready for the next call
        tags.add(tag)
    assert len(tags) == 1 and 0 not in next(iter(tags))


@pytest.mark.parametrize("kernel", ["register", "bulk"])
@pytest.mark.parametrize("stochastic", [False, True])
def test_requests_without_streamed_rows_are_still_finalised(dev, kernel, stochastic):
    wl = (synth.WORKLOADS["stochastic"] if stochastic else synth.WORKLOADS["large_vocab_mixed"])
    wl = wl.with_(B=12, V=2048, tiers=(96,))
    bt = synth.make_batch(wl, seed=7, stochastic=stochastic)
    B, g = bt.B, bt.gamma
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
    cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
    packed = synth.gather_packed(bt.target, B, g, w)
    kw = dict(temperature=1.0, seed=3, step=0) if stochastic else {}
    drf = bt.draft if stochastic else None
    ws = torch.zeros(bd.dspark_verify_workspace_bytes(B, g, wl.V, stochastic), dtype=torch.uint8,
                     device=dev)
    # the packed buffer cut to the first requests' rows: the later requests stream nothing
    # (or only part of their rows) and must come out as bad rows, the earlier ones verified
    for rows in (int(cu[B // 2]), int(cu[B // 2]) + 1, 0):
        tgt = packed[:rows] if rows else packed[:0]
        gres = run(dev, ws, "compact", tgt, bt.tokens, cu, w, stochastic, drf, kernel, **kw)
        rres = ref("compact", tgt, bt.tokens, cu, w, stochastic, drf, **kw)
        check(gres, rres, stochastic, rows)
        assert gres["status"] & bd.STATUS_BAD_ROWS
    # cap-accept with a block buffer short of the last requests' rows
    tgt = bt.target[: (B - 3) * g + 2]
    gres = run(dev, ws, "cap_accept", tgt, bt.tokens, None, w, stochastic, drf, kernel, **kw)
    rres = ref("cap_accept", tgt, bt.tokens, None, w, stochastic, drf, **kw)
    check(gres, rres, stochastic, tgt.shape[0])


@pytest.mark.parametrize("kernel", ["register", "bulk"])
def test_rows_before_the_first_request_are_skipped(dev, kernel):
    wl = synth.WORKLOADS["large_vocab_mixed"].with_(B=9, V=1024, tiers=(80,))
    bt = synth.make_batch(wl, seed=11)
    B, g = bt.B, bt.gamma
    # short windows (a steep theta): the rows with the leading gap still fit B * gamma rows
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, 0.3 * np.arange(B * g + 1))["windows"]
    lead = 5
    assert lead + int(w.sum()) <= B * g
    cu = (lead + np.concatenate([[0], np.cumsum(w)])).astype(np.int32)
    body = synth.gather_packed(bt.target, B, g, w)
    gap = torch.randn(lead, wl.V, generator=torch.Generator().manual_seed(1)).to(body.dtype)
    tgt = torch.cat([gap, body])
    ws = torch.zeros(bd.dspark_verify_workspace_bytes(B, g, wl.V, False), dtype=torch.uint8,
                     device=dev)
    gres = run(dev, ws, "compact", tgt, bt.tokens, cu, w, False, None, kernel)
    rres = ref("compact", tgt, bt.tokens, cu, w, False)
    check(gres, rres, False, tgt.shape[0])
    assert gres["status"] == 0


@pytest.mark.parametrize("kernel", ["register", "bulk"])
@pytest.mark.parametrize("stochastic", [False, True])
def test_a_window_reaching_into_the_next_request(dev, kernel, stochastic):
    # request 3's window claims a row that cu_seqlens gives to request 4: every request reads
    # its rows from cu_seqlens[b] on, as the oracle does (row_prob is not compared: the shared
    # row holds either request's values, and the row after request 4 belongs to no request)
    wl = (synth.WORKLOADS["stochastic"] if stochastic else synth.WORKLOADS["large_vocab_mixed"])
    wl = wl.with_(B=8, V=2048, tiers=(64,))
    bt = synth.make_batch(wl, seed=5, stochastic=stochastic)
    B, g = bt.B, bt.gamma
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, 0.0 * bt.theta)["windows"]   # all gamma
    cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
    cu_bad = cu.copy()
    cu_bad[4] -= 1
    tgt = synth.gather_packed(bt.target, B, g, w)
    drf = bt.draft if stochastic else None
    kw = dict(temperature=1.0, seed=2, step=4) if stochastic else {}
    ws = torch.zeros(bd.dspark_verify_workspace_bytes(B, g, wl.V, stochastic), dtype=torch.uint8,
                     device=dev)
    gres = run(dev, ws, "compact", tgt, bt.tokens, cu_bad, w, stochastic, drf, kernel, **kw)
    rres = ref("compact", tgt, bt.tokens, cu_bad, w, stochastic, drf, **kw)
    check(gres, rres, stochastic, 0)


@pytest.mark.parametrize("kernel", ["register", "bulk"])
@pytest.mark.parametrize("stochastic", [False, True])
def test_fewer_rows_than_requests(dev, kernel, stochastic):
    # cu_seqlens puts two requests on each row, so its total (32) is below B (64): the
    # even requests share their tested row with the next request (bad rows, as the oracle has
    # it), the odd ones share only their last row and are verified
    wl = (synth.WORKLOADS["stochastic"] if stochastic else synth.WORKLOADS["large_vocab_mixed"])
    wl = wl.with_(B=64, V=4096, tiers=(512,))
    bt = synth.make_batch(wl, seed=9, stochastic=stochastic)
    B, g = bt.B, bt.gamma
    w = np.full(B, 2, dtype=np.int32)
    cu = (np.arange(B + 1) // 2).astype(np.int32)
    # a 128-row buffer of which cu_seqlens names 32; the last request's second row lies past
    # them (bad rows, as the oracle has it)
    tgt = synth.gather_packed(bt.target, B, g, w)
    drf = bt.draft if stochastic else None
    kw = dict(temperature=1.0, seed=6, step=1) if stochastic else {}
    ws = torch.zeros(bd.dspark_verify_workspace_bytes(B, g, wl.V, stochastic), dtype=torch.uint8,
                     device=dev)
    for _ in range(2):          # the second call hands out the bulk kernel's tail by ticket
        gres = run(dev, ws, "compact", tgt, bt.tokens, cu, w, stochastic, drf, kernel, **kw)
        rres = ref("compact", tgt, bt.tokens, cu, w, stochastic, drf, **kw)
        check(gres, rres, stochastic, 0)


@pytest.mark.parametrize("case", range(48))
def test_random_cu_seqlens_against_the_oracle(dev, case):
    # non-decreasing cu_seqlens that need not be the scan of the windows: leading rows, gaps,
    # requests sharing rows, totals past or short of the buffer, windows outside [1, gamma];
    # every request verified, flagged or clamped as the oracle has it (compact mode)
    rng = np.random.default_rng(31000 + case)
    kernel = ["register", "bulk"][case % 2]
    stochastic = bool((case // 2) % 2)
    B = int(rng.integers(1, 49))
    g = int(rng.integers(2 if stochastic else 1, 9))
    V = int(rng.choice([1000, 1024, 2048, 4104]))
    w = rng.integers(0, g + 2, size=B).astype(np.int32)
    steps = rng.integers(0, g + 2, size=B)
    cu = np.concatenate([[0], np.cumsum(steps)]).astype(np.int32) + int(rng.integers(0, 4))
    rows = max(0, int(cu[B]) + int(rng.integers(-3, g + 1)))
    tgt = (torch.randn((max(rows, 1), V), generator=torch.Generator().manual_seed(case)) * 2.0)
    tgt = tgt.to(torch.bfloat16)[:rows]
    tokens = rng.integers(0, V, size=(B, g)).astype(np.int32)
    if rows:
        best = tgt.float().argmax(dim=1).numpy()
        for b in range(B):                      # accept some drafts where the rows exist
            for i in range(g - 1):
                r = int(cu[b]) + i
                if r < rows and rng.uniform() < 0.7:
                    tokens[b, i + 1] = best[r]
    drf = None
    kw = {}
    if stochastic:
        drf = (torch.randn((max(B * (g - 1), 1), V), generator=torch.Generator().manual_seed(
            100 + case)) * 2.0).to(torch.bfloat16)[: B * (g - 1)]
        kw = dict(temperature=float(rng.choice([0.7, 1.0])), seed=case, step=3)
    ws = torch.empty(max(bd.dspark_verify_workspace_bytes(B, g, V, stochastic), 16),
                     dtype=torch.uint8, device=dev)
    for _ in range(2):          # the second call finds the head the first one left
        gres = run(dev, ws, "compact", tgt, tokens, cu, w, stochastic, drf, kernel, **kw)
        rres = ref("compact", tgt, tokens, cu, w, stochastic, drf, **kw)
        check(gres, rres, stochastic, 0)


@pytest.mark.parametrize("kernel", ["register", "bulk"])
@pytest.mark.parametrize("T", [0.02, 0.1, 5.0, 20.0])
def test_extreme_temperatures(dev, kernel, T):
    # a very sharp softmax (most exponentials underflow, p/q spans fp32's range) and a very
    # flat one (the bonus draw's tile sums nearly uniform), compact and cap-accept
    wl = synth.WORKLOADS["stochastic"].with_(B=24, V=8192, temperature=T, tiers=(192,))
    bt = synth.make_batch(wl, seed=int(T * 100) + 3, stochastic=True)
    B, g = bt.B, bt.gamma
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
    cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
    kw = dict(temperature=T, seed=11, step=4)
    ws = torch.empty(bd.dspark_verify_workspace_bytes(B, g, wl.V, True), dtype=torch.uint8,
                     device=dev)
    for mode in ("compact", "cap_accept"):
        tgt = synth.gather_packed(bt.target, B, g, w) if mode == "compact" else bt.target
        gres = run(dev, ws, mode, tgt, bt.tokens, cu if mode == "compact" else None, w, True,
                   bt.draft, kernel, **kw)
        rres = ref(mode, tgt, bt.tokens, cu if mode == "compact" else None, w, True, bt.draft,
                   **kw)
        check(gres, rres, True, tgt.shape[0])


def test_register_kernel_with_more_units_than_a_32_bit_split_holds(dev):
    # stochastic compact at the largest batch with full windows: 8192 x 32 target rows and as
    # many draft jobs, one chunk each (V = 256), 524288 units for the register kernel's 4864
    # warps, past 2^31 / warps: the split falls back to 64-bit arithmetic
    B, g, V = 8192, 32, 256
    gen = torch.Generator().manual_seed(17)
    tgt = (torch.randn((B * g, V), generator=gen) * 2.0).to(torch.bfloat16)
    drf = (tgt.view(B, g, V)[:, : g - 1].float()
           + torch.randn((B, g - 1, V), generator=gen) * 0.5).to(torch.bfloat16)
    drf = drf.reshape(B * (g - 1), V)
    rng = np.random.default_rng(17)
    tokens = rng.integers(0, V, size=(B, g)).astype(np.int32)
    w = np.full(B, g, dtype=np.int32)
    cu = (np.arange(B + 1) * g).astype(np.int32)
    kw = dict(temperature=1.0, seed=5, step=2)
    ws = torch.empty(bd.dspark_verify_workspace_bytes(B, g, V, True), dtype=torch.uint8,
                     device=dev)
    gres = run(dev, ws, "compact", tgt, tokens, cu, w, True, drf, "register", **kw)
    rres = ref("compact", tgt, tokens, cu, w, True, drf, **kw)
    near, _ = compare_stochastic(gres, rres, tgt.shape[0])
    assert near <= 2                 # 253952 accept tests: counted near-ties only
    np.testing.assert_array_equal(gres["ceiling_len"], rres["ceiling_len"])


@pytest.mark.parametrize("stochastic", [False, True])
def test_more_than_4096_requests(dev, stochastic):
    wl = (synth.WORKLOADS["stochastic"] if stochastic else synth.WORKLOADS["large_vocab_mixed"])
    wl = wl.with_(B=4099, gamma=3, V=64, tiers=(3 * 4099,))
    bt = synth.make_batch(wl, seed=21, stochastic=stochastic)
    B, g = bt.B, bt.gamma
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
    cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
    tgt = synth.gather_packed(bt.target, B, g, w)
    drf = bt.draft if stochastic else None
    kw = dict(temperature=1.0, seed=8, step=2) if stochastic else {}
    ws = torch.zeros(bd.dspark_verify_workspace_bytes(B, g, wl.V, stochastic), dtype=torch.uint8,
                     device=dev)
    for kernel in ("register", "bulk"):
        gres = run(dev, ws, "compact", tgt, bt.tokens, cu, w, stochastic, drf, kernel, **kw)
        rres = ref("compact", tgt, bt.tokens, cu, w, stochastic, drf, **kw)
        check(gres, rres, stochastic, tgt.shape[0])


def chunks_per_row(V, B, gamma):
    """Chunks per logits row of the streaming plan: about 4096 units per call (1024 when the
    block holds at most 64 rows), chunks of 256 to 12288 elements in multiples of 8."""
    rows = B * gamma
    nc_min = -(-V // 12288)
    nc_max = max(V // 256, 1)
    want = -(-(1024 if rows <= 64 else 4096) // max(rows, 1))
    nc = max(min(want, nc_max), nc_min)
    C = -(-(-(-V // nc)) // 8) * 8
    return -(-V // C)


# (B, gamma, V): the bonus kernel combines a row's partials with 1, 2 or 4 per lane, or one row
# at a time past 128 chunks
COMBINE_CASES = [(40, 8, 4096), (3, 6, 20000), (2, 5, 40000), (1, 2, 131072)]


@pytest.mark.parametrize("B,gamma,V", COMBINE_CASES)
@pytest.mark.parametrize("mode", ["compact", "cap_accept"])
def test_stochastic_every_combine_width(dev, B, gamma, V, mode):
    nc = chunks_per_row(V, B, gamma)
    wl = synth.WORKLOADS["stochastic"].with_(B=B, gamma=gamma, V=V, tiers=(B * gamma,))
    bt = synth.make_batch(wl, seed=B + V, stochastic=True)
    w = oracle.schedule(bt.conf, bt.bias, bt.alpha, 0.0 * bt.theta)["windows"]   # full windows
    cu = np.concatenate([[0], np.cumsum(w)]).astype(np.int32)
    tgt = synth.gather_packed(bt.target, B, gamma, w) if mode == "compact" else bt.target
    kw = dict(temperature=0.8, seed=13, step=2)
    ws = torch.empty(bd.dspark_verify_workspace_bytes(B, gamma, V, True), dtype=torch.uint8,
                     device=dev)
    for kernel in ("register", "bulk"):
        gres = run(dev, ws, mode, tgt, bt.tokens, cu if mode == "compact" else None, w, True,
                   bt.draft, kernel, **kw)
        rres = ref(mode, tgt, bt.tokens, cu if mode == "compact" else None, w, True, bt.draft,
                   **kw)
        check(gres, rres, True, tgt.shape[0])
    assert nc == chunks_per_row(V, B, gamma)
    assert {(40, 8, 4096): nc <= 32, (3, 6, 20000): 32 < nc <= 64,
            (2, 5, 40000): 64 < nc <= 128, (1, 2, 131072): nc > 128}[(B, gamma, V)], nc
