"""dspark_verify_noalloc: the verify entry point for callers that cannot provide scratch
memory (a host that hands a kernel library only its input and output buffers, or a serving
loop that has reserved the device's memory up front and must not call cudaMalloc mid-step).
Its scratch is a static device array inside the library.

The test calls it through the C ABI twice in a row with different inputs and checks each
result against the ordinary dspark_verify with a caller workspace (bit for bit: both run the
same kernels in the same order), then checks that sizes beyond the array are refused. The
greedy case is large enough for the bulk-copy streaming kernel, whose unit counter then sits in
the static array's head: the first call finds it zeroed (no tag: units split evenly), the second
hands out tickets. The file
is named to be collected last, so a run that stops at the first failure has run everything else;
it also passes alone in a fresh process."""
import numpy as np
import pytest
import torch

from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    from speculative_decoding_ragged_gb300 import build
    build.build()
    bd.lib()
    return torch.device("cuda:0")


def outputs(B, gamma, rows, dev):
    i32 = dict(dtype=torch.int32, device=dev)
    return dict(accept_len=torch.full((B,), -7, **i32),
                committed=torch.full((B, gamma), -7, **i32),
                ceiling_len=torch.full((B,), -7, **i32),
                row_prob=torch.full((rows, 2), -7.0, dtype=torch.float32, device=dev),
                status=torch.zeros(1, **i32))


def case(name, seed, dev):
    """(mode, kwargs) of one verify call on a seeded workload, windows from dspark_schedule."""
    if name == "greedy":
        wl = synth.WORKLOADS["large_vocab_mixed"].with_(B=64)
        stochastic = False
    else:
        wl = synth.WORKLOADS["stochastic"]
        stochastic = True
    bt = synth.make_batch(wl, seed=seed)
    w = torch.zeros(bt.B, dtype=torch.int32, device=dev)
    k = torch.zeros(1, dtype=torch.int32, device=dev)
    cost = bd.CostTable(bt.bias, torch.as_tensor(bt.alpha, device=dev),
                        torch.as_tensor(bt.theta, device=dev))
    bd.dspark_schedule(torch.as_tensor(bt.conf, device=dev), cost, w, k)
    cu = torch.zeros(bt.B + 1, dtype=torch.int32, device=dev)
    cu[1:] = torch.cumsum(w, 0)
    packed = synth.gather_packed(bt.target, bt.B, bt.gamma, w.cpu().numpy()).to(dev)
    kw = dict(stochastic=stochastic, cu_seqlens=cu, windows=w,
              draft=bt.draft.to(dev) if stochastic else None, temperature=wl.temperature,
              seed=seed + 11, step=seed)
    return packed, torch.as_tensor(bt.tokens, device=dev), kw


@pytest.mark.parametrize("name", ["greedy", "stochastic"])
def test_noalloc_matches_workspace_verify_on_two_calls(dev, name):
    for seed in (0, 1):        # two calls in a row: the second must not see the first's data
        target, tokens, kw = case(name, seed, dev)
        B, gamma = tokens.shape
        ref = outputs(B, gamma, target.shape[0], dev)
        ws = torch.empty(max(bd.dspark_verify_workspace_bytes(B, gamma, target.shape[1],
                                                              kw["stochastic"]), 16),
                         dtype=torch.uint8, device=dev)
        bd.dspark_verify("compact", target, tokens, ref["accept_len"], ref["committed"], ws,
                         ceiling_len=ref["ceiling_len"], row_prob=ref["row_prob"],
                         status=ref["status"], **kw)
        got = outputs(B, gamma, target.shape[0], dev)
        bd.dspark_verify_noalloc("compact", target, tokens, got["accept_len"], got["committed"],
                                 ceiling_len=got["ceiling_len"], row_prob=got["row_prob"],
                                 status=got["status"], **kw)
        torch.cuda.synchronize()
        for key in ref:
            np.testing.assert_array_equal(got[key].cpu().numpy(), ref[key].cpu().numpy(),
                                          err_msg=f"{name} seed {seed}: {key}")
        assert (got["accept_len"] >= 1).all()


def test_noalloc_refuses_sizes_beyond_its_array(dev):
    B, gamma, V = 1024, 16, 151936        # stochastic partials need about 10 MB
    assert bd.dspark_verify_workspace_bytes(B, gamma, V, True) > bd.NOALLOC_SCRATCH_BYTES
    i32 = dict(dtype=torch.int32, device=dev)
    target = torch.zeros((1, V), dtype=torch.bfloat16, device=dev)   # refused before any read
    with pytest.raises(bd.DSparkError) as err:
        bd.dspark_verify_noalloc("static", target, torch.zeros((B, gamma), **i32),
                                 torch.zeros(B, **i32), torch.zeros((B, gamma), **i32),
                                 stochastic=True)
    assert err.value.code == -2 and "static array holds" in str(err.value)
