"""DP tier agreement on the device ("DSpark in SGLang", A2 ragged verify over full CUDA graphs:
every DP rank replays the largest tier any rank needs). The fused schedule-and-pack writes
meta = {M, tier} on the GPU; TierSync all-reduces meta[1] in place over an NCCL group (of one
rank: the test runs on a single GPU) and hands the agreed tier, still on the device, to
the re-pack as its only tier. The re-pack must equal the oracle's pack with that tier."""
import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd
from speculative_decoding_ragged_gb300 import synth
from speculative_decoding_ragged_gb300.dp import TierSync
from speculative_decoding_ragged_gb300.step import DSparkStep

from gpu_util import device

pytestmark = pytest.mark.gpu


def test_tier_agreement_on_device_meta_feeds_the_repack():
    dev = device()
    store = dist.HashStore()
    dist.init_process_group("nccl", store=store, rank=0, world_size=1,
                            device_id=dev)
    try:
        wl = synth.WORKLOADS["high_load"].with_(B=64, V=64)
        sync = TierSync(device=dev)
        for step, slope in enumerate((0.001, 0.016, 0.004)):
            bt = synth.make_batch(wl, seed=5, step=step, theta_slope=slope)
            st = DSparkStep(wl.B, wl.gamma, wl.V, wl.tiers, bt.bias, bt.alpha, bt.theta,
                            device=dev)
            conf = torch.as_tensor(bt.conf, device=dev)
            tokens = torch.as_tensor(bt.tokens, device=dev)
            st.schedule_pack(conf, tokens)
            tiers = sync.step(st.meta)                 # all-reduce on the pack's own output
            # the re-pack takes the agreed tier where it lies: no host read in between
            bd.dspark_pack(st.windows, tokens, tiers, st.cu, st.packed_ids, st.meta,
                           st.row_req, st.row_pos, st.status)
            torch.cuda.synchronize()
            w = oracle.schedule(bt.conf, bt.bias, bt.alpha, bt.theta)["windows"]
            own = oracle.pack(w, bt.tokens, bt.tiers, st.packed_cap)
            agreed = int(tiers.item())
            assert agreed == own["tier"]              # one rank: the max over ranks is its own
            ref = oracle.pack(w, bt.tokens, np.array([agreed], np.int32), st.packed_cap)
            np.testing.assert_array_equal(st.windows.cpu().numpy(), w)
            np.testing.assert_array_equal(st.meta.cpu().numpy(), [ref["M"], ref["tier"]])
            np.testing.assert_array_equal(st.cu.cpu().numpy(), ref["cu"])
            for name in ("packed_ids", "row_req", "row_pos"):
                np.testing.assert_array_equal(getattr(st, name).cpu().numpy()[:agreed],
                                              ref[name][:agreed], err_msg=name)
            assert int(st.status.item()) == 0
    finally:
        dist.destroy_process_group()
