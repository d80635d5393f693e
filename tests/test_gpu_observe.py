"""GPU parity of dspark_observe against the oracle: the calibration histogram and the
utilisation counters are exact integers, so they must match bit for bit, also when several
calls accumulate into the same counters."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_ragged_gb300 import _binding as bd

from gpu_util import device, i32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    return device()


@pytest.mark.parametrize("B,gamma,nb", [(0, 4, 8), (1, 1, 4), (5, 8, 10), (512, 8, 20),
                                        (3000, 16, 1024), (77, 32, 7)])
def test_observe_parity(dev, B, gamma, nb):
    rng = np.random.default_rng(B + nb)
    hist = torch.zeros((nb, 3), dtype=torch.int64, device=dev)
    util = torch.zeros(2, dtype=torch.int64, device=dev)
    st = torch.zeros(1, dtype=torch.int32, device=dev)
    ref_h, ref_u, ref_s = None, None, 0
    for call in range(3):
        conf = rng.uniform(-0.1, 1.1, size=(B, gamma - 1)).astype(np.float32)
        if B and gamma > 1:
            conf[0, 0] = np.nan
        ceiling = rng.integers(1, gamma + 1, size=B).astype(np.int32)
        accept = np.minimum(ceiling, rng.integers(1, gamma + 1, size=B)).astype(np.int32)
        if call == 2 and B > 2:
            ceiling[1], accept[2] = gamma + 3, -1          # clamped, flagged
        bd.dspark_observe(torch.as_tensor(conf, device=dev), i32(accept, dev), i32(ceiling, dev),
                          hist, util, st)
        r = oracle.observe(conf, accept, ceiling, nb, ref_h, ref_u)
        ref_h, ref_u, ref_s = r["hist"], r["util"], ref_s | r["status"]
    torch.cuda.synchronize()
    np.testing.assert_array_equal(hist.cpu().numpy().astype(np.uint64), ref_h)
    np.testing.assert_array_equal(util.cpu().numpy().astype(np.uint64), ref_u)
    assert int(st.item()) == ref_s
