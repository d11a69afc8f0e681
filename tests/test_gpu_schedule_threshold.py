"""GPU parity of the static-threshold baseline (dspark_schedule_threshold,
DSpark paper section 4.3.3) against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("R,g", [(1, 1), (7, 32), (512, 16), (3000, 16)])
def test_threshold_matches_oracle(dev, R, g):
    conf = workloads.make_confidences(R, g, seed=R + g)
    conf[::5, 2 % g] = 0.5        # ties exactly at a threshold below
    c = torch.from_numpy(conf).to(dev)
    for thr in (-0.5, 0.0, 0.3, 0.5, 0.75, 0.9, 1.0, 1.5):
        out = binding.dspark_schedule_threshold(c, thr, check=True)
        np.testing.assert_array_equal(out["verify_len"].cpu().numpy(),
                                      oracle.schedule_threshold(conf, thr), err_msg=str(thr))


def test_bad_confidence_sets_status(dev):
    conf = np.full((4, 4), 0.9, np.float32)
    conf[2, 1] = np.nan
    out = binding.dspark_schedule_threshold(torch.from_numpy(conf).to(dev), 0.5)
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 5
    assert list(out["verify_len"].cpu().numpy()) == [4, 4, 1, 4]
