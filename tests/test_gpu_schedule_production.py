"""GPU parity of the production scheduler (DSpark paper, section 5.2): the
capacity from the global search without the early-stopping break
(dspark_schedule_capacity) and the dynamic top-K admission
(dspark_schedule_topk), against the oracle. Both scheduler paths are covered:
the rank-and-sweep kernels (up to 6,144 candidates) and the block path
beyond."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._sched import assess_schedule

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def _t(x, dev, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype)).to(dev)


def gpu_capacity(conf, T, dev):
    out = binding.dspark_schedule_capacity(_t(conf, dev, np.float32), _t(T, dev, np.float64),
                                           check=True)
    return (int(out["capacity"].item()), out["verify_len"].cpu().numpy(),
            float(out["theta_best"].item()), int(out["near_tie_count"].item()))


def gpu_topk(conf, K, dev):
    cap = torch.tensor([K], dtype=torch.int32, device=dev)
    out = binding.dspark_schedule_topk(_t(conf, dev, np.float32), cap, check=True)
    return out["verify_len"].cpu().numpy()


def jagged_profile(rng, n):
    """A step-time table with cliffs: base + slope*N plus a jump every few
    tokens, the shape for which the global search beats the early stop."""
    N = np.arange(n, dtype=np.float64)
    period = int(rng.integers(3, 40))
    return rng.uniform(1, 4) + rng.uniform(0.001, 0.05) * N + rng.uniform(0.05, 0.6) * (N // period)


def random_conf(rng, R, g):
    conf = rng.uniform(0, 1, (R, g)).astype(np.float32) ** 0.3
    conf[rng.uniform(size=(R, g)) < 0.1] = 1.0     # equal survival inside a request
    conf[rng.uniform(size=(R, g)) < 0.05] = 0.0
    return conf


def check_capacity(conf, T, dev, no_ties=False):
    """Every request's length against the oracle's admission path: the
    capacity may differ from the oracle's first maximum only where the two
    Theta values lie in the 1e-9 near-tie window. no_ties=True also asserts
    that the oracle sees no near tie, so K and the lengths equal its own."""
    K, ell, theta, ties = gpu_capacity(conf, T, dev)
    ref = oracle.schedule(conf, T, early_stop=False)
    R, g = conf.shape
    assert K == int(ell.sum())
    excused = assess_schedule(ell, theta, oracle.schedule_path(conf, T), R, g, early_stop=False)
    if ref["near_ties"] == 0 or no_ties:
        assert ref["near_ties"] == 0 and excused == 0
        assert K == ref["n_admitted"]
        np.testing.assert_array_equal(ell, ref["verify_len"])
        assert abs(theta - ref["theta_best"]) <= 1e-12 * abs(ref["theta_best"])
        assert ties == 0
    return K, ref


def test_appendix8_capacity(dev):
    g = json.load(open(os.path.join(GOLDEN, "appendix8.json")))
    sps = g["sps"]
    T = np.array([1e300, 1 / sps[0], 1 / sps[1], 1 / sps[2]])
    conf = np.array([[g["a1"], g["case1_c2"]]], np.float32)
    K, ell, theta, _ = gpu_capacity(conf, T, dev)
    # the worked example uses exact decimals; the confidences here are float32
    assert K == 2 and ell[0] == 2 and abs(theta - g["case1_theta2"]) < 1e-6
    ref = oracle.schedule(conf, T, early_stop=False)
    assert abs(theta - ref["theta_best"]) <= 1e-12 * ref["theta_best"]
    # case 2 (c2 = 0): the second token is no candidate, Theta stays at 1.0
    K, ell, theta, _ = gpu_capacity(np.array([[g["a1"], g["case2_c2"]]], np.float32), T, dev)
    assert K == 0 and ell[0] == 0 and abs(theta - g["theta0"]) < 1e-12


@pytest.mark.parametrize("seed", range(16))
def test_capacity_random(dev, seed):
    rng = np.random.default_rng(1000 + seed)
    R, g = int(rng.integers(1, 200)), int(rng.integers(1, 33))
    conf = random_conf(rng, R, g)
    check_capacity(conf, jagged_profile(rng, R * (g + 1) + 1), dev)


@pytest.mark.parametrize("R,g", [(512, 16), (1024, 16), (1100, 16), (3000, 32)])
def test_capacity_named_and_large(dev, R, g):
    """The scheduled workload's 512 x 16 and three larger batches, all on the
    block path (more than 6,144 candidates)."""
    rng = np.random.default_rng(R + g)
    conf = workloads.make_confidences(R, g, seed=7)
    K, ref = check_capacity(conf, jagged_profile(rng, R * (g + 1) + 1), dev, no_ties=True)
    assert K > 0


def test_global_search_steps_over_a_cliff(dev):
    """A profile whose first admission is worse but the later ones better: the
    early stop admits nothing, the global search admits past the cliff."""
    conf = np.full((4, 4), 0.95, np.float32)
    n = 4 * 5 + 1
    T = np.full(n, 4.0)
    T[5] = 6.0           # admitting one token costs a cliff ...
    T[6:] = 4.2          # ... after which admissions are cheap
    es = oracle.schedule(conf, T, early_stop=True)
    assert es["n_admitted"] == 0
    K, ref = check_capacity(conf, T, dev)
    assert K == ref["n_admitted"] > 0


@pytest.mark.parametrize("R,g", [(9, 5), (200, 16), (512, 16), (1100, 16)])
def test_topk_matches_oracle(dev, R, g):
    rng = np.random.default_rng(R * 7 + g)
    conf = random_conf(rng, R, g)
    nE = int((np.cumprod(conf.astype(np.float64), axis=1) > 0).sum())
    for K in sorted({0, 1, 2, nE // 3, nE // 2, nE - 1, nE, nE + 5, 1 << 30}):
        if K < 0:
            continue
        got = gpu_topk(conf, K, dev)
        ref = oracle.schedule_topk(conf, K)
        np.testing.assert_array_equal(got, ref["verify_len"], err_msg=f"K={K}")
        assert int(got.sum()) == min(K, nE)


def test_capacity_then_topk_on_one_stream(dev):
    """The serving pipeline: the capacity of older confidences, then the top-K
    admission of the current ones, with K passed on the device."""
    rng = np.random.default_rng(77)
    R, g = 256, 16
    old = workloads.make_confidences(R, g, seed=11)
    now = workloads.make_confidences(R, g, seed=12)
    T = jagged_profile(rng, R * (g + 1) + 1)
    bufs = binding.ScheduleBuffers(R, g, dev)
    binding.dspark_schedule_capacity(_t(old, dev, np.float32), _t(T, dev, np.float64),
                                     buffers=bufs)
    cap = bufs.capacity.clone()
    out = binding.dspark_schedule_topk(_t(now, dev, np.float32), cap, buffers=bufs, check=True)
    K_ref = oracle.schedule(old, T, early_stop=False)["n_admitted"]
    assert int(cap.item()) == K_ref
    np.testing.assert_array_equal(out["verify_len"].cpu().numpy(),
                                  oracle.schedule_topk(now, K_ref)["verify_len"])


def test_negative_capacity_sets_bad_data(dev):
    conf = workloads.make_confidences(8, 4, seed=3)
    cap = torch.tensor([-3], dtype=torch.int32, device=dev)
    out = binding.dspark_schedule_topk(_t(conf, dev, np.float32), cap)
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 5
    assert not out["verify_len"].cpu().numpy().any()
