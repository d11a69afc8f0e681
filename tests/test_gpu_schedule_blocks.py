"""GPU parity of the scheduler's block path (sorted blocks of 1,024
candidates, ranks against the other blocks, a sweep over tiles of 8,192
positions), which takes the batches whose candidates exceed what the rank
path holds in shared memory. Against the oracle (DSpark paper section 3.2.2,
Algorithm 1; section 5.2 for the capacity and the top-K admission): every
request's length checked along the oracle's admission path, Theta, and the
stopping points that fall on a tile's first and last positions."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._sched import assess_schedule

pytestmark = pytest.mark.gpu
TILE = 8192  # positions per tile of the block path's sweep


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def _t(x, dev, dtype):
    return torch.from_numpy(np.ascontiguousarray(x, dtype)).to(dev)


def run_stop(conf, T, dev):
    out = binding.dspark_schedule(_t(conf, dev, np.float32), _t(T, dev, np.float64), check=True)
    return (out["verify_len"].cpu().numpy(), float(out["theta_best"].item()),
            int(out["near_tie_count"].item()))


def check_stop(conf, T, dev, no_ties=False):
    ell, theta, _ = run_stop(conf, T, dev)
    ref = oracle.schedule(conf, T, early_stop=True)
    R, g = conf.shape
    excused = assess_schedule(ell, theta, oracle.schedule_path(conf, T), R, g, early_stop=True)
    if ref["near_ties"] == 0 or no_ties:
        assert ref["near_ties"] == 0 and excused == 0
        np.testing.assert_array_equal(ell, ref["verify_len"])
        assert abs(theta - ref["theta_best"]) <= 1e-12 * abs(ref["theta_best"])
    return ell, ref


def check_capacity(conf, T, dev):
    out = binding.dspark_schedule_capacity(_t(conf, dev, np.float32), _t(T, dev, np.float64),
                                           check=True)
    K, ell = int(out["capacity"].item()), out["verify_len"].cpu().numpy()
    theta = float(out["theta_best"].item())
    assert K == int(ell.sum())
    ref = oracle.schedule(conf, T, early_stop=False)
    R, g = conf.shape
    excused = assess_schedule(ell, theta, oracle.schedule_path(conf, T), R, g, early_stop=False)
    if ref["near_ties"] == 0:
        assert excused == 0 and K == ref["n_admitted"]
        np.testing.assert_array_equal(ell, ref["verify_len"])
        assert abs(theta - ref["theta_best"]) <= 1e-12 * abs(ref["theta_best"])
    return K, ref


def quantized(rng, R, g):
    """Confidences from four levels: long runs of exactly equal survival
    values, spread over many blocks."""
    return rng.choice(np.array([0.5, 0.75, 0.9, 1.0], np.float32), size=(R, g))


SHAPES = [(1100, 16),   # 17,600 candidates: 18 blocks, the last of 192; 3 tiles
          (20000, 1),   # runs of one candidate, 20,000 requests
          (7001, 3),    # requests straddling block boundaries, a ragged last block
          (700, 32),    # the longest runs
          (6000, 16)]   # 96,000 candidates: 94 blocks, 12 tiles


@pytest.mark.parametrize("R,g", SHAPES)
def test_early_stop_on_named_profiles(dev, R, g):
    conf = workloads.make_confidences(R, g, seed=R + g)
    n = R * (g + 1) + 1
    N = np.arange(n, dtype=np.float64)
    check_stop(conf, workloads.step_time_profile(n), dev)
    check_stop(conf, 2.0 + 1e-5 * N, dev)   # a slow slope: the stop lands late
    check_stop(conf, np.full(n, 4.0), dev)  # flat: every tile, up to the first value
    # that no longer moves tau (Algorithm 1 stops where Theta stops growing)


@pytest.mark.parametrize("R,g", SHAPES)
def test_capacity_and_topk(dev, R, g):
    rng = np.random.default_rng(R * 3 + g)
    conf = workloads.make_confidences(R, g, seed=R * 5 + g)
    n = R * (g + 1) + 1
    N = np.arange(n, dtype=np.float64)
    T = rng.uniform(1, 4) + 1e-4 * N + rng.uniform(0.05, 0.3) * (N // 997)  # cliffs
    K, _ = check_capacity(conf, T, dev)
    nE = int((np.cumprod(conf.astype(np.float64), axis=1) > 0).sum())
    cap_t = torch.empty(1, dtype=torch.int32, device=dev)
    for k in sorted({0, 1, TILE, TILE + 1, K, nE // 2, nE - 1, nE, nE + 3}):
        cap_t.fill_(k)
        out = binding.dspark_schedule_topk(_t(conf, dev, np.float32), cap_t, check=True)
        np.testing.assert_array_equal(out["verify_len"].cpu().numpy(),
                                      oracle.schedule_topk(conf, k)["verify_len"],
                                      err_msg=f"K={k}")


@pytest.mark.parametrize("stop_at", [1, 2, TILE - 1, TILE, TILE + 1, 2 * TILE + 1, 3 * TILE])
def test_stop_at_tile_edges(dev, stop_at):
    """A profile that is flat up to the admission stop_at and then jumps: the
    first non-improving admission is exactly stop_at, so n* = stop_at - 1
    (TILE + 1 stops on the second tile's first position, where tau(n*) is the
    tile's carry)."""
    R, g = 2000, 16  # 32,000 candidates, each survival value above 2.8e-4, so
    # that no admission on the flat part is a near tie
    conf = np.clip(workloads.make_confidences(R, g, seed=5), 0.6, 1.0).astype(np.float32)
    n = R * (g + 1) + 1
    T = np.full(n, 3.0)
    T[R + stop_at:] = 1e9
    ell, ref = check_stop(conf, T, dev, no_ties=True)
    assert ref["n_admitted"] == stop_at - 1 == int(ell.sum())


@pytest.mark.parametrize("R,g", [(1100, 16), (7001, 3)])
def test_equal_values_across_blocks(dev, R, g):
    rng = np.random.default_rng(17)
    conf = quantized(rng, R, g)
    n = R * (g + 1) + 1
    N = np.arange(n, dtype=np.float64)
    for T in (workloads.step_time_profile(n), 2.0 + 2e-5 * N, np.full(n, 4.0)):
        check_stop(conf, T, dev)
    check_capacity(conf, 1.0 + 1e-5 * N + 0.2 * (N // 3001), dev)


def test_all_equal_and_zero_candidates(dev):
    R, g = 1500, 16
    n = R * (g + 1) + 1
    ell, ref = check_stop(np.ones((R, g), np.float32), np.full(n, 4.0), dev)
    assert np.all(ell == g)
    ell, ref = check_stop(np.zeros((R, g), np.float32), workloads.step_time_profile(n), dev)
    assert not ell.any() and ref["n_admitted"] == 0


def test_bad_inputs_set_status(dev):
    R, g = 1100, 16
    n = R * (g + 1) + 1
    conf = workloads.make_confidences(R, g, seed=3)
    conf[1057, 4] = 1.5
    out = binding.dspark_schedule(_t(conf, dev, np.float32),
                                  _t(workloads.step_time_profile(n), dev, np.float64))
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 5
    T = workloads.step_time_profile(n)
    T[R + 12345] = -1.0
    out = binding.dspark_schedule(_t(workloads.make_confidences(R, g, seed=4), dev, np.float32),
                                  _t(T, dev, np.float64))
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 5
