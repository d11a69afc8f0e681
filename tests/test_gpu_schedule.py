"""GPU parity of dspark_schedule against the oracle (DSpark paper section
3.2.2, Algorithm 1), and the scheduled end-to-end workload: the scheduler's
lengths drive a ragged verification that is checked against the oracle."""
import json
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._gpu import PROB_RTOL_QUALITY, compare, oracle_on_requests
from tests._sched import assess_schedule

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def gpu_schedule(conf, T, dev):
    out = binding.dspark_schedule(torch.from_numpy(np.ascontiguousarray(conf, np.float32)).to(dev),
                                  torch.from_numpy(np.ascontiguousarray(T, np.float64)).to(dev),
                                  check=True)
    return (out["verify_len"].cpu().numpy(), float(out["theta_best"].item()),
            int(out["near_tie_count"].item()))


def check(conf, T, dev, no_ties=False):
    """Every request's length against the oracle's admission path: the GPU's
    stopping point may differ from the oracle's only at an admission whose own
    Theta comparison lies in the 1e-9 near-tie window. no_ties=True also
    asserts that the oracle sees no near tie at all (the named workloads), so
    the lengths must equal the oracle's outright."""
    ell, theta, ties = gpu_schedule(conf, T, dev)
    ref = oracle.schedule(conf, T, early_stop=True)
    R, g = conf.shape
    excused = assess_schedule(ell, theta, oracle.schedule_path(conf, T), R, g, early_stop=True)
    if ref["near_ties"] == 0 or no_ties:
        assert ref["near_ties"] == 0 and excused == 0
        np.testing.assert_array_equal(ell, ref["verify_len"])
        assert abs(theta - ref["theta_best"]) <= 1e-12 * abs(ref["theta_best"])
    return ell, ref


def test_appendix8_numbers(dev):
    g = json.load(open(os.path.join(GOLDEN, "appendix8.json")))
    sps = g["sps"]
    T = np.array([1e300, 1 / sps[0], 1 / sps[1], 1 / sps[2]])
    for c2 in (g["case1_c2"], g["case2_c2"]):
        ell, theta, _ = gpu_schedule(np.array([[g["a1"], c2]], np.float32), T, dev)
        assert ell[0] == 0 and abs(theta - g["theta0"]) < 1e-12


@pytest.mark.parametrize("seed", range(12))
def test_random_small(dev, seed):
    rng = np.random.default_rng(seed)
    R, g = int(rng.integers(1, 60)), int(rng.integers(1, 33))
    conf = rng.uniform(0, 1, (R, g)).astype(np.float32) ** 0.3
    conf[rng.uniform(size=(R, g)) < 0.1] = 1.0
    conf[rng.uniform(size=(R, g)) < 0.05] = 0.0
    n = R * (g + 1) + 1
    N = np.arange(n, dtype=np.float64)
    T = (rng.uniform(1, 5) + rng.uniform(0.001, 0.2) * N + rng.uniform(0, 1e-3) * N * N
         if seed % 2 == 0 else rng.uniform(1.0, 1.5, n) + 0.01 * N)
    check(conf, T, dev)


@pytest.mark.parametrize("R,g", [(512, 16), (1024, 16), (3000, 32), (1, 1), (7, 32)])
def test_named_and_large(dev, R, g):
    conf = workloads.make_confidences(R, g, seed=7)
    T = workloads.step_time_profile(R * (g + 1) + 1)
    ell, ref = check(conf, T, dev, no_ties=True)
    assert ell.sum() == ref["n_admitted"]


@pytest.mark.parametrize("R,g", [(256, 16), (4096, 1), (1, 32), (4097, 1),
                                 (257, 16), (255, 16), (129, 31)])
def test_shapes_and_ties(dev, R, g):
    """The headline 256 x 16 and shapes around it: gamma = 1 (runs of one
    candidate), one request of 32, request counts that are not powers of two,
    with ties from repeated confidences and certain tokens (c = 1)."""
    rng = np.random.default_rng(R * 31 + g)
    conf = workloads.make_confidences(R, g, seed=R + g)
    conf[rng.uniform(size=(R, g)) < 0.2] = 1.0
    conf[:, :] = np.where(rng.uniform(size=(R, g)) < 0.1, conf[0, 0], conf)
    N = np.arange(R * (g + 1) + 1, dtype=np.float64)
    for T in (workloads.step_time_profile(R * (g + 1) + 1), 2.0 + 0.01 * N + 0.4 * (N % 7 == 0)):
        check(conf, T, dev)


@pytest.mark.parametrize("kind", ["all_ones", "quantized", "one_outlier"])
def test_many_equal_survival_values(dev, kind):
    """512 x 16 with massive ties in the sort: every confidence 1 (all
    survival values equal); confidences from four levels (thousands of
    exactly equal products across requests); and a dense cluster of distinct
    values near 1 beside one far outlier."""
    R, g = 512, 16
    rng = np.random.default_rng(99)
    if kind == "all_ones":
        conf = np.ones((R, g), np.float32)
    elif kind == "quantized":
        conf = rng.choice(np.array([0.5, 0.75, 0.9, 1.0], np.float32), size=(R, g))
    else:
        conf = (1.0 - rng.uniform(0, 1e-6, (R, g))).astype(np.float32)
        conf[7, 0] = 1e-30
    N = np.arange(R * (g + 1) + 1, dtype=np.float64)
    for T in (workloads.step_time_profile(R * (g + 1) + 1), 2.0 + 0.001 * N,
              np.full(R * (g + 1) + 1, 4.0)):
        check(conf, T, dev)


def test_flat_profile_admits_everything(dev):
    conf = workloads.make_confidences(256, 16, seed=1)
    ell, _ = check(conf, np.full(256 * 17 + 1, 4.0), dev)
    assert np.all(ell == 16)


@pytest.mark.parametrize("R,g", [(37, 9), (1100, 16)])
def test_negative_zero_confidence(dev, R, g):
    """-0.0 lies in [0, 1]: it ends its request's candidates like +0.0 (a > 0
    is false for a = -0), on the rank path (333 candidates) and the block path
    (17,600)."""
    conf = workloads.make_confidences(R, g, seed=R)
    rng = np.random.default_rng(R)
    rows = rng.choice(R, size=max(1, R // 10), replace=False)
    conf[rows, rng.integers(0, g, size=rows.size)] = np.float32(-0.0)
    assert np.signbit(conf).any()
    n = R * (g + 1) + 1
    N = np.arange(n, dtype=np.float64)
    for T in (workloads.step_time_profile(n), np.full(n, 4.0), 2.0 + 1e-4 * N):
        ell, ref = check(conf, T, dev)
        zero_at = np.where(conf[rows] == 0, np.arange(g), g).min(axis=1)
        assert np.all(ell[rows] <= zero_at)
    out = binding.dspark_schedule(torch.from_numpy(conf).to(dev),
                                  torch.from_numpy(workloads.step_time_profile(n)).to(dev))
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 0


def test_bad_confidence_sets_status(dev):
    conf = workloads.make_confidences(8, 4, seed=1)
    conf[3, 2] = np.nan
    out = binding.dspark_schedule(torch.from_numpy(conf).to(dev),
                                  torch.from_numpy(workloads.step_time_profile(41)).to(dev))
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 5
    v = out["verify_len"].cpu().numpy()
    assert v.min() >= 0 and v.max() <= 4


def test_scheduled_workload_end_to_end(dev):
    """R=512, gamma=16: Beta confidences and T(N) = 4 + 0.006 N (+0.02 beyond
    2048) drive the lengths; ragged verification over V=129,280 bf16 follows."""
    R, g = 512, 16
    conf = workloads.make_confidences(R, g, seed=7)
    T = workloads.step_time_profile(R * (g + 1) + 1)
    ell, ref = check(conf, T, dev, no_ties=True)
    vi = workloads.make_config("sched_r512_g16_v129280_bf16", device=dev, verify_len=ell)
    out = binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens, vi.verify_len,
                                vi.uniforms, vi.temperature, vi.target_row_off, vi.draft_row_off,
                                check=True)
    idx = np.arange(R)
    st = compare(out, oracle_on_requests(vi, idx), vi, idx)
    assert st["prob_max_rel_err"] <= PROB_RTOL_QUALITY, st
    assert st["excused"] <= st["mismatch_budget"], st
