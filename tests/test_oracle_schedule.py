"""Pins of the oracle's prefix scheduler (DSpark paper section 3.2.2, and the
Chinese translation page's Algorithm 1) against brute force."""
import numpy as np
import pytest

import oracle
from tests._sched import exhaustive_best, greedy_order, theta_of


def _convex_profile(rng, n):
    a, b, c = rng.uniform(1, 5), rng.uniform(0.01, 1.0), rng.uniform(0, 0.2)
    N = np.arange(n, dtype=np.float64)
    return a + b * N + c * N * N


def _confidences(rng, R, g):
    c = rng.uniform(0, 1, (R, g)).astype(np.float32)
    c[rng.uniform(size=(R, g)) < 0.15] = 1.0   # ties inside a request
    c[rng.uniform(size=(R, g)) < 0.08] = 0.0   # excluded candidates
    return c


@pytest.mark.parametrize("seed", range(40))
def test_early_stop_is_optimal_for_convex_step_time(seed):
    """For increasing convex T(N) Theta is unimodal along the greedy path, so the
    causal early-stopping scheduler reaches the brute-force maximum."""
    rng = np.random.default_rng(seed)
    R, g = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    conf = _confidences(rng, R, g)
    T = _convex_profile(rng, R * (g + 1) + 1)
    s = oracle.schedule(conf, T, early_stop=True)
    best, _ = exhaustive_best(conf, T)
    assert abs(s["theta_best"] - best) <= 1e-12 * best
    assert abs(theta_of(s["verify_len"], conf, T) - s["theta_best"]) <= 1e-12 * best
    assert s["n_admitted"] == int(s["verify_len"].sum())


@pytest.mark.parametrize("seed", range(40))
def test_global_search_is_optimal_for_any_step_time(seed):
    """Without the break (section 5.2) the best greedy prefix is the brute-force
    optimum for any T(N): for a fixed batch size the top survival values are
    optimal and are prefix-closed."""
    rng = np.random.default_rng(100 + seed)
    R, g = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    conf = _confidences(rng, R, g)
    T = rng.uniform(1.0, 3.0, R * (g + 1) + 1)        # jagged profile
    s = oracle.schedule(conf, T, early_stop=False)
    best, _ = exhaustive_best(conf, T)
    assert abs(s["theta_best"] - best) <= 1e-12 * best
    assert abs(theta_of(s["verify_len"], conf, T) - best) <= 1e-12 * best


@pytest.mark.parametrize("seed", range(30))
def test_early_stop_is_first_drop_on_jagged_profile(seed):
    """With a jagged T the causal scheduler stops at the first non-improvement
    along the globally sorted admission path."""
    rng = np.random.default_rng(200 + seed)
    R, g = int(rng.integers(1, 5)), int(rng.integers(1, 6))
    conf = _confidences(rng, R, g)
    T = rng.uniform(1.0, 3.0, R * (g + 1) + 1)
    s = oracle.schedule(conf, T, early_stop=True)
    order = greedy_order(conf)
    ell = np.zeros(R, int)
    prev = theta_of(ell, conf, T)
    n_star = 0
    for n, (r, j, _) in enumerate(order, 1):
        ell[r] = j
        th = theta_of(ell, conf, T)
        if not th > prev:
            break
        prev, n_star = th, n
    assert s["n_admitted"] == n_star
    assert abs(s["theta_best"] - prev) <= 1e-12 * prev
    expect = np.zeros(R, int)
    for r, j, _ in order[:n_star]:
        expect[r] = max(expect[r], j)
    np.testing.assert_array_equal(s["verify_len"], expect)


def test_scheduled_workload_is_sane():
    from speculative_decoding_verification_41_gb300 import workloads
    R, g = 512, 16
    conf = workloads.make_confidences(R, g, seed=7)
    T = workloads.step_time_profile(R * (g + 1) + 1)
    s = oracle.schedule(conf, T, early_stop=True)
    ell = s["verify_len"]
    assert ell.min() >= 0 and ell.max() <= g
    assert s["n_admitted"] == ell.sum() and s["n_admitted"] > 0
    # the admitted candidates are exactly the top n* survival values
    a = np.cumprod(conf.astype(np.float64), axis=1)
    chosen = np.concatenate([a[r, :ell[r]] for r in range(R)])
    rest = np.concatenate([a[r, ell[r]:] for r in range(R)])
    assert chosen.min() >= rest.max()
    # flat profile: every candidate is admitted
    s2 = oracle.schedule(conf, np.full(R * (g + 1) + 1, 4.0), early_stop=True)
    assert np.all(s2["verify_len"] == g)


@pytest.mark.parametrize("seed", range(20))
def test_admission_path_matches_independent_statement(seed):
    """The oracle's admission path equals the sorted order stated independently
    (numpy stable sort of the survival products) and Theta recomputed from the
    objective's definition at every prefix; the early-stop and global-search
    results sit on that path where their rules put them."""
    from tests._sched import assess_schedule, lengths_of_prefix
    rng = np.random.default_rng(300 + seed)
    R, g = int(rng.integers(1, 7)), int(rng.integers(1, 6))
    conf = _confidences(rng, R, g)
    T = (rng.uniform(1.0, 3.0, R * (g + 1) + 1) if seed % 2 else
         _convex_profile(rng, R * (g + 1) + 1))
    p = oracle.schedule_path(conf, T)
    order = greedy_order(conf)
    assert [(int(f // g), int(f % g) + 1) for f in p["order"]] == [(r, j) for r, j, _ in order]
    for n in range(len(order) + 1):
        ell = lengths_of_prefix(p["order"], n, R, g)
        assert int(ell.sum()) == n
        assert abs(p["theta"][n] - theta_of(ell, conf, T)) <= 1e-12 * p["theta"][n]
    for es in (True, False):
        s = oracle.schedule(conf, T, early_stop=es)
        assert assess_schedule(s["verify_len"], s["theta_best"], p, R, g, early_stop=es) == 0
        assert p["theta"][s["n_admitted"]] == s["theta_best"]


def test_assess_rejects_a_wrong_stopping_point():
    """The comparison the GPU tests use refuses a length vector one admission
    short of or past the oracle's, and one that is not a prefix of its order."""
    from tests._sched import assess_schedule, lengths_of_prefix
    rng = np.random.default_rng(5)
    R, g = 6, 4
    conf = _confidences(rng, R, g)
    N = np.arange(R * (g + 1) + 1, dtype=np.float64)
    T = 2.0 + 0.05 * N + 0.004 * N * N   # stops at 5 of 20 candidates
    p = oracle.schedule_path(conf, T)
    s = oracle.schedule(conf, T, early_stop=True)
    n = s["n_admitted"]
    assert 0 < n < len(p["order"])
    for m in (n - 1, n + 1):
        with pytest.raises(AssertionError):
            assess_schedule(lengths_of_prefix(p["order"], m, R, g), None, p, R, g)
    bad = s["verify_len"].copy()
    r = int(np.argmax(bad))
    bad[r] -= 1
    other = int(np.argmin(bad + (np.arange(R) == r) * 99))
    bad[other] += 1
    if not np.array_equal(bad, s["verify_len"]):
        with pytest.raises(AssertionError):
            assess_schedule(bad, None, p, R, g)


def test_negative_zero_confidence_acts_as_zero():
    """-0.0 is a confidence in [0, 1]; its survival product is -0.0, and a > 0
    is false for it as for +0.0: the request's candidates end there. Every
    output of both scheduler variants equals the +0.0 case's."""
    rng = np.random.default_rng(5)
    conf = rng.uniform(0.3, 1.0, (6, 5)).astype(np.float32)
    N = np.arange(6 * 6 + 1, dtype=np.float64)
    T = 2.0 + 0.05 * N
    for r, j in [(0, 0), (2, 3), (5, 4)]:
        neg, pos = conf.copy(), conf.copy()
        neg[r, j], pos[r, j] = np.float32(-0.0), np.float32(0.0)
        for stop in (True, False):
            a, b = oracle.schedule(neg, T, early_stop=stop), oracle.schedule(pos, T, early_stop=stop)
            assert a["verify_len"].tolist() == b["verify_len"].tolist()
            assert a["theta_best"] == b["theta_best"] and a["n_admitted"] == b["n_admitted"]
            assert a["verify_len"][r] <= j
        assert oracle.schedule_path(neg, T)["order"].tolist() == \
            oracle.schedule_path(pos, T)["order"].tolist()
