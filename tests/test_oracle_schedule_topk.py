"""Pins of the oracle's production scheduler (DSpark paper, section 5.2,
"Hardware-Aware Prefix Scheduler in Practice"): the capacity K from the
unconstrained global search, and the dynamic top-K admission of the current
candidates.

The admission is pinned by brute force over every admissible length vector
(the K admitted tokens with the largest total survival), by closed forms at the
edges, by a hand-worked tie example, and by Appendix 8's worked numbers."""
import itertools
import json
import os

import numpy as np
import pytest

import oracle
from tests._sched import survival

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "appendix8.json")


def _distinct_confidences(rng, R, g):
    c = rng.uniform(0.05, 0.999, (R, g)).astype(np.float32)
    c[rng.uniform(size=(R, g)) < 0.1] = 0.0   # excluded tails
    return c


def _caps(conf):
    a = survival(conf)
    return [int((a[r] > 0).sum()) for r in range(a.shape[0])]


@pytest.mark.parametrize("seed", range(30))
def test_topk_admits_the_k_tokens_of_largest_survival(seed):
    """With distinct survival values the top-K admission is the unique length
    vector with sum K (each request a prefix of its positive candidates) whose
    admitted survival probabilities have the largest total."""
    rng = np.random.default_rng(100 + seed)
    R, g = int(rng.integers(1, 4)), int(rng.integers(1, 5))
    conf = _distinct_confidences(rng, R, g)
    a = survival(conf)
    caps = _caps(conf)
    nE = sum(caps)
    for K in range(0, nE + 1):
        best, arg = -1.0, None
        for ell in itertools.product(*[range(c + 1) for c in caps]):
            if sum(ell) != K:
                continue
            tot = sum(a[r, :ell[r]].sum() for r in range(R))
            if tot > best:
                best, arg = tot, ell
        got = oracle.schedule_topk(conf, K)
        assert tuple(int(x) for x in got["verify_len"]) == arg, (K, got, arg)
        assert got["n_admitted"] == K


def test_topk_edges_and_totals():
    rng = np.random.default_rng(7)
    conf = _distinct_confidences(rng, 6, 5)
    caps = _caps(conf)
    nE = sum(caps)
    zero = oracle.schedule_topk(conf, 0)
    assert not zero["verify_len"].any() and zero["n_admitted"] == 0
    for K in (nE, nE + 1, 10 ** 6):   # capacity at or above |E|: every candidate
        full = oracle.schedule_topk(conf, K)
        assert list(full["verify_len"]) == caps and full["n_admitted"] == nE
    prev = np.zeros(6, np.int32)
    for K in range(nE + 1):
        ell = oracle.schedule_topk(conf, K)["verify_len"]
        assert int(ell.sum()) == K
        assert (ell >= prev).all()      # a larger capacity never drops a token
        prev = ell


def test_topk_equal_survival_follows_flattened_order():
    """Two requests with a = (0.5, 0.5) each: the order is (0,1), (0,2), (1,1),
    (1,2), so capacities 1..4 give (1,0), (2,0), (2,1), (2,2)."""
    conf = np.array([[0.5, 1.0], [0.5, 1.0]], np.float32)
    want = {1: [1, 0], 2: [2, 0], 3: [2, 1], 4: [2, 2]}
    for K, ell in want.items():
        assert list(oracle.schedule_topk(conf, K)["verify_len"]) == ell


def test_topk_rejects_bad_inputs():
    conf = np.array([[0.5, 1.5]], np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.schedule_topk(conf, 1)
    with pytest.raises(oracle.OracleError):
        oracle.schedule_topk(np.array([[0.5]], np.float32), -1)


def test_production_pipeline_on_appendix8():
    """Appendix 8, case 1 (c2 = 0.9): the global search admits both draft
    tokens (Theta = 1.134 against 1.0 and 0.9), so the capacity is 2 and the
    top-K admission of the same confidences verifies both."""
    g = json.load(open(GOLDEN))
    conf = np.array([[g["a1"], g["case1_c2"]]], np.float32)
    sps = np.array(g["sps"], np.float64)
    T = np.concatenate([[1.0], 1.0 / sps])   # T(N) = 1/SPS(N) for N = 1..3
    s = oracle.schedule(conf, T, early_stop=False)
    assert s["n_admitted"] == 2
    assert abs(s["theta_best"] - g["case1_theta2"]) < 1e-6
    assert list(oracle.schedule_topk(conf, s["n_admitted"])["verify_len"]) == [2]
    # the causal scheduler stops after Theta1 = 0.9 <= Theta0 = 1.0
    assert list(oracle.schedule(conf, T, early_stop=True)["verify_len"]) == [0]


@pytest.mark.parametrize("seed", range(10))
def test_topk_at_global_capacity_is_the_global_schedule(seed):
    """Admitting the global search's capacity from the same confidences gives
    the global search's lengths (both take a prefix of the same order)."""
    rng = np.random.default_rng(500 + seed)
    R, g = int(rng.integers(2, 8)), int(rng.integers(2, 8))
    conf = rng.uniform(0, 1, (R, g)).astype(np.float32)
    N = np.arange(R * (g + 1) + 1, dtype=np.float64)
    T = 2.0 + 0.05 * N + 0.3 * (N % 3 == 0)        # jagged step-time profile
    s = oracle.schedule(conf, T, early_stop=False)
    t = oracle.schedule_topk(conf, s["n_admitted"])
    assert (t["verify_len"] == s["verify_len"]).all()
