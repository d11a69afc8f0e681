"""Pins of the oracle's per-position acceptance probability (DSpark paper,
equation 8: P(accept x_k) = sum_v min(p_t^k(v), p_d^k(v)) = 1 - TV(p_t^k,
p_d^k)). The rates are pinned to Appendix 8's worked number, to the total
variation written with a library softmax, to special cases, and to the
verifier itself: the probability that the oracle's ratio test accepts, found
by locating each token's uniform threshold by bisection."""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "appendix8.json")


def _rates(tl, dl, T, ell=None):
    gamma = dl.shape[0]
    ell = gamma if ell is None else ell
    return oracle.acceptance(tl, dl, np.array([ell], np.int32), T, gamma,
                             target_row_off=np.array([0, tl.shape[0]], np.int64),
                             draft_row_off=np.array([0, dl.shape[0]], np.int64))[0]


def test_appendix8_acceptance_is_0_8():
    g = json.load(open(GOLDEN))
    tl = np.log(np.array([g["p_t"], g["p_t"]], np.float64))
    dl = np.log(np.array([g["p_d"]], np.float64))
    assert abs(_rates(tl, dl, 1.0)[0] - g["acceptance"]) < 1e-15


@pytest.mark.parametrize("seed", range(12))
def test_rates_equal_one_minus_total_variation(seed):
    rng = np.random.default_rng(seed)
    V, gamma, T = int(rng.integers(2, 300)), int(rng.integers(1, 6)), float(rng.uniform(0.3, 2))
    tl = rng.normal(0, 3, (gamma + 1, V))
    dl = 0.7 * tl[:gamma] + rng.normal(0, 2, (gamma, V))
    got = _rates(tl, dl, T)
    for k in range(gamma):
        pt = scipy.special.softmax(tl[k] / T)
        pd = scipy.special.softmax(dl[k] / T)
        assert abs(got[k] - (1.0 - 0.5 * np.abs(pt - pd).sum())) < 1e-13


def test_special_cases():
    V = 16
    z = np.random.default_rng(1).normal(0, 2, (2, V))
    assert abs(_rates(z, z[:1], 0.8)[0] - 1.0) < 1e-14            # identical rows
    tl = np.full((2, V), -np.inf)
    dl = np.full((1, V), -np.inf)
    tl[:, :8] = 0.0
    dl[:, 8:] = 0.0
    assert _rates(tl, dl, 1.0)[0] == 0.0                             # disjoint supports
    # temperature only scales the logits
    a = _rates(z, 0.5 * z[:1], 0.7)[0]
    b = _rates(z / 0.7, 0.5 * z[:1] / 0.7, 1.0)[0]
    assert abs(a - b) < 1e-14


def test_positions_beyond_the_verify_length():
    rng = np.random.default_rng(5)
    tl = rng.normal(size=(5, 20))
    dl = rng.normal(size=(4, 20))
    r = _rates(tl, dl, 1.0, ell=2)
    assert (r[:2] >= 0).all() and (r[2:] == -1.0).all()
    assert (_rates(tl, dl, 1.0, ell=0) == -1.0).all()


@pytest.mark.parametrize("seed", range(6))
def test_rate_is_the_verifiers_acceptance_probability(seed):
    """P(the first ratio test accepts) = sum_x p_d(x) * P(u < threshold(x)),
    with each threshold located by bisection on the oracle's own decision."""
    rng = np.random.default_rng(50 + seed)
    V, T = int(rng.integers(2, 9)), float(rng.uniform(0.5, 1.5))
    tl = rng.normal(0, 2, (2, V))
    dl = rng.normal(0, 2, (1, V))
    pd = scipy.special.softmax(dl[0] / T)
    zeros = np.zeros(2, np.int64)
    total = 0.0
    for x in range(V):
        lo, hi = 0.0, 1.0

        def accepts(u):
            out = oracle.verify(tl, dl, np.array([[x]], np.int32), np.array([1], np.int32),
                                np.array([[u, 0.5]]), T, target_row_off=zeros,
                                draft_row_off=zeros)
            return out["accepted_len"][0] == 1

        if accepts(np.nextafter(1.0, 0.0)):
            thr = 1.0
        else:
            for _ in range(60):
                mid = 0.5 * (lo + hi)
                lo, hi = (mid, hi) if accepts(mid) else (lo, mid)
            thr = hi
        total += pd[x] * thr
    assert abs(_rates(tl, dl, T)[0] - total) < 1e-12
