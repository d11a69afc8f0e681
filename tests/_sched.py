"""Independent statements of the prefix scheduler's objective, for pins.

The objective of the DSpark paper, section 3.2.2: for verify lengths l_r,
B = sum_r (1 + l_r), tau = sum_r (1 + sum_{j<=l_r} a_{r,j}) with
a_{r,j} = prod_{i<=j} c_{r,i}, and Theta = tau * SPS(B), SPS(B) = 1 / T(B).
"""
import itertools

import numpy as np


def survival(conf):
    return np.cumprod(np.asarray(conf, np.float64), axis=1)


def theta_of(ell, conf, T):
    a = survival(conf)
    R = a.shape[0]
    tau = R + sum(a[r, :ell[r]].sum() for r in range(R))
    return tau / T[R + int(np.sum(ell))]


def exhaustive_best(conf, T):
    """max of Theta over every length vector whose admitted tokens all have
    a > 0 (the candidate space E of Algorithm 1), by brute force."""
    a = survival(conf)
    R, g = a.shape
    cap = [int((a[r] > 0).sum()) for r in range(R)]   # a is non-increasing in j
    best, arg = -np.inf, None
    for ell in itertools.product(*[range(c + 1) for c in cap]):
        th = theta_of(ell, conf, T)
        if th > best:
            best, arg = th, ell
    return best, arg


def greedy_order(conf):
    """Candidates (r, j) with a > 0 sorted by a descending, ties by flat index."""
    a = survival(conf)
    R, g = a.shape
    flat = a.reshape(-1)
    idx = [i for i in np.argsort(-flat, kind="stable") if flat[i] > 0]
    return [(i // g, i % g + 1, flat[i]) for i in idx]


TIE_REL = 1e-9   # the oracle's scheduler near-tie window (relative)


def lengths_of_prefix(order, n, R, gamma):
    """l_r = the largest j among the first n candidates of request r (0 if none)."""
    ell = np.zeros(R, np.int64)
    for f in np.asarray(order[:n], np.int64):
        r, j = int(f // gamma), int(f % gamma) + 1
        ell[r] = max(ell[r], j)
    return ell


def assess_schedule(ell, theta, path, R, gamma, early_stop=True):
    """Assess another implementation's scheduler output against the oracle's
    admission path (oracle.schedule_path). Every request's length must be the
    one its admitted count n = sum(l) gives along the oracle's order; n itself
    must be where the oracle's rule stops, except where the comparison that
    decides it lies within the 1e-9 near-tie window.

    early_stop=True (Algorithm 1): admissions 1..n each improve Theta, and
    admission n+1 (if any) does not. early_stop=False (the global search): n
    is the first maximum of Theta over the path.

    Returns the number of admissions whose decision was excused as a near tie
    (0 when the result is exactly the oracle's). Raises AssertionError
    otherwise."""
    th = np.asarray(path["theta"], np.float64)
    nE = len(th) - 1
    ell = np.asarray(ell, np.int64)
    n = int(ell.sum())
    assert 0 <= n <= nE, (n, nE)
    np.testing.assert_array_equal(ell, lengths_of_prefix(path["order"], n, R, gamma))

    def tie(x, y):
        return abs(x - y) <= TIE_REL * max(abs(x), abs(y))

    excused = 0
    if early_stop:
        for i in range(1, n + 1):          # admitted: each improved on the one before
            if not th[i] > th[i - 1]:
                assert tie(th[i], th[i - 1]), f"admission {i} does not improve Theta"
                excused += 1
        if n < nE and th[n + 1] > th[n]:   # stopped: the next one must not improve
            assert tie(th[n + 1], th[n]), f"stopped at {n} before an improving admission"
            excused += 1
    else:
        for i in range(nE + 1):
            better = th[i] > th[n] if i > n else th[i] >= th[n]
            if i != n and better:
                assert tie(th[i], th[n]), f"Theta({i}) beats the chosen Theta({n})"
                excused += 1
    if theta is not None:
        assert abs(theta - th[n]) <= 1e-12 * abs(th[n]), (theta, th[n])
    return excused
