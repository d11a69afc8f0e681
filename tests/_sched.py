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
