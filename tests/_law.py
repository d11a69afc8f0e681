"""Exact law of the oracle's emitted tokens, by interval integration.

The verifier's output is a deterministic function of its uniforms: each ratio
test is a threshold on its own uniform, and the resampled token is a
non-decreasing step function of the resample uniform. This helper treats the
oracle as a black box, locates every threshold and step by bisection on the
uniforms (double precision, so to ~1e-16), and sums the interval lengths,
weighting each draft-token combination by its probability under the drafter.
The result is the exact law of the emitted sequence (up to rounding), which the
tests compare with the target distribution (losslessness, DSpark paper section
2.1) and with closed forms.
"""
from __future__ import annotations

import itertools

import numpy as np
import scipy.special

import oracle

U_MAX = np.nextafter(1.0, 0.0)  # largest uniform below 1


def softmax(z, T):
    return scipy.special.softmax(np.asarray(z, np.float64) / T)


class Probe:
    """Batched calls of oracle.verify on one request's rows (all probes share
    the rows through zero offsets)."""

    def __init__(self, tl, dl, gamma, ell, T, lib=None):
        self.tl = np.ascontiguousarray(tl, np.float64)  # [gamma+1, V]
        self.dl = np.ascontiguousarray(dl, np.float64)  # [gamma, V]
        self.gamma, self.ell, self.T = gamma, ell, T
        self.lib = lib
        self.calls = 0

    def run(self, x, u):
        """x: [n, gamma] draft tokens, u: [n, gamma+1] uniforms."""
        n = x.shape[0]
        self.calls += 1
        zeros = np.zeros(n + 1, np.int64)
        return oracle.verify(self.tl, self.dl, x, np.full(n, self.ell, np.int32), u, self.T,
                             target_row_off=zeros, draft_row_off=zeros, lib=self.lib)


def _bisect(f, lo, hi, iters=60):
    """Vectorised bisection: f(u) -> bool array, True at lo, False at hi.
    Returns the boundary (largest True within precision)."""
    for _ in range(iters):
        mid = 0.5 * (lo + hi)
        t = f(mid)
        lo = np.where(t, mid, lo)
        hi = np.where(t, hi, mid)
    return hi


def emitted_law(tl, dl, gamma, ell, T, fixed_x=None, lib=None):
    """Exact law {tuple(emitted tokens): probability} of one verification step
    with verify length ell, draft tokens x_k ~ softmax(dl[k-1]/T); with
    fixed_x (a tuple of ell tokens) the law conditional on those draft tokens."""
    V = tl.shape[1]
    probe = Probe(tl, dl, gamma, ell, T, lib=lib)
    pd = [softmax(dl[k], T) for k in range(gamma)]
    if fixed_x is not None:
        combos = [tuple(fixed_x[:ell])]
    else:
        combos = [c for c in itertools.product(range(V), repeat=ell)
                  if np.prod([pd[k][c[k]] for k in range(ell)]) > 0] if ell else [()]
    X = np.zeros((len(combos), gamma), np.int32)
    for i, c in enumerate(combos):
        X[i, :ell] = c
    wx = (np.ones(len(combos)) if fixed_x is not None else
          np.array([np.prod([pd[k][c[k]] for k in range(ell)]) for c in combos]))

    # acceptance threshold t_k(x): accept at k iff u_k < t_k (earlier positions forced to accept)
    thr = np.ones((len(combos), max(ell, 1)))
    for k in range(ell):
        def accepted(uk, k=k):
            u = np.zeros((len(combos), gamma + 1))
            u[:, k] = uk
            return probe.run(X, u)["accepted_len"] >= k + 1
        always = accepted(np.full(len(combos), U_MAX))
        b = _bisect(accepted, np.zeros(len(combos)), np.full(len(combos), U_MAX))
        thr[:, k] = np.where(always, 1.0, b)

    law: dict = {}
    for m in range(ell + 1):
        # probability of stopping with exactly m accepted
        mass = wx.copy()
        for k in range(m):
            mass *= np.minimum(thr[:, k], 1.0)
        if m < ell:
            mass *= 1.0 - np.minimum(thr[:, m], 1.0)
        live = np.nonzero(mass > 0)[0]
        if live.size == 0:
            continue
        Xl = X[live]
        u_base = np.zeros((live.size, gamma + 1))
        if m < ell:
            # a uniform inside the rejection interval of position m+1
            u_base[:, m] = 0.5 * (thr[live, m] + 1.0)

        def y_at(ur):
            u = u_base.copy()
            u[:, gamma] = ur
            out = probe.run(Xl, u)
            assert np.all(out["accepted_len"] == m)
            return out["emitted"][np.arange(live.size), m]

        lo = np.zeros(live.size)
        active = np.ones(live.size, bool)
        while active.any():
            y_lo = y_at(lo)
            y_hi = y_at(np.full(live.size, U_MAX))
            done = active & (y_hi == y_lo)
            hi = np.where(done, 1.0, 0.0)
            need = active & ~done
            if need.any():
                b = _bisect(lambda uu: y_at(uu) == y_lo, lo.copy(), np.full(live.size, U_MAX))
                hi = np.where(need, b, hi)
            for i in np.nonzero(active)[0]:
                seq = tuple(int(t) for t in Xl[i, :m]) + (int(y_lo[i]),)
                law[seq] = law.get(seq, 0.0) + mass[live[i]] * (hi[i] - lo[i])
            lo = np.where(need, hi, lo)
            active = need
    return law


def first_token_law(law, V):
    p = np.zeros(V)
    for seq, w in law.items():
        p[seq[0]] += w
    return p
