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


def chisq_pvalue(samples, p, minimum=5.0):
    """Chi-square p-value of integer samples against the law p (cells whose
    expected count is below `minimum` pooled into one)."""
    from scipy import stats
    n = len(samples)
    counts = np.bincount(np.asarray(samples, np.int64), minlength=len(p))
    keep = np.asarray(p) * n >= minimum
    obs = np.append(counts[keep], counts[~keep].sum())
    exp = np.append(np.asarray(p)[keep] * n, np.asarray(p)[~keep].sum() * n)
    if exp[-1] == 0:
        obs, exp = obs[:-1], exp[:-1]
    return float(stats.chisquare(obs, exp).pvalue)


def one_position_trials(V, T, seed, n):
    """Trials of one request with a block of one position: bf16 target rows 1
    and 2, draft row 1, n draft tokens drawn from p_d by inverse CDF and n
    uniform pairs, all seeded. Returns (zt [2, V] and zd [V] as bf16 bit
    patterns, x [n], uniforms [n, 2], pt1, pt2, pd1 in float64)."""
    import torch
    from scipy import special
    from speculative_decoding_verification_41_gb300 import workloads
    rng = np.random.default_rng(seed)
    zt = torch.tensor(2.0 * rng.standard_normal((2, V)), dtype=torch.float32).to(torch.bfloat16)
    zd = torch.tensor(0.6 * zt[0].float().numpy() + rng.standard_normal(V),
                      dtype=torch.float32).to(torch.bfloat16)
    pt1 = special.softmax(zt[0].double().numpy() / T)
    pt2 = special.softmax(zt[1].double().numpy() / T)
    pd1 = special.softmax(zd.double().numpy() / T)
    u_draft = workloads.philox_uniforms(seed, workloads.PURPOSE_DRAFT_SAMPLING, n).astype(np.float64)
    x = np.minimum(np.searchsorted(np.cumsum(pd1), u_draft, side="right"), V - 1).astype(np.int32)
    uni = workloads.philox_uniforms(seed, workloads.PURPOSE_VERIFY_UNIFORMS, 2 * n).reshape(n, 2)
    bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    return bits(zt), bits(zd), x, uni, pt1, pt2, pd1


def law_pvalues(acc, em, x, pt1, pt2, pd1):
    """The three checks of a block of one position: the acceptance rate's
    distance from sum min(p_t, p_d) in standard deviations, and the chi-square
    p-values of the first emitted token against p_t of row 1 and of the bonus
    (after an accepted token) against p_t of row 2."""
    acc = np.asarray(acc)
    em = np.asarray(em)
    n = len(acc)
    alpha = np.minimum(pt1, pd1).sum()
    z = abs(acc.mean() - alpha) / np.sqrt(alpha * (1 - alpha) / n)
    return z, chisq_pvalue(em[:, 0], pt1), chisq_pvalue(em[acc == 1, 1], pt2)
