"""Pins of the CPU oracle against what the pages and mathematics fix.

Each test checks the oracle against something other than itself: the worked
numbers of the DSpark paper's Appendix 8, the closed form of equation 8
(acceptance = sum_v min(p_t, p_d)), losslessness (the emitted law equals the
target distribution, section 2.1) by exact interval integration, and scipy's
softmax. A mistake such as a swapped row, a dropped temperature, the wrong
residual sign or the wrong bonus row fails at least one of them (see
test_oracle_mutants.py, which plants such mistakes and checks they are caught).
"""
import json
import os

import numpy as np
import pytest
import scipy.special

import oracle
from speculative_decoding_verification_41_gb300 import workloads
from tests._law import emitted_law, first_token_law, softmax

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _logits(p):
    return np.log(np.asarray(p, np.float64))


# --------------------------------------------------------------------------
# softmax
# --------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
@pytest.mark.parametrize("dtype", ["f32", "f64", "bf16"])
def test_softmax_matches_scipy(T, dtype):
    rng = np.random.default_rng(3)
    z = (3 * rng.standard_normal(1000)).astype(np.float64)
    if dtype == "f32":
        z_in = z.astype(np.float32)
        z_ref = z_in.astype(np.float64)
    elif dtype == "bf16":
        bits = (z.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
        z_in = bits
        z_ref = (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    else:
        z_in, z_ref = z, z
    p = oracle.softmax_row(z_in, T)
    np.testing.assert_allclose(p, scipy.special.softmax(z_ref / T), rtol=1e-13, atol=1e-300)


def test_softmax_special_cases():
    V = 37
    np.testing.assert_allclose(oracle.softmax_row(np.full(V, 1.25), 0.7), np.full(V, 1.0 / V),
                               rtol=1e-15)
    z = np.zeros(V)
    z[5] = 60.0
    p = oracle.softmax_row(z, 1.0)
    assert abs(p[5] - 1.0 / (1.0 + (V - 1) * np.exp(-60.0))) < 1e-15
    # temperature scaling: p_T(z) = p_1(z / T)
    rng = np.random.default_rng(1)
    z = rng.standard_normal(50) * 4
    np.testing.assert_allclose(oracle.softmax_row(z, 0.35), oracle.softmax_row(z / 0.35, 1.0),
                               rtol=1e-13)
    # masked entries (-inf) carry no mass
    z[::3] = -np.inf
    p = oracle.softmax_row(z, 1.0)
    assert np.all(p[::3] == 0.0) and abs(p.sum() - 1) < 1e-14


# --------------------------------------------------------------------------
# Appendix 8 worked example
# --------------------------------------------------------------------------
def test_appendix8_verification():
    g = json.load(open(os.path.join(GOLDEN, "appendix8.json")))
    pt, pd = g["p_t"], g["p_d"]
    tl = _logits([pt, pt])          # row 1: p_t; row 2 (bonus) unused here
    dl = _logits([pd])
    law = emitted_law(tl, dl, gamma=1, ell=1, T=1.0)
    # acceptance probability at position 1 = sum_x min(p_t, p_d) = 0.8
    acc = sum(w for seq, w in law.items() if len(seq) == 2)
    assert abs(acc - g["acceptance"]) < 1e-12
    # lossless: the first emitted token is distributed as p_t = (0.7, 0.3)
    np.testing.assert_allclose(first_token_law(law, 2), g["lossless_first_token_law"], atol=1e-12)
    # the residual max(0, p_t - p_d) = (0.2, 0) always yields token A after a rejection of B
    for ures in (0.0, 0.3, 0.999999):
        out = oracle.verify(tl, dl, [[1]], [1], [[0.99, ures]], 1.0)
        assert out["accepted_len"][0] == 0 and out["emitted"][0, 0] == 0


def test_appendix8_retrospective_scheduler_is_biased():
    """The worked counterexample: with the early-stopping break removed the
    admission of x_1 depends on x_1 and the first token law becomes
    (0.85, 0.15); with the break it stays (0.7, 0.3)."""
    g = json.load(open(os.path.join(GOLDEN, "appendix8.json")))
    sps = g["sps"]                                # SPS(1), SPS(2), SPS(3)
    T = np.array([1e300, 1 / sps[0], 1 / sps[1], 1 / sps[2]])  # T(N) = 1/SPS(N), N = 0..3
    pt, pd = g["p_t"], g["p_d"]
    tl = _logits([pt, [0.5, 0.5], [0.5, 0.5]])
    dl = _logits([pd, [0.5, 0.5]])
    c2 = {0: g["case1_c2"], 1: g["case2_c2"]}     # x_1 = A -> 0.9, x_1 = B -> 0
    for early_stop, expect in ((False, g["retrospective_first_token_law"]),
                               (True, g["lossless_first_token_law"])):
        p = np.zeros(2)
        for x1 in (0, 1):                         # x_1 ~ p_d = (0.5, 0.5)
            conf = np.array([[g["a1"], c2[x1]]], np.float32)
            ell = int(oracle.schedule(conf, T, early_stop=early_stop)["verify_len"][0])
            law = emitted_law(tl, dl, gamma=2, ell=ell, T=1.0, fixed_x=(x1, 0))
            p += pd[x1] * first_token_law(law, 2)
        np.testing.assert_allclose(p, expect, atol=1e-12)


def test_appendix8_scheduler_numbers():
    g = json.load(open(os.path.join(GOLDEN, "appendix8.json")))
    sps = g["sps"]
    T = np.array([1e300, 1 / sps[0], 1 / sps[1], 1 / sps[2]])
    # early stop: Theta_0 = 1.0, Theta_1 = 0.9 -> stop, l = 0
    for c2 in (g["case1_c2"], g["case2_c2"]):
        s = oracle.schedule(np.array([[g["a1"], c2]], np.float32), T, early_stop=True)
        assert s["verify_len"][0] == 0
        assert abs(s["theta_best"] - g["theta0"]) < 1e-12
    # no break (global search): case 1 -> l = 2, Theta = 1.134; case 2 -> l = 0, Theta = 1.0
    s = oracle.schedule(np.array([[g["a1"], g["case1_c2"]]], np.float32), T, early_stop=False)
    assert s["verify_len"][0] == 2
    assert abs(s["theta_best"] - g["case1_theta2"]) < 1e-7   # a's are float32 inputs
    s = oracle.schedule(np.array([[g["a1"], g["case2_c2"]]], np.float32), T, early_stop=False)
    assert s["verify_len"][0] == 0 and abs(s["theta_best"] - g["theta0"]) < 1e-12


# --------------------------------------------------------------------------
# closed form and losslessness by exact enumeration
# --------------------------------------------------------------------------
@pytest.mark.parametrize("V,T,seed", [(2, 1.0, 0), (3, 0.7, 1), (5, 1.0, 2), (8, 1.3, 3)])
def test_acceptance_closed_form_and_lossless_gamma1(V, T, seed):
    rng = np.random.default_rng(seed)
    tl = 2 * rng.standard_normal((2, V))
    dl = 0.6 * tl[:1] + rng.standard_normal((1, V))
    law = emitted_law(tl, dl, gamma=1, ell=1, T=T)
    pt1, pd1 = softmax(tl[0], T), softmax(dl[0], T)
    acc = sum(w for seq, w in law.items() if len(seq) == 2)
    assert abs(acc - np.minimum(pt1, pd1).sum()) < 1e-12                 # equation 8
    assert abs(acc - (1 - 0.5 * np.abs(pt1 - pd1).sum())) < 1e-12
    np.testing.assert_allclose(first_token_law(law, V), pt1, atol=1e-12)  # lossless
    # after acceptance of all drafts the bonus token comes from target row 2
    cont = np.zeros(V)
    for seq, w in law.items():
        if len(seq) == 2:
            cont[seq[1]] += w
    np.testing.assert_allclose(cont / acc, softmax(tl[1], T), atol=1e-12)


@pytest.mark.parametrize("V,ell,T,seed", [(3, 2, 1.0, 4), (4, 2, 0.7, 5), (5, 1, 1.0, 6),
                                          (6, 0, 0.9, 7)])
def test_lossless_gamma2(V, ell, T, seed):
    """gamma = 2: the first token ~ p_t^1; given x_1 was accepted the next token
    ~ p_t^2 (tested draft or bonus); with ell = 0 a fresh token from p_t^1."""
    rng = np.random.default_rng(seed)
    tl = 2 * rng.standard_normal((3, V))
    dl = 0.7 * tl[:2] + rng.standard_normal((2, V))
    law = emitted_law(tl, dl, gamma=2, ell=ell, T=T)
    assert abs(sum(law.values()) - 1.0) < 1e-12
    np.testing.assert_allclose(first_token_law(law, V), softmax(tl[0], T), atol=1e-12)
    if ell >= 1:
        pt1, pd1 = softmax(tl[0], T), softmax(dl[0], T)
        joint = np.zeros((V, V))
        for seq, w in law.items():
            if len(seq) >= 2:
                joint[seq[0], seq[1]] += w
        # P(x_1 = v accepted) = min(p_t^1(v), p_d^1(v))
        np.testing.assert_allclose(joint.sum(1), np.minimum(pt1, pd1), atol=1e-12)
        cond = joint / np.maximum(joint.sum(1, keepdims=True), 1e-300)
        for v in range(V):
            if joint[v].sum() > 0:
                np.testing.assert_allclose(cond[v], softmax(tl[1], T), atol=1e-11)
    if ell == 2:
        trip = np.zeros(V)
        tot = 0.0
        for seq, w in law.items():
            if len(seq) == 3:
                trip[seq[2]] += w
                tot += w
        np.testing.assert_allclose(trip / tot, softmax(tl[2], T), atol=1e-11)


def test_monte_carlo_acceptance_rate():
    """Empirical acceptance at position 1 with Philox uniforms agrees with the
    closed form sum min(p_t, p_d) within 4 sigma."""
    V, n, T = 400, 20000, 0.8
    rng = np.random.default_rng(11)
    zt = 2 * rng.standard_normal((1, V))
    zd = 0.7 * zt + rng.standard_normal((1, V))
    pd = softmax(zd[0], T)
    cdf = np.cumsum(pd)
    us = workloads.philox_uniforms(5, workloads.PURPOSE_DRAFT_SAMPLING, n).astype(np.float64)
    x = np.minimum(np.searchsorted(cdf, us * cdf[-1], side="right"), V - 1).astype(np.int32)
    u = workloads.philox_uniforms(5, workloads.PURPOSE_VERIFY_UNIFORMS, 2 * n).reshape(n, 2)
    zeros = np.zeros(n + 1, np.int64)
    out = oracle.verify(np.vstack([zt, zt]), zd, x[:, None], np.ones(n, np.int32), u, T,
                        target_row_off=zeros, draft_row_off=zeros)
    rate = out["accepted_len"].mean()
    c = np.minimum(softmax(zt[0], T), pd).sum()
    assert abs(rate - c) < 4 * np.sqrt(c * (1 - c) / n)
    # first emitted token ~ p_t (chi-square, generous bound)
    counts = np.bincount(out["emitted"][:, 0], minlength=V)
    pt = softmax(zt[0], T)
    big = pt * n > 20
    chi2 = ((counts[big] - n * pt[big]) ** 2 / (n * pt[big])).sum()
    assert chi2 < big.sum() + 6 * np.sqrt(2 * big.sum())


# --------------------------------------------------------------------------
# tiny workload: structure of the outputs
# --------------------------------------------------------------------------
def test_tiny_workload_structure():
    w = workloads.make_tiny("cpu")
    out = oracle.verify(w.target_logits.numpy(), w.draft_logits.numpy(), w.draft_tokens.numpy(),
                        w.verify_len.numpy(), w.uniforms.numpy(), w.temperature)
    B, g = w.B, w.gamma
    x = w.draft_tokens.numpy()
    u = w.uniforms.numpy().astype(np.float64)
    for r in range(B):
        m = out["accepted_len"][r]
        assert 0 <= m <= g
        assert np.all(out["emitted"][r, :m] == x[r, :m])
        assert 0 <= out["emitted"][r, m] < w.V
        assert np.all(out["emitted"][r, m + 1:] == -1)
        ratios = out["probs"][r, :, 0] / out["probs"][r, :, 1]
        # the first m tests passed, test m+1 (if any) failed
        assert np.all(u[r, :m] < ratios[:m])
        if m < g:
            assert not u[r, m] < ratios[m]
        # probabilities agree with scipy's softmax of the rows
        zt = w.target_logits.numpy().reshape(B, g + 1, -1)[r]
        zd = w.draft_logits.numpy().reshape(B, g, -1)[r]
        for k in range(g):
            assert abs(out["probs"][r, k, 0] - softmax(zt[k], 1.0)[x[r, k]]) < 1e-14
            assert abs(out["probs"][r, k, 1] - softmax(zd[k], 1.0)[x[r, k]]) < 1e-14


def test_invalid_inputs_rejected():
    tl = np.zeros((2, 4), np.float32)
    dl = np.zeros((1, 4), np.float32)
    with pytest.raises(oracle.OracleError):
        oracle.verify(tl, dl, [[7]], [1], [[0.5, 0.5]], 1.0)          # token out of range
    with pytest.raises(oracle.OracleError):
        oracle.verify(tl, dl, [[1]], [2], [[0.5, 0.5]], 1.0)          # verify_len > gamma
    with pytest.raises(oracle.OracleError):
        oracle.verify(tl, dl, [[1]], [1], [[0.5, 0.5]], 0.0)          # temperature
    with pytest.raises(oracle.OracleError):
        oracle.schedule(np.array([[0.5, 1.5]], np.float32), np.ones(4))  # confidence > 1
    with pytest.raises(oracle.OracleError):
        oracle.schedule(np.array([[0.5, 0.5]], np.float32), np.ones(3))  # profile too short
