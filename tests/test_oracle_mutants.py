"""Plant plausible mistakes in a copy of the oracle and check that the pins
catch every one of them (and pass on the unmodified source).

Each mutant replaces one exact snippet of oracle/dspark_oracle.c, compiles the
copy into a temporary library and runs the pin checks against it on the CPU.
"""
import os

import numpy as np
import pytest
import scipy.special

import oracle
from tests._law import emitted_law, first_token_law, softmax
from tests._sched import exhaustive_best, greedy_order, lengths_of_prefix, theta_of

SRC = os.path.join(os.path.dirname(oracle.__file__), "dspark_oracle.c")

MUTANTS = {
    "residual_sign": ("q[v] = pt[v] - pd[v] > 0.0 ? pt[v] - pd[v] : 0.0;",
                      "q[v] = pd[v] - pt[v] > 0.0 ? pd[v] - pt[v] : 0.0;"),
    "residual_row_off_by_one": ("if ((rc = softmax_row(tl, dtype, trow0 + kstar - 1, V, T, pt))) return rc;",
                                "if ((rc = softmax_row(tl, dtype, trow0 + kstar, V, T, pt))) return rc;"),
    "bonus_row_off_by_one": ("if ((rc = softmax_row(tl, dtype, trow0 + ell, V, T, pt))) return rc;",
                             "if ((rc = softmax_row(tl, dtype, trow0 + (ell ? ell - 1 : 0), V, T, pt))) return rc;"),
    "draft_temperature_dropped": ("if ((rc = softmax_row(dl, dtype, drow0 + k - 1, V, T, pd))) return rc;",
                                  "if ((rc = softmax_row(dl, dtype, drow0 + k - 1, V, 1.0, pd))) return rc;"),
    "ratio_inverted": ("ratio = ptx / pdx;", "ratio = pdx / ptx;"),
    "no_truncation": ("if (!(u[k - 1] < ratio)) break;", "if (!(u[k - 1] < ratio)) continue;"),
    "temperature_multiplies": ("p[v] = exp(logit_at(base, dtype, off + v) / T - M);",
                               "p[v] = exp(logit_at(base, dtype, off + v) * T - M);"),
    "residual_uses_target_only": ("y = inverse_cdf(q, V, Z, u[gamma], &flags[gamma]);",
                                  "y = inverse_cdf(pt, V, 1.0, u[gamma], &flags[gamma]);"),
    "sort_ascending": ("if (x->a > y->a) return -1;\n  if (x->a < y->a) return 1;",
                       "if (x->a > y->a) return 1;\n  if (x->a < y->a) return -1;"),
    "survival_not_cumulative": ("prod *= (double)confidences[(int64_t)r * gamma + j];",
                                "prod = (double)confidences[(int64_t)r * gamma + j];"),
    # the scheduler and its written-out admission path take the same steps, so
    # these two mistakes are planted in both (two occurrences each)
    "batch_not_counted": ("    Bsz += 1;\n", "\n", 2),
    "anchor_token_dropped": ("double tau = (double)R;", "double tau = 0.0;", 2),
    "path_theta_not_cumulative": ("theta[i + 1] = tau / step_time[Bsz];",
                                  "theta[i + 1] = (R + E[i].a) / step_time[Bsz];"),
    "path_order_off_by_one": ("order[i] = E[i].flat;", "order[i] = E[i].flat + 1;"),
    "draft_embedding_from_w2": ("a[j] = bf16_to_double(W1[(int64_t)prev * r + j]);",
                                "a[j] = bf16_to_double(W2t[(int64_t)prev * r + j]);"),
    "draft_projection_from_w1": ("const uint16_t* col = W2t + v * r;",
                                 "const uint16_t* col = W1 + v * r;"),
    "draft_prev_stays_anchor": ("    prev = y;\n", "    prev = x0;\n"),
    "draft_base_row_off_by_one": ("const uint16_t* Uk = U + (int64_t)k * V;",
                                  "const uint16_t* Uk = U + (int64_t)(k ? k - 1 : 0) * V;"),
    "draft_no_binary32_step": ("const float s = (float)(bf16_to_double(Uk[v]) + bias);",
                               "const double s = bf16_to_double(Uk[v]) + bias;"),
    "draft_round_half_up": ("const double q = rint(n);", "const double q = floor(n + 0.5);"),
    "draft_temperature_dropped": ("w[v] = exp(L[v] / T - M);", "w[v] = exp(L[v] - M / T);"),
    "draft_first_uniform_reused": ("const double uk = (double)u[k];",
                                   "const double uk = (double)u[0];"),
}


def check_softmax(lib):
    rng = np.random.default_rng(0)
    z = 3 * rng.standard_normal(64)
    for T in (0.7, 1.0):
        np.testing.assert_allclose(oracle.softmax_row(z, T, lib=lib),
                                   scipy.special.softmax(z / T), rtol=1e-12)


def check_verify(lib):
    rng = np.random.default_rng(5)
    V, T = 4, 0.7
    tl = 2 * rng.standard_normal((3, V))
    dl = 0.7 * tl[:2] + rng.standard_normal((2, V))
    for ell in (0, 1, 2):
        law = emitted_law(tl, dl, gamma=2, ell=ell, T=T, lib=lib)
        assert abs(sum(law.values()) - 1) < 1e-12
        np.testing.assert_allclose(first_token_law(law, V), softmax(tl[0], T), atol=1e-12)
        for depth in range(1, ell + 1):
            cond = np.zeros(V)
            for seq, w in law.items():
                if len(seq) > depth:
                    cond[seq[depth]] += w
            np.testing.assert_allclose(cond / cond.sum(), softmax(tl[depth], T), atol=1e-11)
    # equation 8: acceptance probability at position 1
    law = emitted_law(tl, dl, gamma=2, ell=1, T=T, lib=lib)
    acc = sum(w for seq, w in law.items() if len(seq) == 2)
    assert abs(acc - np.minimum(softmax(tl[0], T), softmax(dl[0], T)).sum()) < 1e-12


def check_schedule(lib):
    sps = (1.0, 0.5, 0.45)
    T = np.array([1e300, 1 / sps[0], 1 / sps[1], 1 / sps[2]])
    s = oracle.schedule(np.array([[0.8, 0.9]], np.float32), T, early_stop=False, lib=lib)
    assert s["verify_len"][0] == 2 and abs(s["theta_best"] - 1.134) < 1e-7
    s = oracle.schedule(np.array([[0.8, 0.9]], np.float32), T, early_stop=True, lib=lib)
    assert s["verify_len"][0] == 0 and abs(s["theta_best"] - 1.0) < 1e-12
    for seed in range(12):
        rng = np.random.default_rng(seed)
        R, g = int(rng.integers(2, 4)), int(rng.integers(2, 5))
        conf = rng.uniform(0, 1, (R, g)).astype(np.float32)
        n = R * (g + 1) + 1
        N = np.arange(n, dtype=np.float64)
        T = rng.uniform(1, 5) + rng.uniform(0.05, 1.0) * N + rng.uniform(0, 0.2) * N * N
        s = oracle.schedule(conf, T, early_stop=True, lib=lib)
        best, _ = exhaustive_best(conf, T)
        assert abs(s["theta_best"] - best) <= 1e-12 * best
        # the written-out admission path: the independent order, and Theta of
        # every prefix from the objective's definition
        p = oracle.schedule_path(conf, T, lib=lib)
        order = greedy_order(conf)
        assert [(int(f // g), int(f % g) + 1) for f in p["order"]] == [(r, j) for r, j, _ in order]
        for k in range(len(order) + 1):
            ell = lengths_of_prefix(p["order"], k, R, g)
            assert abs(p["theta"][k] - theta_of(ell, conf, T)) <= 1e-12 * p["theta"][k]


def _bits(vals):
    return (np.asarray(vals, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def check_draft(lib):
    """Compact forms of the drafter pins (tests/test_oracle_markov_draft.py)."""
    V, r = 16, 64
    # successor chain: each token forces succ(a) = (5a + 3) mod 16
    succ = [(5 * a + 3) % V for a in range(V)]
    W1 = np.zeros((V, r), np.uint16)
    W2t = np.zeros((V, r), np.uint16)
    for a in range(V):
        W1[a, 4 * a:4 * a + 4] = _bits([0.5] * 4)
        W2t[succ[a], 4 * a:4 * a + 4] = _bits([0.5] * 4)
    g = 6
    U = np.zeros((2, g, V), np.uint16)
    u = np.full((2, g), 0.5, np.float32)
    out = oracle.markov_draft(U, W1, W2t, np.array([3, 11], np.int32), u, 0.05, lib=lib)
    for b, x in enumerate((3, 11)):
        for k in range(g):
            x = succ[x]
            assert out["tokens"][b, k] == x
    # rounding: ties to even, binary32 first
    for terms, want in [([(0.5, 2.0 ** -7)], 1.0), ([(0.5, 2.0 ** -7), (2.0 ** -15, 2.0 ** -15)], 1.0),
                        ([(0.5, 2.0 ** -7), (2.0 ** -10, 2.0 ** -10)], 1.0078125)]:
        W1 = np.zeros((8, r), np.uint16)
        W2t = np.zeros((8, r), np.uint16)
        for j, (a, b) in enumerate(terms):
            W1[0, j], W2t[1, j] = _bits([a])[0], _bits([b])[0]
        L = oracle.markov_draft(np.tile(_bits([1.0] * 8), (1, 1, 1)), W1, W2t,
                                np.array([0], np.int32), np.array([[0.5]], np.float32), 1.0,
                                want_logits=True, lib=lib)["logits"][0, 0]
        got = (L.astype(np.uint32) << 16).view(np.float32)
        assert got[1] == want and got[0] == 1.0
    # two tokens: p(0) = 1 / (1 + exp((L1 - L0) / T)) at T = 0.5
    W1 = np.zeros((2, r), np.uint16)
    W2t = np.zeros((2, r), np.uint16)
    W1[0, 0], W2t[0, 0], W2t[1, 0] = _bits([0.5, 0.25, -0.5])
    out = oracle.markov_draft(np.zeros((1, 1, 2), np.uint16), W1, W2t, np.array([0], np.int32),
                              np.array([[0.1]], np.float32), 0.5, lib=lib)
    assert abs(out["probs"][0, 0] - 1.0 / (1.0 + np.exp(-0.375 / 0.5))) < 1e-15
    # zero head: the block samples softmax(U_k / T) by the inverse CDF, row k at step k
    rng = np.random.default_rng(2)
    V, g, T = 40, 4, 0.8
    Uf = (3 * rng.standard_normal((1, g, V))).astype(np.float32)
    U = _bits((Uf.view(np.uint32) & 0xFFFF0000).view(np.float32))
    u = rng.uniform(0, 1, (1, g)).astype(np.float32)
    out = oracle.markov_draft(U, np.zeros((V, r), np.uint16), np.zeros((V, r), np.uint16),
                              np.array([0], np.int32), u, T, want_logits=True, lib=lib)
    assert np.array_equal(out["logits"], U)
    for k in range(g):
        z = (U[0, k].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        y = int(np.searchsorted(np.cumsum(scipy.special.softmax(z / T)), u[0, k], side="right"))
        assert out["flags"][0, k] or out["tokens"][0, k] == y


def _all_checks(lib):
    failures = []
    for chk in (check_softmax, check_verify, check_schedule, check_draft):
        try:
            chk(lib)
        except (AssertionError, oracle.OracleError) as e:
            failures.append(f"{chk.__name__}: {str(e).splitlines()[0] if str(e) else type(e).__name__}")
    return failures


def test_unmodified_oracle_passes_all_checks():
    assert _all_checks(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new, *count = MUTANTS[name]
    count = count[0] if count else 1
    src = open(SRC).read()
    assert src.count(old) == count, f"mutation anchor for {name} not found {count} time(s)"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / "libmutant.so")))
    assert _all_checks(lib), f"planted mistake '{name}' passed every pin"


def test_law_check_has_power():
    """The statistical check the GPU losslessness test applies passes on the
    oracle and rejects a planted wrong residual (p_t in place of the normalised
    max(0, p_t - p_d)) at the same trial count."""
    from tests._law import law_pvalues, one_position_trials
    V, T, n = 8, 1.0, 65535
    zt, zd, x, uni, pt1, pt2, pd1 = one_position_trials(V, T, 1, n)
    tl = np.tile(zt, (n, 1))
    dl = np.tile(zd.reshape(1, V), (n, 1))
    ell = np.ones(n, np.int32)
    good = oracle.verify(tl, dl, x.reshape(n, 1), ell, uni, T, nthreads=4)
    z, p1, p2 = law_pvalues(good["accepted_len"], good["emitted"], x, pt1, pt2, pd1)
    assert z <= 5.0 and p1 > 1e-4 and p2 > 1e-4, (z, p1, p2)
    old, new = MUTANTS["residual_uses_target_only"][:2]
    import tempfile
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "mutant.c")
        open(path, "w").write(open(SRC).read().replace(old, new))
        lib = oracle.load(oracle.build(path, os.path.join(tmp, "libmutant.so")))
        bad = oracle.verify(tl, dl, x.reshape(n, 1), ell, uni, T, nthreads=4, lib=lib)
    z, p1, p2 = law_pvalues(bad["accepted_len"], bad["emitted"], x, pt1, pt2, pd1)
    assert p1 < 1e-4, p1
