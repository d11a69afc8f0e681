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
from tests._sched import exhaustive_best

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
    "batch_not_counted": ("    Bsz += 1;\n", "\n"),
    "anchor_token_dropped": ("double tau = (double)R;", "double tau = 0.0;"),
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


def _all_checks(lib):
    failures = []
    for chk in (check_softmax, check_verify, check_schedule):
        try:
            chk(lib)
        except (AssertionError, oracle.OracleError) as e:
            failures.append(f"{chk.__name__}: {str(e).splitlines()[0] if str(e) else type(e).__name__}")
    return failures


def test_unmodified_oracle_passes_all_checks():
    assert _all_checks(oracle.load()) == []


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(SRC).read()
    assert src.count(old) == 1, f"mutation anchor for {name} not found exactly once"
    path = tmp_path / "mutant.c"
    path.write_text(src.replace(old, new))
    lib = oracle.load(oracle.build(str(path), str(tmp_path / "libmutant.so")))
    assert _all_checks(lib), f"planted mistake '{name}' passed every pin"
