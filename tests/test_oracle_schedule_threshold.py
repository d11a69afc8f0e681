"""Pins of the oracle's static-threshold baseline (DSpark paper, section
4.3.3, "Static Threshold Sweep"): each request verifies its draft tokens while
their confidence reaches the threshold."""
import numpy as np
import pytest

import oracle


def test_hand_worked_rows():
    conf = np.array([[0.9, 0.8, 0.95, 0.1],
                     [0.4, 0.99, 0.99, 0.99],
                     [0.7, 0.7, 0.7, 0.7],
                     [1.0, 0.0, 1.0, 1.0]], np.float32)
    # threshold 0.7: stop at the first confidence below it (equal passes)
    assert list(oracle.schedule_threshold(conf, 0.7)) == [3, 0, 4, 1]
    assert list(oracle.schedule_threshold(conf, 0.85)) == [1, 0, 0, 1]


def test_extreme_thresholds():
    rng = np.random.default_rng(3)
    conf = rng.uniform(0, 1, (20, 9)).astype(np.float32)
    assert (oracle.schedule_threshold(conf, 0.0) == 9).all()    # every c >= 0
    assert (oracle.schedule_threshold(conf, -1.0) == 9).all()
    assert not oracle.schedule_threshold(conf, 1.01).any()      # no c reaches it


@pytest.mark.parametrize("seed", range(10))
def test_prefix_property_and_monotonicity(seed):
    """Every admitted position reaches the threshold, the next one (if any)
    does not, and a higher threshold never admits more."""
    rng = np.random.default_rng(seed)
    R, g = int(rng.integers(1, 30)), int(rng.integers(1, 17))
    conf = rng.uniform(0, 1, (R, g)).astype(np.float32) ** 0.4
    prev = np.full(R, g + 1)
    for thr in np.linspace(0.0, 1.0, 11):
        ell = oracle.schedule_threshold(conf, thr)
        for r in range(R):
            assert (conf[r, :ell[r]] >= np.float32(thr)).all()
            if ell[r] < g:
                assert conf[r, ell[r]] < np.float32(thr)
        assert (ell <= prev).all()
        prev = ell


def test_rejects_bad_inputs():
    with pytest.raises(oracle.OracleError):
        oracle.schedule_threshold(np.array([[0.5, np.nan]], np.float32), 0.5)
    with pytest.raises(oracle.OracleError):
        oracle.schedule_threshold(np.array([[0.5]], np.float32), float("nan"))
