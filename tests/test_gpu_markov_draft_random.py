"""The drafter's sequential stage on seeded random shapes against the oracle.

Each case draws the batch (1..300, so one request tile, two, or more), the
block length (1..8), the vocabulary (a multiple of 8 up to 6,000, with ragged
last tiles), the rank (64, 128, 192 or 256) and the temperature (0.1..5,
log-uniform). The weights are on the 2^-8 grid: rows bit-exact, tokens equal
except after a draw the oracle flags as a near tie (as in test_gpu_markov_draft).
"""
import numpy as np
import pytest

from speculative_decoding_verification_41_gb300 import workloads
from tests.test_gpu_markov_draft import compare_chains, dev, run_gpu, run_oracle  # noqa: F401

pytestmark = pytest.mark.gpu


def draw_case(seed):
    rng = np.random.default_rng(2000 + seed)
    B = int(rng.integers(1, 301))
    gamma = int(rng.integers(1, 9))
    V = 8 * int(rng.integers(1, 751))
    r = int(rng.choice([64, 128, 192, 256]))
    T = float(np.exp(rng.uniform(np.log(0.1), np.log(5.0))))
    return B, gamma, V, r, T


@pytest.mark.parametrize("seed", range(10))
def test_random_shapes(dev, seed):
    B, gamma, V, r, T = draw_case(seed)
    d = workloads.make_markov_draft(B, gamma, V, r, temperature=T, seed=seed + 40, device="cpu")
    L, x = run_gpu(d, dev)
    ref = run_oracle(d)
    excused = compare_chains(L, x, ref, range(B))
    assert excused <= max(1, B // 100), (B, gamma, V, r, T, excused)
