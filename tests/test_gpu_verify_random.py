"""dspark_verify (and dspark_acceptance) on seeded random shapes against the
CPU oracle.

Each case draws, from its own generator:
- the batch size, the block length gamma (1..32) and the vocabulary (8..6,000).
  Odd sizes give rows that are not 16-byte multiples, which take the
  plain-load path.
- the dtype, the temperature (0.05..5, log-uniform) and the range of the
  per-request draft/target correlation.
- the verify lengths: every position, uniform, or any value in 0..gamma
  (zero-length requests included).
- the layout, dense or ragged.

The bar is that of the fixed shapes in test_gpu_verify: accepted lengths and
emitted tokens equal request by request, except requests the oracle flags at
a near tie; probabilities within the stated tolerance.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._gpu import PROB_RTOL_QUALITY, compare, oracle_on_requests

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def draw_case(seed):
    rng = np.random.default_rng(1000 + seed)
    B = int(rng.integers(1, 200))
    gamma = int(rng.integers(1, 33))
    V = int(rng.integers(8, 6001))
    dt = torch.float32 if rng.random() < 0.35 else torch.bfloat16
    T = float(np.exp(rng.uniform(np.log(0.05), np.log(5.0))))
    lo = float(rng.uniform(0.0, 0.9))
    rho = (lo, float(rng.uniform(lo, 0.99)))
    kind = int(rng.integers(0, 3))
    if kind == 0:
        ell = "full"
    elif kind == 1:
        ell = "uniform"
    else:
        ell = rng.integers(0, gamma + 1, size=B).astype(np.int32)
    ragged = bool(rng.random() < 0.5)
    return B, gamma, V, dt, T, rho, ell, ragged


@pytest.mark.parametrize("seed", range(24))
def test_random_shapes(dev, seed):
    B, g, V, dt, T, rho, ell, ragged = draw_case(seed)
    vi = workloads.make_verify(B, g, V, dt, T, rho=rho, verify_len=ell, ragged=ragged,
                               seed=seed + 3, device=dev)
    out = binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                                vi.verify_len, vi.uniforms, vi.temperature, vi.target_row_off,
                                vi.draft_row_off, check=True)
    idx = np.arange(B)
    ref = oracle_on_requests(vi, idx)
    st = compare(out, ref, vi, idx)
    assert st["prob_max_rel_err"] <= PROB_RTOL_QUALITY, (B, g, V, dt, T, ragged, st)


@pytest.mark.parametrize("seed", range(12))
def test_random_shapes_acceptance(dev, seed):
    """dspark_acceptance (every verified position's sum_v min(p_t, p_d)) on
    the same random shapes, within the probability tolerance of the oracle."""
    from tests.test_gpu_acceptance import check as check_acceptance
    B, g, V, dt, T, rho, ell, ragged = draw_case(100 + seed)
    vi = workloads.make_verify(B, g, V, dt, T, rho=rho, verify_len=ell, ragged=ragged,
                               seed=seed + 5, device=dev)
    check_acceptance(vi)
