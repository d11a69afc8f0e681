"""The law of the GPU path itself, not its agreement with the oracle: on a
tiny vocabulary, many independent trials of one request (the same target and
draft rows, fresh uniforms each) must emit tokens distributed as the target
distribution says.

Speculative verification is lossless (DSpark paper, section 2.1: accept x
with probability min(1, p_t(x)/p_d(x)), otherwise draw from the normalised
max(0, p_t - p_d); Appendix 8: the per-position acceptance probability is
sum_v min(p_t(v), p_d(v))). With draft tokens drawn from p_d:
  - the first emitted token follows p_t of target row 1;
  - the acceptance rate of position 1 is sum_v min(p_t, p_d) (equation 8);
  - given an accepted first token, the token after a block of one position
    (the bonus) follows p_t of target row 2.
The expected laws are computed here from the bf16 logits by scipy in float64;
the counts are compared by chi-square tests at a fixed seed.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._law import law_pvalues, one_position_trials

pytestmark = pytest.mark.gpu

N = 65535        # trials: requests of one call, the largest batch the call takes
P_MIN = 1e-4     # smallest chi-square p-value accepted (seeded: the outcome is fixed)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("V,T,seed", [(8, 1.0, 1), (16, 0.7, 2), (24, 1.5, 3)])
def test_emitted_law_is_the_target_law(dev, V, T, seed):
    zt, zd, x, uni, pt1, pt2, pd1 = one_position_trials(V, T, seed, N)
    as_bf16 = lambda b: torch.from_numpy(b.view(np.int16)).view(torch.bfloat16)
    tl = as_bf16(zt).repeat(N, 1).to(dev)              # dense: request r's target rows 2r, 2r + 1
    dl = as_bf16(zd).reshape(1, V).repeat(N, 1).to(dev)  # request r's draft row r
    out = binding.dspark_verify(tl, dl, torch.from_numpy(x).reshape(N, 1).to(dev),
                                torch.ones(N, dtype=torch.int32, device=dev),
                                torch.from_numpy(uni).to(dev), T, check=True)
    acc = out["accepted_len"].cpu().numpy()
    em = out["emitted_tokens"].cpu().numpy()
    assert set(np.unique(acc)) <= {0, 1}
    assert np.all(em[acc == 1, 0] == x[acc == 1])
    z, p_first, p_bonus = law_pvalues(acc, em, x, pt1, pt2, pd1)
    assert z <= 5.0, z                      # equation 8
    assert p_first > P_MIN, p_first         # first token ~ p_t of row 1
    assert p_bonus > P_MIN, p_bonus         # bonus ~ p_t of row 2
