"""Edge values of dspark_verify's inputs (DSpark paper section 2.1 for the
ratio test and the draws; the data-error contract of the C-ABI header):

- a NaN or an infinite logit in a row the call verifies makes that row's
  statistics non-finite: the call sets DSPARK_ERR_BAD_DATA, every output stays
  inside its buffer, and the other requests still equal the oracle;
- rows past a request's verify length are never read, so non-finite values
  there change nothing;
- uniforms of exactly 0 and of the largest float below 1 (the ends of the
  interval the header allows), against the oracle.
"""
import numpy as np
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._gpu import compare, oracle_on_requests

pytestmark = pytest.mark.gpu
BAD_DATA = 5


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def run(vi):
    out = binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                                vi.verify_len, vi.uniforms, vi.temperature, vi.target_row_off,
                                vi.draft_row_off)
    torch.cuda.synchronize()
    return out


def in_bounds(out, vi):
    acc = out["accepted_len"].cpu().numpy()
    ell = vi.verify_len.cpu().numpy()
    em = out["emitted_tokens"].cpu().numpy()
    assert np.all((acc >= 0) & (acc <= ell))
    assert np.all((em >= -1) & (em < vi.V))


def row_of(vi, r, k, target):
    """Global row index of request r's target (k = 0..g) or draft (k = 0..g-1) row."""
    off = vi.target_row_off if target else vi.draft_row_off
    if off is None:
        return r * (vi.gamma + 1) + k if target else r * vi.gamma + k
    return int(off[r].item()) + k


@pytest.mark.parametrize("dt", [torch.bfloat16, torch.float32])
@pytest.mark.parametrize("what", ["target_nan", "target_inf", "draft_inf", "draft_neg_inf_row"])
def test_non_finite_verified_row(dev, dt, what):
    V = 3000 if dt == torch.bfloat16 else 3001  # bulk-copy and plain-load paths
    vi = workloads.make_verify(6, 4, V, dt, 1.0, rho=(0.5, 0.95), verify_len="full",
                               ragged=dt == torch.float32, seed=70, device=dev)
    r = 2
    if what == "target_nan":
        vi.target_logits[row_of(vi, r, 1, True), 17] = float("nan")
    elif what == "target_inf":
        vi.target_logits[row_of(vi, r, 0, True), V - 1] = float("inf")
    elif what == "draft_inf":
        vi.draft_logits[row_of(vi, r, 3, False), 1000] = float("inf")
    else:
        vi.draft_logits[row_of(vi, r, 0, False), :] = float("-inf")
    out = run(vi)
    assert int(out["device_status"].item()) == BAD_DATA
    in_bounds(out, vi)
    others = np.array([i for i in range(vi.B) if i != r])
    compare(out, oracle_on_requests(vi, others), vi, others, mismatch_budget=False)


def test_rows_past_the_verify_length_are_not_read(dev):
    ell = np.array([0, 1, 3, 2, 4, 1], np.int32)
    vi = workloads.make_verify(6, 4, 3000, torch.bfloat16, 0.8, rho=(0.5, 0.95),
                               verify_len=ell, seed=71, device=dev)
    ref = oracle_on_requests(vi, np.arange(vi.B))
    for r in range(vi.B):
        for k in range(ell[r] + 1, vi.gamma + 1):   # target rows after the bonus row
            vi.target_logits[row_of(vi, r, k, True), :] = float("nan")
        for k in range(ell[r], vi.gamma):           # draft rows after the verified ones
            vi.draft_logits[row_of(vi, r, k, False), 5] = float("inf")
    out = run(vi)
    assert int(out["device_status"].item()) == 0
    compare(out, ref, vi, np.arange(vi.B))


@pytest.mark.parametrize("u", [0.0, float(np.nextafter(np.float32(1.0), np.float32(0.0)))])
def test_extreme_uniforms(dev, u):
    vi = workloads.make_verify(16, 8, 5000, torch.bfloat16, 0.8, rho=(0.5, 0.95),
                               verify_len="uniform", seed=72, device=dev)
    vi.uniforms.fill_(u)
    out = run(vi)
    assert int(out["device_status"].item()) == 0
    in_bounds(out, vi)
    idx = np.arange(vi.B)
    st = compare(out, oracle_on_requests(vi, idx), vi, idx, mismatch_budget=False)
    if u == 0.0:
        # every finite logit has p > 0: all verified positions pass, and the
        # draw's cut at 0 takes the first token of positive weight, token 0
        acc = out["accepted_len"].cpu().numpy()
        np.testing.assert_array_equal(acc, vi.verify_len.cpu().numpy())
        em = out["emitted_tokens"].cpu().numpy()
        assert np.all(em[np.arange(vi.B), acc] == 0)
        assert st["excused"] == 0
