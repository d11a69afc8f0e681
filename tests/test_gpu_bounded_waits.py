"""Failure detection without a GPU fault: every wait in the library is
bounded by about a second of the device's global timer; when it runs out the
kernel records DSPARK_ERR_TIMEOUT in the status word and returns. Here a
diagnostic entry point runs each kind of wait on a condition that never comes
true (an mbarrier that nothing completes, a grid barrier missing a CTA) and
the test reads the status; the context stays usable, which the verification
call that follows shows."""
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("which", [0, 1])
def test_wait_gives_up_with_timeout_status(dev, which):
    vi = workloads.make_verify(16, 8, 9000, torch.bfloat16, 1.0, seed=2, device=dev)
    bufs = binding.VerifyBuffers(16, 8, 9000, dev)
    args = (vi.target_logits, vi.draft_logits, vi.draft_tokens, vi.verify_len, vi.uniforms,
            vi.temperature)
    ref = {k: v.clone() for k, v in binding.dspark_verify(*args, buffers=bufs, check=True).items()
           if v is not None}

    r = binding.wait_selftest(which, dev)
    assert r["status"] == binding.DSPARK_ERR_TIMEOUT, r
    assert 0.9 <= r["seconds"] <= 10.0, r  # about a second of wall time

    out = binding.dspark_verify(*args, buffers=bufs, check=True)  # the context still works
    for k in ref:
        assert torch.equal(out[k], ref[k]), k
