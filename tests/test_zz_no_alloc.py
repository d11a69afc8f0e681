"""dspark_verify_static: verification for callers that cannot allocate device
memory (framework plugins handed only their buffers, serving loops that must
not call cudaMalloc because it can synchronise the device, processes under a
fixed device-memory budget). Its scratch is a fixed array inside libdspark.

Each case calls the entry point through the C-ABI twice in a row and checks
that both calls give exactly the results of dspark_verify with a caller
workspace: the same kernels run on the same inputs, so every output (accepted
lengths, tokens, probabilities, near-tie count) is compared bit for bit. The
cases cover both dtypes, both load paths (rows whose byte length is a multiple
of 16 stream by bulk copies, other rows by plain loads), dense and ragged
layouts, and batches whose scratch fills the array exactly. A batch one
request larger is rejected before anything runs. This file is collected last
so that a run that stops at the first failure has already run every other
test.
"""
import ctypes
import os
import re

import numpy as np
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu

TOO_LARGE = 6  # DSPARK_ERR_TOO_LARGE
HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "dspark.h")


def static_ws_bytes() -> int:
    m = re.search(r"#define DSPARK_STATIC_WS_BYTES \(\(size_t\)(\d+)u << (\d+)\)",
                  open(HEADER).read())
    return int(m.group(1)) << int(m.group(2))


def largest_batch(gamma: int, V: int) -> int:
    """The largest B whose DSPARK_VERIFY_WS_BYTES(B, gamma, V) fits the array."""
    lim, lo, hi = static_ws_bytes(), 1, 65535
    while lo < hi:
        mid = (lo + hi + 1) // 2
        if binding.verify_workspace_bytes(mid, gamma, V) <= lim:
            lo = mid
        else:
            hi = mid - 1
    return lo


@pytest.fixture(scope="module")
def lib():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return binding.load()


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def dtype_code(t):
    return binding.DSPARK_BF16 if t.dtype == torch.bfloat16 else binding.DSPARK_F32


def call_static(lib, vi, outs):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dspark_verify_static(
        _p(vi.target_logits), _p(vi.draft_logits), _p(vi.draft_tokens), _p(vi.verify_len),
        _p(vi.uniforms), float(vi.temperature), dtype_code(vi.target_logits), vi.B, vi.gamma,
        vi.V, _p(vi.target_row_off), _p(vi.draft_row_off), _p(outs["accepted_len"]),
        _p(outs["emitted_tokens"]), _p(outs["probs"]), _p(outs["near_tie_count"]),
        _p(outs["device_status"]), stream)


def random_batch(B, gamma, V, dtype, seed, dev):
    """Many short requests, made in bulk (any valid inputs serve: the two entry
    points are compared with each other, not with the oracle)."""
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    tl = (3 * torch.randn(B * (gamma + 1), V, generator=g, device=dev)).to(dtype)
    dl = (3 * torch.randn(B * gamma, V, generator=g, device=dev)).to(dtype)
    tok = torch.randint(0, V, (B, gamma), generator=g, device=dev, dtype=torch.int32)
    ell = torch.randint(0, gamma + 1, (B,), generator=g, device=dev, dtype=torch.int32)
    uni = torch.randint(0, 1 << 24, (B, gamma + 1), generator=g, device=dev).float() * 2.0 ** -24
    return workloads.VerifyInputs(tl, dl, tok, ell, uni, 0.8)


def check_matches_caller_workspace(lib, vi, dev):
    ref = binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                                vi.verify_len, vi.uniforms, vi.temperature, vi.target_row_off,
                                vi.draft_row_off, check=True)
    ref = {k: v.clone() for k, v in ref.items() if v is not None}
    for _ in range(2):  # two calls in a row share the static array
        outs = {"accepted_len": torch.full((vi.B,), -7, dtype=torch.int32, device=dev),
                "emitted_tokens": torch.full((vi.B, vi.gamma + 1), -7, dtype=torch.int32,
                                             device=dev),
                "probs": torch.full((vi.B, vi.gamma, 2), 7.0, dtype=torch.float32, device=dev),
                "near_tie_count": torch.full((1,), 99, dtype=torch.int32, device=dev),
                "device_status": torch.full((1,), 99, dtype=torch.int32, device=dev)}
        assert call_static(lib, vi, outs) == 0
        torch.cuda.synchronize()
        assert int(outs["device_status"].item()) == 0
        for k in ("accepted_len", "emitted_tokens", "probs", "near_tie_count"):
            assert torch.equal(outs[k], ref[k]), k


@pytest.mark.parametrize("B,gamma,V,dtype,ragged", [
    (24, 16, 20000, torch.bfloat16, True),   # bulk copies, ragged rows
    (12, 16, 5000, torch.float32, True),     # fp32, rows of 20,000 bytes
    (6, 4, 4099, torch.float32, False),      # fp32 rows of 16,396 bytes: plain loads
    (9, 8, 3001, torch.bfloat16, False),     # bf16 rows of 6,002 bytes: plain loads
])
def test_static_scratch_matches_caller_workspace(lib, B, gamma, V, dtype, ragged):
    dev = torch.device("cuda:0")
    vi = workloads.make_verify(B, gamma, V, dtype, 0.7, rho=(0.6, 0.95), verify_len="uniform",
                               ragged=ragged, seed=21 + B, device=dev)
    check_matches_caller_workspace(lib, vi, dev)


@pytest.mark.parametrize("V,dtype", [(64, torch.bfloat16), (63, torch.float32)])
def test_batch_that_fills_the_array(lib, V, dtype):
    """The largest batch the array holds (tens of thousands of short requests,
    scratch within 256 bytes of the 16 MiB), on both load paths."""
    dev = torch.device("cuda:0")
    gamma = 4
    B = largest_batch(gamma, V)
    need = binding.verify_workspace_bytes(B, gamma, V)
    assert static_ws_bytes() - 256 < need <= static_ws_bytes()
    vi = random_batch(B, gamma, V, dtype, seed=V, dev=dev)
    check_matches_caller_workspace(lib, vi, dev)


def test_static_scratch_rejects_oversized_batch(lib):
    dev = torch.device("cuda:0")
    for B, g, V in [(1024, 16, 151936), (largest_batch(4, 64) + 1, 4, 64)]:
        assert binding.verify_workspace_bytes(B, g, V) > static_ws_bytes()
        tl = torch.zeros(1, V, dtype=torch.bfloat16, device=dev)
        small = torch.zeros(B * (g + 1), dtype=torch.int32, device=dev)
        status = torch.full((1,), 99, dtype=torch.int32, device=dev)
        rc = lib.dspark_verify_static(
            _p(tl), _p(tl), _p(small), _p(small), _p(small), 1.0, binding.DSPARK_BF16, B, g, V,
            None, None, _p(small), _p(small), None, None, _p(status),
            ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
        assert rc == TOO_LARGE
        torch.cuda.synchronize()
        assert int(status.item()) == 99  # nothing was launched
