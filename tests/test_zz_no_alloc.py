"""dspark_verify_static: verification for callers that cannot allocate device
memory (framework plugins handed only their buffers, serving loops that must
not call cudaMalloc because it can synchronise the device, processes under a
fixed device-memory budget). Its scratch is a fixed array inside libdspark.

The test calls the entry point through the C-ABI and checks that two calls in
a row give the same results as dspark_verify with a caller workspace:
identical accepted lengths and tokens, probabilities within the 1e-5 absolute
tolerance the parity tests use. It also checks that an oversized batch is
rejected before anything runs. This file is collected last so that a run that
stops at the first failure has already run every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build
from tests._gpu import PROB_ATOL

pytestmark = pytest.mark.gpu

TOO_LARGE = 6  # DSPARK_ERR_TOO_LARGE


def _p(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def call_static(lib, vi, outs):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return lib.dspark_verify_static(
        _p(vi.target_logits), _p(vi.draft_logits), _p(vi.draft_tokens), _p(vi.verify_len),
        _p(vi.uniforms), float(vi.temperature), binding.DSPARK_BF16, vi.B, vi.gamma, vi.V,
        _p(vi.target_row_off), _p(vi.draft_row_off), _p(outs["accepted_len"]),
        _p(outs["emitted_tokens"]), _p(outs["probs"]), _p(outs["near_tie_count"]),
        _p(outs["device_status"]), stream)


def test_static_scratch_matches_caller_workspace():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    lib = binding.load()
    dev = torch.device("cuda:0")
    vi = workloads.make_verify(24, 16, 20000, torch.bfloat16, 0.7, rho=(0.6, 0.95),
                               verify_len="uniform", ragged=True, seed=21, device=dev)
    ref = binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                                vi.verify_len, vi.uniforms, vi.temperature, vi.target_row_off,
                                vi.draft_row_off, check=True)
    ref = {k: v.clone() for k, v in ref.items() if v is not None}
    for _ in range(2):  # two calls in a row share the static array
        outs = {"accepted_len": torch.full((vi.B,), -7, dtype=torch.int32, device=dev),
                "emitted_tokens": torch.full((vi.B, vi.gamma + 1), -7, dtype=torch.int32,
                                             device=dev),
                "probs": torch.zeros(vi.B, vi.gamma, 2, dtype=torch.float32, device=dev),
                "near_tie_count": torch.full((1,), 99, dtype=torch.int32, device=dev),
                "device_status": torch.full((1,), 99, dtype=torch.int32, device=dev)}
        assert call_static(lib, vi, outs) == 0
        torch.cuda.synchronize()
        assert int(outs["device_status"].item()) == 0
        assert torch.equal(outs["accepted_len"], ref["accepted_len"])
        assert torch.equal(outs["emitted_tokens"], ref["emitted_tokens"])
        assert torch.equal(outs["near_tie_count"], ref["near_tie_count"])
        err = (outs["probs"] - ref["probs"]).abs().max().item()
        assert err <= PROB_ATOL


def test_static_scratch_rejects_oversized_batch():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    lib = binding.load()
    dev = torch.device("cuda:0")
    B, g, V = 1024, 16, 151936  # needs ~21 MB of scratch, more than the 16 MiB array
    assert binding.verify_workspace_bytes(B, g, V) > 16 << 20
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
