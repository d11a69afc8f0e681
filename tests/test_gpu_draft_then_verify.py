"""The drafter and the verifier chained on the device: dspark_draft_markov
writes its rows in dspark_verify's dense draft layout, so one speculative
step is the two calls on one stream with no copy between them (DSpark paper,
section 3.1 drafts the block, section 2.1 verifies it).

The oracle runs the same pipeline from its own outputs (its drafter's rows
and tokens feed its verifier); nothing it reads comes from the GPU."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


@pytest.mark.parametrize("B,gamma,V,r,T", [(8, 8, 4096, 64, 1.0), (33, 16, 3000, 128, 0.7)])
def test_draft_then_verify(dev, B, gamma, V, r, T):
    d = workloads.make_markov_draft(B, gamma, V, r, temperature=T, seed=B + gamma, device="cpu")
    # target rows: the verifier's target recipe, B * (gamma + 1) rows in bf16
    vi = workloads.make_verify(B, gamma, V, torch.bfloat16, T, seed=B + V, device="cpu")
    target = vi.target_logits
    uni = vi.uniforms
    ell = torch.full((B,), gamma, dtype=torch.int32)

    # GPU: draft, then verify the emitted rows and tokens in place
    g = d.to(dev)
    dr = binding.dspark_draft_markov(g.base_logits, g.w1, g.w2t, g.anchors, g.uniforms, T,
                                     check=True)
    rows = dr["draft_logits"].view(B * gamma, V)
    out = binding.dspark_verify(target.to(dev), rows, dr["draft_tokens"], ell.to(dev),
                                uni.to(dev), T, check=True)

    # oracle: the same two steps, from its own drafter
    od = oracle.markov_draft(workloads.bf16_bits(d.base_logits), workloads.bf16_bits(d.w1),
                             workloads.bf16_bits(d.w2t), d.anchors.numpy(), d.uniforms.numpy(),
                             T, want_logits=True)
    ov = oracle.verify(workloads.bf16_bits(target), od["logits"].reshape(B * gamma, V),
                       od["tokens"], ell.numpy(), uni.numpy(), T)

    draft_tie = od["flags"].any(axis=1)
    verify_tie = ov["flags"].any(axis=1)
    gx = dr["draft_tokens"].cpu().numpy()
    acc = out["accepted_len"].cpu().numpy()
    em = out["emitted_tokens"].cpu().numpy()
    # every request compared; a difference only where the oracle flags a near
    # tie in that request's draft or verification, and at most one such request
    differ = 0
    for b in range(B):
        same = (np.array_equal(gx[b], od["tokens"][b]) and acc[b] == ov["accepted_len"][b]
                and np.array_equal(em[b], ov["emitted"][b]))
        if not same:
            assert draft_tie[b] or verify_tie[b], (b, gx[b], od["tokens"][b], acc[b], em[b])
            differ += 1
    assert differ <= 1, differ
