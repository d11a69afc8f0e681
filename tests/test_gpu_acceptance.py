"""GPU parity of dspark_acceptance (the acceptance probability sum_v
min(p_t^k, p_d^k) of every verified position, DSpark paper equation 8)
against the oracle: both load paths, both dtypes, dense and ragged layouts,
invalid requests and the named workloads (sampled)."""
import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu
ATOL = 1e-5  # the probability tolerance of the verification outputs


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def host(t):
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def check(vi, idx=None):
    out = binding.dspark_acceptance(vi.target_logits, vi.draft_logits, vi.verify_len,
                                    vi.temperature, vi.gamma, vi.target_row_off,
                                    vi.draft_row_off, check=True)
    got = out["rates"].cpu().numpy()
    toff = None if vi.target_row_off is None else vi.target_row_off.cpu().numpy()
    doff = None if vi.draft_row_off is None else vi.draft_row_off.cpu().numpy()
    ell = vi.verify_len.cpu().numpy()
    if idx is None:
        ref = oracle.acceptance(host(vi.target_logits), host(vi.draft_logits), ell,
                                vi.temperature, vi.gamma, toff, doff, nthreads=oracle.max_threads())
        sel = np.arange(vi.B)
    else:  # sampled requests: the oracle sees only their rows, through their offsets
        B, g = vi.B, vi.gamma
        t0 = toff if toff is not None else np.arange(B + 1, dtype=np.int64) * (g + 1)
        d0 = doff if doff is not None else np.arange(B + 1, dtype=np.int64) * g
        ref = oracle.acceptance(host(vi.target_logits), host(vi.draft_logits), ell[idx],
                                vi.temperature, g,
                                np.concatenate([t0[idx], [0]]).astype(np.int64),
                                np.concatenate([d0[idx], [0]]).astype(np.int64),
                                nthreads=oracle.max_threads())
        sel = idx
    g = got[sel]
    assert ((g == -1.0) == (ref == -1.0)).all()
    valid = ref >= 0
    assert np.abs(g[valid] - ref[valid]).max() <= ATOL, np.abs(g[valid] - ref[valid]).max()
    return g, ref


SHAPES = [
    # B, gamma, V, dtype, T, verify_len, ragged
    (8, 16, 10000, torch.bfloat16, 1.0, "full", False),     # aligned: bulk-copy path
    (16, 8, 20011, torch.bfloat16, 0.7, "uniform", True),   # odd V: plain-load path
    (12, 16, 5000, torch.float32, 1.3, "uniform", True),    # fp32, ragged rows
    (6, 4, 4099, torch.float32, 0.7, "full", False),        # fp32 odd V: plain path
    (5, 32, 9000, torch.bfloat16, 1.0, "full", False),      # gamma = 32
    (8, 16, 10000, torch.bfloat16, 0.05, "full", False),    # cold: nearly one-hot rows
    (8, 16, 10000, torch.bfloat16, 20.0, "uniform", False), # hot: nearly flat rows
    (7, 5, 1, torch.bfloat16, 0.9, "uniform", False),       # one token: every rate is 1
    (7, 5, 3, torch.float32, 0.9, "uniform", True),         # three tokens, ragged
]


@pytest.mark.parametrize("B,g,V,dt,T,vl,ragged", SHAPES)
def test_shapes(dev, B, g, V, dt, T, vl, ragged):
    vi = workloads.make_verify(B, g, V, dt, T, rho=(0.5, 0.95), verify_len=vl, ragged=ragged,
                               seed=21 + B + g, device=dev)
    check(vi)


def test_zero_lengths_and_identical_rows(dev):
    vi = workloads.make_verify(4, 8, 6000, torch.bfloat16, 1.0, seed=3, device=dev)
    vi.draft_logits.copy_(vi.target_logits.view(4, 9, -1)[:, :8].reshape(32, -1))
    vi.verify_len[1] = 0
    g, _ = check(vi)
    assert (g[1] == -1.0).all()
    assert np.abs(g[[0, 2, 3]] - 1.0).max() < 1e-5


@pytest.mark.parametrize("name,sample", [("b256_g16_v129280_bf16", 24),
                                         ("ragged_b1024_g16_v151936_f32", 16)])
def test_named_workloads(dev, name, sample):
    vi = workloads.make_config(name, device=dev)
    idx = np.sort(np.random.default_rng(0).choice(vi.B, sample, replace=False))
    check(vi, idx)


# ---------------------------------------------------------------------------
# dspark_verify_rates: the verification and the rates from one statistics pass
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("B,g,V,dt,T,vl,ragged", SHAPES + [
    (64, 16, 40000, torch.bfloat16, 0.7, "uniform", False),  # items claimed past the fixed rounds
])
def test_verify_rates_equal_the_separate_calls(dev, B, g, V, dt, T, vl, ragged):
    """Outputs bit-identical to dspark_verify's, rates bit-identical to
    dspark_acceptance's (the same kernels on the same statistics), and so
    within the oracle's tolerance."""
    vi = workloads.make_verify(B, g, V, dt, T, rho=(0.5, 0.95), verify_len=vl, ragged=ragged,
                               seed=31 + B + g, device=dev)
    args = (vi.target_logits, vi.draft_logits, vi.draft_tokens, vi.verify_len, vi.uniforms,
            vi.temperature, vi.target_row_off, vi.draft_row_off)
    plain = {k: v.clone() for k, v in binding.dspark_verify(*args, check=True).items()
             if v is not None}
    both = binding.dspark_verify(*args, check=True, with_rates=True)
    for k in plain:
        assert torch.equal(plain[k], both[k]), k
    sep, _ = check(vi)  # dspark_acceptance against the oracle
    assert np.array_equal(both["rates"].cpu().numpy(), np.asarray(sep))


def test_verify_rates_repeated_with_buffers(dev):
    """Reused buffers (and their counters) give the same rates call after call."""
    vi = workloads.make_verify(24, 16, 30000, torch.bfloat16, 0.7, rho=(0.6, 0.95), seed=8,
                               device=dev)
    bufs = binding.VerifyBuffers(24, 16, 30000, dev, with_rates=True)
    args = (vi.target_logits, vi.draft_logits, vi.draft_tokens, vi.verify_len, vi.uniforms,
            vi.temperature)
    a = binding.dspark_verify(*args, buffers=bufs, check=True, with_rates=True)["rates"].clone()
    for _ in range(3):
        b = binding.dspark_verify(*args, buffers=bufs, check=True, with_rates=True)["rates"]
        assert torch.equal(a, b)


def test_verify_rates_headline_size(dev):
    """The headline workload (256 x 16 x 129,280 bf16) in the bench's launch
    configuration: the combined call equals the two separate calls bit for bit."""
    vi = workloads.make_config("b256_g16_v129280_bf16", device=dev)
    args = (vi.target_logits, vi.draft_logits, vi.draft_tokens, vi.verify_len, vi.uniforms,
            vi.temperature)
    plain = {k: v.clone() for k, v in binding.dspark_verify(*args, check=True).items()
             if v is not None}
    rates = binding.dspark_acceptance(vi.target_logits, vi.draft_logits, vi.verify_len,
                                      vi.temperature, vi.gamma, check=True)["rates"].clone()
    both = binding.dspark_verify(*args, check=True, with_rates=True)
    for k in plain:
        assert torch.equal(plain[k], both[k]), k
    assert torch.equal(rates, both["rates"])
