"""GPU parity of the drafter's sequential stage with the Markov head (DSpark
paper, section 3.1, equations 4 and 5) against the oracle.

The weights are on the 2^-8 grid (workloads.make_markov_draft, weights="grid"),
where every partial sum of the bias is exact in binary32: the emitted bf16
rows must then equal the oracle's bit for bit, and the tokens must agree
except at a draw the oracle flags as a near tie (|u*Z - C| < 1e-6 Z), after
which that request's chain is no longer compared. Sizes span several request
and vocabulary tiles with ragged tails; the 256 x 16 x 129,280 x 256 case is
checked on a sample of requests, each drafted by the oracle in full."""
import os

import numpy as np
import pytest
import torch

import oracle
from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu
NTHREADS = max(1, min(16, os.cpu_count() or 1))


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def run_gpu(d, dev, **kw):
    g = d.to(dev)
    out = binding.dspark_draft_markov(g.base_logits, g.w1, g.w2t, g.anchors, g.uniforms,
                                      d.temperature, check=True, **kw)
    return (workloads.bf16_bits(out["draft_logits"]), out["draft_tokens"].cpu().numpy())


def run_oracle(d, requests=None):
    return oracle.markov_draft(workloads.bf16_bits(d.base_logits), workloads.bf16_bits(d.w1),
                               workloads.bf16_bits(d.w2t), d.anchors.cpu().numpy(),
                               d.uniforms.cpu().numpy(), d.temperature, requests=requests,
                               want_logits=True, nthreads=NTHREADS)


def compare_chains(L_gpu, x_gpu, ref, requests):
    """Rows bit-exact and tokens equal while the chains agree; a divergence is
    allowed only at a flagged draw. Returns the number of excused requests."""
    excused = 0
    for i, b in enumerate(requests):
        for k in range(x_gpu.shape[1]):
            np.testing.assert_array_equal(L_gpu[b, k], ref["logits"][i, k],
                                          err_msg=f"request {b} position {k + 1}")
            if x_gpu[b, k] != ref["tokens"][i, k]:
                assert ref["flags"][i, k] != 0, (
                    f"request {b} position {k + 1}: gpu {x_gpu[b, k]} oracle {ref['tokens'][i, k]}")
                excused += 1
                break
    return excused


@pytest.mark.parametrize("B,gamma,V,r,T", [
    (1, 1, 8, 64, 1.0),          # one token tile, mostly out of bounds
    (5, 4, 1000, 64, 0.7),       # ragged vocabulary tail: the last tile holds 40 tokens
    (130, 3, 1064, 128, 1.0),    # two request tiles; the last tile holds 40 tokens
    (200, 6, 4096, 256, 0.7),    # whole tiles only
    (3, 2, 1032, 64, 1.0),       # the last tile holds 8 tokens
    (257, 2, 2048, 192, 2.0),    # three request tiles, rank 192
    (40, 16, 20000, 256, 0.7),   # the full block length
    (150, 4, 30000, 128, 0.9),   # two request tiles, 3 or 4 vocabulary tiles per CTA's range
    (24, 8, 6000, 128, 0.05),    # cold: the draws nearly argmax
    (24, 8, 6000, 128, 25.0),    # hot: the draws nearly uniform over the tiles
])
def test_matches_oracle(dev, B, gamma, V, r, T):
    d = workloads.make_markov_draft(B, gamma, V, r, temperature=T, seed=B + V, device="cpu")
    L, x = run_gpu(d, dev)
    ref = run_oracle(d)
    excused = compare_chains(L, x, ref, range(B))
    assert excused <= max(1, B // 100)


def test_batch_too_large_for_one_resident_grid(dev):
    """B = 20,000 needs 157 request tiles, more than one CTA per SM can hold at
    once, so the call takes the per-launch path (gather, then a step and a
    draw kernel per position); results as on the single-launch path."""
    B, gamma, V, r = 20000, 2, 64, 64
    d = workloads.make_markov_draft(B, gamma, V, r, temperature=1.0, seed=21, device="cpu")
    L, x = run_gpu(d, dev)
    ref = run_oracle(d)
    excused = compare_chains(L, x, ref, range(B))
    assert excused <= B // 100


def test_in_place(dev):
    d = workloads.make_markov_draft(33, 5, 3000, 256, seed=3, device="cpu")
    g = d.to(dev)
    U = g.base_logits.clone()
    out = binding.dspark_draft_markov(U, g.w1, g.w2t, g.anchors, g.uniforms, d.temperature,
                                      draft_logits=U, check=True)
    assert out["draft_logits"].data_ptr() == U.data_ptr()
    ref = run_oracle(d)
    compare_chains(workloads.bf16_bits(U), out["draft_tokens"].cpu().numpy(), ref, range(33))


def test_deterministic(dev):
    d = workloads.make_markov_draft(64, 8, 8192, 256, seed=5, device="cpu")
    L1, x1 = run_gpu(d, dev)
    L2, x2 = run_gpu(d, dev)
    np.testing.assert_array_equal(L1, L2)
    np.testing.assert_array_equal(x1, x2)


def test_timed_entry_matches(dev):
    d = workloads.make_markov_draft(20, 4, 5000, 128, seed=8, device="cpu")
    L1, x1 = run_gpu(d, dev)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * 4 + 2)]
    L2, x2 = run_gpu(d, dev, events=ev)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(L1, L2)
    np.testing.assert_array_equal(x1, x2)
    times = [ev[i].elapsed_time(ev[i + 1]) for i in range(len(ev) - 1)]
    assert all(t >= 0 for t in times)


def test_headline_size_on_sampled_requests(dev):
    """256 requests x 16 positions x 129,280 tokens, rank 256, T = 0.7 (the
    drafter's share of the 256 x 16 x 129,280 bf16 verification workload): the
    whole batch on the GPU, eight requests drafted by the oracle in full."""
    B, gamma, V, r = 256, 16, 129280, 256
    d = workloads.make_markov_draft(B, gamma, V, r, temperature=0.7, seed=7, device=dev)
    out = binding.dspark_draft_markov(d.base_logits, d.w1, d.w2t, d.anchors, d.uniforms,
                                      d.temperature, check=True)
    x = out["draft_tokens"].cpu().numpy()
    sample = [0, 1, 127, 128, 129, 200, 254, 255]
    idx = torch.tensor(sample, device=dev)
    sub = workloads.MarkovDraftInputs(d.base_logits.index_select(0, idx), d.w1, d.w2t,
                                      d.anchors.index_select(0, idx), d.uniforms.index_select(0, idx),
                                      d.temperature)
    ref = run_oracle(sub)
    L = workloads.bf16_bits(out["draft_logits"].index_select(0, idx))
    excused = compare_chains(L, x[sample], ref, range(len(sample)))
    assert excused <= 1
    assert (x >= 0).all() and (x < V).all()


def _as_float(bits):
    return (np.asarray(bits, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def test_gaussian_weights_within_the_binary32_error_bound(dev):
    """Off the grid the device's binary32 sum of the bias can differ from the
    exact one by up to about (r + 1) 2^-24 sum_j |W1[a][j] W2[j][v]|; after
    rounding to bf16 the two rows then differ by at most that bound plus one
    bf16 spacing (several spacings where U_k + bias nearly cancels), and are
    equal almost everywhere. Position 1 is compared (same anchor on both
    sides)."""
    B, V, r = 64, 8192, 256
    d = workloads.make_markov_draft(B, 1, V, r, seed=12, device="cpu", weights="gauss")
    L, x = run_gpu(d, dev)
    ref = run_oracle(d)
    a = _as_float(L[:, 0])
    b = _as_float(ref["logits"][:, 0])
    w1 = _as_float(workloads.bf16_bits(d.w1))
    w2t = _as_float(workloads.bf16_bits(d.w2t))
    s_abs = np.abs(w1[d.anchors.numpy()]) @ np.abs(w2t).T            # [B, V]
    u_abs = np.abs(_as_float(workloads.bf16_bits(d.base_logits))[:, 0])
    spacing = np.exp2(np.floor(np.log2(np.maximum(np.abs(b), 2.0 ** -126))) - 7)
    bound = spacing + 2.0 * (r + 2) * 2.0 ** -24 * (s_abs + u_abs)
    assert (np.abs(a - b) <= bound).all()
    assert (L[:, 0] == ref["logits"][:, 0]).mean() > 0.999
    agree = (x[:, 0] == ref["tokens"][:, 0]) | (ref["flags"][:, 0] != 0)
    assert agree.mean() >= 0.95


@pytest.mark.parametrize("what", ["anchor", "uniform", "nan", "neg_inf_row"])
def test_bad_data_sets_status(dev, what):
    d = workloads.make_markov_draft(6, 3, 1024, 64, seed=2, device="cpu")
    U, x0, u = d.base_logits.clone(), d.anchors.clone(), d.uniforms.clone()
    if what == "anchor":
        x0[2] = 1024
    elif what == "uniform":
        u[4, 1] = 1.0
    elif what == "nan":
        U[1, 0, 77] = float("nan")
    else:
        U[3, 2, :] = float("-inf")
    out = binding.dspark_draft_markov(U.to(dev), d.w1.to(dev), d.w2t.to(dev), x0.to(dev),
                                      u.to(dev), d.temperature)
    torch.cuda.synchronize()
    assert int(out["device_status"].item()) == 5
    tok = out["draft_tokens"].cpu().numpy()
    assert (tok >= 0).all() and (tok < 1024).all()


def test_draw_law_is_the_emitted_rows_softmax(dev):
    """The law of the device's draw itself: 16,384 requests with the same base
    rows and anchor but their own uniforms draw x_1 from softmax(L_1 / T) of
    the (shared) emitted row; chi-square against that law in float64."""
    from scipy import special
    from tests._law import chisq_pvalue
    B, gamma, V, r, T = 16384, 1, 64, 64, 0.8
    one = workloads.make_markov_draft(1, gamma, V, r, temperature=T, seed=31, device="cpu")
    u = torch.from_numpy(workloads.philox_uniforms(31, workloads.PURPOSE_DRAFT_SAMPLING, B)
                         .reshape(B, gamma))
    d = workloads.MarkovDraftInputs(one.base_logits.repeat(B, 1, 1), one.w1, one.w2t,
                                    one.anchors.repeat(B), u, T)
    L, x = run_gpu(d, dev)
    assert (L == L[0]).all()  # every request emits the same row
    z = (L[0, 0].astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    pv = chisq_pvalue(x[:, 0], special.softmax(z / T))
    assert pv > 1e-4, pv
