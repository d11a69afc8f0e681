"""Pins of the oracle's sequential drafter with the Markov head (DSpark paper,
section 3.1, "Sequential stage": equation 4, p_k = softmax(U_k + B_k), and
equation 5, B(x_{k-1}, .) = W1[x_{k-1}] W2).

Each pin checks the oracle against something other than itself:
  - bfloat16 rounding against torch's float32 -> bfloat16 conversion and a
    brute-force nearest search over all 65,536 bfloat16 patterns;
  - ties to even and the binary32-then-bfloat16 order on hand-built cases
    whose answers are stated in the test;
  - a zero head (W1 = 0) against scipy's softmax and numpy's searchsorted;
  - the two-token closed form p(0) = 1 / (1 + exp((L1 - L0) / T));
  - a head built so that each token forces a known successor (the chain is
    then x_k = succ^k(x_0), a closed form that a transposed W1/W2, a wrong
    previous token or a wrong row would break);
  - the block equals gamma one-position blocks chained by hand;
  - the law of each draw: the uniform-measure of every outcome equals the
    probability the oracle reports, and those probabilities equal scipy's
    softmax of the emitted row.
"""
import numpy as np
import pytest
import torch
from scipy.special import softmax

import oracle
from speculative_decoding_verification_41_gb300 import workloads


def bits(vals) -> np.ndarray:
    """bfloat16 patterns of values that bfloat16 holds exactly."""
    f = np.asarray(vals, np.float32)
    b = (f.view(np.uint32) >> 16).astype(np.uint16)
    back = (b.astype(np.uint32) << 16).view(np.float32)
    assert np.array_equal(back, f, equal_nan=True), "value not exact in bfloat16"
    return b


def as_float(b) -> np.ndarray:
    with np.errstate(invalid="ignore"):
        return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def draft(U, W1, W2t, x0, u, T, **kw):
    U = np.asarray(U, np.uint16)
    return oracle.markov_draft(U, W1, W2t, np.asarray(x0, np.int32),
                               np.asarray(u, np.float32).reshape(U.shape[0], U.shape[1]), T, **kw)


# ---------------------------------------------------------------------------
# bfloat16 rounding
# ---------------------------------------------------------------------------
def test_bf16_round_matches_torch_on_float32_values():
    rng = np.random.default_rng(0)
    x = np.concatenate([
        rng.standard_normal(20000) * 10.0 ** rng.integers(-30, 30, 20000),
        rng.uniform(-1, 1, 5000) * 2.0 ** -126,         # subnormal range
        [0.0, -0.0, 1.0, -1.0, 3.3895313892515355e38, 1e-45],
    ]).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = oracle.bf16_round(x.astype(np.float64))
    np.testing.assert_array_equal(got, ref)


def test_bf16_round_is_the_nearest_pattern_ties_to_even():
    """Brute force: every finite bfloat16 value, sorted; the oracle's result
    must be a nearest one, and at an exact midpoint the even significand."""
    allb = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    vals = as_float(allb)
    fin = np.isfinite(vals) & ~((allb == 0x8000))
    vals, pats = vals[fin], allb[fin]
    order = np.argsort(vals, kind="stable")
    vals, pats = vals[order], pats[order]
    rng = np.random.default_rng(1)
    x = rng.standard_normal(3000) * 2.0 ** rng.integers(-20, 20, 3000)
    mids = (vals[1000:1100] + vals[1001:1101]) / 2.0     # exact midpoints
    x = np.concatenate([x, mids, -mids])
    got = as_float(oracle.bf16_round(x))
    i = np.searchsorted(vals, x)
    lo, hi = vals[np.clip(i - 1, 0, len(vals) - 1)], vals[np.clip(i, 0, len(vals) - 1)]
    dlo, dhi = np.abs(x - lo), np.abs(hi - x)
    best = np.minimum(dlo, dhi)
    assert np.all(np.abs(got - x) == best)
    tie = dlo == dhi
    got_p = oracle.bf16_round(x[tie])
    assert np.all((got_p & 1) == 0)


# ---------------------------------------------------------------------------
# emitted logits: rounding order
# ---------------------------------------------------------------------------
def _one_position(u_val, bias_terms, T=1.0, V=8, r=64):
    """U_1 = u_val at every token; W1[0] . W2t[v] = sum of bias_terms for token
    v = 1 only (products of exact bfloat16 factors)."""
    U = np.tile(bits([u_val] * V), (1, 1, 1))
    W1 = np.zeros((V, r), np.uint16)
    W2t = np.zeros((V, r), np.uint16)
    for j, (a, b) in enumerate(bias_terms):
        W1[0, j] = bits([a])[0]
        W2t[1, j] = bits([b])[0]
    return draft(U, W1, W2t, [0], [0.5], T, want_logits=True)["logits"][0, 0]


@pytest.mark.parametrize("u_val,terms,want", [
    (1.0, [(0.5, 2.0 ** -7)], 1.0),                    # 1 + 2^-8: tie -> even (1.0)
    (1.0, [(0.5, 3 * 2.0 ** -7)], 1.015625),           # 1 + 3*2^-8: tie -> even (1 + 2^-6)
    (-1.0, [(0.5, -(2.0 ** -7))], -1.0),               # negative tie
    # 1 + 2^-8 + 2^-20 lies above the midpoint and binary32 holds it: rounds up
    (1.0, [(0.5, 2.0 ** -7), (2.0 ** -10, 2.0 ** -10)], 1.0078125),
    # 1 + 2^-8 + 2^-30 also lies above the midpoint, but binary32 holds only
    # 1 + 2^-8: rounding to binary32 first (the device's order) makes it a tie,
    # which goes to the even significand, 1.0
    (1.0, [(0.5, 2.0 ** -7), (2.0 ** -15, 2.0 ** -15)], 1.0),
])
def test_emitted_logit_rounding(u_val, terms, want):
    L = _one_position(u_val, terms)
    assert as_float(L[1]) == want
    assert as_float(L[0]) == u_val     # token 0 gets no bias


# ---------------------------------------------------------------------------
# zero head: the draw is the inverse CDF of softmax(U_k / T)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("T", [1.0, 0.7, 2.5])
def test_zero_head_samples_base_logits(T):
    B, g, V, r = 6, 5, 300, 64
    d = workloads.make_markov_draft(B, g, V, r, temperature=T, seed=3, device="cpu")
    U = workloads.bf16_bits(d.base_logits)
    W1 = np.zeros((V, r), np.uint16)
    out = draft(U, W1, workloads.bf16_bits(d.w2t), d.anchors.numpy(), d.uniforms.numpy(), T,
                want_logits=True)
    np.testing.assert_array_equal(out["logits"], U)        # bias 0: L = U exactly
    u = d.uniforms.numpy().astype(np.float64)
    for b in range(B):
        for k in range(g):
            p = softmax(as_float(U[b, k]) / T)
            y = int(np.searchsorted(np.cumsum(p), u[b, k], side="right"))
            if out["flags"][b, k]:
                continue
            assert out["tokens"][b, k] == y
            assert abs(out["probs"][b, k] - p[y]) < 1e-12
    # with no head the anchors cannot matter
    out2 = draft(U, W1, workloads.bf16_bits(d.w2t), (d.anchors.numpy() + 1) % V,
                 d.uniforms.numpy(), T)
    np.testing.assert_array_equal(out2["tokens"], out["tokens"])


@pytest.mark.parametrize("T", [1.0, 0.5, 3.0])
def test_two_token_closed_form(T):
    """L = (0.125, -0.25): W1[0] = (0.5, 0, ...), W2t[0] = (0.25, ...),
    W2t[1] = (-0.5, ...), U = 0. p(0) = 1 / (1 + exp((L1 - L0) / T)); the draw
    is token 0 below u = p(0) and token 1 above it."""
    V, r = 2, 64
    W1 = np.zeros((V, r), np.uint16)
    W2t = np.zeros((V, r), np.uint16)
    W1[0, 0] = bits([0.5])[0]
    W2t[0, 0] = bits([0.25])[0]
    W2t[1, 0] = bits([-0.5])[0]
    p0 = 1.0 / (1.0 + np.exp((-0.25 - 0.125) / T))
    U = np.zeros((1, 1, V), np.uint16)
    f0, f1 = np.float32(0), np.float32(1)
    below = np.nextafter(np.float32(p0), f0)                      # >= half an ulp below p(0)
    above = np.nextafter(np.nextafter(np.float32(p0), f1), f1)    # >= 1.5 ulp above
    for u, want in [(below, 0), (above, 1), (f0, 0), (np.nextafter(f1, f0), 1)]:
        out = draft(U, W1, W2t, [0], [u], T, want_logits=True)
        assert out["tokens"][0, 0] == want, (u, p0)
        assert abs(out["probs"][0, 0] - (p0 if want == 0 else 1 - p0)) < 1e-15
    np.testing.assert_array_equal(as_float(out["logits"][0, 0]), [0.125, -0.25])


# ---------------------------------------------------------------------------
# the Markov chain: each token forces its successor
# ---------------------------------------------------------------------------
def _successor_head(V, r, succ):
    """W1[a] = 0.5 on the 4 indices 4a..4a+3; W2t[succ(a)] = 0.5 on the same
    indices: B(a, succ(a)) = 1, every other bias 0."""
    W1 = np.zeros((V, r), np.uint16)
    W2t = np.zeros((V, r), np.uint16)
    for a in range(V):
        W1[a, 4 * a:4 * a + 4] = bits([0.5] * 4)
        W2t[succ[a], 4 * a:4 * a + 4] = bits([0.5] * 4)
    return W1, W2t


def test_chain_follows_the_successor_map():
    V, r, g, T = 16, 64, 12, 0.05      # bias / T = 20: the successor has p > 0.99999
    succ = [(5 * a + 3) % V for a in range(V)]
    W1, W2t = _successor_head(V, r, succ)
    rng = np.random.default_rng(4)
    B = 8
    U = (rng.uniform(-0.01, 0.01, (B, g, V)).astype(np.float32).view(np.uint32) >> 16
         ).astype(np.uint16)        # truncated to bfloat16
    x0 = rng.integers(0, V, B)
    u = rng.uniform(0.01, 0.99, (B, g)).astype(np.float32)
    out = draft(U, W1, W2t, x0, u, T)
    for b in range(B):
        x = int(x0[b])
        for k in range(g):
            x = succ[x]
            assert out["tokens"][b, k] == x
            assert out["probs"][b, k] > 0.9999


def test_block_is_the_chain_of_single_positions():
    B, g, V, r, T = 5, 6, 200, 64, 0.8
    d = workloads.make_markov_draft(B, g, V, r, temperature=T, seed=11, device="cpu")
    U = workloads.bf16_bits(d.base_logits)
    W1, W2t = workloads.bf16_bits(d.w1), workloads.bf16_bits(d.w2t)
    u = d.uniforms.numpy()
    blk = draft(U, W1, W2t, d.anchors.numpy(), u, T, want_logits=True)
    prev = d.anchors.numpy().copy()
    for k in range(g):
        one = draft(U[:, k:k + 1], W1, W2t, prev, u[:, k:k + 1], T, want_logits=True)
        np.testing.assert_array_equal(one["tokens"][:, 0], blk["tokens"][:, k])
        np.testing.assert_array_equal(one["logits"][:, 0], blk["logits"][:, k])
        prev = one["tokens"][:, 0]


def test_request_subset_matches_the_full_batch():
    B, g, V, r = 7, 3, 120, 128
    d = workloads.make_markov_draft(B, g, V, r, seed=5, device="cpu")
    args = (workloads.bf16_bits(d.base_logits), workloads.bf16_bits(d.w1),
            workloads.bf16_bits(d.w2t), d.anchors.numpy(), d.uniforms.numpy(), d.temperature)
    full = draft(*args, want_logits=True)
    sub = draft(*args, requests=[6, 2, 2], want_logits=True)
    for i, b in enumerate([6, 2, 2]):
        np.testing.assert_array_equal(sub["tokens"][i], full["tokens"][b])
        np.testing.assert_array_equal(sub["logits"][i], full["logits"][b])


# ---------------------------------------------------------------------------
# the law of each draw
# ---------------------------------------------------------------------------
def test_each_draw_has_the_softmax_law():
    """Position 1 of a 5-token vocabulary: sweeping the uniform over a fine
    grid, the fraction of the unit interval mapped to each token equals the
    probability reported for it, which equals scipy's softmax of the emitted
    row at T."""
    V, r, T = 5, 64, 0.9
    d = workloads.make_markov_draft(1, 1, V, r, temperature=T, seed=9, device="cpu")
    U = workloads.bf16_bits(d.base_logits)
    W1, W2t = workloads.bf16_bits(d.w1), workloads.bf16_bits(d.w2t)
    n = 4096
    grid = ((np.arange(n) + 0.5) / n).astype(np.float32)
    Ub = np.repeat(U, n, axis=0)
    out = draft(Ub, W1, W2t, np.repeat(d.anchors.numpy(), n), grid.reshape(n, 1), T,
                want_logits=True)
    p = softmax(as_float(out["logits"][0, 0]) / T)
    freq = np.bincount(out["tokens"][:, 0], minlength=V) / n
    assert np.abs(freq - p).max() <= 1.0 / n + 1e-12
    for y in range(V):
        sel = out["tokens"][:, 0] == y
        if sel.any():
            assert np.allclose(out["probs"][sel, 0], p[y], rtol=1e-12)


# ---------------------------------------------------------------------------
# bad inputs
# ---------------------------------------------------------------------------
def test_bad_inputs_are_errors():
    V, r = 16, 64
    U = np.zeros((1, 2, V), np.uint16)
    W = np.zeros((V, r), np.uint16)
    with pytest.raises(oracle.OracleError):
        draft(U, W, W, [V], [[0.1, 0.2]], 1.0)            # anchor outside [0, V)
    with pytest.raises(oracle.OracleError):
        draft(U, W, W, [0], [[0.1, 1.0]], 1.0)            # uniform not below 1
    U2 = U.copy()
    U2[0, 1, 3] = 0x7FC0                                   # NaN base logit
    with pytest.raises(oracle.OracleError):
        draft(U2, W, W, [0], [[0.1, 0.2]], 1.0)
    U3 = U.copy()
    U3[0, 0, :] = 0xFF80                                   # a row of -inf
    with pytest.raises(oracle.OracleError):
        draft(U3, W, W, [0], [[0.1, 0.2]], 1.0)
