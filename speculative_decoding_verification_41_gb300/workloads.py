"""Seeded synthetic workloads for DSpark verification and scheduling.

This module only generates inputs. It holds none of the verifier's or the
scheduler's arithmetic: the CUDA library and the CPU oracle both consume what it
produces. Randomness that the method itself consumes (the ratio-test and
resample uniforms) is drawn here and passed in as an input.

Counter-based generator: Philox4x32-10 as published by Salmon, Moraes, Dror and
Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11): 10 rounds of
(hi, lo) = mulhilo(M, x) with multipliers 0xD2511F53 / 0xCD9E8D57 and a Weyl key
schedule with increments 0x9E3779B9 / 0xBB67AE85. Streams are split as
key = (seed, 0), counter = (index, purpose, 0, 0); a uniform is
(word >> 8) * 2^-24, a value on the 2^-24 grid that float32 holds exactly.

Purposes: 0 logit normals (tiny case only), 1 draft-token sampling,
2 verification uniforms, 3 per-request rho / verify-length draws, 4 anchor
tokens of the sequential drafter.

The workload shapes stand in for the DSpark paper's evaluation (section 4.1:
Qwen3-class vocabularies of 151,936 tokens, temperature 1.0; section 5.1:
DeepSeek-V4-class vocabulary of 129,280; block size gamma = 16 as in section
2.2). No benchmark item or trained weight is used: logits are Gaussian with a
Zipf log-frequency bias, and the draft logits are a noisy copy of the target's.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np
import torch

# ---------------------------------------------------------------------------
# Philox4x32-10 (Salmon et al., SC'11)
# ---------------------------------------------------------------------------
_PHILOX_M0 = np.uint64(0xD2511F53)
_PHILOX_M1 = np.uint64(0xCD9E8D57)
_PHILOX_W0 = np.uint64(0x9E3779B9)
_PHILOX_W1 = np.uint64(0xBB67AE85)
_MASK32 = np.uint64(0xFFFFFFFF)

PURPOSE_NORMALS = 0
PURPOSE_DRAFT_SAMPLING = 1
PURPOSE_VERIFY_UNIFORMS = 2
PURPOSE_REQUEST_PARAMS = 3
PURPOSE_ANCHORS = 4


def philox4x32_10(counters: np.ndarray, key) -> np.ndarray:
    """Philox4x32 with 10 rounds. counters: [N, 4] uint32; key: 2 uint32 words.
    Returns [N, 4] uint32."""
    c = np.asarray(counters, dtype=np.uint64).reshape(-1, 4)
    x0, x1, x2, x3 = (c[:, i].copy() for i in range(4))
    k0 = np.uint64(int(key[0]) & 0xFFFFFFFF)
    k1 = np.uint64(int(key[1]) & 0xFFFFFFFF)
    for rnd in range(10):
        if rnd:
            k0 = (k0 + _PHILOX_W0) & _MASK32
            k1 = (k1 + _PHILOX_W1) & _MASK32
        p0 = _PHILOX_M0 * x0
        p1 = _PHILOX_M1 * x2
        x0, x1, x2, x3 = ((p1 >> np.uint64(32)) ^ x1 ^ k0, p1 & _MASK32,
                          (p0 >> np.uint64(32)) ^ x3 ^ k1, p0 & _MASK32)
    return np.stack([x0, x1, x2, x3], axis=1).astype(np.uint32)


def philox_words(seed: int, purpose: int, n: int, start: int = 0) -> np.ndarray:
    """n consecutive 32-bit words of stream (seed, purpose), from word `start`."""
    first = start // 4
    last = (start + n + 3) // 4
    idx = np.arange(first, last, dtype=np.uint64)
    ctr = np.zeros((idx.shape[0], 4), np.uint64)
    ctr[:, 0] = idx & _MASK32
    ctr[:, 1] = np.uint64(purpose)
    ctr[:, 2] = idx >> np.uint64(32)
    words = philox4x32_10(ctr, (seed, 0)).reshape(-1)
    off = start - first * 4
    return words[off:off + n]


def philox_uniforms(seed: int, purpose: int, n: int, start: int = 0) -> np.ndarray:
    """Uniforms in [0, 1) on the 2^-24 grid (exact in float32), float32 [n]."""
    w = philox_words(seed, purpose, n, start)
    return ((w >> np.uint32(8)).astype(np.float64) * 2.0 ** -24).astype(np.float32)


def philox_normals(seed: int, purpose: int, n: int) -> np.ndarray:
    """Standard normals by the Box-Muller transform of Philox uniforms, float64."""
    m = (n + 1) // 2
    w = philox_words(seed, purpose, 2 * m).reshape(m, 2).astype(np.float64)
    u1 = (np.floor(w[:, 0] / 256.0) + 1.0) * 2.0 ** -24  # (0, 1]
    u2 = np.floor(w[:, 1] / 256.0) * 2.0 ** -24          # [0, 1)
    rad = np.sqrt(-2.0 * np.log(u1))
    z = np.empty(2 * m)
    z[0::2] = rad * np.cos(2.0 * math.pi * u2)
    z[1::2] = rad * np.sin(2.0 * math.pi * u2)
    return z[:n]


# ---------------------------------------------------------------------------
# Workload containers
# ---------------------------------------------------------------------------
@dataclass
class VerifyInputs:
    """Inputs of one batched verification call (all tensors on one device).

    target_logits [rows_t, V] and draft_logits [rows_d, V] are row-major; request
    r's target rows start at target_row_off[r] (dense when None: r*(gamma+1)) and
    its draft rows at draft_row_off[r] (dense: r*gamma)."""
    target_logits: torch.Tensor
    draft_logits: torch.Tensor
    draft_tokens: torch.Tensor      # [B, gamma] int32
    verify_len: torch.Tensor        # [B] int32
    uniforms: torch.Tensor          # [B, gamma+1] float32
    temperature: float              # a binary32 value (see __post_init__)
    target_row_off: Optional[torch.Tensor] = None  # [B+1] int64
    draft_row_off: Optional[torch.Tensor] = None   # [B+1] int64
    name: str = ""
    meta: dict = field(default_factory=dict)

    def __post_init__(self):
        # the verification call takes the temperature as a binary32 value:
        # the value kept here is that one, so that every consumer (the call,
        # the oracle) is handed the same temperature
        self.temperature = float(np.float32(self.temperature))

    @property
    def B(self) -> int:
        return int(self.draft_tokens.shape[0])

    @property
    def gamma(self) -> int:
        return int(self.draft_tokens.shape[1])

    @property
    def V(self) -> int:
        return int(self.target_logits.shape[-1])

    def to(self, device) -> "VerifyInputs":
        mv = lambda t: None if t is None else t.to(device)
        return VerifyInputs(mv(self.target_logits), mv(self.draft_logits), mv(self.draft_tokens),
                            mv(self.verify_len), mv(self.uniforms), self.temperature,
                            mv(self.target_row_off), mv(self.draft_row_off), self.name,
                            dict(self.meta))

    def logit_bytes(self, ell: Optional[np.ndarray] = None) -> int:
        """Algorithmic bytes of one verification: every verified target row
        (l_r + 1 per request) and draft row (l_r) read once."""
        if ell is None:
            ell = self.verify_len.cpu().numpy()
        rows = int((2 * ell.astype(np.int64) + 1).sum())
        return rows * self.V * self.target_logits.element_size()


@dataclass
class ScheduleInputs:
    confidences: torch.Tensor   # [R, gamma] float32 in [0, 1]
    step_time_ms: torch.Tensor  # [n_profile] float64, T(N) for N = 0..n_profile-1
    name: str = ""

    @property
    def R(self) -> int:
        return int(self.confidences.shape[0])

    @property
    def gamma(self) -> int:
        return int(self.confidences.shape[1])


# ---------------------------------------------------------------------------
# Generators
# ---------------------------------------------------------------------------
def _request_params(seed: int, B: int):
    """Per-request uniform pair (for rho and for a verify length), purpose 3."""
    w = philox_uniforms(seed, PURPOSE_REQUEST_PARAMS, 2 * B).astype(np.float64).reshape(B, 2)
    return w[:, 0], w[:, 1]


def zipf_bias(V: int, s: float = 1.1) -> np.ndarray:
    """Log-frequency bias -s*ln(v+1): token id 0 is the most frequent."""
    return -s * np.log(np.arange(1, V + 1, dtype=np.float64))


def _sample_rows_inverse_cdf(logits: torch.Tensor, temperature: float, u: torch.Tensor,
                             chunk: int = 512) -> torch.Tensor:
    """Draw one token per row from softmax(logits / T) with the given uniforms.
    This is the drafter's sampling (it produces the draft tokens under test)."""
    out = torch.empty(logits.shape[0], dtype=torch.int64, device=logits.device)
    for s in range(0, logits.shape[0], chunk):
        z = logits[s:s + chunk].float() / temperature
        p = torch.softmax(z, dim=-1)
        c = torch.cumsum(p, dim=-1)
        tgt = (u[s:s + chunk].to(c.dtype) * c[:, -1]).unsqueeze(1)
        idx = torch.searchsorted(c, tgt, right=True).squeeze(1)
        out[s:s + chunk] = idx.clamp_(0, logits.shape[1] - 1)
    return out


def make_tiny(device="cpu") -> VerifyInputs:
    """B=4 requests, gamma=4, V=32, float32. Target logits ~ N(0, 2^2) (seed 0);
    draft = 0.8*target + N(0, 1); draft tokens sampled from the draft softmax at
    T=1 with Philox seed 1; verification uniforms Philox seed 1 (purpose 2);
    every position verified."""
    B, gamma, V, T = 4, 4, 32, 1.0
    n_t = B * (gamma + 1) * V
    n_d = B * gamma * V
    z = philox_normals(0, PURPOSE_NORMALS, n_t + n_d)
    zt = (2.0 * z[:n_t]).reshape(B, gamma + 1, V)
    zd = 0.8 * zt[:, :gamma, :] + z[n_t:].reshape(B, gamma, V)
    zt32 = zt.astype(np.float32)
    zd32 = zd.astype(np.float32)
    us = philox_uniforms(1, PURPOSE_DRAFT_SAMPLING, B * gamma).astype(np.float64)
    tokens = np.zeros((B, gamma), np.int32)
    for i in range(B * gamma):
        row = zd32.reshape(B * gamma, V)[i].astype(np.float64) / T
        w = np.exp(row - row.max())
        cdf = np.cumsum(w)
        tokens.reshape(-1)[i] = min(int(np.searchsorted(cdf, us[i] * cdf[-1], side="right")), V - 1)
    uni = philox_uniforms(1, PURPOSE_VERIFY_UNIFORMS, B * (gamma + 1)).reshape(B, gamma + 1)
    dev = torch.device(device)
    return VerifyInputs(
        torch.from_numpy(zt32.reshape(B * (gamma + 1), V)).to(dev),
        torch.from_numpy(zd32.reshape(B * gamma, V)).to(dev),
        torch.from_numpy(tokens).to(dev),
        torch.full((B,), gamma, dtype=torch.int32, device=dev),
        torch.from_numpy(uni).to(dev), T, name="tiny_b4_g4_v32_f32")


def make_verify(B: int, gamma: int, V: int, dtype: torch.dtype, temperature: float,
                rho=(0.85, 0.85), verify_len="full", ragged: bool = False, seed: int = 7,
                device="cuda", name: str = "", pad_rows: int = 0) -> VerifyInputs:
    """Synthetic verification batch shaped like the paper's workloads.

    Target logits: 3*N(0,1) - 1.1*ln(v+1). Draft logits: rho_r*target +
    sqrt(1-rho_r^2)*3*N(0,1), with rho_r ~ U(rho[0], rho[1]) per request.
    verify_len: "full" (every position), "uniform" (l_r ~ U{1..gamma}), or an
    int array. ragged=True packs the rows with offsets (l_r+1 target rows and
    l_r draft rows per request); otherwise rows are laid out dense."""
    dev = torch.device(device)
    u_rho, u_len = _request_params(seed, B)
    rho_r = rho[0] + (rho[1] - rho[0]) * u_rho
    if isinstance(verify_len, str):
        if verify_len == "full":
            ell = np.full(B, gamma, np.int32)
        elif verify_len == "uniform":
            ell = (1 + np.floor(u_len * gamma)).astype(np.int32)
        else:
            raise ValueError(verify_len)
    else:
        ell = np.asarray(verify_len, np.int32).reshape(B)
    if ragged:
        t_cnt = ell.astype(np.int64) + 1
        d_cnt = ell.astype(np.int64)
    else:
        t_cnt = np.full(B, gamma + 1, np.int64)
        d_cnt = np.full(B, gamma, np.int64)
    t_off = np.concatenate([[0], np.cumsum(t_cnt)]).astype(np.int64)
    d_off = np.concatenate([[0], np.cumsum(d_cnt)]).astype(np.int64)
    rows_t = int(t_off[-1]) + pad_rows
    rows_d = int(d_off[-1]) + pad_rows

    gen = torch.Generator(device=dev)
    gen.manual_seed(seed * 1000003 + 17)
    bias = torch.from_numpy(zipf_bias(V)).to(dev, torch.float32)
    tl = torch.empty(rows_t, V, dtype=dtype, device=dev)
    dl = torch.empty(rows_d, V, dtype=dtype, device=dev)
    # pad rows (never referenced) still hold finite logits
    for r0 in range(0, B, 64):
        r1 = min(B, r0 + 64)
        for r in range(r0, r1):
            nt, nd = int(t_cnt[r]), int(d_cnt[r])
            zt = 3.0 * torch.randn(nt, V, generator=gen, device=dev) + bias
            tl[t_off[r]:t_off[r] + nt] = zt.to(dtype)
            if nd:
                noise = torch.randn(nd, V, generator=gen, device=dev)
                zd = float(rho_r[r]) * zt[:nd] + math.sqrt(1.0 - float(rho_r[r]) ** 2) * 3.0 * noise
                dl[d_off[r]:d_off[r] + nd] = zd.to(dtype)
    if pad_rows:
        tl[rows_t - pad_rows:] = (3.0 * torch.randn(pad_rows, V, generator=gen, device=dev)).to(dtype)
        dl[rows_d - pad_rows:] = (3.0 * torch.randn(pad_rows, V, generator=gen, device=dev)).to(dtype)

    # draft tokens: one draw per draft position from the draft softmax at T
    us = torch.from_numpy(philox_uniforms(seed, PURPOSE_DRAFT_SAMPLING, B * gamma)).to(dev)
    tokens = torch.zeros(B, gamma, dtype=torch.int32, device=dev)
    rows, which = [], []
    for r in range(B):
        for k in range(int(d_cnt[r])):
            rows.append(int(d_off[r]) + k)
            which.append(r * gamma + k)
    if rows:
        ridx = torch.tensor(rows, dtype=torch.int64, device=dev)
        widx = torch.tensor(which, dtype=torch.int64, device=dev)
        sampled = torch.empty(len(rows), dtype=torch.int64, device=dev)
        for s in range(0, len(rows), 1024):
            sub = dl.index_select(0, ridx[s:s + 1024])
            sampled[s:s + 1024] = _sample_rows_inverse_cdf(sub, temperature, us[widx[s:s + 1024]])
        tokens.view(-1)[widx] = sampled.to(torch.int32)

    uni = torch.from_numpy(
        philox_uniforms(seed, PURPOSE_VERIFY_UNIFORMS, B * (gamma + 1)).reshape(B, gamma + 1)).to(dev)
    vi = VerifyInputs(tl, dl, tokens, torch.from_numpy(ell).to(dev), uni, float(temperature),
                      torch.from_numpy(t_off).to(dev) if ragged else None,
                      torch.from_numpy(d_off).to(dev) if ragged else None,
                      name=name or f"b{B}_g{gamma}_v{V}_{str(dtype).split('.')[-1]}",
                      meta={"rho": rho_r, "seed": seed})
    return vi


def step_time_profile(n: int, base_ms=4.0, slope_ms=0.006, knee=2048, slope2_ms=0.02) -> np.ndarray:
    """Step-time table T(N) in ms for N = 0..n-1: base + slope*min(N, knee) +
    slope2*max(N - knee, 0) (continuous piecewise linear)."""
    N = np.arange(n, dtype=np.float64)
    return base_ms + slope_ms * np.minimum(N, knee) + slope2_ms * np.maximum(N - knee, 0.0)


def make_confidences(R: int, gamma: int, seed: int = 7) -> np.ndarray:
    """c_{r,k} ~ Beta(8 * 0.9^k, 2), k = 1..gamma (numpy PCG64 stream)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    k = np.arange(1, gamma + 1, dtype=np.float64)
    c = rng.beta(8.0 * 0.9 ** k, 2.0, size=(R, gamma))
    return c.astype(np.float32)


def make_schedule(R: int = 512, gamma: int = 16, seed: int = 7, device="cuda",
                  flat_profile: bool = False) -> ScheduleInputs:
    """Scheduler inputs: Beta confidences and the piecewise-linear T(N) profile
    (flat_profile=True: constant T, every candidate admitted)."""
    n = R * (gamma + 1) + 1
    prof = np.full(n, 4.0) if flat_profile else step_time_profile(n)
    dev = torch.device(device)
    return ScheduleInputs(torch.from_numpy(make_confidences(R, gamma, seed)).to(dev),
                          torch.from_numpy(prof).to(dev),
                          name=f"sched_r{R}_g{gamma}" + ("_flat" if flat_profile else ""))


@dataclass
class MarkovDraftInputs:
    """Inputs of the sequential stage with the Markov head (DSpark paper,
    section 3.1): base logits U [B, gamma, V] bf16 from the parallel stage, the
    head's factors W1 [V, r] and W2 stored transposed as w2t [V, r] (row v =
    column v of W2), both bf16, anchor tokens [B] int32 and one uniform per
    position [B, gamma] float32."""
    base_logits: torch.Tensor
    w1: torch.Tensor
    w2t: torch.Tensor
    anchors: torch.Tensor
    uniforms: torch.Tensor
    temperature: float              # a binary32 value, as the drafter's call takes it
    name: str = ""

    def __post_init__(self):
        self.temperature = float(np.float32(self.temperature))

    @property
    def B(self) -> int:
        return int(self.base_logits.shape[0])

    @property
    def gamma(self) -> int:
        return int(self.base_logits.shape[1])

    @property
    def V(self) -> int:
        return int(self.base_logits.shape[2])

    @property
    def r(self) -> int:
        return int(self.w1.shape[1])

    def to(self, device) -> "MarkovDraftInputs":
        return MarkovDraftInputs(self.base_logits.to(device), self.w1.to(device),
                                 self.w2t.to(device), self.anchors.to(device),
                                 self.uniforms.to(device), self.temperature, self.name)


def make_markov_draft(B: int, gamma: int, V: int, r: int = 256, temperature: float = 0.7,
                      seed: int = 7, device="cuda", weights: str = "grid",
                      name: str = "") -> MarkovDraftInputs:
    """Synthetic drafter inputs (random weights: the pages publish no trained head).

    Base logits: 3*N(0,1) - 1.1*ln(v+1), rounded to bf16, like the verifier's
    target rows. weights="grid": W1 and W2 entries k/256 with k uniform on
    {-127..127} (an int8-like grid; the bias B(a, v) then has a standard
    deviation of about 1.3 and every partial sum of W1[a] . W2[:, v] is exact in
    binary32). weights="gauss": N(0, 0.29^2) entries rounded to bf16.
    Anchors: Philox words (purpose 4) mod V; uniforms: Philox (purpose 1)."""
    dev = torch.device(device)
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed * 7919 + 101)
    if weights == "grid":
        w1 = (torch.randint(-127, 128, (V, r), generator=gen, device=dev).float() / 256.0)
        w2t = (torch.randint(-127, 128, (V, r), generator=gen, device=dev).float() / 256.0)
    elif weights == "gauss":
        w1 = 0.29 * torch.randn(V, r, generator=gen, device=dev)
        w2t = 0.29 * torch.randn(V, r, generator=gen, device=dev)
    else:
        raise ValueError(weights)
    bias = torch.from_numpy(zipf_bias(V)).to(dev, torch.float32)
    U = torch.empty(B, gamma, V, dtype=torch.bfloat16, device=dev)
    for b in range(B):
        U[b] = (3.0 * torch.randn(gamma, V, generator=gen, device=dev) + bias).to(torch.bfloat16)
    anchors = (philox_words(seed, PURPOSE_ANCHORS, B).astype(np.int64) % V).astype(np.int32)
    uni = philox_uniforms(seed, PURPOSE_DRAFT_SAMPLING, B * gamma).reshape(B, gamma)
    return MarkovDraftInputs(U, w1.to(torch.bfloat16), w2t.to(torch.bfloat16),
                             torch.from_numpy(anchors).to(dev), torch.from_numpy(uni).to(dev),
                             float(temperature),
                             name or f"draft_b{B}_g{gamma}_v{V}_r{r}_{weights}")


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """bfloat16 tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# The five named workloads (names state the sizes).
CONFIGS = {
    "tiny_b4_g4_v32_f32": dict(kind="tiny"),
    "b64_g16_v151936_bf16": dict(B=64, gamma=16, V=151936, dtype=torch.bfloat16, temperature=1.0,
                                 rho=(0.85, 0.85), verify_len="full", ragged=False),
    "b256_g16_v129280_bf16": dict(B=256, gamma=16, V=129280, dtype=torch.bfloat16, temperature=0.7,
                                  rho=(0.6, 0.95), verify_len="full", ragged=False),
    "ragged_b1024_g16_v151936_f32": dict(B=1024, gamma=16, V=151936, dtype=torch.float32,
                                         temperature=1.0, rho=(0.5, 0.95), verify_len="uniform",
                                         ragged=True),
    "sched_r512_g16_v129280_bf16": dict(kind="scheduled", R=512, gamma=16, V=129280,
                                        dtype=torch.bfloat16, temperature=1.0, rho=(0.6, 0.95)),
}


def make_config(name: str, device="cuda", verify_len=None) -> VerifyInputs:
    """Build a named workload. For the scheduled workload, pass the verify
    lengths that the scheduler chose (host int array)."""
    cfg = dict(CONFIGS[name])
    kind = cfg.pop("kind", "verify")
    if kind == "tiny":
        return make_tiny(device)
    if kind == "scheduled":
        if verify_len is None:
            raise ValueError("the scheduled workload needs the scheduler's verify lengths")
        return make_verify(cfg["R"], cfg["gamma"], cfg["V"], cfg["dtype"], cfg["temperature"],
                           rho=cfg["rho"], verify_len=np.asarray(verify_len), ragged=True,
                           device=device, name=name)
    return make_verify(device=device, name=name, **cfg)
