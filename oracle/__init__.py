"""CPU oracle for DSpark verification and scheduling (plain C, IEEE double).

TEST INFRASTRUCTURE. Only the test suite, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / reference leg of ``bench.py`` may import this module. It
shares no code with the CUDA library in ``speculative_decoding_verification_41_gb300``
and is never called by it.

The C source (``dspark_oracle.c``) states the definitions it follows:
"DSpark: Confidence-Scheduled Speculative Decoding with Semi-Autoregressive
Generation", section 2.1 (ratio test, first-reject truncation), section 1
(bonus token), Appendix 8 (fresh token from p_t, acceptance = sum min), section
3.2.2 and the Chinese translation page's Algorithm 1 (prefix scheduler), and
section 5.2 (global search without the early-stopping break).

Parity pins (tests/test_oracle_*.py): Appendix 8's worked numbers, the closed
form sum_v min(p_t, p_d) of equation 8, exact interval enumeration of the
emitted law (= p_t) on vocabularies of at most 8, scipy's softmax, and an
exhaustive search of the scheduler objective on tiny batches.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dspark_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

F32, BF16, F64 = 0, 1, 2
FLAG_CDF_NEAR_TIE, FLAG_ZERO_RESIDUAL, FLAG_CDF_OVERRUN = 1, 2, 4

_lock = threading.Lock()
_lib = None

# IEEE semantics on both build hosts: no fast-math, no a*b+c contraction into
# fused multiply-adds (aarch64 gcc contracts by default).
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
          "-fno-fast-math", "-Wall", "-Wextra"]


def build(src: str = _SRC, out: str = _LIB_PATH, extra_flags=()) -> str:
    """Compile the oracle into a shared library with gcc; returns its path."""
    os.makedirs(os.path.dirname(out), exist_ok=True)
    cmd = ["gcc", *CFLAGS, *extra_flags, "-o", out, src, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return out


def _setup(lib):
    c_i32p = ctypes.POINTER(ctypes.c_int32)
    c_i64p = ctypes.POINTER(ctypes.c_int64)
    c_f64p = ctypes.POINTER(ctypes.c_double)
    lib.oracle_verify.restype = ctypes.c_int
    lib.oracle_verify.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, c_i32p, c_i32p, c_f64p,
        ctypes.c_double, ctypes.c_int32, ctypes.c_int32, ctypes.c_int64,
        c_i64p, c_i64p, c_i32p, c_i32p, c_f64p, c_i32p, ctypes.c_int32]
    lib.oracle_softmax_row.restype = ctypes.c_int
    lib.oracle_softmax_row.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int64,
                                       ctypes.c_double, c_f64p]
    lib.oracle_schedule.restype = ctypes.c_int
    lib.oracle_schedule.argtypes = [
        ctypes.POINTER(ctypes.c_float), c_f64p, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int32, c_i32p, c_f64p, c_i64p, c_i32p]
    lib.oracle_schedule_path.restype = ctypes.c_int
    lib.oracle_schedule_path.argtypes = [
        ctypes.POINTER(ctypes.c_float), c_f64p, ctypes.c_int64, ctypes.c_int32,
        ctypes.c_int32, c_i64p, c_f64p, c_i64p]
    lib.oracle_acceptance.restype = ctypes.c_int
    lib.oracle_acceptance.argtypes = [
        ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, c_i32p, ctypes.c_double, ctypes.c_int32,
        ctypes.c_int32, ctypes.c_int64, c_i64p, c_i64p, c_f64p, ctypes.c_int32]
    lib.oracle_schedule_topk.restype = ctypes.c_int
    lib.oracle_schedule_topk.argtypes = [
        ctypes.POINTER(ctypes.c_float), ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, c_i32p,
        c_i64p]
    lib.oracle_schedule_threshold.restype = ctypes.c_int
    lib.oracle_schedule_threshold.argtypes = [
        ctypes.POINTER(ctypes.c_float), ctypes.c_int32, ctypes.c_int32, ctypes.c_float, c_i32p]
    c_u16p = ctypes.POINTER(ctypes.c_uint16)
    lib.oracle_bf16_round.restype = ctypes.c_int
    lib.oracle_bf16_round.argtypes = [c_f64p, ctypes.c_int64, c_u16p]
    lib.oracle_markov_draft.restype = ctypes.c_int
    lib.oracle_markov_draft.argtypes = [
        c_u16p, c_u16p, c_u16p, c_i32p, ctypes.POINTER(ctypes.c_float), ctypes.c_double,
        ctypes.c_int32, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, c_i32p, ctypes.c_int32,
        c_i32p, c_f64p, c_i32p, c_u16p, ctypes.c_int32]
    lib.oracle_max_threads.restype = ctypes.c_int
    lib.oracle_max_threads.argtypes = []
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library."""
    global _lib
    with _lock:
        if path is not None:
            return _setup(ctypes.CDLL(path))
        if _lib is None:
            if (not os.path.exists(_LIB_PATH)
                    or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC)):
                build()
            _lib = _setup(ctypes.CDLL(_LIB_PATH))
        return _lib


def _ptr(a, ctype):
    return a.ctypes.data_as(ctypes.POINTER(ctype))


def _logits_and_dtype(a: np.ndarray):
    """Accept float32, float64 or bfloat16 stored as uint16 bit patterns."""
    if a.dtype == np.float32:
        return np.ascontiguousarray(a), F32
    if a.dtype == np.float64:
        return np.ascontiguousarray(a), F64
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a), BF16
    raise TypeError(f"oracle logits must be float32, float64 or uint16 (bf16 bits), got {a.dtype}")


class OracleError(RuntimeError):
    pass


def verify(target_logits, draft_logits, draft_tokens, verify_len, uniforms, temperature,
           target_row_off=None, draft_row_off=None, nthreads=1, lib=None):
    """Batched verification. Shapes: target [rows_t, V], draft [rows_d, V]
    (dense: rows_t = B*(gamma+1), rows_d = B*gamma), draft_tokens [B, gamma],
    verify_len [B], uniforms [B, gamma+1] (widened exactly to float64).

    Returns a dict: accepted_len [B], emitted [B, gamma+1], probs [B, gamma, 2],
    flags [B, gamma+1] (flags[:, k-1] = near tie at decision k; flags[:, gamma]
    = resample flag bits FLAG_*)."""
    lib = lib or load()
    tl, dtype = _logits_and_dtype(target_logits)
    dl, dtype_d = _logits_and_dtype(draft_logits)
    if dtype != dtype_d:
        raise TypeError("target and draft logits must share a dtype")
    V = tl.shape[-1]
    if dl.shape[-1] != V:
        raise ValueError("vocabulary mismatch")
    x = np.ascontiguousarray(draft_tokens, dtype=np.int32)
    B, gamma = x.shape
    ell = np.ascontiguousarray(verify_len, dtype=np.int32).reshape(B)
    u = np.ascontiguousarray(uniforms, dtype=np.float64).reshape(B, gamma + 1)
    toff = None if target_row_off is None else np.ascontiguousarray(target_row_off, dtype=np.int64)
    doff = None if draft_row_off is None else np.ascontiguousarray(draft_row_off, dtype=np.int64)
    acc = np.zeros(B, np.int32)
    emitted = np.zeros((B, gamma + 1), np.int32)
    probs = np.zeros((B, gamma, 2), np.float64)
    flags = np.zeros((B, gamma + 1), np.int32)
    rc = lib.oracle_verify(
        tl.ctypes.data, dl.ctypes.data, dtype, _ptr(x, ctypes.c_int32), _ptr(ell, ctypes.c_int32),
        _ptr(u, ctypes.c_double), float(temperature), B, gamma, V,
        None if toff is None else _ptr(toff, ctypes.c_int64),
        None if doff is None else _ptr(doff, ctypes.c_int64),
        _ptr(acc, ctypes.c_int32), _ptr(emitted, ctypes.c_int32), _ptr(probs, ctypes.c_double),
        _ptr(flags, ctypes.c_int32), int(nthreads))
    if rc != 0:
        raise OracleError(f"oracle_verify returned {rc}")
    return {"accepted_len": acc, "emitted": emitted, "probs": probs, "flags": flags}


def softmax_row(logits, temperature, lib=None):
    """p(v) of one row at temperature T, float64."""
    lib = lib or load()
    z, dtype = _logits_and_dtype(np.asarray(logits).reshape(-1))
    out = np.zeros(z.shape[0], np.float64)
    rc = lib.oracle_softmax_row(z.ctypes.data, dtype, z.shape[0], float(temperature),
                                _ptr(out, ctypes.c_double))
    if rc != 0:
        raise OracleError(f"oracle_softmax_row returned {rc}")
    return out


def schedule(confidences, step_time, early_stop=True, lib=None):
    """Prefix scheduler. confidences [R, gamma] (float32), step_time T(N) for
    N = 0..len-1. Returns dict: verify_len [R], theta_best, n_admitted, near_ties."""
    lib = lib or load()
    c = np.ascontiguousarray(confidences, dtype=np.float32)
    R, gamma = c.shape
    T = np.ascontiguousarray(step_time, dtype=np.float64)
    ell = np.zeros(R, np.int32)
    theta = ctypes.c_double(0.0)
    n_adm = ctypes.c_int64(0)
    ties = ctypes.c_int32(0)
    rc = lib.oracle_schedule(_ptr(c, ctypes.c_float), _ptr(T, ctypes.c_double), T.shape[0], R,
                             gamma, 1 if early_stop else 0, _ptr(ell, ctypes.c_int32),
                             ctypes.byref(theta), ctypes.byref(n_adm), ctypes.byref(ties))
    if rc != 0:
        raise OracleError(f"oracle_schedule returned {rc}")
    return {"verify_len": ell, "theta_best": theta.value, "n_admitted": n_adm.value,
            "near_ties": ties.value}


def schedule_path(confidences, step_time, lib=None):
    """Algorithm 1's greedy admission path without the break. Returns dict:
    order [|E|] (flattened index r*gamma + j - 1 of each candidate in admission
    order) and theta [|E| + 1] (Theta after the first n admissions)."""
    lib = lib or load()
    c = np.ascontiguousarray(confidences, dtype=np.float32)
    R, gamma = c.shape
    T = np.ascontiguousarray(step_time, dtype=np.float64)
    order = np.zeros(R * gamma, np.int64)
    theta = np.zeros(R * gamma + 1, np.float64)
    nE = ctypes.c_int64(0)
    rc = lib.oracle_schedule_path(_ptr(c, ctypes.c_float), _ptr(T, ctypes.c_double), T.shape[0],
                                  R, gamma, _ptr(order, ctypes.c_int64),
                                  _ptr(theta, ctypes.c_double), ctypes.byref(nE))
    if rc != 0:
        raise OracleError(f"oracle_schedule_path returned {rc}")
    return {"order": order[:nE.value], "theta": theta[:nE.value + 1]}


def acceptance(target_logits, draft_logits, verify_len, temperature, gamma,
               target_row_off=None, draft_row_off=None, nthreads=1, lib=None):
    """Acceptance probability sum_v min(p_t^k(v), p_d^k(v)) of every verified
    position k = 1..l_r (equation 8), from the same row layout as verify.
    Returns rates [B, gamma] float64, -1 beyond each l_r."""
    lib = lib or load()
    tl, dtype = _logits_and_dtype(target_logits)
    dl, dtype_d = _logits_and_dtype(draft_logits)
    if dtype != dtype_d:
        raise TypeError("target and draft logits must share a dtype")
    V = tl.shape[-1]
    if dl.shape[-1] != V:
        raise ValueError("vocabulary mismatch")
    ell = np.ascontiguousarray(verify_len, dtype=np.int32).reshape(-1)
    B = ell.shape[0]
    toff = None if target_row_off is None else np.ascontiguousarray(target_row_off, dtype=np.int64)
    doff = None if draft_row_off is None else np.ascontiguousarray(draft_row_off, dtype=np.int64)
    rates = np.zeros((B, gamma), np.float64)
    rc = lib.oracle_acceptance(
        tl.ctypes.data, dl.ctypes.data, dtype, _ptr(ell, ctypes.c_int32), float(temperature), B,
        gamma, V, None if toff is None else _ptr(toff, ctypes.c_int64),
        None if doff is None else _ptr(doff, ctypes.c_int64), _ptr(rates, ctypes.c_double),
        int(nthreads or 1))
    if rc != 0:
        raise OracleError(f"oracle_acceptance returned {rc}")
    return rates


def schedule_topk(confidences, K: int, lib=None):
    """Top-K admission of the production scheduler: the first min(K, |E|)
    candidates in Algorithm 1's order. Returns dict: verify_len [R], n_admitted."""
    lib = lib or load()
    c = np.ascontiguousarray(confidences, dtype=np.float32)
    R, gamma = c.shape
    ell = np.zeros(R, np.int32)
    n_adm = ctypes.c_int64(0)
    rc = lib.oracle_schedule_topk(_ptr(c, ctypes.c_float), R, gamma, int(K),
                                  _ptr(ell, ctypes.c_int32), ctypes.byref(n_adm))
    if rc != 0:
        raise OracleError(f"oracle_schedule_topk returned {rc}")
    return {"verify_len": ell, "n_admitted": n_adm.value}


def schedule_threshold(confidences, threshold: float, lib=None):
    """Static-threshold baseline: l_r = the number of leading draft tokens whose
    confidence reaches the threshold. Returns verify_len [R] int32."""
    lib = lib or load()
    c = np.ascontiguousarray(confidences, dtype=np.float32)
    R, gamma = c.shape
    ell = np.zeros(R, np.int32)
    rc = lib.oracle_schedule_threshold(_ptr(c, ctypes.c_float), R, gamma, float(threshold),
                                       _ptr(ell, ctypes.c_int32))
    if rc != 0:
        raise OracleError(f"oracle_schedule_threshold returned {rc}")
    return ell


def bf16_round(x, lib=None):
    """Nearest bfloat16 (ties to even) of each float64 value, as uint16 bits."""
    lib = lib or load()
    a = np.ascontiguousarray(x, dtype=np.float64)
    out = np.zeros(a.shape, np.uint16)
    rc = lib.oracle_bf16_round(_ptr(a, ctypes.c_double), a.size, _ptr(out, ctypes.c_uint16))
    if rc != 0:
        raise OracleError(f"oracle_bf16_round returned {rc}")
    return out


def markov_draft(base_logits, w1, w2t, anchors, uniforms, temperature, requests=None,
                 want_logits=False, nthreads=1, lib=None):
    """Sequential stage with the Markov head (section 3.1, equations 4 and 5).

    base_logits [B, gamma, V] bf16 bits (uint16); w1, w2t [V, r] bf16 bits
    (w2t row v = column v of W2); anchors [B]; uniforms [B, gamma] float32.
    requests: indices of the requests to draft (None: all). Returns a dict:
    tokens [n, gamma], probs [n, gamma] (p_k of the drawn token), flags
    [n, gamma] (FLAG_* bits of each draw), logits [n, gamma, V] bf16 bits if
    want_logits."""
    lib = lib or load()
    U = np.ascontiguousarray(base_logits, dtype=np.uint16)
    B, gamma, V = U.shape
    W1 = np.ascontiguousarray(w1, dtype=np.uint16)
    W2t = np.ascontiguousarray(w2t, dtype=np.uint16)
    if W1.shape[0] != V or W2t.shape != W1.shape:
        raise ValueError("w1 and w2t must both be [V, r]")
    r = W1.shape[1]
    x0 = np.ascontiguousarray(anchors, dtype=np.int32).reshape(B)
    u = np.ascontiguousarray(uniforms, dtype=np.float32).reshape(B, gamma)
    req = None if requests is None else np.ascontiguousarray(requests, dtype=np.int32).reshape(-1)
    n = B if req is None else req.shape[0]
    tokens = np.zeros((n, gamma), np.int32)
    probs = np.zeros((n, gamma), np.float64)
    flags = np.zeros((n, gamma), np.int32)
    logits = np.zeros((n, gamma, V), np.uint16) if want_logits else None
    u16 = ctypes.c_uint16
    rc = lib.oracle_markov_draft(
        _ptr(U, u16), _ptr(W1, u16), _ptr(W2t, u16), _ptr(x0, ctypes.c_int32),
        _ptr(u, ctypes.c_float), float(temperature), B, gamma, V, r,
        None if req is None else _ptr(req, ctypes.c_int32), n, _ptr(tokens, ctypes.c_int32),
        _ptr(probs, ctypes.c_double), _ptr(flags, ctypes.c_int32),
        None if logits is None else _ptr(logits, u16), int(nthreads or 1))
    if rc != 0:
        raise OracleError(f"oracle_markov_draft returned {rc}")
    out = {"tokens": tokens, "probs": probs, "flags": flags}
    if want_logits:
        out["logits"] = logits
    return out


def max_threads(lib=None) -> int:
    lib = lib or load()
    return int(lib.oracle_max_threads())
