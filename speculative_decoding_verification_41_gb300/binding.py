"""Thin Python binding of libdspark (ctypes). Argument marshalling only: every
step of verification and scheduling runs in the CUDA kernels of libdspark.so;
there is no CPU path. Torch supplies device memory and the current stream.

The two calls mirror include/dspark.h:
  dspark_verify(...)   -- batched speculative verification (DSpark paper, section 2.1)
  dspark_schedule(...) -- hardware-aware prefix scheduler (section 3.2.2, Algorithm 1)
"""
from __future__ import annotations

import ctypes
import os
import re
import threading
from typing import Optional

import torch

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
HEADER = os.path.join(ROOT, "include", "dspark.h")
LIB_PATH = os.path.join(PKG, "libdspark.so")

STATUS_NAMES = {0: "DSPARK_OK", 1: "DSPARK_ERR_INVALID_ARG", 2: "DSPARK_ERR_CUDA",
                3: "DSPARK_ERR_WORKSPACE", 4: "DSPARK_ERR_TIMEOUT", 5: "DSPARK_ERR_BAD_DATA",
                6: "DSPARK_ERR_TOO_LARGE"}
DSPARK_OK, DSPARK_ERR_TIMEOUT, DSPARK_ERR_BAD_DATA = 0, 4, 5
DSPARK_F32, DSPARK_BF16 = 0, 1
EXPORTED = ("dspark_verify", "dspark_acceptance", "dspark_schedule", "dspark_schedule_capacity",
            "dspark_schedule_topk", "dspark_schedule_threshold", "dspark_verify_static",
            "dspark_verify_timed", "dspark_verify_rates", "dspark_draft_markov",
            "dspark_draft_markov_timed", "dspark_wait_selftest")


class DsparkError(RuntimeError):
    def __init__(self, where: str, code: int):
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")
        self.code = code


def _header_consts() -> dict:
    txt = open(HEADER).read()
    out = {}
    for name in ("DSPARK_TILE_BYTES", "DSPARK_RESAMPLE_SEG", "DSPARK_MAX_GAMMA",
                 "DSPARK_DRAFT_TILE", "DSPARK_DRAFT_MAX_RANK"):
        out[name] = int(re.search(rf"#define {name} (\d+)", txt).group(1))
    return out


_CONSTS = _header_consts()
MAX_GAMMA = _CONSTS["DSPARK_MAX_GAMMA"]


def _a256(x: int) -> int:
    return (x + 255) & ~255


def _cdiv(a: int, b: int) -> int:
    return (a + b - 1) // b


def verify_workspace_bytes(B: int, gamma: int, V: int) -> int:
    """Python statement of DSPARK_VERIFY_WS_BYTES (include/dspark.h)."""
    rows = B * (2 * gamma + 1)
    tiles = _cdiv(V, _CONSTS["DSPARK_TILE_BYTES"] // 4)
    segs = _cdiv(V, _CONSTS["DSPARK_RESAMPLE_SEG"])
    return (256 + _a256((B + 1) * 4) + _a256(rows * 8) + _a256(rows * tiles * 16)
            + _a256(B * 64) + _a256(B * segs * 8) + _a256(B * 4))


def acceptance_workspace_bytes(B: int, gamma: int, V: int) -> int:
    """Python statement of DSPARK_ACCEPTANCE_WS_BYTES (include/dspark.h)."""
    segs = _cdiv(V, _CONSTS["DSPARK_RESAMPLE_SEG"])
    return verify_workspace_bytes(B, gamma, V) + _a256(B * gamma * 64) + _a256(B * gamma * segs * 8)


def draft_workspace_bytes(B: int, r: int, V: int) -> int:
    """Python statement of DSPARK_DRAFT_WS_BYTES (include/dspark.h)."""
    return (_a256(B * r * 2) + 2 * _a256(B * _cdiv(V, _CONSTS["DSPARK_DRAFT_TILE"]) * 8) + 256
            + _a256(B * 128) + 4096 + (2 << 20))


def schedule_workspace_bytes(R: int, gamma: int) -> int:
    """Python statement of DSPARK_SCHEDULE_WS_BYTES (include/dspark.h)."""
    n = R * gamma
    return 256 + 2 * _a256(n * 8) + 2 * _a256(n * 4) + _a256(R * 4)


_lock = threading.Lock()
_lib = None


def load(path: Optional[str] = None):
    """Load libdspark.so. Raises if it has not been built: there is no fallback."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB_PATH
        if not os.path.exists(p):
            raise RuntimeError(f"libdspark.so is not built ({p}); run "
                               "`python -c 'import __graft_entry__ as g; g.build()'`")
        lib = ctypes.CDLL(p)
        vp, i32, i64, f32, sz = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                                 ctypes.c_size_t)
        lib.dspark_verify.restype = ctypes.c_int
        lib.dspark_verify.argtypes = [vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, vp, vp, vp, vp,
                                      vp, vp, vp, vp, sz, vp]
        lib.dspark_acceptance.restype = ctypes.c_int
        lib.dspark_acceptance.argtypes = [vp, vp, vp, f32, i32, i32, i32, i32, vp, vp, vp, vp, vp,
                                          sz, vp]
        lib.dspark_verify_timed.restype = ctypes.c_int
        lib.dspark_verify_timed.argtypes = [vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, vp, vp, vp,
                                            vp, vp, vp, vp, vp, sz, vp, vp]
        lib.dspark_verify_rates.restype = ctypes.c_int
        lib.dspark_verify_rates.argtypes = [vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, vp, vp,
                                            vp, vp, vp, vp, vp, vp, vp, sz, vp]
        lib.dspark_wait_selftest.restype = ctypes.c_int
        lib.dspark_wait_selftest.argtypes = [i32, vp, vp, vp]
        lib.dspark_verify_static.restype = ctypes.c_int
        lib.dspark_verify_static.argtypes = [vp, vp, vp, vp, vp, f32, i32, i32, i32, i32, vp, vp,
                                             vp, vp, vp, vp, vp, vp]
        lib.dspark_schedule.restype = ctypes.c_int
        lib.dspark_schedule.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp, vp, vp, sz, vp]
        lib.dspark_schedule_capacity.restype = ctypes.c_int
        lib.dspark_schedule_capacity.argtypes = [vp, vp, i64, i32, i32, vp, vp, vp, vp, vp, vp, sz,
                                                 vp]
        lib.dspark_schedule_topk.restype = ctypes.c_int
        lib.dspark_schedule_topk.argtypes = [vp, vp, i32, i32, vp, vp, vp, sz, vp]
        lib.dspark_schedule_threshold.restype = ctypes.c_int
        lib.dspark_schedule_threshold.argtypes = [vp, f32, i32, i32, vp, vp, vp]
        lib.dspark_draft_markov.restype = ctypes.c_int
        lib.dspark_draft_markov.argtypes = [vp, vp, vp, vp, vp, f32, i32, i32, i64, i32, vp, vp,
                                            vp, vp, sz, vp]
        lib.dspark_draft_markov_timed.restype = ctypes.c_int
        lib.dspark_draft_markov_timed.argtypes = [vp, vp, vp, vp, vp, f32, i32, i32, i64, i32, vp,
                                                  vp, vp, vp, sz, vp, vp]
        if path is None:
            _lib = lib
        return lib


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream_handle(stream) -> ctypes.c_void_p:
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _require_cuda(name: str, t: torch.Tensor, dtype=None, device=None):
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (libdspark has no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


class VerifyBuffers:
    """Outputs and workspace of dspark_verify for a fixed (B, gamma, V), so that
    repeated calls (and CUDA-graph capture) allocate nothing. with_rates=True
    adds the rates output and the larger workspace of dspark_verify_rates."""

    def __init__(self, B: int, gamma: int, V: int, device, with_probs: bool = True,
                 with_rates: bool = False):
        self.B, self.gamma, self.V = B, gamma, V
        dev = torch.device(device)
        self.accepted_len = torch.empty(B, dtype=torch.int32, device=dev)
        self.emitted_tokens = torch.empty(B, gamma + 1, dtype=torch.int32, device=dev)
        self.probs = torch.empty(B, gamma, 2, dtype=torch.float32, device=dev) if with_probs else None
        self.near_tie_count = torch.zeros(1, dtype=torch.int32, device=dev)
        self.device_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.rates = torch.empty(B, gamma, dtype=torch.float32, device=dev) if with_rates else None
        ws = acceptance_workspace_bytes(B, gamma, V) if with_rates else verify_workspace_bytes(B, gamma, V)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=dev)
        assert self.workspace.data_ptr() % 256 == 0


def dspark_verify(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                  draft_tokens: torch.Tensor, verify_len: torch.Tensor, uniforms: torch.Tensor,
                  temperature: float, target_row_off: Optional[torch.Tensor] = None,
                  draft_row_off: Optional[torch.Tensor] = None, *, with_probs: bool = True,
                  buffers: Optional[VerifyBuffers] = None, stream=None, check: bool = False,
                  events=None, with_rates: bool = False) -> dict:
    """Batched speculative verification through libdspark (see include/dspark.h).

    Returns a dict of device tensors: accepted_len [B] int32, emitted_tokens
    [B, gamma+1] int32, probs [B, gamma, 2] float32 (or None), near_tie_count
    [1], device_status [1]. With check=True the call synchronises and raises on
    a non-OK device status. With events (four torch.cuda.Event made with
    enable_timing=True) the call goes through dspark_verify_timed, which records
    them around the planning, streaming and decision passes. With
    with_rates=True it goes through dspark_verify_rates and the dict also holds
    rates [B, gamma] float32, the acceptance probability of every verified
    position (-1 beyond l_r), from the same row statistics."""
    dev = target_logits.device
    if target_logits.dtype == torch.bfloat16:
        dtype = DSPARK_BF16
    elif target_logits.dtype == torch.float32:
        dtype = DSPARK_F32
    else:
        raise ValueError(f"logits must be bfloat16 or float32, got {target_logits.dtype}")
    _require_cuda("target_logits", target_logits)
    _require_cuda("draft_logits", draft_logits, target_logits.dtype, dev)
    _require_cuda("draft_tokens", draft_tokens, torch.int32, dev)
    _require_cuda("verify_len", verify_len, torch.int32, dev)
    _require_cuda("uniforms", uniforms, torch.float32, dev)
    if (target_row_off is None) != (draft_row_off is None):
        raise ValueError("pass both row-offset tensors or neither")
    if target_row_off is not None:
        _require_cuda("target_row_off", target_row_off, torch.int64, dev)
        _require_cuda("draft_row_off", draft_row_off, torch.int64, dev)
    B, gamma = draft_tokens.shape
    V = target_logits.shape[-1]
    if draft_logits.shape[-1] != V:
        raise ValueError("target and draft vocabularies differ")
    if uniforms.shape != (B, gamma + 1) or verify_len.shape != (B,):
        raise ValueError("uniforms must be [B, gamma+1] and verify_len [B]")
    if with_rates and events is not None:
        raise ValueError("with_rates and events are separate entry points")
    buf = buffers or VerifyBuffers(B, gamma, V, dev, with_probs, with_rates)
    if (buf.B, buf.gamma, buf.V) != (B, gamma, V):
        raise ValueError("buffers were made for another shape")
    if with_rates and buf.rates is None:
        raise ValueError("buffers were made without rates (VerifyBuffers(..., with_rates=True))")
    lib = load()
    args = (_ptr(target_logits), _ptr(draft_logits), _ptr(draft_tokens), _ptr(verify_len),
            _ptr(uniforms), float(temperature), dtype, B, gamma, V, _ptr(target_row_off),
            _ptr(draft_row_off), _ptr(buf.accepted_len), _ptr(buf.emitted_tokens),
            _ptr(buf.probs if with_probs else None), _ptr(buf.near_tie_count),
            _ptr(buf.device_status), _ptr(buf.workspace), buf.workspace.numel())
    with torch.cuda.device(dev):
        s = _stream_handle(stream)
        if with_rates:
            rargs = args[:16] + (_ptr(buf.rates),) + args[16:]
            rc = lib.dspark_verify_rates(*rargs, s)
        elif events is None:
            rc = lib.dspark_verify(*args, s)
        else:
            if len(events) != 4:
                raise ValueError("events must hold four torch.cuda.Event")
            st = stream if stream is not None else torch.cuda.current_stream(dev)
            for e in events:  # a torch event's handle exists once it has been recorded
                e.record(st)
            handles = (ctypes.c_void_p * 4)(*[ctypes.c_void_p(e.cuda_event) for e in events])
            rc = lib.dspark_verify_timed(*args, s, handles)
    if rc != 0:
        name = ("dspark_verify_rates" if with_rates else
                "dspark_verify_timed" if events is not None else "dspark_verify")
        raise DsparkError(name, rc)
    out = {"accepted_len": buf.accepted_len, "emitted_tokens": buf.emitted_tokens,
           "probs": buf.probs if with_probs else None, "near_tie_count": buf.near_tie_count,
           "device_status": buf.device_status}
    if with_rates:
        out["rates"] = buf.rates
    if check:
        torch.cuda.synchronize(dev)
        st = int(buf.device_status.item())
        if st != 0:
            raise DsparkError("dspark_verify (device)", st)
    return out


def dspark_acceptance(target_logits: torch.Tensor, draft_logits: torch.Tensor,
                      verify_len: torch.Tensor, temperature: float, gamma: int,
                      target_row_off: Optional[torch.Tensor] = None,
                      draft_row_off: Optional[torch.Tensor] = None, *,
                      rates: Optional[torch.Tensor] = None,
                      workspace: Optional[torch.Tensor] = None, stream=None,
                      check: bool = False) -> dict:
    """Acceptance probability sum_v min(p_t^k, p_d^k) of every verified position
    (equation 8) through libdspark. Returns rates [B, gamma] float32 (-1 beyond
    each l_r) and device_status [1] (device tensors)."""
    dev = target_logits.device
    if target_logits.dtype == torch.bfloat16:
        dtype = DSPARK_BF16
    elif target_logits.dtype == torch.float32:
        dtype = DSPARK_F32
    else:
        raise ValueError(f"logits must be bfloat16 or float32, got {target_logits.dtype}")
    _require_cuda("target_logits", target_logits)
    _require_cuda("draft_logits", draft_logits, target_logits.dtype, dev)
    _require_cuda("verify_len", verify_len, torch.int32, dev)
    if (target_row_off is None) != (draft_row_off is None):
        raise ValueError("pass both row-offset tensors or neither")
    if target_row_off is not None:
        _require_cuda("target_row_off", target_row_off, torch.int64, dev)
        _require_cuda("draft_row_off", draft_row_off, torch.int64, dev)
    B = verify_len.shape[0]
    V = target_logits.shape[-1]
    out = rates if rates is not None else torch.empty(B, gamma, dtype=torch.float32, device=dev)
    ws_bytes = acceptance_workspace_bytes(B, gamma, V)
    ws = workspace if workspace is not None else torch.empty(ws_bytes, dtype=torch.uint8,
                                                             device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lib = load()
    with torch.cuda.device(dev):
        rc = lib.dspark_acceptance(_ptr(target_logits), _ptr(draft_logits), _ptr(verify_len),
                                   float(temperature), dtype, B, gamma, V, _ptr(target_row_off),
                                   _ptr(draft_row_off), _ptr(out), _ptr(status), _ptr(ws),
                                   ws.numel(), _stream_handle(stream))
    if rc != 0:
        raise DsparkError("dspark_acceptance", rc)
    if check:
        torch.cuda.synchronize(dev)
        if int(status.item()) != 0:
            raise DsparkError("dspark_acceptance (device)", int(status.item()))
    return {"rates": out, "device_status": status}


class ScheduleBuffers:
    def __init__(self, R: int, gamma: int, device):
        dev = torch.device(device)
        self.R, self.gamma = R, gamma
        self.capacity = torch.zeros(1, dtype=torch.int32, device=dev)
        self.verify_len = torch.empty(R, dtype=torch.int32, device=dev)
        self.theta_best = torch.empty(1, dtype=torch.float64, device=dev)
        self.near_tie_count = torch.zeros(1, dtype=torch.int32, device=dev)
        self.device_status = torch.zeros(1, dtype=torch.int32, device=dev)
        self.workspace = torch.empty(schedule_workspace_bytes(R, gamma), dtype=torch.uint8, device=dev)


def dspark_schedule(confidences: torch.Tensor, step_time_ms: torch.Tensor, *,
                    buffers: Optional[ScheduleBuffers] = None, stream=None,
                    check: bool = False) -> dict:
    """Hardware-aware prefix scheduler through libdspark (see include/dspark.h).
    Returns verify_len [R] int32, theta_best [1] float64, near_tie_count [1],
    device_status [1] (device tensors)."""
    dev = confidences.device
    _require_cuda("confidences", confidences, torch.float32)
    _require_cuda("step_time_ms", step_time_ms, torch.float64, dev)
    R, gamma = confidences.shape
    buf = buffers or ScheduleBuffers(R, gamma, dev)
    lib = load()
    with torch.cuda.device(dev):
        rc = lib.dspark_schedule(_ptr(confidences), _ptr(step_time_ms), step_time_ms.numel(), R,
                                 gamma, _ptr(buf.verify_len), _ptr(buf.theta_best),
                                 _ptr(buf.near_tie_count), _ptr(buf.device_status),
                                 _ptr(buf.workspace), buf.workspace.numel(), _stream_handle(stream))
    if rc != 0:
        raise DsparkError("dspark_schedule", rc)
    return _schedule_out(buf, dev, check, "dspark_schedule")


def _schedule_out(buf, dev, check, name):
    out = {"verify_len": buf.verify_len, "theta_best": buf.theta_best, "capacity": buf.capacity,
           "near_tie_count": buf.near_tie_count, "device_status": buf.device_status}
    if check:
        torch.cuda.synchronize(dev)
        st = int(buf.device_status.item())
        if st != 0:
            raise DsparkError(f"{name} (device)", st)
    return out


def dspark_schedule_capacity(confidences: torch.Tensor, step_time_ms: torch.Tensor, *,
                             buffers: Optional[ScheduleBuffers] = None, stream=None,
                             check: bool = False) -> dict:
    """Production scheduler, capacity (section 5.2): the global search without the
    early-stopping break. Returns capacity [1] int32 (n*), verify_len [R] of the
    best prefix, theta_best, near_tie_count, device_status (device tensors)."""
    dev = confidences.device
    _require_cuda("confidences", confidences, torch.float32)
    _require_cuda("step_time_ms", step_time_ms, torch.float64, dev)
    R, gamma = confidences.shape
    buf = buffers or ScheduleBuffers(R, gamma, dev)
    lib = load()
    with torch.cuda.device(dev):
        rc = lib.dspark_schedule_capacity(
            _ptr(confidences), _ptr(step_time_ms), step_time_ms.numel(), R, gamma,
            _ptr(buf.capacity), _ptr(buf.verify_len), _ptr(buf.theta_best),
            _ptr(buf.near_tie_count), _ptr(buf.device_status), _ptr(buf.workspace),
            buf.workspace.numel(), _stream_handle(stream))
    if rc != 0:
        raise DsparkError("dspark_schedule_capacity", rc)
    return _schedule_out(buf, dev, check, "dspark_schedule_capacity")


def dspark_schedule_topk(confidences: torch.Tensor, capacity: torch.Tensor, *,
                         buffers: Optional[ScheduleBuffers] = None, stream=None,
                         check: bool = False) -> dict:
    """Production scheduler, admission (section 5.2): the first min(K, |E|)
    candidates of the current confidences, K = capacity[0] read on the device.
    Returns verify_len [R] and device_status (device tensors)."""
    dev = confidences.device
    _require_cuda("confidences", confidences, torch.float32)
    _require_cuda("capacity", capacity, torch.int32, dev)
    R, gamma = confidences.shape
    buf = buffers or ScheduleBuffers(R, gamma, dev)
    lib = load()
    with torch.cuda.device(dev):
        rc = lib.dspark_schedule_topk(_ptr(confidences), _ptr(capacity), R, gamma,
                                      _ptr(buf.verify_len), _ptr(buf.device_status),
                                      _ptr(buf.workspace), buf.workspace.numel(),
                                      _stream_handle(stream))
    if rc != 0:
        raise DsparkError("dspark_schedule_topk", rc)
    return _schedule_out(buf, dev, check, "dspark_schedule_topk")


def dspark_schedule_threshold(confidences: torch.Tensor, threshold: float, *,
                              verify_len: Optional[torch.Tensor] = None,
                              device_status: Optional[torch.Tensor] = None, stream=None,
                              check: bool = False) -> dict:
    """Static-threshold baseline (section 4.3.3): l_r = the number of leading
    draft tokens whose confidence reaches the threshold. Returns verify_len [R]
    int32 and device_status [1] (device tensors)."""
    dev = confidences.device
    _require_cuda("confidences", confidences, torch.float32)
    R, gamma = confidences.shape
    ell = verify_len if verify_len is not None else torch.empty(R, dtype=torch.int32, device=dev)
    st = device_status if device_status is not None else torch.zeros(1, dtype=torch.int32,
                                                                      device=dev)
    lib = load()
    with torch.cuda.device(dev):
        rc = lib.dspark_schedule_threshold(_ptr(confidences), float(threshold), R, gamma,
                                           _ptr(ell), _ptr(st), _stream_handle(stream))
    if rc != 0:
        raise DsparkError("dspark_schedule_threshold", rc)
    if check:
        torch.cuda.synchronize(dev)
        if int(st.item()) != 0:
            raise DsparkError("dspark_schedule_threshold (device)", int(st.item()))
    return {"verify_len": ell, "device_status": st}


def dspark_draft_markov(base_logits: torch.Tensor, w1: torch.Tensor, w2t: torch.Tensor,
                        anchors: torch.Tensor, uniforms: torch.Tensor, temperature: float, *,
                        draft_logits: Optional[torch.Tensor] = None,
                        draft_tokens: Optional[torch.Tensor] = None,
                        workspace: Optional[torch.Tensor] = None, stream=None,
                        check: bool = False, events=None) -> dict:
    """Sequential stage of the drafter with the Markov head (section 3.1,
    equations 4 and 5) through libdspark.

    base_logits [B, gamma, V] bf16, w1 and w2t [V, r] bf16 (w2t row v = column v
    of W2), anchors [B] int32, uniforms [B, gamma] float32. draft_logits may be
    base_logits itself (in place). Returns device tensors: draft_logits [B,
    gamma, V] bf16, draft_tokens [B, gamma] int32, device_status [1]. With
    events (2*gamma + 2 torch.cuda.Event made with enable_timing=True) the call
    goes through dspark_draft_markov_timed."""
    dev = base_logits.device
    _require_cuda("base_logits", base_logits, torch.bfloat16)
    _require_cuda("w1", w1, torch.bfloat16, dev)
    _require_cuda("w2t", w2t, torch.bfloat16, dev)
    _require_cuda("anchors", anchors, torch.int32, dev)
    _require_cuda("uniforms", uniforms, torch.float32, dev)
    if base_logits.dim() != 3:
        raise ValueError("base_logits must be [B, gamma, V]")
    B, gamma, V = base_logits.shape
    if w1.dim() != 2 or w1.shape[0] != V or w2t.shape != w1.shape:
        raise ValueError("w1 and w2t must both be [V, r]")
    r = w1.shape[1]
    if anchors.shape != (B,) or uniforms.shape != (B, gamma):
        raise ValueError("anchors must be [B] and uniforms [B, gamma]")
    out = draft_logits if draft_logits is not None else torch.empty_like(base_logits)
    _require_cuda("draft_logits", out, torch.bfloat16, dev)
    if out.shape != base_logits.shape:
        raise ValueError("draft_logits must be [B, gamma, V]")
    tok = draft_tokens if draft_tokens is not None else torch.empty(B, gamma, dtype=torch.int32,
                                                                     device=dev)
    ws = workspace if workspace is not None else torch.empty(
        max(draft_workspace_bytes(B, r, V), 256), dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    lib = load()
    args = (_ptr(base_logits), _ptr(w1), _ptr(w2t), _ptr(anchors), _ptr(uniforms),
            float(temperature), B, gamma, V, r, _ptr(out), _ptr(tok), _ptr(status), _ptr(ws),
            ws.numel())
    with torch.cuda.device(dev):
        s = _stream_handle(stream)
        if events is None:
            rc = lib.dspark_draft_markov(*args, s)
        else:
            if len(events) != 2 * gamma + 2:
                raise ValueError("events must hold 2*gamma + 2 torch.cuda.Event")
            st = stream if stream is not None else torch.cuda.current_stream(dev)
            for e in events:
                e.record(st)
            handles = (ctypes.c_void_p * len(events))(*[ctypes.c_void_p(e.cuda_event)
                                                        for e in events])
            rc = lib.dspark_draft_markov_timed(*args, s, handles)
    if rc != 0:
        raise DsparkError("dspark_draft_markov", rc)
    if check:
        torch.cuda.synchronize(dev)
        st = int(status.item())
        if st != 0:
            raise DsparkError("dspark_draft_markov (device)", st)
    return {"draft_logits": out, "draft_tokens": tok, "device_status": status}


def wait_selftest(which: int, device="cuda", stream=None) -> dict:
    """Run dspark_wait_selftest (include/dspark.h): one bounded wait that never
    completes. Returns the device status it left (DSPARK_ERR_TIMEOUT expected)
    and the seconds the call took on the device."""
    dev = torch.device(device)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    sync = torch.zeros(2, dtype=torch.int32, device=dev)
    lib = load()
    with torch.cuda.device(dev):
        st = stream if stream is not None else torch.cuda.current_stream(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(st)
        rc = lib.dspark_wait_selftest(int(which), _ptr(sync), _ptr(status), _stream_handle(st))
        b.record(st)
        if rc != 0:
            raise DsparkError("dspark_wait_selftest", rc)
        torch.cuda.synchronize(dev)
    return {"status": int(status.item()), "seconds": a.elapsed_time(b) / 1e3}
