"""The C-ABI boundary, checked on the CPU: the library loads and exports every
entry point include/dspark.h and include/dspark_testing.h declare, the workspace macros agree with the
Python binding's statement of them, and host-side argument checks reject bad
calls before anything is launched."""
import ctypes
import os
import re
import subprocess

import pytest

from speculative_decoding_verification_41_gb300 import binding
from speculative_decoding_verification_41_gb300 import build as cuda_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dspark.h")
TESTING_HEADER = os.path.join(ROOT, "include", "dspark_testing.h")
# the method's calls (the two of the verification path and the rows after
# them) and the no-allocation variant; the testing header holds the rest
METHOD_CALLS = {"dspark_verify", "dspark_schedule", "dspark_acceptance", "dspark_verify_rates",
                "dspark_schedule_capacity", "dspark_schedule_topk", "dspark_schedule_threshold",
                "dspark_draft_markov", "dspark_verify_static"}
TESTING_CALLS = {"dspark_wait_selftest", "dspark_verify_timed", "dspark_draft_markov_timed"}


@pytest.fixture(scope="module")
def lib():
    cuda_build.build()
    return binding.load()


def declared_functions(headers=(HEADER, TESTING_HEADER)):
    txt = "".join(open(h).read() for h in headers)
    return sorted(set(re.findall(r"^int\s+(dspark_\w+)\s*\(", txt, flags=re.M)))


def test_header_declares_the_exported_calls():
    assert declared_functions() == sorted(binding.EXPORTED)


def test_method_header_holds_only_the_methods_calls():
    assert set(declared_functions((HEADER,))) == METHOD_CALLS
    assert set(declared_functions((TESTING_HEADER,))) == TESTING_CALLS


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", binding.LIB_PATH], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(dspark_\w+)", out))
    for name in declared_functions():
        assert name in exported, name
        assert getattr(lib, name) is not None


def test_header_compiles_as_c_and_macros_match_binding(tmp_path):
    shapes = [(1, 1, 1), (4, 4, 32), (64, 16, 151936), (256, 16, 129280), (1024, 16, 151936),
              (7, 32, 1001), (0, 3, 5)]
    src = ['#include <stdio.h>', '#include "dspark.h"', '#include "dspark_testing.h"',
           "int main(void) {"]
    for B, g, V in shapes:
        src.append(f'  printf("%zu %zu %zu\\n", DSPARK_VERIFY_WS_BYTES({B}, {g}, {V}), '
                   f'DSPARK_SCHEDULE_WS_BYTES({max(B, 1)}, {g}), '
                   f'DSPARK_ACCEPTANCE_WS_BYTES({B}, {g}, {V}));')
    draft_shapes = [(1, 64, 8), (5, 128, 1000), (256, 256, 129280), (1000, 192, 151936)]
    for B, r, V in draft_shapes:
        src.append(f'  printf("%zu\\n", DSPARK_DRAFT_WS_BYTES({B}, {r}, {V}));')
    src.append("  return 0; }")
    c = tmp_path / "probe.c"
    c.write_text("\n".join(src))
    exe = tmp_path / "probe"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", f"-I{os.path.dirname(HEADER)}", str(c),
                    "-o", str(exe)], check=True)
    lines = subprocess.run([str(exe)], capture_output=True, text=True, check=True).stdout.split("\n")
    for (B, g, V), line in zip(shapes, lines):
        v, s, a = map(int, line.split())
        assert v == binding.verify_workspace_bytes(B, g, V)
        assert s == binding.schedule_workspace_bytes(max(B, 1), g)
        assert a == binding.acceptance_workspace_bytes(B, g, V)
    for (B, r, V), line in zip(draft_shapes, lines[len(shapes):]):
        assert int(line) == binding.draft_workspace_bytes(B, r, V)


def _verify_call(lib, **kw):
    args = dict(tl=1, dl=1, tok=1, vlen=1, uni=1, T=1.0, dtype=1, B=4, gamma=4, V=32, toff=None,
                doff=None, acc=1, em=1, probs=None, ties=None, status=1, ws=256, ws_bytes=1 << 30)
    args.update(kw)
    p = lambda x: None if x is None else ctypes.c_void_p(x)
    return lib.dspark_verify(p(args["tl"]), p(args["dl"]), p(args["tok"]), p(args["vlen"]),
                             p(args["uni"]), args["T"], args["dtype"], args["B"], args["gamma"],
                             args["V"], p(args["toff"]), p(args["doff"]), p(args["acc"]),
                             p(args["em"]), p(args["probs"]), p(args["ties"]), p(args["status"]),
                             p(args["ws"]), args["ws_bytes"], None)


@pytest.mark.parametrize("bad,code", [
    (dict(gamma=0), 1), (dict(gamma=33), 1), (dict(V=0), 1), (dict(B=-1), 1), (dict(B=70000), 1),
    (dict(T=0.0), 1), (dict(T=float("inf")), 1), (dict(T=float("nan")), 1), (dict(dtype=7), 1),
    (dict(status=None), 1), (dict(toff=64), 1), (dict(tl=None), 1), (dict(em=None), 1),
    (dict(ws=None), 3), (dict(ws=128), 3), (dict(ws_bytes=100), 3)])
def test_verify_rejects_bad_arguments_on_host(lib, bad, code):
    assert _verify_call(lib, **bad) == code


def test_schedule_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    call = lambda R, g, n, ws=256, wsb=1 << 30, conf=1: lib.dspark_schedule(
        None if conf is None else p(conf), p(1), n, R, g, p(1), None, None, p(1),
        None if ws is None else p(ws), wsb, None)
    assert call(0, 4, 100) == 1
    assert call(4, 0, 100) == 1
    assert call(4, 33, 1000) == 1
    assert call(4, 4, 20) == 1          # profile shorter than R*(gamma+1)+1
    assert call(4, 4, 21, conf=None) == 1
    assert call(4, 4, 21, ws=None) == 3
    assert call(4, 4, 21, wsb=10) == 3


def test_timed_verify_rejects_missing_events_on_host(lib):
    p = ctypes.c_void_p
    args = [p(1), p(1), p(1), p(1), p(1), 1.0, 1, 4, 4, 32, None, None, p(1), p(1), None, None,
            p(1), p(256), 1 << 30, None]
    assert lib.dspark_verify_timed(*args, None) == 1
    some_null = (ctypes.c_void_p * 4)(1, 1, None, 1)
    assert lib.dspark_verify_timed(*args, some_null) == 1
    # the timed entry runs the same host checks as dspark_verify
    good_events = (ctypes.c_void_p * 4)(1, 1, 1, 1)
    bad = list(args)
    bad[8] = 33  # gamma
    assert lib.dspark_verify_timed(*bad, good_events) == 1


def test_production_scheduler_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    cap = lambda R=4, g=4, n=21, capacity=1, T=1, ws=256: lib.dspark_schedule_capacity(
        p(1), None if T is None else p(T), n, R, g, None if capacity is None else p(capacity),
        p(1), None, None, p(1), None if ws is None else p(ws), 1 << 30, None)
    assert cap(capacity=None) == 1
    assert cap(T=None) == 1
    assert cap(n=20) == 1
    assert cap(R=0) == 1
    assert cap(ws=None) == 3
    topk = lambda R=4, g=4, capacity=1, ws=256, wsb=1 << 30: lib.dspark_schedule_topk(
        p(1), None if capacity is None else p(capacity), R, g, p(1), p(1),
        None if ws is None else p(ws), wsb, None)
    assert topk(capacity=None) == 1
    assert topk(g=33) == 1
    assert topk(wsb=10) == 3


def test_threshold_baseline_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    call = lambda thr=0.5, R=4, g=4, conf=1, out=1, st=1: lib.dspark_schedule_threshold(
        None if conf is None else p(conf), thr, R, g, None if out is None else p(out),
        None if st is None else p(st), None)
    assert call(thr=float("nan")) == 1
    assert call(thr=float("inf")) == 1
    assert call(R=0) == 1
    assert call(g=33) == 1
    assert call(conf=None) == 1
    assert call(st=None) == 1


def test_acceptance_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    def call(**kw):
        a = dict(tl=1, dl=1, vlen=1, T=1.0, dtype=1, B=4, g=4, V=32, toff=None, doff=None,
                 rates=1, st=1, ws=256, wsb=1 << 30)
        a.update(kw)
        q = lambda x: None if x is None else p(x)
        return lib.dspark_acceptance(q(a["tl"]), q(a["dl"]), q(a["vlen"]), a["T"], a["dtype"],
                                     a["B"], a["g"], a["V"], q(a["toff"]), q(a["doff"]),
                                     q(a["rates"]), q(a["st"]), q(a["ws"]), a["wsb"], None)
    assert call(T=0.0) == 1
    assert call(g=33) == 1
    assert call(rates=None) == 1
    assert call(st=None) == 1
    assert call(toff=64) == 1
    assert call(ws=None) == 3
    assert call(wsb=100) == 3


def test_verify_rates_rejects_bad_arguments_on_host(lib):
    """dspark_verify_rates: dspark_verify's checks, a rates pointer, and the
    larger workspace of dspark_acceptance (no device is needed)."""
    p = ctypes.c_void_p
    B, g, V = 4, 4, 32

    def call(**kw):
        a = dict(tl=256, dl=256, tok=256, vlen=256, uni=256, T=1.0, dtype=1, toff=None,
                 doff=None, acc=256, em=256, pr=None, ties=None, rates=256, st=256, ws=256,
                 wsb=1 << 30)
        a.update(kw)
        q = lambda x: None if x is None else p(x)
        return lib.dspark_verify_rates(q(a["tl"]), q(a["dl"]), q(a["tok"]), q(a["vlen"]),
                                       q(a["uni"]), a["T"], a["dtype"], B, g, V, q(a["toff"]),
                                       q(a["doff"]), q(a["acc"]), q(a["em"]), q(a["pr"]),
                                       q(a["ties"]), q(a["rates"]), q(a["st"]), q(a["ws"]),
                                       a["wsb"], None)
    assert call(rates=None) == 1
    assert call(T=0.0) == 1
    assert call(st=None) == 1
    assert call(toff=64) == 1
    assert call(ws=None) == 3
    # enough for dspark_verify, not for the rates' jobs and sums
    assert call(wsb=binding.verify_workspace_bytes(B, g, V)) == 3
    assert binding.acceptance_workspace_bytes(B, g, V) > binding.verify_workspace_bytes(B, g, V)


def test_wait_selftest_rejects_bad_arguments_on_host(lib):
    p = ctypes.c_void_p
    assert lib.dspark_wait_selftest(2, p(256), p(256), None) == 1
    assert lib.dspark_wait_selftest(-1, p(256), p(256), None) == 1
    assert lib.dspark_wait_selftest(0, p(256), None, None) == 1
    assert lib.dspark_wait_selftest(1, None, p(256), None) == 1
    assert lib.dspark_wait_selftest(1, p(260), p(256), None) == 1  # sync words not 8-byte aligned


def _draft_call(lib, timed=False, events=None, **kw):
    a = dict(U=256, w1=256, w2t=256, x0=256, uni=256, T=1.0, B=4, g=4, V=1024, r=256, L=256,
             tok=256, st=256, ws=256, wsb=1 << 30)
    a.update(kw)
    q = lambda x: None if x is None else ctypes.c_void_p(x)
    args = (q(a["U"]), q(a["w1"]), q(a["w2t"]), q(a["x0"]), q(a["uni"]), a["T"], a["B"], a["g"],
            a["V"], a["r"], q(a["L"]), q(a["tok"]), q(a["st"]), q(a["ws"]), a["wsb"], None)
    if timed:
        return lib.dspark_draft_markov_timed(*args, events)
    return lib.dspark_draft_markov(*args)


@pytest.mark.parametrize("bad,code", [
    (dict(g=0), 1), (dict(g=33), 1), (dict(V=4), 1), (dict(V=1001), 1), (dict(B=-1), 1),
    (dict(r=0), 1), (dict(r=100), 1), (dict(r=320), 1), (dict(T=0.0), 1),
    (dict(T=float("nan")), 1), (dict(T=float("inf")), 1), (dict(U=None), 1), (dict(w2t=None), 1),
    (dict(L=None), 1), (dict(tok=None), 1), (dict(st=None), 1), (dict(ws=None), 1),
    (dict(U=264), 1), (dict(w1=8), 1), (dict(L=1032), 1), (dict(ws=128), 1),
    (dict(wsb=1000), 3),
])
def test_draft_rejects_bad_arguments_on_host(lib, bad, code):
    """Every check runs before the first CUDA call (no device is needed)."""
    assert _draft_call(lib, **bad) == code


def test_draft_with_no_requests_does_nothing(lib):
    assert _draft_call(lib, B=0, U=None, w1=None, w2t=None, x0=None, uni=None, L=None, tok=None,
                       st=None, ws=None, wsb=0) == 0


def test_timed_draft_rejects_missing_events_on_host(lib):
    assert _draft_call(lib, timed=True, events=None) == 1
    ev = (ctypes.c_void_p * 10)(*([ctypes.c_void_p(64)] * 9 + [None]))
    assert _draft_call(lib, timed=True, events=ev) == 1      # one of 2*4 + 2 is NULL
