"""Benchmark of the DSpark verification hot path on GB300.

A step is one pass of the whole path over one batch: the prefix scheduler
(dspark_schedule) on per-position confidences, then batched verification
(dspark_verify) of the lengths it chose, over B=256 requests, gamma=16 draft
positions, V=129,280 bf16 logits, temperature 0.7 (the headline workload). The
step-time profile is flat, so the scheduler admits every candidate and all 16
positions of every request are verified, as that workload specifies.

Metric: verified draft positions per second (sum of verify lengths / step time).
Inputs are resident in HBM before timing; the logits (2.18 GB) exceed L2, so no
flush is needed between steps. `e2e` repeats the step through the same C-ABI
calls from pinned host buffers, host->device copies and the device->host read
of the results inside the timed region.

The line's `configs` object measures the other named workloads the same way,
each through its own calls: B=64 x V=151,936 bf16, the ragged B=1,024 fp32
workload, the scheduled R=512 workload (dspark_schedule on its step-time
profile T(N) = 4 + 0.006 min(N, 2048) + 0.02 max(N - 2048, 0) ms, then ragged
verification of the lengths it chose) and the tiny B=4 case. For every
workload the oracle runs on the host cores over a host copy of the very bytes
the GPU verified (the input checksums match), and its outputs are compared
with the GPU's request by request.

--impl reference times the CPU oracle (the plain fp64 C implementation under
oracle/) on the host cores, on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

WORKLOAD = "b256_g16_v129280_bf16"
METRIC = "verified draft positions/sec (B=256, gamma=16, V=129280, bf16)"
UNIT = "positions/s"
OTHER_CONFIGS = ("b64_g16_v151936_bf16", "ragged_b1024_g16_v151936_f32",
                 "sched_r512_g16_v129280_bf16", "tiny_b4_g4_v32_f32")


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=30)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["native", "reference"], default="native")
    p.add_argument("--e2e-steps", type=int, default=5)
    p.add_argument("--cpu-sample", type=int, default=256, help="requests in the oracle's sample")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-drafter", action="store_true",
                   help="skip the drafter's sequential stage (dspark_draft_markov)")
    p.add_argument("--drafter-only", action="store_true",
                   help="measure only the drafter's sequential stage (the ncu capture case)")
    p.add_argument("--draft-batch", type=int, default=None,
                   help="requests of the drafter measurement (default 256)")
    p.add_argument("--batch", type=int, default=None,
                   help="requests per step (default: the headline 256); a smaller batch of the "
                        "same recipe serves the ncu capture case")
    p.add_argument("--configs", default=",".join(OTHER_CONFIGS),
                   help="comma-separated other workloads measured beside the headline "
                        "(empty: none)")
    p.add_argument("--only", default=None, choices=OTHER_CONFIGS,
                   help="measure this one named workload alone and print its line (the "
                        "headline is not run)")
    return p.parse_args()


# ---------------------------------------------------------------------------
# distributed plumbing (one process per GPU, independent replicas)
# ---------------------------------------------------------------------------
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def shard_seed(rank: int) -> int:
    """Seed of rank r's shard. Requests are independent, so N ranks verify a
    global batch of N x B requests without any collective: rank r generates its
    own B requests of the same recipe from seed 7 + r (rank 0's shard is the
    headline workload itself)."""
    return 7 + rank


def aggregate_value(positions_per_step: int, world_size: int, steps: int,
                    max_total_ms: float) -> float:
    """Whole-job throughput: positions verified by all ranks over the slowest
    rank's timed region (weak scaling: every rank verifies its own shard)."""
    return positions_per_step * world_size * steps / (max_total_ms * 1e-3)


def barrier(dist, device=None):
    if dist is not None:
        if device is not None and device.type == "cuda":
            dist.barrier(device_ids=[device.index])
        else:
            dist.barrier()


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for name, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# the oracle on the host, over the bytes the GPU verified
# ---------------------------------------------------------------------------
def checksum(tensors) -> str:
    """64-bit sums of the bit patterns of each tensor (device or host, signed
    integers of the element's width), joined: equal strings mean equal bytes."""
    out = []
    for t in tensors:
        b = t.contiguous().view({2: torch.int16, 4: torch.int32}[t.element_size()]).reshape(-1)
        acc = 0
        for s0 in range(0, b.numel(), 1 << 27):
            part = b[s0:s0 + (1 << 27)]
            if part.is_cuda:
                acc += int(part.to(torch.int64).sum().item())
            else:
                acc += int(part.numpy().sum(dtype=np.int64))
        out.append(f"{acc & 0xFFFFFFFFFFFFFFFF:016x}")
    return "-".join(out)


def input_tensors(vi):
    return (vi.target_logits, vi.draft_logits, vi.draft_tokens, vi.uniforms)


def logits_np(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).numpy().view(np.uint16) if t.dtype == torch.bfloat16 else t.numpy()


def oracle_verify_host(h, nthreads: int, n_req=None):
    """The oracle over the first n_req requests (default: all) of a host copy
    of a workload. Returns (outputs, wall seconds)."""
    import oracle
    B = h.B if n_req is None else min(int(n_req), h.B)
    toff = None if h.target_row_off is None else h.target_row_off.numpy()[:B + 1]
    doff = None if h.draft_row_off is None else h.draft_row_off.numpy()[:B + 1]
    t0 = time.perf_counter()
    ref = oracle.verify(logits_np(h.target_logits), logits_np(h.draft_logits),
                        h.draft_tokens.numpy()[:B], h.verify_len.numpy()[:B],
                        h.uniforms.numpy()[:B], h.temperature, toff, doff, nthreads=nthreads)
    return ref, time.perf_counter() - t0


def agreement(out: dict, ref: dict, ell: np.ndarray) -> dict:
    """Request-by-request agreement of the GPU's outputs with the oracle's:
    requests that differ at all, those that differ without a near-tie flag of
    the oracle (must be 0), and the decisions they are counted against (the
    oracle's ratio tests, positions 1..min(m+1, l), plus one draw per
    request)."""
    acc = out["accepted_len"].cpu().numpy()
    em = out["emitted_tokens"].cpu().numpy()
    same = (acc == ref["accepted_len"]) & (em == ref["emitted"]).all(axis=1)
    flagged = ref["flags"].any(axis=1)
    ell = np.asarray(ell, np.int64)
    ratio_tests = int(np.minimum(ref["accepted_len"].astype(np.int64) + 1, ell).sum())
    res = {"requests": int(len(acc)), "mismatches": int((~same).sum()),
           "mismatches_unflagged": int((~same & ~flagged).sum()),
           "oracle_flagged_requests": int(flagged.sum()), "ratio_tests": ratio_tests,
           "draws": int(len(acc))}
    res["mismatch_rate"] = res["mismatches"] / max(1, ratio_tests + len(acc))
    if out.get("probs") is not None:
        pr = out["probs"].cpu().numpy().astype(np.float64)
        verified = np.arange(pr.shape[1])[None, :] < ell[:, None]
        err = np.abs(pr - ref["probs"])[verified]
        res["prob_max_abs_err"] = float(err.max()) if err.size else 0.0
    return res


def cpu_model() -> str:
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name"):
                return ln.split(":", 1)[1].strip()
    except OSError:
        pass
    return "unknown"


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle
# ---------------------------------------------------------------------------
def reference_inputs():
    """The headline workload on the host. With a GPU present it is generated
    there with the native arm's seeds and copied over, so the oracle reads the
    very bytes the native arm verifies; without one, the same recipe runs on the
    host (the torch CPU generator gives other values)."""
    from speculative_decoding_verification_41_gb300 import workloads
    if torch.cuda.is_available():
        vi = workloads.make_config(WORKLOAD, device=torch.device("cuda", 0))
        h = vi.to("cpu")
        del vi
        torch.cuda.empty_cache()
        return h, "generated on the GPU with the native arm's seeds, copied to the host"
    cfg = workloads.CONFIGS[WORKLOAD]
    h = workloads.make_verify(cfg["B"], cfg["gamma"], cfg["V"], cfg["dtype"], cfg["temperature"],
                              rho=cfg["rho"], verify_len="full", ragged=False, seed=7,
                              device="cpu")
    return h, "host-generated with the same recipe (no GPU: other values)"


def reference_arm(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    cores = oracle.max_threads()
    h, where = reference_inputs()
    n_req = max(1, min(args.cpu_sample, h.B))
    positions = int(h.verify_len.numpy()[:n_req].sum())
    for _ in range(args.warmup):
        oracle_verify_host(h, cores, n_req)
    times = [oracle_verify_host(h, cores, n_req)[1] for _ in range(args.steps)]
    per = statistics.median(times)
    value = positions / per
    sample = (f"{n_req} of {h.B} requests of {WORKLOAD} per step (all {h.gamma} positions, "
              f"{where}), fp64 oracle, OpenMP over requests")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
            "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": per * 1e3, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "B": h.B, "gamma": h.gamma, "V": h.V,
                       "temperature": h.temperature, "sample_requests": n_req,
                       "input_checksum": checksum(input_tensors(h))},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": sample, "cpu": cpu_model()},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


# ---------------------------------------------------------------------------
# the other named workloads
# ---------------------------------------------------------------------------
SCHEDULED = "sched_r512_g16_v129280_bf16"


def measure_config(name: str, args, dev, stream, peak: float, peak_src: str, want_cpu: bool):
    """One named workload measured like the headline: the median CUDA-event
    time of its step (the verification call; for the scheduled workload
    dspark_schedule on its step-time profile, then dspark_verify of the lengths
    it chose), its passes through the timed entry, the roofline of the
    streaming pass and of the call, and -- on the host cores -- the oracle over
    a host copy of the same bytes, compared request by request."""
    from speculative_decoding_verification_41_gb300 import binding, workloads
    import oracle
    n = max(5, min(args.steps, 20))
    sched = sbuf = None
    if name == SCHEDULED:
        cfg = workloads.CONFIGS[name]
        sched = workloads.make_schedule(cfg["R"], cfg["gamma"], seed=7, device=dev)
        sbuf = binding.ScheduleBuffers(cfg["R"], cfg["gamma"], dev)
        binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbuf, check=True)
        vi = workloads.make_config(name, device=dev, verify_len=sbuf.verify_len.cpu().numpy())
    else:
        vi = workloads.make_config(name, device=dev)
    ell = vi.verify_len.cpu().numpy()
    vbuf = binding.VerifyBuffers(vi.B, vi.gamma, vi.V, dev)

    def verify(verify_len, events=None):
        return binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                                     verify_len, vi.uniforms, vi.temperature, vi.target_row_off,
                                     vi.draft_row_off, buffers=vbuf, stream=stream, events=events)

    def step(ev=None, events=None):
        if ev is not None:
            ev[0].record(stream)
        if sched is not None:
            s = binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbuf,
                                        stream=stream)
            lens = s["verify_len"]
        else:
            lens = vi.verify_len
        if ev is not None:
            ev[1].record(stream)
        verify(lens, events)
        if ev is not None:
            ev[2].record(stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    if int(vbuf.device_status.item()) != 0 or (sbuf is not None and
                                               int(sbuf.device_status.item()) != 0):
        raise SystemExit(f"{name}: device status not OK during warm-up")
    if sbuf is not None and not np.array_equal(sbuf.verify_len.cpu().numpy(), ell):
        raise SystemExit(f"{name}: the scheduler's lengths moved between calls")
    out = {k: v.clone() for k, v in (("accepted_len", vbuf.accepted_len),
                                     ("emitted_tokens", vbuf.emitted_tokens),
                                     ("probs", vbuf.probs))}
    ties = int(vbuf.near_tie_count.item())
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
    for i in range(n):
        step(ev[i])
    torch.cuda.synchronize(dev)
    step_ms = [e[0].elapsed_time(e[2]) for e in ev]
    sched_ms = [e[0].elapsed_time(e[1]) for e in ev]
    verify_ms = [e[1].elapsed_time(e[2]) for e in ev]
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(n)]
    for i in range(n):
        step(events=pev[i])
    torch.cuda.synchronize(dev)
    pass_ms = {nm: statistics.median([e[j].elapsed_time(e[j + 1]) for e in pev])
               for j, nm in enumerate(("k_plan", "k_rowstats", "decision"))}
    positions = int(ell.sum())
    logit_bytes = vi.logit_bytes(ell)
    t_step, t_verify = statistics.median(step_ms), statistics.median(verify_ms)
    kern = logit_bytes / (pass_ms["k_rowstats"] * 1e-3) / 1e9
    call = logit_bytes / (t_verify * 1e-3) / 1e9
    res = {
        "workload": name, "B": vi.B, "gamma": vi.gamma, "V": vi.V,
        "dtype": "bf16" if vi.target_logits.dtype == torch.bfloat16 else "f32",
        "temperature": vi.temperature,
        "layout": "ragged" if vi.target_row_off is not None else "dense",
        "positions_per_step": positions, "logit_bytes_per_step": logit_bytes,
        "value": positions / (t_step * 1e-3), "unit": UNIT, "ms_per_step": t_step,
        "steps": n,
        "timing_ms": {"verify_median": t_verify,
                      "verify_p10": float(np.percentile(verify_ms, 10)),
                      "verify_p90": float(np.percentile(verify_ms, 90)),
                      "passes_median": pass_ms},
        "roofline": {"bound": "hbm", "achieved": kern, "peak": peak, "unit": "GB/s",
                     "frac": kern / peak, "frac_of_nominal": kern / 7900.0,
                     "kernel": "streaming pass (k_rowstats_tma, or k_rowstats_plain for rows "
                               "that are not 16-byte multiples)", "peak_source": peak_src},
        "roofline_call": {"bound": "hbm", "achieved": call, "peak": peak, "unit": "GB/s",
                          "frac": call / peak, "frac_of_nominal": call / 7900.0,
                          "scope": "whole dspark_verify call, logit bytes only"},
        "near_ties": ties,
        "input_checksum": checksum(input_tensors(vi)),
        "l2": ("inputs larger than L2, no flush" if logit_bytes > 129e6 else
               "inputs smaller than L2: repeated calls find them in L2"),
    }
    if sched is not None:
        conf = sched.confidences.cpu().numpy()
        prof = sched.step_time_ms.cpu().numpy()
        ref_s = oracle.schedule(conf, prof, early_stop=True)
        ts = []
        for _ in range(20):
            t0 = time.perf_counter()
            oracle.schedule(conf, prof, early_stop=True)
            ts.append(time.perf_counter() - t0)
        res["ms_per_step_note"] = "dspark_schedule then dspark_verify, serial on one stream"
        res["schedule"] = {
            "profile": "T(N) = 4 + 0.006 min(N, 2048) + 0.02 max(N - 2048, 0) ms",
            "median_us": statistics.median(sched_ms) * 1e3,
            "oracle_single_core_us": statistics.median(ts) * 1e6,
            "n_admitted": positions, "theta_best": float(sbuf.theta_best.item()),
            "equals_oracle": bool(np.array_equal(ell, ref_s["verify_len"])
                                  and ref_s["near_ties"] == 0),
            # the scheduler's rank path (two launches) takes up to 6,144
            # candidates, its block path (four) larger batches
            "gpu_launches_per_step": 2 if sched.R * sched.gamma <= 6144 else 4}
    if want_cpu:
        cores = oracle.max_threads()
        h = vi.to("cpu")
        runs = [oracle_verify_host(h, cores) for _ in range(3)]
        t_or = statistics.median(r[1] for r in runs)
        extra_s = res["schedule"]["oracle_single_core_us"] * 1e-6 if sched is not None else 0.0
        res["agreement"] = agreement(out, runs[0][0], ell)
        res["cpu_baseline"] = {
            "value": positions / (t_or + extra_s), "unit": UNIT, "cores": cores,
            "kind": "oracle",
            "sample": (f"all {h.B} requests, a host copy of the bytes the GPU verified, median "
                       f"of 3 passes ({t_or:.2f} s wall each), OpenMP over requests"
                       + (", plus Algorithm 1 on one core" if sched is not None else "")),
            "input_checksum": checksum(input_tensors(h)), "cpu": cpu_model()}
        del h
    del vi, vbuf
    torch.cuda.empty_cache()
    return res


# ---------------------------------------------------------------------------
# native arm
# ---------------------------------------------------------------------------
def native_arm(args):
    ws, rank, local = dist_env()
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    dist = init_dist(ws, "nccl")
    from speculative_decoding_verification_41_gb300 import binding, workloads
    from speculative_decoding_verification_41_gb300 import build as cuda_build
    if rank == 0 or not os.path.exists(cuda_build.LIB_PATH):
        cuda_build.build()
    barrier(dist, dev)
    binding.load()
    if args.drafter_only:
        res = drafter_measure(args, dev, torch.cuda.current_stream(dev), rank, ws)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return
    if args.only:
        peak, peak_src = measured_hbm_peak()
        res = measure_config(args.only, args, dev, torch.cuda.current_stream(dev), peak, peak_src,
                             want_cpu=rank == 0 and not args.no_cpu_baseline)
        if rank == 0:
            print(json.dumps(res), flush=True)
        return

    if args.batch is None and rank == 0:
        vi = workloads.make_config(WORKLOAD, device=dev)
    else:
        cfg = workloads.CONFIGS[WORKLOAD]
        vi = workloads.make_verify(args.batch or cfg["B"], cfg["gamma"], cfg["V"], cfg["dtype"],
                                   cfg["temperature"], rho=cfg["rho"], verify_len="full",
                                   seed=shard_seed(rank), device=dev,
                                   name=f"{WORKLOAD}_b{args.batch or cfg['B']}_shard{rank}")
    sched = workloads.make_schedule(vi.B, vi.gamma, seed=shard_seed(rank), device=dev,
                                    flat_profile=True)
    vbuf = binding.VerifyBuffers(vi.B, vi.gamma, vi.V, dev)
    sbuf = binding.ScheduleBuffers(vi.B, vi.gamma, dev)
    stream = torch.cuda.current_stream(dev)
    B, gamma, V, temperature = vi.B, vi.gamma, vi.V, vi.temperature

    def step():
        s = binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbuf)
        binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens, s["verify_len"],
                              vi.uniforms, vi.temperature, buffers=vbuf)

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize(dev)
    if int(sbuf.device_status.item()) != 0 or int(vbuf.device_status.item()) != 0:
        raise SystemExit("device status not OK during warm-up")
    ell = sbuf.verify_len.cpu().numpy()
    positions = int(ell.sum())
    logit_bytes = vi.logit_bytes(ell)
    # bytes beyond the algorithmic ones: the draw re-reads two rows per
    # rejected request (target and draft at k* = m + 1) and the bonus target row
    # otherwise; B_min is what a left-to-right early-exit design would read
    m_acc = vbuf.accepted_len.cpu().numpy().astype(np.int64)
    rej = m_acc < ell
    row_bytes = vi.V * vi.target_logits.element_size()
    resample_bytes = int((np.where(rej, 2, 1)).sum()) * row_bytes
    b_min_bytes = int(np.where(rej, 2 * (m_acc + 1), 2 * ell + 1).sum()) * row_bytes
    # a checksum of the inputs (64-bit sums of their bit patterns)
    input_checksum = checksum(input_tensors(vi))
    # the outputs of one step, for the request-by-request comparison with the
    # oracle on the host
    step_out = {k: v.clone() for k, v in (("accepted_len", vbuf.accepted_len),
                                          ("emitted_tokens", vbuf.emitted_tokens),
                                          ("probs", vbuf.probs))}
    step_ties = int(vbuf.near_tie_count.item())

    # timed region: the serving loop, pipelined as section 5.2's asynchronous
    # scheduler is -- step i+1's schedule runs on a side stream beside step i's
    # verification (the lengths double-buffered); every step does all its work
    # inside the region, whose events sit on the launching stream
    side = torch.cuda.Stream(dev)
    sbufs = [sbuf, binding.ScheduleBuffers(vi.B, vi.gamma, dev)]
    ready = [torch.cuda.Event() for _ in range(args.steps)]
    done = [torch.cuda.Event() for _ in range(args.steps)]

    def schedule_on_side(i):
        with torch.cuda.stream(side):
            if i >= 2:
                side.wait_event(done[i - 2])  # its buffer was read by verification i-2
            binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbufs[i % 2],
                                    stream=side)
            ready[i].record(side)

    clocks = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else local)
    clocks.start()
    time.sleep(0.3)
    barrier(dist, dev)
    torch.cuda.synchronize(dev)
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    _nvtx("push", "timed steps")  # for a profiler's timeline
    t_start.record(stream)
    side.wait_event(t_start)
    schedule_on_side(0)
    for i in range(args.steps):
        if i + 1 < args.steps:
            schedule_on_side(i + 1)
        stream.wait_event(ready[i])
        binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                              sbufs[i % 2].verify_len, vi.uniforms, vi.temperature, buffers=vbuf,
                              stream=stream)
        done[i].record(stream)
    t_end.record(stream)
    _nvtx("pop")
    torch.cuda.synchronize(dev)
    barrier(dist, dev)
    clk = clocks.stop()
    for b in sbufs[:min(2, args.steps)]:  # the buffers the loop wrote
        if int(b.device_status.item()) != 0 or not torch.equal(b.verify_len, sbuf.verify_len):
            raise SystemExit("schedule buffers disagree in the pipelined loop")
    total_ms = t_start.elapsed_time(t_end)
    total_ms = max_over_ranks(dist, total_ms, dev)
    ms_per_step = total_ms / args.steps
    value = aggregate_value(positions, ws, args.steps, total_ms)

    # per-call durations: the same calls one after the other on one stream,
    # with events between them
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(args.steps)]
    for i in range(args.steps):
        ev[i][0].record(stream)
        s = binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbuf)
        ev[i][1].record(stream)
        binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                              s["verify_len"], vi.uniforms, vi.temperature, buffers=vbuf)
        ev[i][2].record(stream)
    torch.cuda.synchronize(dev)
    sched_ms = [e[0].elapsed_time(e[1]) for e in ev]
    verify_ms = [e[1].elapsed_time(e[2]) for e in ev]
    serial_step_ms = statistics.median([e[0].elapsed_time(e[2]) for e in ev])

    # per-pass durations: the same steps again, the verify call through
    # dspark_verify_timed (events before k_plan, k_rowstats, k_decide and after)
    pev = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(args.steps)]
    for i in range(args.steps):
        s = binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbuf)
        binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                              s["verify_len"], vi.uniforms, vi.temperature, buffers=vbuf,
                              events=pev[i])
    torch.cuda.synchronize(dev)
    pass_ms = {name: statistics.median([e[j].elapsed_time(e[j + 1]) for e in pev])
               for j, name in enumerate(("k_plan", "k_rowstats_tma", "decision"))}

    # the acceptance probabilities of every verified position (a separate call,
    # not part of the step): its own median over a few calls
    acc_ws = torch.empty(binding.acceptance_workspace_bytes(vi.B, vi.gamma, vi.V),
                         dtype=torch.uint8, device=dev)
    acc_rates = torch.empty(vi.B, vi.gamma, dtype=torch.float32, device=dev)
    acc_ms = []
    for i in range(6):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        binding.dspark_acceptance(vi.target_logits, vi.draft_logits, sbuf.verify_len,
                                  vi.temperature, vi.gamma, rates=acc_rates, workspace=acc_ws)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        if i > 0:
            acc_ms.append(a0.elapsed_time(a1))
    del acc_ws
    # the verification and the rates in one call (one statistics pass for both)
    rbuf = binding.VerifyBuffers(vi.B, vi.gamma, vi.V, dev, with_rates=True)
    vr_ms = []
    for i in range(6):
        a0, a1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a0.record(stream)
        binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                              sbuf.verify_len, vi.uniforms, vi.temperature, buffers=rbuf,
                              with_rates=True)
        a1.record(stream)
        torch.cuda.synchronize(dev)
        if i > 0:
            vr_ms.append(a0.elapsed_time(a1))
    if not torch.equal(rbuf.rates, acc_rates):
        raise SystemExit("dspark_verify_rates and dspark_acceptance disagree")
    del rbuf

    drafter = None if args.no_drafter else drafter_measure(args, dev, stream, rank, ws)

    # end to end: pinned host buffers -> device, both calls, results back
    e2e = None
    if args.e2e_steps > 0:
        host = {k: getattr(vi, k).cpu().pin_memory() for k in
                ("target_logits", "draft_logits", "draft_tokens", "uniforms")}
        host_conf = sched.confidences.cpu().pin_memory()
        host_prof = sched.step_time_ms.cpu().pin_memory()
        # two sets of device inputs: step i+1's inputs cross the host link on a
        # copy stream while step i is verified (every step still copies its
        # own inputs in and its results out inside the timed region)
        dbufs = [{k: torch.empty_like(getattr(vi, k)) for k in host} for _ in range(2)]
        dconfs = [torch.empty_like(sched.confidences) for _ in range(2)]
        dprofs = [torch.empty_like(sched.step_time_ms) for _ in range(2)]
        out_acc = torch.empty(vi.B, dtype=torch.int32).pin_memory()
        out_em = torch.empty(vi.B, vi.gamma + 1, dtype=torch.int32).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values()) + \
            host_conf.numel() * 4 + host_prof.numel() * 8
        d2h = out_acc.numel() * 4 + out_em.numel() * 4
        copy_stream = torch.cuda.Stream(dev)
        n_e2e = args.e2e_steps + 1  # one untimed step first
        copied = [torch.cuda.Event() for _ in range(n_e2e)]
        used = [torch.cuda.Event() for _ in range(n_e2e)]

        def copy_in(i):
            j = i % 2
            with torch.cuda.stream(copy_stream):
                if i >= 2:
                    copy_stream.wait_event(used[i - 2])  # step i-2 is done with this set
                for k, t in host.items():
                    dbufs[j][k].copy_(t, non_blocking=True)
                dconfs[j].copy_(host_conf, non_blocking=True)
                dprofs[j].copy_(host_prof, non_blocking=True)
                copied[i].record(copy_stream)

        def compute(i):
            j = i % 2
            stream.wait_event(copied[i])
            s = binding.dspark_schedule(dconfs[j], dprofs[j], buffers=sbuf)
            d = dbufs[j]
            o = binding.dspark_verify(d["target_logits"], d["draft_logits"], d["draft_tokens"],
                                      s["verify_len"], d["uniforms"], vi.temperature,
                                      buffers=vbuf)
            used[i].record(stream)
            out_acc.copy_(o["accepted_len"], non_blocking=True)
            out_em.copy_(o["emitted_tokens"], non_blocking=True)

        copy_in(0)
        compute(0)
        torch.cuda.synchronize(dev)
        barrier(dist, dev)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(stream)
        copy_stream.wait_event(a)
        copy_in(1)
        for i in range(1, n_e2e):
            if i + 1 < n_e2e:
                copy_in(i + 1)
            compute(i)
        b.record(stream)
        torch.cuda.synchronize(dev)
        e2e_ms = max_over_ranks(dist, a.elapsed_time(b), dev)
        e2e = {"value": positions * ws * args.e2e_steps / (e2e_ms * 1e-3), "unit": UNIT,
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h),
               "ms_per_step": e2e_ms / args.e2e_steps,
               "copies": "step i+1's inputs copied on a second stream while step i is verified"}
        del host, dbufs

    cpu = agree = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        cores = oracle.max_threads()
        h = vi.to("cpu")   # the very bytes the GPU verified
        n_req = max(1, min(args.cpu_sample, vi.B))
        runs = [oracle_verify_host(h, cores, n_req) for _ in range(3)]
        t = statistics.median(r[1] for r in runs)
        if n_req == vi.B:
            agree = agreement(step_out, runs[0][0], ell)
        n1 = max(1, min(16, n_req))
        _, t1 = oracle_verify_host(h, 1, n1)
        cpu = {"value": int(ell[:n_req].sum()) / t, "unit": UNIT, "cores": cores,
               "kind": "oracle",
               "sample": f"{n_req} of {vi.B} requests of {WORKLOAD}, a host copy of the bytes "
                         f"the GPU verified, median of 3 passes, {t:.2f} s wall each, OpenMP "
                         f"over requests",
               "input_checksum": checksum(input_tensors(h)),
               "single_thread_value": int(ell[:n1].sum()) / t1,
               "single_thread_sample": f"the first {n1} requests, one pass, {t1:.2f} s wall",
               "cpu": cpu_model()}
        del h

    # the other named workloads, one at a time (the headline's inputs freed)
    configs = {}
    names = [c for c in args.configs.split(",") if c] if ws == 1 else []
    if names:
        del vi
        torch.cuda.empty_cache()
    peak, peak_src = measured_hbm_peak()
    for nm in names:
        configs[nm] = measure_config(nm, args, dev, stream, peak, peak_src,
                                     want_cpu=rank == 0 and not args.no_cpu_baseline)

    if rank != 0:
        return
    v_med = statistics.median(verify_ms)
    achieved_call = logit_bytes / (v_med * 1e-3) / 1e9
    achieved = logit_bytes / (pass_ms["k_rowstats_tma"] * 1e-3) / 1e9
    traffic = measured_traffic(logit_bytes)
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": ws, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B, "gamma": gamma, "V": V,
                   "temperature": temperature, "positions_per_step": positions,
                   "logit_bytes_per_step": logit_bytes,
                   "input_checksum": input_checksum,
                   "l2": "inputs (2.18 GB) larger than L2, no flush",
                   "step": "dspark_schedule (flat profile) + dspark_verify; step i+1's "
                           "schedule on a side stream beside step i's verify"},
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "nominal_peak": 7900.0, "frac_of_nominal": achieved / 7900.0,
                     "kernel": "k_rowstats_tma (streaming pass; median CUDA-event interval "
                               "around its launch, dspark_verify_timed)",
                     "peak_source": peak_src,
                     "peak_note": "the measured peak is a copy, which moves every byte both "
                                  "ways; a read-only stream can exceed it, so the nominal "
                                  "7.9 TB/s fraction is given beside it"},
        "bytes_per_step": {"algorithmic": logit_bytes, "resample_reread": resample_bytes,
                           "actual": logit_bytes + resample_bytes, "b_min_early_exit": b_min_bytes},
        "roofline_call": {"bound": "hbm", "achieved": achieved_call, "peak": peak,
                          "unit": "GB/s", "frac": achieved_call / peak,
                          "scope": "whole dspark_verify call (k_plan, k_rowstats_tma, k_desc, "
                                   "k_resid, k_pick), median CUDA-event time, logit bytes only"},
        "timing_ms": {"verify_median": v_med, "verify_p10": float(np.percentile(verify_ms, 10)),
                      "verify_p90": float(np.percentile(verify_ms, 90)),
                      "schedule_median": statistics.median(sched_ms),
                      "serial_step_median": serial_step_ms,
                      "passes_median": pass_ms,
                      "acceptance_median": statistics.median(acc_ms),
                      "verify_rates_median": statistics.median(vr_ms)},
        "gpu_launches": args.steps * 7,  # per step: k_sched_rank, k_sched_sweep, k_plan, k_rowstats_tma, k_desc, k_resid, k_pick
        "near_ties": step_ties,
        "agreement": agree,
        "clocks": clk,
        "e2e": e2e,
        "cpu_baseline": cpu,
        "drafter": drafter,
        "configs": configs,
    }
    if drafter is not None and drafter.get("roofline"):
        drafter["roofline"]["peak"] = peak
        drafter["roofline"]["frac"] = drafter["roofline"]["achieved"] / peak
        drafter["roofline"]["peak_source"] = peak_src
        drafter["block"]["frac"] = drafter["block"]["achieved"] / peak
    print(json.dumps(line), flush=True)


DRAFT_SHAPE = dict(B=256, gamma=16, V=129280, r=256, temperature=0.7)


def draft_algorithmic_bytes(B, gamma, V, r) -> int:
    """Compulsory DRAM bytes of one k_draft_step launch: U_k read and L_k written
    (bf16), one statistic per (request, 128-token tile) written, the batch's
    W1 rows read, and W2 once per call spread over its gamma launches."""
    tiles = -(-V // 128)
    return 2 * B * V * 2 + B * tiles * 8 + B * r * 2 + V * r * 2 // gamma


def drafter_measure(args, dev, stream, rank, ws):
    """The drafter's sequential stage with the Markov head (dspark_draft_markov)
    on 256 requests x 16 positions x 129,280 tokens, rank 256: its own median
    call time (separate from the verification step), per-kernel medians through
    dspark_draft_markov_timed, and the oracle on a host sample."""
    from speculative_decoding_verification_41_gb300 import binding, workloads
    sh = dict(DRAFT_SHAPE, B=args.draft_batch or DRAFT_SHAPE["B"])
    d = workloads.make_markov_draft(sh["B"], sh["gamma"], sh["V"], sh["r"],
                                    temperature=sh["temperature"], seed=shard_seed(rank),
                                    device=dev)
    out_L = torch.empty_like(d.base_logits)
    out_x = torch.empty(sh["B"], sh["gamma"], dtype=torch.int32, device=dev)
    wsp = torch.empty(binding.draft_workspace_bytes(sh["B"], sh["r"], sh["V"]), dtype=torch.uint8,
                      device=dev)

    def call(events=None):
        return binding.dspark_draft_markov(d.base_logits, d.w1, d.w2t, d.anchors, d.uniforms,
                                           d.temperature, draft_logits=out_L, draft_tokens=out_x,
                                           workspace=wsp, events=events)

    for _ in range(3):
        o = call()
    torch.cuda.synchronize(dev)
    if int(o["device_status"].item()) != 0:
        raise SystemExit("drafter device status not OK during warm-up")
    # calls issued back to back with an event pair around each, one
    # synchronisation at the end (as the verification steps are timed): the
    # host stays ahead of the GPU, so an interval holds the call's device work,
    # not the host's time to submit it to an idle GPU
    n = max(5, min(args.steps, 20))
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
           for _ in range(n)]
    for a0, a1 in evs:
        a0.record(stream)
        call()
        a1.record(stream)
    torch.cuda.synchronize(dev)
    ms = [a0.elapsed_time(a1) for a0, a1 in evs]
    # a soak of back-to-back calls with the clocks sampled during it
    clocks = ClockSampler(dev.index if "CUDA_VISIBLE_DEVICES" not in os.environ else
                          int(os.environ.get("LOCAL_RANK", "0")))
    clocks.start()
    time.sleep(0.3)
    s0, s1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    n_soak = max(20, int(1.2 / max(statistics.median(ms) * 1e-3, 1e-4)))
    s0.record(stream)
    for _ in range(n_soak):
        call()
    s1.record(stream)
    torch.cuda.synchronize(dev)
    clk = clocks.stop()
    soak_ms = s0.elapsed_time(s1) / n_soak
    g = sh["gamma"]
    step_ms, pick_ms = [], []
    for _ in range(3):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(2 * g + 2)]
        call(events=ev)
        torch.cuda.synchronize(dev)
        step_ms += [ev[1 + 2 * k].elapsed_time(ev[2 + 2 * k]) for k in range(g)]
        pick_ms += [ev[2 + 2 * k].elapsed_time(ev[3 + 2 * k]) for k in range(g)]
    t_call = statistics.median(ms)
    t_step = statistics.median(step_ms)
    positions = sh["B"] * g
    alg = draft_algorithmic_bytes(sh["B"], g, sh["V"], sh["r"])
    flops = 2.0 * sh["B"] * sh["V"] * sh["r"]
    res = {
        "metric": "draft_positions_per_s", "value": positions * ws / (t_call * 1e-3),
        "unit": "positions/s", "ms_per_call": t_call,
        "config": {"workload": f"draft_b{sh['B']}_g{g}_v{sh['V']}_r{sh['r']}_bf16",
                   "weights": "random on the 2^-8 grid", "temperature": sh["temperature"],
                   "l2": "base logits (1.06 GB) larger than L2, no flush"},
        "clocks": clk,
        "timing_ms": {"call_median": t_call, "call_p90": float(np.percentile(ms, 90)),
                      "call_soak_mean": soak_ms,
                      "k_draft_step_median": t_step, "k_draft_pick_median":
                          statistics.median(pick_ms)},
        "roofline": {"bound": "hbm", "achieved": alg / (t_step * 1e-3) / 1e9, "unit": "GB/s",
                     "traffic": None, "algorithmic_bytes_per_launch": alg,
                     "kernel": "k_draft_step (median CUDA-event interval around each of the 16 "
                               "launches, dspark_draft_markov_timed)",
                     "tensor_tflops": flops / (t_step * 1e-3) / 1e12},
        # the product path, the whole block as one cooperative launch
        # (k_draft_pair for two request tiles, 128 < B <= 256; k_draft_block
        # for one): the same bytes per position (W2 counted once) over the
        # call time, the chain between positions included
        "block": {"kernel": "k_draft_pair" if 128 < sh["B"] <= 256 else "k_draft_block",
                  "algorithmic_bytes": alg * g,
                  "achieved": alg * g / (t_call * 1e-3) / 1e9, "unit": "GB/s",
                  "tensor_tflops": flops * g / (t_call * 1e-3) / 1e12},
        "gpu_launches_per_call": 1,  # one cooperative launch, after one memset
        "gpu_launches_per_call_timed_path": 1 + 2 * g,
        "cpu_baseline": None,
    }
    del out_L
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        cores = oracle.max_threads()
        nreq = max(1, min(cores, 16))
        U = workloads.bf16_bits(d.base_logits[:nreq])
        W1, W2t = workloads.bf16_bits(d.w1), workloads.bf16_bits(d.w2t)
        x0, u = d.anchors[:nreq].cpu().numpy(), d.uniforms[:nreq].cpu().numpy()
        t0 = time.perf_counter()
        oracle.markov_draft(U, W1, W2t, x0, u, d.temperature, nthreads=cores)
        t = time.perf_counter() - t0
        res["cpu_baseline"] = {"value": nreq * g / t, "unit": "positions/s", "cores": cores,
                               "kind": "oracle",
                               "sample": f"{nreq} of 256 requests, all 16 positions, "
                                         f"{t:.2f} s wall, OpenMP over requests"}
    return res


# DRAM traffic of the streaming kernel from one ncu capture (dram__bytes_read.sum +
# dram__bytes_write.sum) on the B = 32 case of the headline recipe, scaled per
# logit byte; valid only for the sources the kernel is built from (the headers
# hashed below), as they were at the capture.
TRAFFIC_CAPTURE = {
    "sources_sha256": "118816c64befe0531575031839ed371c052b6efabab2261d94be4f2980d328a1",
    "dram_bytes": 273095936 + 3616768,  # read + write, one launch at B = 32
    "logit_bytes": 273039360,
}


def kernel_sources_sha256() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "speculative_decoding_verification_41_gb300", "csrc")
    for f in ("dspark_rowstats.cuh", "dspark_verify_types.cuh", "dspark_common.cuh"):
        h.update(open(os.path.join(csrc, f), "rb").read())
    return h.hexdigest()


def measured_traffic(logit_bytes: int):
    cap = TRAFFIC_CAPTURE
    if not cap["sources_sha256"] or cap["sources_sha256"] != kernel_sources_sha256():
        return None
    return cap["dram_bytes"] / cap["logit_bytes"] * logit_bytes


def measured_hbm_peak():
    """The HBM peak of the GB300s (a measured copy, burst), else the
    fallback figure; returns (GB/s, "measured" | "fallback")."""
    try:
        peak = json.load(open(os.path.join(ROOT, "MEASURED_PEAKS.json"))).get("hbm_gbs")
    except (OSError, ValueError):
        peak = None
    return (peak, "measured") if peak else (6800.0, "fallback")


def _nvtx(op: str, name: str = "") -> None:
    """An NVTX range mark, if this torch build has NVTX (it only labels a
    profiler's timeline)."""
    try:
        if op == "push":
            torch.cuda.nvtx.range_push(name)
        else:
            torch.cuda.nvtx.range_pop()
    except Exception:
        pass


def main():
    args = parse()
    if args.impl == "reference":
        reference_arm(args)
    else:
        native_arm(args)


if __name__ == "__main__":
    main()
