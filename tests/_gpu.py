"""Helpers of the GPU parity tests: run the oracle on a sample of requests of a
device-resident workload and compare the CUDA outputs with it."""
from __future__ import annotations

import numpy as np
import torch

import oracle

PROB_ATOL = 1e-5          # probabilities: absolute agreement required
PROB_RTOL_QUALITY = 2e-6  # relative agreement the kernels are expected to reach
MISMATCH_RATE = 1e-4      # actual disagreements allowed per (ratio test + draw)


def logits_to_numpy(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)
    return t.contiguous().cpu().numpy()


def offsets(vi):
    B, g = vi.B, vi.gamma
    if vi.target_row_off is None:
        return np.arange(B + 1, dtype=np.int64) * (g + 1), np.arange(B + 1, dtype=np.int64) * g
    return vi.target_row_off.cpu().numpy(), vi.draft_row_off.cpu().numpy()


def oracle_on_requests(vi, idx, nthreads=None):
    """Run the oracle on requests `idx` of `vi`, gathering only their rows."""
    idx = np.asarray(idx, np.int64)
    ell = vi.verify_len.cpu().numpy().astype(np.int64)
    toff, doff = offsets(vi)
    trows = np.concatenate([toff[r] + np.arange(ell[r] + 1) for r in idx]) if len(idx) else np.zeros(0, np.int64)
    drows = [doff[r] + np.arange(ell[r]) for r in idx]
    drows = np.concatenate(drows) if drows else np.zeros(0, np.int64)
    dev = vi.target_logits.device
    tsub = logits_to_numpy(vi.target_logits.index_select(0, torch.from_numpy(trows).to(dev)))
    if drows.size:
        dsub = logits_to_numpy(vi.draft_logits.index_select(0, torch.from_numpy(drows).to(dev)))
    else:
        dsub = logits_to_numpy(vi.draft_logits[:1])
    t_new = np.concatenate([[0], np.cumsum(ell[idx] + 1)]).astype(np.int64)
    d_new = np.concatenate([[0], np.cumsum(ell[idx])]).astype(np.int64)
    if nthreads is None:
        nthreads = oracle.max_threads()
    ref = oracle.verify(tsub, dsub, vi.draft_tokens.cpu().numpy()[idx], ell[idx].astype(np.int32),
                        vi.uniforms.cpu().numpy()[idx], vi.temperature, t_new, d_new,
                        nthreads=nthreads)
    return ref


def compare(out, ref, vi, idx, mismatch_budget=True):
    """Element-by-element comparison. Returns statistics; raises on a mismatch
    that no near-tie flag of the oracle excuses, on a probability error above
    PROB_ATOL, and (mismatch_budget) on more excused mismatches -- requests
    whose outputs actually differ at a flagged near tie -- than MISMATCH_RATE
    of the decisions the oracle took: its ratio tests (positions 1..min(m+1, l)
    of each request) plus one draw per request."""
    idx = np.asarray(idx, np.int64)
    ell = vi.verify_len.cpu().numpy()[idx]
    acc = out["accepted_len"].cpu().numpy()[idx]
    em = out["emitted_tokens"].cpu().numpy()[idx]
    flagged = ref["flags"].any(axis=1)
    same = (acc == ref["accepted_len"]) & (em == ref["emitted"]).all(axis=1)
    bad = np.nonzero(~same & ~flagged)[0]
    assert bad.size == 0, (
        f"{bad.size} unexcused mismatches, e.g. request {idx[bad[0]]}: gpu m={acc[bad[0]]} "
        f"{em[bad[0]].tolist()} oracle m={ref['accepted_len'][bad[0]]} {ref['emitted'][bad[0]].tolist()}")
    ratio_tests = int(np.minimum(ref["accepted_len"].astype(np.int64) + 1, ell).sum())
    stats = {"requests": int(len(idx)), "excused": int((~same & flagged).sum()),
             "flagged": int(flagged.sum()), "ratio_tests": ratio_tests, "draws": int(len(idx))}
    stats["mismatch_budget"] = int(MISMATCH_RATE * (ratio_tests + len(idx)))
    if mismatch_budget:
        assert stats["excused"] <= stats["mismatch_budget"], (
            f"{stats['excused']} requests differ at flagged near ties, more than "
            f"{MISMATCH_RATE} of {ratio_tests} ratio tests + {len(idx)} draws")
    if out.get("probs") is not None:
        pr = out["probs"].cpu().numpy()[idx].astype(np.float64)
        g = pr.shape[1]
        verified = np.arange(g)[None, :] < ell[:, None]
        err = np.abs(pr - ref["probs"])[verified]
        stats["prob_max_abs_err"] = float(err.max()) if err.size else 0.0
        assert stats["prob_max_abs_err"] <= PROB_ATOL
        denom = np.maximum(ref["probs"][verified], 1e-300)
        rel = np.abs(pr[verified] - ref["probs"][verified]) / denom
        big = ref["probs"][verified] > 1e-30
        stats["prob_max_rel_err"] = float(rel[big].max()) if big.any() else 0.0
        assert np.all(pr[~verified] == -1.0)
    stats["decisions"] = ratio_tests + int(len(idx))
    return stats


def near_tie_budget(out, vi):
    """Decisions taken by one verification call: the ratio tests actually
    evaluated (positions 1..min(m+1, l)) and the comparisons of each inverse-CDF
    scan (tokens 0..y, i.e. y + 1 per draw)."""
    acc = out["accepted_len"].cpu().numpy().astype(np.int64)
    em = out["emitted_tokens"].cpu().numpy().astype(np.int64)
    ell = vi.verify_len.cpu().numpy().astype(np.int64)
    y = em[np.arange(len(acc)), acc]
    ratio = int(np.minimum(acc + 1, ell).sum())
    cdf = int((y + 1).sum())
    return {"ratio_tests": ratio, "cdf_comparisons": cdf, "draws": int(len(acc)),
            "decisions": ratio + cdf}
