"""The calls captured in a CUDA graph and replayed: the library allocates
nothing, never synchronises and launches only on the caller's stream, so a
serving loop can capture a whole step (scheduler, verification, drafter) once
and replay it. Replays must give the eager calls' outputs bit for bit, replay
after replay (the per-call counters are reset inside the captured work)."""
import pytest
import torch

from speculative_decoding_verification_41_gb300 import binding, workloads
from speculative_decoding_verification_41_gb300 import build as cuda_build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    cuda_build.build()
    return torch.device("cuda:0")


def test_schedule_and_verify_replay(dev):
    B, g, V = 48, 16, 30000
    vi = workloads.make_verify(B, g, V, torch.bfloat16, 0.7, rho=(0.6, 0.95), seed=9, device=dev)
    sched = workloads.make_schedule(B, g, seed=9, device=dev)
    sbuf = binding.ScheduleBuffers(B, g, dev)
    vbuf = binding.VerifyBuffers(B, g, V, dev, with_rates=True)

    def step():
        s = binding.dspark_schedule(sched.confidences, sched.step_time_ms, buffers=sbuf)
        return binding.dspark_verify(vi.target_logits, vi.draft_logits, vi.draft_tokens,
                                     s["verify_len"], vi.uniforms, vi.temperature,
                                     buffers=vbuf, with_rates=True)

    out = step()  # eager: also sets the kernel attributes before capture
    torch.cuda.synchronize()
    assert int(vbuf.device_status.item()) == 0 and int(sbuf.device_status.item()) == 0
    ref = {k: v.clone() for k, v in out.items() if v is not None}
    ref_len = sbuf.verify_len.clone()

    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        cap = step()  # the buffers' tensors
    for _ in range(3):
        for t in (vbuf.accepted_len, vbuf.emitted_tokens, vbuf.rates, sbuf.verify_len):
            t.fill_(-7)
        graph.replay()
        torch.cuda.synchronize()
        assert int(vbuf.device_status.item()) == 0
        assert torch.equal(sbuf.verify_len, ref_len)
        for k in ref:
            assert torch.equal(cap[k], ref[k]), k


def test_drafter_replay(dev):
    d = workloads.make_markov_draft(40, 8, 6000, 128, temperature=0.8, seed=5, device=dev)
    ws = torch.empty(binding.draft_workspace_bytes(40, 128, 6000), dtype=torch.uint8, device=dev)
    logits = torch.empty_like(d.base_logits)
    tokens = torch.empty(40, 8, dtype=torch.int32, device=dev)

    def draft():
        return binding.dspark_draft_markov(d.base_logits, d.w1, d.w2t, d.anchors, d.uniforms,
                                           d.temperature, draft_logits=logits,
                                           draft_tokens=tokens, workspace=ws)

    draft()
    torch.cuda.synchronize()
    ref_l, ref_t = logits.clone(), tokens.clone()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        draft()
    for _ in range(3):
        logits.zero_()
        tokens.fill_(-1)
        graph.replay()
        torch.cuda.synchronize()
        assert torch.equal(tokens, ref_t)
        assert torch.equal(logits, ref_l)
