"""The multi-rank path of bench.py, on the CPU with two gloo ranks.

Verification shards without any data-path collective: each rank verifies its
own requests. What the ranks share is host logic: the timing barrier, the
maximum of the timed regions over ranks, the shard each rank generates, and
the whole-job throughput. The GPU arm itself needs CUDA; here the same
functions run under torch.distributed with the gloo backend, world size 2.
"""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
WORLD = 2


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, port: int, out_dir: str):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(WORLD), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (WORLD, rank, rank)
    d = bench.init_dist(ws, "gloo")
    assert d is not None and d.get_world_size() == WORLD
    bench.barrier(d)
    # each rank times a different region; the job takes the slowest
    mx = bench.max_over_ranks(d, 10.0 + 5.0 * rank, torch.device("cpu"))
    seeds = [None] * WORLD
    d.all_gather_object(seeds, bench.shard_seed(rank))
    bench.barrier(d)
    with open(os.path.join(out_dir, f"rank{rank}.json"), "w") as f:
        json.dump({"max": mx, "seeds": seeds}, f)
    d.destroy_process_group()


@pytest.fixture(scope="module")
def rank_results(tmp_path_factory):
    out = tmp_path_factory.mktemp("ranks")
    mp.start_processes(_rank_main, args=(free_port(), str(out)), nprocs=WORLD,
                       start_method="spawn", join=True)
    return [json.load(open(out / f"rank{r}.json")) for r in range(WORLD)]


def test_max_over_ranks_is_the_slowest_region(rank_results):
    for res in rank_results:
        assert res["max"] == 15.0


def test_ranks_verify_distinct_shards(rank_results):
    seeds = rank_results[0]["seeds"]
    assert seeds == rank_results[1]["seeds"]
    assert len(set(seeds)) == WORLD
    assert seeds[0] == 7  # rank 0's shard is the headline workload's seed


def test_whole_job_throughput_counts_every_rank():
    sys.path.insert(0, ROOT)
    import bench
    one = bench.aggregate_value(4096, 1, 30, 12.0)
    two = bench.aggregate_value(4096, 2, 30, 12.0)
    assert two == pytest.approx(2 * one)
    assert one == pytest.approx(4096 * 30 / 12e-3)


def test_reference_arm_under_torchrun_prints_one_line_on_rank0():
    port = free_port()
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes", "1", "--nproc-per-node",
           str(WORLD), "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py",
           "--impl", "reference", "--gpus", str(WORLD), "--steps", "1", "--warmup", "0",
           "--cpu-sample", "2"]
    env = dict(os.environ, OMP_NUM_THREADS="2")
    p = subprocess.run(cmd, cwd=ROOT, capture_output=True, text=True, timeout=600, env=env)
    assert p.returncode == 0, p.stderr[-2000:]
    lines = [ln for ln in p.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, p.stdout
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == WORLD
    assert rec["value"] > 0 and rec["e2e"]["h2d_bytes_per_step"] == 0
    assert rec["cpu_baseline"]["kind"] == "oracle"
