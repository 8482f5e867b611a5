"""Multi-rank logic of bench.py on CPU (gloo, world size 2).

The decode path shards by batch with no exchange step, so the only
cross-rank code is the timing: every rank times its own replica batch, the
job is timed by the slowest rank (an all-reduce MAX), and the whole-job value
is world x the per-rank bytes over that time.  These tests run that same code
over the gloo backend in two spawned processes; the GPU run uses NCCL.
"""
import json
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, q) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench as b
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r reports elapsed 10+r ms and attend 5-r ms: the job takes the max of each
        got = b.max_over_ranks([10.0 + rank, 5.0 - rank], dist)
        dist.barrier()
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = {}
    try:
        for _ in procs:
            rank, got = q.get(timeout=180)
            results[rank] = got
    finally:
        for p in procs:
            p.join(timeout=60)
            if p.is_alive():
                p.kill()
    assert all(p.exitcode == 0 for p in procs)
    assert results == {0: [11.0, 5.0], 1: [11.0, 5.0]}


def test_max_over_ranks_without_group_is_identity():
    assert bench.max_over_ranks([3.0, 4.5]) == [3.0, 4.5]


def test_job_throughput_is_weak_scaling():
    one = bench.job_throughput(603_979_776, 1, 0.25)
    assert one == pytest.approx(603_979_776 / 0.25e-3 / 1e9)
    # twice the ranks in the same (slowest-rank) time: twice the job's bytes per second
    assert bench.job_throughput(603_979_776, 2, 0.25) == pytest.approx(2 * one)


def test_reference_arm_prints_on_rank_zero_only(monkeypatch, capsys):
    args = ["--impl", "reference", "--workload", "v2lite_batch", "--seqlen", "64", "--steps", "1", "--warmup", "3",
            "--gpus", "2"]
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    assert bench.main(args) == 0
    assert capsys.readouterr().out.strip() == ""
    monkeypatch.setenv("RANK", "0")
    assert bench.main(args) == 0
    lines = [l for l in capsys.readouterr().out.splitlines() if l.strip()]
    assert len(lines) == 1
    rec = json.loads(lines[0])
    assert rec["impl"] == "reference" and rec["n_gpus"] == 2 and rec["value"] > 0
    assert rec["e2e"]["h2d_bytes_per_step"] == 0 and rec["cpu_baseline"]["kind"] == "oracle"
