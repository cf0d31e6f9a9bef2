"""The multi-rank (replica) path of bench.py on CPU: world_size 2 over gloo.

Query rows are independent, so N GPUs run N replicas with no collective on
the data path; the only exchange is the timing (the max over ranks), and the
job's rate counts every rank's units. The reference arm runs on rank 0 only.
"""
import os
import socket
import sys

import pytest
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, times: list, out) -> None:
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        slowest = bench.max_over_ranks(times[rank], world)
        args = type("A", (), {"k": 512, "steps": 1, "warmup": 1})()
        ref = bench.run_reference(args, world, rank) if rank != 0 else "rank0"
        out.put((rank, slowest, ref))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_replicas_take_the_max_time_and_sum_the_units():
    world, times = 2, [0.040, 0.047]
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[1] for g in got] == pytest.approx([0.047, 0.047])   # every rank sees the slowest
    assert got[1][2] is None                                      # the reference arm: rank 0 alone
    rate = bench.whole_job_rate(world, 256 * 65536, 0.047)
    assert rate == pytest.approx(2 * 256 * 65536 / 47e-6)


def test_single_rank_rate_and_env(monkeypatch):
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench.dist_env() == (1, 0, 0)
    assert bench.max_over_ranks(1.5, 1) == 1.5
    assert bench.whole_job_rate(1, 1000, 2.0) == pytest.approx(5e5)
