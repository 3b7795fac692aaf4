"""Multi-rank host logic of the benchmark on CPU (gloo, two ranks).

The path shards by block (or head) with no collective on the data path: every
rank runs an independent workload, and the only cross-rank step is the
max-over-ranks timing reduction at the end.  These checks run that logic
in two real processes over the gloo backend.
"""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        per_rank_ms = 10.0 + 5.0 * rank
        total = bench.max_over_ranks(per_rank_ms, world, torch.device("cpu"))
        value = bench.whole_job_value(1e12, world, 4, total)
        blocks = [None] * world
        dist.all_gather_object(blocks, bench.rank_block(rank))
        q.put((rank, total, value, blocks))
    finally:
        dist.destroy_process_group()


def test_two_rank_timing_reduction_and_independent_blocks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, total, value, blocks in res:
        assert total == 15.0                                   # slowest rank's time on every rank
        assert value == pytest.approx(1e12 * 2 * 4 / 15e-3 / 1e12)  # all ranks' work / slowest time
        assert sorted(blocks) == [0, 1]                        # each rank seeds a different block


def test_reference_arm_is_rank0_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.main() == 0
    assert capsys.readouterr().out == ""
