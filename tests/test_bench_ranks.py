"""The multi-rank host logic of bench.py on CPU: N independent replicas
(one per rank, no data-path collective), the step time taken as the maximum
over the ranks and the job throughput as every rank's units over that time;
under torchrun the reference arm runs on rank 0 only. World size 2 over the
gloo backend on 127.0.0.1."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = [2.5, 4.0][rank]                    # rank 1 is the slower replica
        slow = bench.max_over_ranks(ms, world)   # a collective: both ranks call it
        out[rank] = (slow, bench.job_tops(1.0e12, slow, world))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_rank_max_and_job_throughput():
    world = 2
    out = mp.Manager().dict()
    mp.spawn(_worker, args=(world, _free_port(), out), nprocs=world, join=True)
    for rank in range(world):
        slow, tops = out[rank]
        assert slow == 4.0                       # every rank sees the slowest rank's time
        assert tops == pytest.approx(2 * 1.0e12 / 4.0e-3 / 1e12)   # both ranks' units over it


def test_single_rank_is_its_own_time():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.job_tops(2.0e12, 1.0, 1) == pytest.approx(2000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.main(["--impl", "reference", "--gpus", "2", "--steps", "1", "--warmup", "3"]) == 0
    assert capsys.readouterr().out == ""         # rank 1 does no work and prints nothing
