"""bench.py's multi-rank plumbing on CPU: two gloo ranks reduce their timings
(max of the elapsed times, sum of the verified positions), and the reference
arm runs on rank 0 only."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out_dir):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        elapsed, units = bench.reduce_timing(0.5 + rank, 100.0 * (rank + 1))
        bench.barrier()
        with open(os.path.join(out_dir, f"r{rank}.txt"), "w") as f:
            f.write(f"{elapsed} {units}")
    finally:
        dist.destroy_process_group()


def test_reduce_timing_two_gloo_ranks(tmp_path):
    import torch.multiprocessing as mp
    port = _free_port()
    mp.start_processes(_rank_main, args=(2, port, str(tmp_path)), nprocs=2, join=True,
                       start_method="spawn")
    for r in range(2):
        elapsed, units = map(float, open(tmp_path / f"r{r}.txt").read().split())
        assert elapsed == 1.5      # the slowest rank's time
        assert units == 300.0      # every rank's positions


def test_reduce_timing_without_process_group():
    import bench
    assert bench.reduce_timing(0.25, 7.0) == (0.25, 7.0)


def test_reference_arm_runs_on_rank0_only(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    bench.main(["--impl", "reference", "--steps", "1", "--warmup", "0"])
    assert capsys.readouterr().out == ""
