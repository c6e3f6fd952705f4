"""The multi-GPU path of the bench is replicas only (each rank runs its own
GEMMs; no collective on the data path).  Its host logic -- the job time as the
maximum over ranks and the whole-job throughput -- runs here on CPU ranks over
gloo, world size 2."""
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


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t_max = bench.max_over_ranks(times[rank], dist, torch, "cpu")
        out[rank] = (t_max, bench.job_value(world, 1000.0, t_max))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value_gloo():
    world, times = 2, [0.5, 0.8]
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_rank_main, args=(world, _free_port(), times, out), nprocs=world, start_method="spawn")
    for r in range(world):
        t_max, value = out[r]
        assert t_max == max(times)
        assert value == pytest.approx(world * 1000.0 / max(times))


def test_reference_arm_other_ranks_exit_without_work(monkeypatch, capsys):
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setattr(sys, "argv", ["bench.py", "--impl", "reference", "--gpus", "2"])
    assert bench.run_reference(bench.parse_args()) == 0
    assert capsys.readouterr().out == ""
