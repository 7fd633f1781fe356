"""Multi-rank host logic of bench.py on CPU: gloo, world size 2.

The path shards by output rows with no collective; bench.py runs one replica
per rank, takes the slowest rank's time and reports the whole-job weight
GB/s. Here two gloo ranks check the barrier, the max-over-ranks reduction
and the aggregation, without a GPU.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "LOCAL_RANK": str(rank),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    import bench
    import torch.distributed as dist
    r, w = bench.dist_init("gloo")
    assert (r, w) == (rank, world)
    bench.barrier(w)
    t = 1.0 + rank                      # rank 1 is the slow one
    tmax = bench.max_over_ranks(t, w)
    value = bench.aggregate_value(4e9, w, tmax)
    out[rank] = (tmax, value)
    dist.destroy_process_group()


def test_two_rank_timing_and_aggregation():
    port = _free_port()
    mgr = mp.get_context("spawn").Manager()
    out = mgr.dict()
    mp.start_processes(_worker, args=(2, port, out), nprocs=2, join=True, start_method="spawn")
    assert out[0] == out[1]
    tmax, value = out[0]
    assert tmax == 2.0
    assert value == pytest.approx(2 * 4e9 / 2.0 / 1e9)


def test_reference_arm_only_rank0_prints(capsys, monkeypatch):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    assert bench.reference_arm(bench.parse_args(["--impl", "reference", "--steps", "1", "--warmup", "0"])) == 0
    assert capsys.readouterr().out == ""
