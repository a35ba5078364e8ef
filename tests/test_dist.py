"""Replica aggregation of bench.py on CPU: two gloo ranks, each with its own
units and time; the job value is all units over the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE="2", LOCAL_RANK=str(rank))
    import bench
    ws, r, local = bench.dist_env()
    bench.init_dist(ws, "gloo")
    units = [1440.0, 1440.0][rank]
    secs = [2.0, 3.0][rank]
    value, tmax = bench.aggregate(units, secs)
    q.put((rank, value, tmax))
    torch.distributed.destroy_process_group()


def test_two_rank_replica_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, tmax in out:
        assert tmax == 3.0
        assert value == pytest.approx(2880.0 / 3.0)


def test_single_process_aggregation_is_identity():
    import bench
    v, t = bench.aggregate(100.0, 4.0)
    assert v == 25.0 and t == 4.0


def test_product_arm_refuses_more_than_one_rank_without_touching_a_gpu():
    """The product runs on one GPU (its GEMMs use cluster-multicast loads,
    kept to single-GPU runs): with WORLD_SIZE > 1, rank 0 reports the line
    as unavailable and the other ranks print nothing."""
    import argparse
    import bench
    args = argparse.Namespace()
    line = bench.run_fg(args, 2, 0, 0)
    assert line["unavailable"] == bench.MULTI_GPU_REFUSAL and line["n_gpus"] == 2
    assert bench.run_fg(args, 2, 1, 1) is None
