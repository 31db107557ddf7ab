"""bench.py's multi-GPU path on the CPU: two gloo ranks (one replica each, as torchrun would
launch them) agree on the slowest rank's time and on the whole-job value; no data crosses ranks."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    os.environ.update({"RANK": str(rank), "LOCAL_RANK": str(rank), "WORLD_SIZE": str(world),
                       "MASTER_ADDR": "127.0.0.1", "MASTER_PORT": str(port)})
    import bench
    import torch.distributed as dist
    w, r, local = bench.dist_setup()
    assert (w, r, local) == (world, rank, rank) and dist.get_backend() == "gloo"
    bench.dist_barrier(w)
    slowest = bench.dist_max(times[rank], w)
    out[rank] = slowest
    dist.destroy_process_group()


def test_two_rank_replicas_reduce_to_the_slowest_rank():
    ctx = mp.get_context("spawn")
    port = _free_port()
    manager = ctx.Manager()
    out = manager.dict()
    times = [0.125, 0.5]
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0] == out[1] == 0.5


def test_whole_job_value_counts_every_replica():
    import numpy as np
    sys.path.insert(0, ROOT)
    import bench
    import pkv_workloads as W
    w = W.make_workload("c1")
    nb = bench.algorithmic_bytes(w)
    # value = world * bytes per replica step / slowest step time (weak scaling)
    world, ms = 2, 0.1
    value = world * nb["step"] / (ms * 1e-3) / 1e9
    assert np.isclose(value, 2 * (nb["step"] / 1e-4) / 1e9)
    assert nb["kv"] == w.kv_read_bytes() and nb["step"] > nb["attention"] > nb["kv"]
