"""Multi-rank host logic of the benchmark, on CPU with two gloo processes.

The path shards by request with no exchange step, so ranks run independent
replicas (own seed, same shape) and the job time is the max over ranks.
"""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    import workloads as wl
    w = bench.replica_workload(bench.get_workload("lru_pressure_64k_fp8"), rank, world)
    small = w.with_(batch=1, n_layers=1, ctx=64 * 4)
    k, _, _ = wl.store_batch(small, 0)
    t = bench.reduce_max(1.0 + 0.5 * rank, dist, "cpu")
    q.put((rank, w.seed, w.batch, float(k[0, 0, 0]), t))
    dist.barrier()
    dist.destroy_process_group()


def test_two_rank_replicas_and_max_time():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(2))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, s0, b0, k0, t0), (r1, s1, b1, k1, t1) = res
    assert s0 != s1 and b0 == b1 == 4          # own seed, same shape
    assert k0 != k1                             # different inputs per replica
    assert t0 == t1 == 1.5                      # max over ranks


def test_single_rank_is_the_workload_itself():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    w = bench.get_workload("lru_pressure_64k_fp8")
    assert bench.replica_workload(w, 0, 1) is w
    assert bench.reduce_max(3.0, None, "cpu") == 3.0
