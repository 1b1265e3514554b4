"""World-size-2 gloo runs on CPU of the multi-rank plumbing.

* The natural sharding of the type 1 transform: it is linear in the
  strengths, so each rank transforms its share of the points and one sum
  all-reduce of the modes gives the full result ("A Hybrid MPI-CUDA Approach
  for NDFT", Sec. 3 eq. (8) and Alg. 3).  Checked with the oracle's direct sum.
* The benchmark's aggregation: max over ranks of the timed region, and
  whole-job throughput = units all ranks processed / that time.
"""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import oracle
        rng = np.random.default_rng(0)
        M, N = 3000, (12, 10)
        pts = [rng.uniform(-np.pi, np.pi, M) for _ in range(2)]
        c = rng.standard_normal(M) + 1j * rng.standard_normal(M)
        lo, hi = rank * M // world, (rank + 1) * M // world
        part = oracle.direct_type1([p[lo:hi] for p in pts], c[lo:hi], N, -1)
        t = torch.from_numpy(np.ascontiguousarray(part).view(np.float64).copy())
        dist.all_reduce(t, op=dist.ReduceOp.SUM)
        full = t.numpy().view(np.complex128).reshape(part.shape)
        err = oracle.rel_l2(full, oracle.direct_type1(pts, c, N, -1))
        tmax = bench.reduce_max(10.0 + rank)          # rank 1 is the slower one
        val = bench.job_throughput(world, 2 * M, 4, tmax)
        q.put((rank, err, tmax, val))
    finally:
        dist.destroy_process_group()


def test_two_rank_point_sharding_and_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, err, tmax, val in res:
        assert err < 1e-13
        assert tmax == 11.0
        assert val == pytest.approx(2 * 2 * 3000 * 4 / 11.0)
