"""The N > 1 path on CPU: two gloo ranks.

Sequences are independent, so a batch shards across ranks with no data-path
collective: each rank runs its half of the batch, forward and backward, and the
concatenation equals the single-process result bit for bit.  The benchmark's only collectives (a
barrier and the max-over-ranks of the step time) are exercised with gloo.
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
    p = s.getsockname()[1]
    s.close()
    return p


GRADS = ("dq", "dk", "dv", "dbeta", "dS0")


def _dO(x):
    g = torch.Generator().manual_seed(7)
    return torch.randn(x["v"].shape, generator=g, dtype=torch.float64).to(x["v"].dtype)


def _worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import efla_workloads as wl
        import oracle
        w = wl.resized(wl.LM340M_FWD, B=4, H=2, L=96, dk=16, dv=16, chunk=32)
        x = wl.make_inputs(w)
        per = w.B // world
        sl = slice(rank * per, (rank + 1) * per)      # this rank's batch shard
        o, Sf = oracle.fwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], nthreads=1)
        np.save(os.path.join(out_dir, f"o{rank}.npy"), o)
        np.save(os.path.join(out_dir, f"S{rank}.npy"), Sf)
        grads = oracle.bwd(x["q"][sl], x["k"][sl], x["v"][sl], x["beta"][sl], _dO(x)[sl], None)
        for name, g in zip(GRADS, grads):
            np.save(os.path.join(out_dir, f"{name}{rank}.npy"), g)
        bench.barrier(world)
        m = bench.max_over_ranks(float(rank + 1) * 1.5, world, torch.device("cpu"))
        np.save(os.path.join(out_dir, f"max{rank}.npy"), np.array([m]))
    finally:
        dist.destroy_process_group()


def test_two_rank_batch_shards_need_no_exchange(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    import efla_workloads as wl
    import oracle
    w = wl.resized(wl.LM340M_FWD, B=4, H=2, L=96, dk=16, dv=16, chunk=32)
    x = wl.make_inputs(w)
    o_full, S_full = oracle.fwd(x["q"], x["k"], x["v"], x["beta"], nthreads=1)
    o = np.concatenate([np.load(tmp_path / f"o{r}.npy") for r in range(world)], 0)
    S = np.concatenate([np.load(tmp_path / f"S{r}.npy") for r in range(world)], 0)
    assert np.array_equal(o, o_full) and np.array_equal(S, S_full)
    g_full = oracle.bwd(x["q"], x["k"], x["v"], x["beta"], _dO(x), None)
    for name, gf in zip(GRADS, g_full):
        g = np.concatenate([np.load(tmp_path / f"{name}{r}.npy") for r in range(world)], 0)
        assert np.array_equal(g, gf), name
    for r in range(world):
        assert float(np.load(tmp_path / f"max{r}.npy")[0]) == 3.0   # max over ranks of 1.5, 3.0
