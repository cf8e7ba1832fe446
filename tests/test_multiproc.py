"""The N > 1 path on CPU: two gloo ranks.

Sequences are independent, so a batch shards across ranks with no data-path
collective: each rank runs its half of the batch, forward and backward, and the
concatenation equals the single-process result bit for bit.

The benchmark's own multi-rank code runs here too, as it runs under torchrun:
bench.dist_setup (process group from the RANK / WORLD_SIZE environment; gloo where
there is no GPU), the per-rank seeding of the inputs, the barrier, the max over ranks
of the step time and the whole-job value; and bench.py --impl reference launched by
torch.distributed.run on two ranks, where rank 0 alone prints the line.
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


def _bench_worker(rank, world, port, out_dir):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import argparse
    import bench
    import efla_workloads as wl
    ws, r, local = bench.dist_setup(argparse.Namespace(impl="gb300"))
    try:
        assert (ws, r, local) == (world, rank, rank)
        assert dist.get_backend() == "gloo"
        w = wl.LM340M_FWD
        small = wl.resized(w, B=1, H=1, L=8, dk=16, dv=16)
        x = wl.make_inputs(small, seed=bench.rank_seed(w, rank))
        np.save(os.path.join(out_dir, f"q{rank}.npy"), x["q"].float().numpy())
        bench.barrier(ws)
        step_ms = 2.0 if rank == 0 else 5.0          # the slower rank sets the time
        ms, value = bench.headline_value(ws, w.B * w.L, step_ms, torch.device("cpu"))
        cfg = bench.headline_config(w, ws)
        np.save(os.path.join(out_dir, f"agg{rank}.npy"), np.array([ms, value, cfg["global_batch"]]))
        with open(os.path.join(out_dir, f"par{rank}.txt"), "w") as f:
            f.write(cfg["parallelism"])
    finally:
        dist.destroy_process_group()


def test_bench_multi_rank_pieces_under_gloo(tmp_path):
    world = 2
    mp.start_processes(_bench_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    import efla_workloads as wl
    w = wl.LM340M_FWD
    q0, q1 = (np.load(tmp_path / f"q{r}.npy") for r in range(world))
    assert not np.array_equal(q0, q1)                 # each rank draws its own batch
    for r in range(world):
        ms, value, gb = np.load(tmp_path / f"agg{r}.npy")
        assert ms == 5.0                              # max over ranks
        assert value == world * w.B * w.L / 5e-3      # every rank's tokens / slowest time
        assert gb == w.B * world
        assert (tmp_path / f"par{r}.txt").read_text() == "batch shards x2, no collective"


def test_bench_reference_arm_under_torchrun():
    """torch.distributed.run, two ranks: rank 0 alone times the oracle and prints one JSON
    line (n_gpus 2, the same config as the GPU arm's); rank 1 exits 0 without output."""
    import json
    import subprocess
    import sys
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node=2",
           "--master-addr=127.0.0.1", f"--master-port={_free_port()}",
           os.path.join(ROOT, "bench.py"), "--impl", "reference", "--gpus", "2", "--steps", "1",
           "--warmup", "3"]
    r = subprocess.run(cmd, capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    line = json.loads(lines[0])
    import bench
    import efla_workloads as wl
    assert line["impl"] == "reference" and line["n_gpus"] == 2
    assert line["config"] == bench.headline_config(wl.LM340M_FWD, 2)
    assert line["value"] > 0 and line["cpu_baseline"]["kind"] == "oracle"
