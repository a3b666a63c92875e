"""The multi-GPU path's host logic, on CPU: two gloo ranks (no GPU).

Lanes are independent, so `bench.py --gpus N` runs one replica per GPU (weak
scaling) and no collective touches the data; the ranks only agree on the
timing (the slowest rank's step time) and add up the work.  Checked here:
the aggregation over two real gloo ranks, and that every rank gets its own
seeded workload of the same shape (rank 0 keeps the single-GPU seed)."""
import os
import socket

import pytest
import torch
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        from workloads import Workload, shape
        ms, nbytes, tokens = bench.aggregate_over_ranks(1.5 + rank, 100.0 * (rank + 1), 10.0 * (rank + 1))
        shp = bench.rank_shape(shape("h2o_toy"), rank)
        K, _ = Workload(shp).context(0)
        q.put((rank, ms, nbytes, tokens, shp.seed, float(K.double().sum())))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_timing_and_own_workloads():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = {}
    for _ in procs:
        r = q.get(timeout=120)
        res[r[0]] = r
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for r in (0, 1):
        _, ms, nbytes, tokens, _, _ = res[r]
        assert ms == 2.5            # the slower rank's step time
        assert nbytes == 300.0      # work of both ranks
        assert tokens == 30.0
    from workloads import shape
    assert res[0][4] == shape("h2o_toy").seed
    assert res[1][4] != res[0][4]
    assert res[1][5] != res[0][5]   # rank 1 serves other sequences


def test_single_process_aggregation_is_identity():
    import bench
    assert bench.aggregate_over_ranks(3.0, 7.0, 2.0) == (3.0, 7.0, 2.0)


def test_bench_gpus_flag_launches_ranks_itself():
    """`bench.py --gpus 2` started without a launcher re-runs itself as two
    ranks (torch.distributed.run, 127.0.0.1 rendezvous); rank 0 prints one
    line aggregated over both (here on CPU ranks with stand-in work)."""
    import json
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = {k: v for k, v in os.environ.items() if k not in ("WORLD_SIZE", "RANK", "LOCAL_RANK")}
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--gpus", "2", "--selftest-cpu"],
                       capture_output=True, text=True, timeout=240, env=env, cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    d = json.loads(lines[0])
    assert d["n_gpus"] == 2 and d["config"]["ranks"] == 2
    assert d["value"] > 0 and d["ms_per_step"] > 0
