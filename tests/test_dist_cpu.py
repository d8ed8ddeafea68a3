"""The multi-rank path of bench.py on CPU: two gloo ranks check the barrier,
the max-over-ranks time reduction and the weak-scaling unit count, and that
the reference arm runs on rank 0 only. Replicas share nothing on the data
path, so no collective beyond these is involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import bench
    w, r = bench.init_dist("gloo")
    assert (w, r) == (world, rank)
    bench.barrier()
    # Each rank reports a different time; every rank must see the slowest.
    t = bench.max_over_ranks(10.0 + rank)
    units = bench.units_for_world(131072, world)
    # The reference arm prints only on rank 0.
    ref = bench.bench_reference(bench.argparse.Namespace(
        workload="long", T=64, steps=1, warmup=0, cpu_seconds=0.01)) if rank else None
    results[rank] = (t, units, ref)
    dist.destroy_process_group()


def test_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    mgr = ctx.Manager()
    results = mgr.dict()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=180)
        assert p.exitcode == 0
    assert results[0][0] == pytest.approx(11.0) and results[1][0] == pytest.approx(11.0)
    assert results[0][1] == results[1][1] == 2 * 131072
    assert results[1][2] is None  # non-zero ranks do no reference work
