"""The N > 1 benchmark path on the CPU: two `gloo` ranks run the benchmark's
cross-rank logic.  Sequences are independent, so each rank gets its own copy of
the workload, and the only cross-rank operations are barriers and the max of the
step time; the reported value is all ranks' tokens over the slowest rank."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, q):
    import sys
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    import bench
    import workloads
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = bench.rank_workload(workloads.PREFILL, rank)
        my_ms = 1.0 + rank  # rank 1 is the slow one
        ms = bench.max_over_ranks(my_ms, world)
        value = bench.weak_scaling_value(w.B * w.S, world, ms)
        dist.barrier()
        q.put((rank, w.seed, ms, value))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=10) for _ in range(world))
    seeds = [r[1] for r in res]
    assert len(set(seeds)) == world  # independent inputs per rank
    for _, _, ms, value in res:
        assert ms == 2.0  # the slowest rank decides
        assert value == pytest.approx(4 * 4096 * world / 2.0e-3)
