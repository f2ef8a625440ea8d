"""The multi-rank path of bench.py on CPU: two gloo ranks, barrier, max-over-ranks
timing and the whole-job weak-scaling aggregate (no GPU, no data-path collective)."""

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


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    w, r, lr = bench.dist_env()
    assert (w, r, lr) == (world, rank, rank)
    bench.barrier()
    local_ms = 10.0 + 5.0 * rank  # rank 1 is the slow one
    ms = bench.max_over_ranks(local_ms)
    rows = 914 + rank  # per-rank batches differ (own seed), the job counts rows_per_rank * world
    val = bench.whole_job_rows_per_s(914, world, ms, 4)
    out[rank] = (ms, val)
    bench.barrier()
    dist.destroy_process_group()


def test_two_ranks_gloo():
    world = 2
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    assert out[0][0] == out[1][0] == 15.0
    assert abs(out[0][1] - 2 * 914 / (15.0e-3 / 4)) < 1e-6
    assert out[0][1] == out[1][1]
