"""The multi-rank bookkeeping of bench.py on CPU: world_size-2 gloo ranks, the
job time is the slowest rank's, throughput counts every rank's units, and the
ranks draw distinct token batches (data parallel over M, no data-path
collective)."""
import os
import socket

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
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        my_ms = 10.0 + 5.0 * rank
        job_ms = bench.max_over_ranks(my_ms, world, "cpu")
        thr = bench.job_throughput(1e12, job_ms, world)
        from nvfp4_bit_quantized_gb300 import inputs
        x = inputs.normal((4, 8), 1.0, bench.rank_seed(rank), dtype=torch.float32)
        gathered = [torch.zeros_like(x) for _ in range(world)]
        dist.all_gather(gathered, x)
        q.put((rank, job_ms, thr, all(not torch.equal(gathered[0], g) for g in gathered[1:])))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, job_ms, thr, distinct in res:
        assert job_ms == 15.0                         # the slower rank decides
        assert thr == pytest.approx(2 * 1e12 / 15e-3 / 1e12)
        assert distinct


def test_single_rank_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.5, 1) == 3.5
    assert bench.job_throughput(2e12, 1.0, 1) == pytest.approx(2000.0)
