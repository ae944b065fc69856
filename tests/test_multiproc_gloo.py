"""World-size-2 gloo test of the benchmark's multi-replica logic (CPU only).

The path shards as independent replicas (one per GPU, no data-path
collective); what runs across ranks is the host-side aggregation: the job's
time is the slowest rank's, its tokens the sum over ranks.
"""

import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [120.0, 80.0][rank]           # rank 0 is the slow one
        local_tokens = [64 * 200, 64 * 200][rank]
        value, ms = bench.job_throughput(local_tokens, local_ms, world, device="cpu")
        mx = bench.max_over_ranks(float(rank), world, device="cpu")
        sm = bench.sum_over_ranks(float(rank + 1), world, device="cpu")
        q.put((rank, value, ms, mx, sm))
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, value, ms, mx, sm in out:
        assert ms == 120.0                         # slowest replica
        assert value == pytest.approx(2 * 64 * 200 / 0.120)
        assert mx == 1.0 and sm == 3.0


def test_single_rank_is_identity():
    import bench
    value, ms = bench.job_throughput(1000, 50.0, 1, device="cpu")
    assert ms == 50.0 and value == pytest.approx(1000 / 0.05)
