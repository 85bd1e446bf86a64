"""Multi-rank host logic on CPU with the gloo backend (world size 2): row
shards tile [0, M) exactly once on tile boundaries, and the bench's whole-job
throughput divides every rank's work by the slowest rank's time."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from tile_scheduled_tensor_gb300.shard import m_shard


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, M, align, local_ms, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        lo, hi = m_shard(M, world, rank, align)
        got = [None] * world
        dist.all_gather_object(got, (lo, hi))

        def max_reduce(x):
            t = torch.tensor([x], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t.item())

        import bench
        value, ms = bench.aggregate(1e12, local_ms[rank], world, max_reduce)
        if rank == 0:
            out.put((got, value, ms))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("M,align", [(4096, 256), (16384, 128), (1000, 256), (128, 256)])
def test_two_rank_shards_and_aggregate(M, align):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    local_ms = [2.0, 4.0]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, M, align, local_ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, value, ms = q.get(timeout=120)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == 0 and got[-1][1] == M
    assert all(a[1] == b[0] for a, b in zip(got, got[1:]))          # contiguous, no overlap
    assert all(lo % align == 0 for lo, _ in got)                    # tile-aligned starts
    assert ms == 4.0 and value == pytest.approx(2 * 1e12 / 4e-3 / 1e12)


def test_shard_edge_cases():
    assert m_shard(0, 4, 3) == (0, 0)
    assert [m_shard(300, 3, r, 128) for r in range(3)] == [(0, 128), (128, 256), (256, 300)]
    assert [m_shard(200, 3, r, 128) for r in range(3)] == [(0, 0), (0, 128), (128, 200)]
    assert [m_shard(1024, 4, r) for r in range(4)] == [(0, 256), (256, 512), (512, 768), (768, 1024)]
    with pytest.raises(ValueError):
        m_shard(10, 2, 2)
