"""Multi-rank host logic on CPU with the gloo backend (world size 2): row
shards tile [0, M) exactly once on tile boundaries, the bench's whole-job
throughput divides every rank's work by the slowest rank's time, and the
bench's --split rows rank path (each rank's workload and its host-only plan)
covers the problem once."""
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


def _rows_worker(rank, world, port, name, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import tile_scheduled_tensor_gb300 as tst
        w_full = bench.WORKLOADS[name]
        lo, hi, w = bench.shard_rows(w_full, world, rank)
        # the rank's plan, as bench.py builds it on its GPU, made host-only here
        plan = tst.gemm_plan_create(w["M"], w["N"], w["K"], dtype=w["dtype"], mapping=w["mapping"],
                                    schedule=w["schedule"], out_dtype=w["out"], bn=w["bn"],
                                    cta_group=w["cta_group"], use_scales=w.get("use_scales", False),
                                    host_only=True, num_sms=152)
        info = plan.info
        got = [None] * world
        dist.all_gather_object(got, (lo, hi, int(info.M), int(info.bm), bench.flops(w)))

        def max_reduce(x):
            t = torch.tensor([x], dtype=torch.float64)
            dist.all_reduce(t, op=dist.ReduceOp.MAX)
            return float(t.item())
        # rank r is slower by r ms: the job's time is the slowest rank's
        value, ms = bench.job_throughput(bench.flops(w_full), 10.0 + rank, max_reduce)
        if rank == 0:
            out.put((got, value, ms, bench.flops(w_full), w_full["M"]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("name", ["c3_e4m3_8192", "c5_bf16_epilogue", "c4_bf16_streamk_pairs"])
def test_two_rank_row_split_rank_path(name):
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rows_worker, args=(r, 2, port, name, q)) for r in range(2)]
    for p in procs:
        p.start()
    got, value, ms, job_flops, M = q.get(timeout=180)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert got[0][0] == 0 and got[-1][1] == M
    assert all(a[1] == b[0] for a, b in zip(got, got[1:]))
    for lo, hi, plan_m, bm, _ in got:
        assert plan_m == hi - lo and lo % bm == 0          # each shard's plan starts on a tile row
    assert sum(g[4] for g in got) == pytest.approx(job_flops)   # the shards' work adds up to the job
    assert ms == 11.0 and value == pytest.approx(job_flops / 11e-3 / 1e12)
