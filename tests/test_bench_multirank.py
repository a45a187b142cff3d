"""Host logic of bench.py's multi-GPU run (one process per GPU, replicas of
the path on independent batches), exercised as two gloo ranks on the CPU:
rank-dependent seeds, the max-over-ranks time, the whole-job throughput and
the reference arm running on rank 0 only."""

import contextlib
import io
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, ws, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(ws),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=ws)
    try:
        got_ws, got_rank, got_local = bench._dist()
        w, _ = bench.make_workload("chain_single", bench.rank_seed(0, got_rank))
        digest = torch.tensor([float(w.Lp.float().sum()), float(w.x.sum())], dtype=torch.float64)
        digests = [torch.zeros(2, dtype=torch.float64) for _ in range(ws)]
        dist.all_gather(digests, digest)
        slowest = bench.max_over_ranks(1.0 + 2.5 * got_rank, got_ws)
        buf = io.StringIO()
        with contextlib.redirect_stdout(buf):
            args = type("A", (), dict(workload="chain_batched", seed=0, steps=0, warmup=0))()
            if got_rank != 0:
                bench.run_reference(args)  # must return at once, printing nothing
        q.put((rank, got_ws, got_rank, got_local, [d.tolist() for d in digests], slowest, buf.getvalue()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks():
    ws, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, ws, port, q)) for r in range(ws)]
    for p in procs:
        p.start()
    res = [q.get(timeout=240) for _ in range(ws)]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    res.sort()
    for rank, got_ws, got_rank, got_local, digests, slowest, out in res:
        assert (got_ws, got_rank, got_local) == (ws, rank, rank)
        assert digests[0] != digests[1]  # each rank verifies its own batch
        assert slowest == pytest.approx(1.0 + 2.5 * (ws - 1))  # every rank sees the slowest time
        if rank != 0:
            assert out == ""
    assert res[0][4] == res[1][4]  # the gathered digests agree across ranks


def test_throughput_is_whole_job():
    import bench

    # two ranks, 10 steps of 512 positions each, slowest rank 2 ms
    assert bench.throughput(512, 10, 2, 2.0) == pytest.approx(512 * 10 * 2 / 2e-3)
    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.rank_seed(7, 3) == 10
