"""bench.py's multi-rank logic on two CPU ranks (gloo): the max-over-ranks timing, the
barrier, the whole-job aggregation and the reference arm's rank-0-only rule.

The path does not shard (every rank runs an independent replica), so these are the only
collectives: they never touch the data path.
"""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
import torch.distributed as dist  # noqa: E402
import torch.multiprocessing as mp  # noqa: E402


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench

        w, r, local = bench.dist_env()
        got = bench.reduce_max(10.0 + 5.0 * rank, w, torch.device("cpu"))
        bench.barrier(w)

        class Args:
            steps, warmup, gpus = 1, 0, world

        ref_rc = bench.run_reference(Args, w, r) if r != 0 else None
        out.put((rank, w, r, local, got, ref_rc))
    finally:
        dist.destroy_process_group()


def test_two_ranks_reduce_to_the_slowest_and_only_rank0_reports():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, w, r, local, got, ref_rc in res:
        assert (w, r, local) == (world, rank, rank)
        assert got == 15.0  # the max over ranks: the slowest rank decides the job time
    assert res[1][5] == 0  # rank 1's reference arm exits 0 without work


def test_job_value_counts_every_rank():
    import bench

    one = bench.job_value(1, 2.0 * 16384**3, 10, 777.0)
    assert bench.job_value(2, 2.0 * 16384**3, 10, 777.0) == pytest.approx(2 * one)
    assert one == pytest.approx(2.0 * 16384**3 * 10 / 0.777 / 1e12)
