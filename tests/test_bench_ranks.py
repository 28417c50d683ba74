"""Multi-rank plumbing of bench.py on CPU: two gloo ranks.

The bench shards requests over ranks with no data-path exchange; the only
collectives are the timing reductions (max of the per-rank time, sum of the
per-rank units).  These run here on the gloo backend with world size 2.
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


def _rank_main(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        r, w, lr = bench.rank_env()
        t_local = 1.0 + 0.5 * rank                   # rank 1 is the slow one
        units = 10.0 * (rank + 1)
        t_max = bench.max_over_ranks(t_local, w, "cpu")
        u_all = bench.sum_over_ranks(units, w, "cpu")
        seeds = [bench.rank_round_index(r, s) for s in range(4)]
        out[rank] = (r, w, lr, t_max, u_all, bench.job_rate(u_all, t_max), tuple(seeds))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_units():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
        assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
        res = dict(out)
    for rank in range(world):
        r, w, lr, t_max, u_all, rate, seeds = res[rank]
        assert (r, w, lr) == (rank, world, rank)
        assert t_max == 1.5                       # max over ranks, seen by every rank
        assert u_all == 30.0                      # units of all ranks
        assert rate == pytest.approx(20.0)        # whole-job throughput: all units / slowest rank
    # every rank verifies its own requests: no seed is shared between ranks
    assert not set(res[0][6]) & set(res[1][6])


def test_single_rank_needs_no_process_group():
    import bench
    assert bench.max_over_ranks(2.5, 1) == 2.5
    assert bench.sum_over_ranks(7.0, 1) == 7.0
    assert bench.job_rate(10.0, 0.0) == 0.0


def test_other_ranks_skip_the_reference_arm(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    bench.main(["--impl", "reference", "--steps", "4", "--warmup", "3"])
    assert capsys.readouterr().out == ""          # only rank 0 runs and prints
