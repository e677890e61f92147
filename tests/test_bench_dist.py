"""Multi-rank logic of bench.py on the host: two gloo ranks on CPU.

bench.py runs one replica of the whole workload per GPU (weak scaling, no
data-path collective); its only cross-rank steps are the barrier and the
max-over-ranks of the timed region, and `value` is the units all ranks
processed divided by that time.  These tests run those steps with the gloo
backend in two processes, and check that the reference arm's non-zero ranks
exit without work.
"""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out_q):
    import torch.distributed as dist

    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ws, r, local = bench.dist_env()
        dist.barrier()
        t_max = bench.max_over_ranks(dist, times[rank], "cpu")
        rate = bench.whole_job_rate(ws, 1000, 10, t_max)
        out_q.put((rank, ws, r, local, t_max, rate))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_two_gloo_ranks():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.25, 0.5]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    for p in procs:
        if p.is_alive():
            p.kill()
    assert all(p.exitcode == 0 for p in procs), [p.exitcode for p in procs]
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, (r0, ws, r, local, t_max, rate) in enumerate(res):
        assert (r0, ws, r, local) == (rank, 2, rank, rank)
        assert t_max == 0.5                       # the slower rank's time, on every rank
        assert rate == pytest.approx(2 * 1000 * 10 / 0.5)


def test_not_distributed_keeps_own_time():
    import bench
    assert bench.max_over_ranks(None, 0.125, "cpu") == 0.125
    assert bench.whole_job_rate(1, 8, 4, 2.0) == 16.0


def test_reference_arm_nonzero_rank_exits_without_work(monkeypatch, capsys):
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = bench.parse_args_from([])
    assert bench.run_reference(args) == 0
    assert capsys.readouterr().out == ""
