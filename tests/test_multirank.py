"""The N > 1 path of bench.py on CPU.  Under torchrun every rank runs its own
copy of the workload (the path shards by request, with no exchange on the
data path); the ranks meet only to take the slowest rank's time, and the
whole-job rate counts every rank's units over that time.  Two gloo ranks on
127.0.0.1 check the rank/world parsing, the max-over-ranks timing and the
rate; the reference arm's other ranks exit without output."""

import argparse
import datetime
import os
import socket
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    ws, r, local = bench._dist()
    dist.init_process_group("gloo", rank=rank, world_size=world,
                            timeout=datetime.timedelta(seconds=60))
    ms = bench.max_over_ranks(10.0 + 5.0 * rank, ws, "cpu")      # rank 1 is the slower
    rate = bench.job_rate(ws, 4160, 200, ms)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, ws, r, local, ms, rate))


def test_two_gloo_ranks_report_the_slowest_time_and_the_whole_job_rate():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    try:
        out = sorted(q.get(timeout=120) for _ in procs)
    finally:
        for p in procs:
            p.join(timeout=60)
    assert [p.exitcode for p in procs] == [0, 0]
    for rank, (r, ws, rr, local, ms, rate) in enumerate(out):
        assert (r, ws, rr, local) == (rank, 2, rank, rank)
        assert ms == 15.0
        assert rate == 2 * 4160 * 200 / (15.0 / 1e3)


def test_single_rank_defaults(monkeypatch):
    import bench
    for k in ("WORLD_SIZE", "RANK", "LOCAL_RANK"):
        monkeypatch.delenv(k, raising=False)
    assert bench._dist() == (1, 0, 0)
    assert bench.max_over_ranks(12.5, 1, "cpu") == 12.5
    assert bench.job_rate(1, 4160, 10, 1000.0) == 41600.0


def test_reference_arm_prints_only_on_rank_0(capsys):
    import bench
    args = argparse.Namespace(steps=1, warmup=3, ref_budget=1.0)
    bench.reference_run(args, 2, 1)
    assert capsys.readouterr().out == ""
