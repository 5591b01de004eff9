"""The benchmark's multi-rank bookkeeping on CPU (gloo, two processes): every
rank ends up with the slowest rank's step time, the whole-job value sums the
ranks' work over that time, and the reference arm does no work off rank 0."""
import os
import socket
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, times, out):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], world, torch.device("cpu"))
        dist.barrier()
        out.put((rank, ms, bench.job_tflops(world, 1e12, ms)))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_processes():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [12.5, 40.0]
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [r[1] for r in res] == [40.0, 40.0]                  # both ranks see the slowest time
    assert res[0][2] == pytest.approx(2 * 1e12 / 40e-3 / 1e12)   # 2 ranks of work over it


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(3.25, 1, "cpu") == 3.25
    assert bench.job_tflops(1, 2e12, 1000.0) == pytest.approx(2.0)


def test_reference_arm_off_rank_zero_does_nothing(capsys):
    sys.path.insert(0, ROOT)
    import bench

    class Args:
        steps, warmup = 1, 0
    assert bench.run_reference(Args(), rank=1, world=2) is None
    assert capsys.readouterr().out == ""
