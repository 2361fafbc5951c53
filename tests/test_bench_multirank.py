"""The N > 1 path of bench.py on CPU: two gloo ranks (127.0.0.1) agree on the
slowest rank's step time and on the whole-job throughput, and the reference
arm runs on rank 0 alone.  The GPU path is the same code with NCCL and
device="cuda"; this run never has more than one GPU, so it is checked here."""
import contextlib
import io
import multiprocessing as mp
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, times, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    import bench
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w, r, _ = bench.dist_env()
        slowest = bench.reduce_max(times[rank], w, "cpu")
        q.put((r, slowest, bench.job_throughput(68.7e9 / 1e12, slowest, w)))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_step():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    times = [0.031, 0.027]        # ms per step seen by ranks 0 and 1
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, times, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slowest, value in out:
        assert slowest == max(times)
        # two replicas, each 68.7 GFLOP per step, in the slowest rank's time
        assert value == pytest.approx(2 * 0.0687 / (0.031e-3))


def test_one_rank_reduces_to_itself():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(1.25, 1, "cpu") == 1.25
    assert bench.job_throughput(2.0, 1000.0, 1) == pytest.approx(2.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    """Under torchrun the reference arm's ranks > 0 exit at once, printing nothing."""
    sys.path.insert(0, ROOT)
    import bench
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("LOCAL_RANK", "1")
    args = bench.parse_args(["--impl", "reference"])
    buf = io.StringIO()
    with contextlib.redirect_stdout(buf):
        assert bench.main_reference(args) is None
    assert buf.getvalue() == ""
