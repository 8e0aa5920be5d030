"""Multi-process host logic of the bench (replicas: one independent model per GPU, no
data-path collective), on CPU ranks over gloo: the timed region is the slowest rank's and
the reported value is the whole job's units per second."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, times, out):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(times[rank], dist, "cpu")
        rate = bench.whole_job_rate(64, ms, world, 8)
        dist.barrier()
        out.put((rank, ms, rate))
    finally:
        dist.destroy_process_group()


def test_single_process_is_the_identity():
    assert bench.max_over_ranks(3.25) == 3.25
    assert bench.whole_job_rate(10, 1000.0, 1, 1) == pytest.approx(10.0)
    assert bench.whole_job_rate(64, 20.0, 2, 8) == pytest.approx(51200.0)


@pytest.mark.timeout(120)
def test_slowest_rank_sets_the_time_on_every_rank():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    times = [12.5, 20.0]
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, times, out)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=90) for _ in procs)
    for p in procs:
        p.join(timeout=30)
        assert p.exitcode == 0
    assert [r for r, _, _ in res] == [0, 1]
    for _, ms, rate in res:
        assert ms == 20.0
        # 64 steps of 8 streams on each of 2 ranks within the slower rank's 20 ms
        assert rate == pytest.approx(64 / 0.020 * 2 * 8)


@pytest.mark.timeout(120)
def test_reference_arm_runs_on_rank_zero_only():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1", MASTER_ADDR="127.0.0.1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "3"], env=env, capture_output=True, text=True, timeout=100)
    assert r.returncode == 0, r.stderr[-2000:]
    assert r.stdout.strip() == ""
