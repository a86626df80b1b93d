"""bench.py's multi-rank logic without a GPU: two gloo ranks on the host.
The job's time is its slowest rank's, the whole-job rate counts every rank's
units (weak scaling: each rank runs the full sweep), and the reference arm
runs on rank 0 alone."""
import multiprocessing as mp
import os
import socket
import subprocess
import sys

from tests.rank_util import bench_rank

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_two_ranks_time_is_the_slowest_and_rate_counts_both():
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    port = free_port()
    local_ms = {0: 3.0, 1: 5.0}
    units = 1.0e6
    procs = [ctx.Process(target=bench_rank, args=(r, 2, port, local_ms[r], units, out)) for r in (0, 1)]
    for p in procs:
        p.start()
    got = sorted(out.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate in got:
        assert ms == 5.0, (rank, ms)
        assert rate == 2 * units / 5.0e-3


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(4.25, 1, None) == 4.25
    assert bench.whole_job_rate(10.0, 2.0, 1) == 5.0


def test_reference_arm_other_ranks_exit_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "1"], env=env, capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""
