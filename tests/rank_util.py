"""Rank body for the two-process gloo test of bench.py's cross-rank logic
(module-level, so that a spawned process can run it by name)."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def bench_rank(rank: int, world: int, port: int, local_ms: float, units: float, out) -> None:
    """Init gloo, reduce this rank's time with bench.max_over_ranks, form the
    whole-job rate, and report (rank, job ms, rate) on `out`."""
    import torch
    import torch.distributed as dist
    if ROOT not in sys.path:
        sys.path.insert(0, ROOT)
    import bench
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        ms = bench.max_over_ranks(local_ms, world, torch.device("cpu"))
        out.put((rank, ms, bench.whole_job_rate(units, ms * 1e-3, world)))
    finally:
        dist.destroy_process_group()
