"""One rank of a CPU run of bench.py's multi-rank host logic, launched by torch.distributed.run.

Joins a gloo process group from the launcher's environment, reports a per-rank time of
10 * (rank + 1) ms, and reports (as one JSON line per rank) what bench.py's helpers make of it:
the slowest rank's time and the whole-job rate for 1000 units per rank.  Rank 0 gathers and prints
every rank's line, so that lines of two processes never interleave on the shared output.
"""
from __future__ import annotations

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main() -> None:
    dist.init_process_group("gloo")
    try:
        rank, world = dist.get_rank(), dist.get_world_size()
        bench.rank_barrier(dist)
        slowest = bench.rank_max(10.0 * (rank + 1), dist, "cpu")
        rate = bench.whole_job_rate(world, 1000.0, slowest)
        bench.rank_barrier(dist)
        lines = [None] * world
        dist.all_gather_object(lines, json.dumps({"rank": rank, "world": world, "slowest_ms": slowest, "rate": rate}))
        if rank == 0:
            print("\n".join(lines), flush=True)
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
