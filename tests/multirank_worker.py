"""Worker for the two-rank CPU tests: one process per rank under torchrun,
gloo backend.  Exercises bench.py's rank aggregation (max over ranks of the
step time, whole-job throughput) and writes one JSON file per rank into the directory
given as its argument."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    world, rank, _ = bench.dist_setup(2)
    dist.init_process_group("gloo")
    assert dist.get_world_size() == world and dist.get_rank() == rank
    step_ms = 10.0 + 5.0 * rank            # rank 1 is the slower one
    max_ms = bench.reduce_max_over_ranks(step_ms, "cpu")
    rate = bench.job_rate(world, 1000, 4, max_ms)
    dist.barrier()
    with open(os.path.join(sys.argv[1], f"rank{rank}.json"), "w") as f:
        json.dump({"rank": rank, "world": world, "max_ms": max_ms, "rate": rate}, f)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
