"""Run by tests/test_bench_multirank.py through bench.launch_command (torch.distributed.run,
gloo on the CPU): each rank builds its own batch the way the benchmark does, and the ranks
reduce a per-rank step time (max) and K/V byte count (sum) with the benchmark's helpers.
Rank 0 prints one JSON line. No library call, no GPU."""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402


def main():
    world, rank, local = bench.rank_env()
    dist.init_process_group("gloo")
    try:
        wl = bench.rank_workload(rank)
        kv = sum(wl.meta["final_lens"]) * wl.spec.kv_token_bytes
        seeds = [torch.zeros(1, dtype=torch.int64) for _ in range(world)]
        dist.all_gather(seeds, torch.tensor([wl.seed], dtype=torch.int64))
        step_ms, = bench.max_over_ranks([1.0 + rank], dist, "cpu")
        job_bytes, = bench.sum_over_ranks([kv], dist, "cpu")
        if rank == 0:
            print(json.dumps({"world": world, "local_ranks": local, "seeds": [int(x) for x in seeds],
                              "step_ms": step_ms, "job_bytes": job_bytes}))
    finally:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
