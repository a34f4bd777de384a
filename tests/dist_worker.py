"""One rank of the two-process gloo test of bench.py's multi-process path
(launched by tests/test_bench_dist_cpu.py through torch.distributed.run)."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

import bench  # noqa: E402


def main():
    dist, rank, world, local = bench.dist_setup(torch)
    assert dist is not None and world == 2 and rank in (0, 1)
    dev = torch.device("cpu")
    bench.barrier(dist, torch, dev)
    # each replica times its own steps; the job's time is the slowest rank's
    ms_local = 1.25 if rank == 0 else 2.5
    ms_max = bench.max_over_ranks(torch, dist, ms_local, dev)
    tokens = bench.replica_throughput(world, 4096, ms_max)
    # the reference arm runs on rank 0 only: other ranks return without work
    # (rank 0 would run the CPU oracle for minutes; it is not called here)
    ref_skipped = None
    if rank == 1:
        ref = bench.run_reference(bench.parse_args(["--impl", "reference", "--gpus", "2"]))
        ref_skipped = ref is None
    bench.barrier(dist, torch, dev)
    dist.destroy_process_group()
    with open(os.path.join(os.environ["DIST_TEST_OUT"], "rank%d.json" % rank), "w") as fh:
        json.dump({"rank": rank, "world": world, "ms_max": ms_max, "tokens_s": tokens,
                   "ref_skipped": ref_skipped}, fh)


if __name__ == "__main__":
    main()
