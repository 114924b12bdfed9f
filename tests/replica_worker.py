"""One rank of the replica-harness test: launched by torch.distributed.run with the gloo backend
on CPU; checks the max-over-ranks timing and the whole-job rate that bench.py reports."""
import json
import os
import sys

import torch.distributed as dist

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402


def main():
    rank, world, _ = bench.dist_env()
    dist.init_process_group("gloo")
    dist.barrier()
    # rank r "took" 10 + r ms for the timed region and 20 + 3 r ms end to end
    ms, e2e = bench.max_over_ranks([10.0 + rank, 20.0 + 3 * rank], world)
    value = bench.whole_job_rate(world, 5, 1024, ms)
    dist.barrier()
    out = os.environ["REPLICA_OUT"]
    with open(f"{out}.{rank}", "w") as f:
        json.dump({"rank": rank, "world": world, "ms": ms, "e2e": e2e, "value": value}, f)
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
