"""One rank of the two-process sharding test (launched by tests/test_shard.py through
torch.distributed.run with the gloo backend, on the CPU).

Each rank filters its shard of a small stream with the float64 oracle, using its halo as the
state; the ranks gather their outputs and final states, and rank 0 checks them against one
oracle call over the whole stream and writes the result to the JSON file named on the command
line.  The step-time reduction of bench.py (max over ranks) is exercised with the same group.
"""
import json
import os
import sys

import numpy as np
import torch.distributed as dist

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import oracle  # noqa: E402
import workloads as W  # noqa: E402
from frequency_domain_order_gb300.shard import halo, shard_ranges  # noqa: E402


def main(out_path: str) -> int:
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    result = {}
    for name in ("C1", "C4"):
        w = W.WORKLOADS[name]
        if name == "C4":
            w = W.scaled(w, 9, 333)
        x = W.make_x(w)
        h = W.oracle_h(w)
        s0 = W.make_x(W.scaled(w, 1))[: w.M - 1]  # nonzero, so rank 0's halo comes from it
        ranges = shard_ranges(len(x), w.L, world, real=w.real)
        a, b = ranges[rank]
        y, s_next = oracle.direct(x[a:b], h, halo(x, s0, a, w.M))
        parts = [None] * world
        dist.all_gather_object(parts, (a, b, y, s_next))
        if rank == 0:
            y1, s1 = oracle.direct(x, h, s0)
            ys = np.concatenate([p[2] for p in sorted(parts, key=lambda t: t[0])])
            result[name] = {
                "ranges": [list(p[:2]) for p in parts],
                "outputs_equal": bool(np.array_equal(ys, y1)),
                "state_equal": bool(np.array_equal(parts[-1][3], s1)),
            }
    # bench.py's timing reduction over ranks
    result["reduce_max"] = bench.reduce_max(float(rank + 1), world, "cpu")
    bench.barrier(world)
    if rank == 0:
        with open(out_path, "w") as f:
            json.dump(result, f)
    dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main(sys.argv[1]))
