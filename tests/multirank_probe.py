"""Run under torchrun (world size 2, gloo, no GPU): bench.py's rank set-up, barrier and
max-over-ranks reduction; every rank writes one JSON file into the directory given as
the first argument."""

import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402

world, rank, local = bench.dist_setup()
bench.barrier(world)
v = bench.max_over_ranks(world, 1.5 + 10.0 * rank, "cpu")
bench.barrier(world)
with open(os.path.join(sys.argv[1], f"rank_{rank}.json"), "w", encoding="utf-8") as f:
    json.dump({"rank": rank, "local": local, "world": world, "max": v}, f)
if world > 1:
    import torch.distributed as dist
    dist.destroy_process_group()
