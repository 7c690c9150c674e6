"""Rank body of the benchmark's replica-launch test: started by
torch.distributed.run through bench.replica_command, it joins the ranks as
bench.py does, derives its replica's seed and takes the max over ranks."""
import json
import os
import sys

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import bench  # noqa: E402
from synth import WORKLOADS  # noqa: E402

dist = bench.init_ranks()
rank, world = dist.get_rank(), dist.get_world_size()
seed = bench.replica_workload(WORKLOADS["tiny"], rank).seed_id
seeds = [None] * world
dist.all_gather_object(seeds, seed)
step = bench.max_over_ranks(1.0 + rank, dist, "cpu")
if rank == 0:
    print(json.dumps({"world": world, "backend": dist.get_backend(), "seeds": seeds, "max": step}),
          flush=True)
dist.destroy_process_group()
