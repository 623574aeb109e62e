"""One rank of the two-rank CPU check of bench.py's cross-rank reduction
(launched by test_bench_dist.py under torch.distributed.run, gloo backend)."""
import json
import os
import sys

import torch
import torch.distributed as dist

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
slowest = bench.world_max(1.5 + rank, dist, torch.device("cpu"))
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "slowest_ms": slowest,
                  "value": bench.job_throughput(21, world, slowest)}), flush=True)
dist.destroy_process_group()
