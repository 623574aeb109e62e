"""One rank of the two-rank CPU check of gather_row_sums (launched by
test_row_split_dist.py under torch.distributed.run, gloo backend): every
rank contributes its slice's sums and gets all slices' sums in rank order."""
import json
import os
import sys

import torch
import torch.distributed as dist

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import post_weight_quantization_32_b300 as awq  # noqa: E402

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
mine = torch.arange(5, dtype=torch.float64) + 10.0 * rank
stacked = awq.gather_row_sums(mine)
dist.barrier()
print(json.dumps({"rank": rank, "world": world, "stacked": stacked.tolist()}), flush=True)
dist.destroy_process_group()
