"""One rank of the replicas path, on CPU over gloo (driven by test_replicas_gloo.py).

Each rank draws its own batch of the tiny workload with the bench's per-rank seed, steps it
with the oracle (no data crosses ranks), then does the bench's host-side bookkeeping: a
barrier on both sides of the "timed region", the max of the ranks' times and the sum of
their tokens. Writes its view as JSON to argv[1].
"""

import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
import oracle  # noqa: E402
from speculative_decoding_tree_parent_gb300 import workloads as W  # noqa: E402

INDEX = 1


def main(out_path):
    ws, rank, _ = bench._dist()
    dist.init_process_group("gloo")
    inp = W.generate_index(INDEX, seed=bench.replica_seed(INDEX, rank))
    dist.barrier()
    acc = oracle.greedy_accept(inp.parent, inp.draft_tokens, inp.target_logits, inp.qo_indptr, inp.path_cap)
    own_ms = 10.0 * (rank + 1) + 0.25          # a fixed per-rank "time", so the max is known
    dist.barrier()
    max_ms = bench.reduce_over_ranks(own_ms, "max", ws)
    tokens = bench.reduce_over_ranks(inp.total_nodes, "sum", ws)
    value = bench.job_throughput(tokens * 3, max_ms)   # three steps
    json.dump({"rank": rank, "ws": ws, "own_ms": own_ms, "max_ms": max_ms, "tokens_all": tokens,
               "own_tokens": int(inp.total_nodes), "value": value,
               "accept_len": np.asarray(acc.accept_len).tolist(), "path": np.asarray(acc.path).tolist(),
               "out_tokens": np.asarray(acc.out_tokens).tolist(),
               "parent_digest": int(np.asarray(inp.parent, np.int64).sum() * 131 + inp.draft_tokens.sum())},
              open(out_path, "w"))
    dist.destroy_process_group()


if __name__ == "__main__":
    main(sys.argv[1])
