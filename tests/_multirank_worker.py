"""One rank of a world-size-2 run on CPU (gloo), started by torchrun: the
per-rank pieces of bench.py's multi-GPU path (independent batches, the
slowest rank's time, the whole-job value), one JSON line per rank."""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import torch  # noqa: E402
import torch.distributed as dist  # noqa: E402

import bench  # noqa: E402
from kda_inputs import make_inputs, small_workload  # noqa: E402


def main():
    dist.init_process_group("gloo")
    ws, rank, _ = bench.dist_env()
    base = bench.WORKLOADS["b2_h32_t32k"]
    w = bench.rank_workload(base, rank)
    # a small batch with the rank's seed: the ranks' inputs differ
    x = make_inputs(bench.rank_workload(small_workload("mr", B=1, T=64, H=1, dk=16, dv=16,
                                                       seed=5), rank))
    ms = 10.0 + 5.0 * rank          # this rank's step time
    slowest = bench.max_over_ranks(ms, ws, torch.device("cpu"))
    value = bench.job_value(ws, w.B * w.T, slowest)
    # one write per line: the ranks share the pipe, and print() may write
    # the text and its newline separately when the stream is unbuffered
    line = json.dumps({"rank": rank, "ws": ws, "seed": w.seed, "slowest_ms": slowest,
                       "value": value, "q0": float(x["q"].flatten()[0])})
    sys.stdout.write(line + "\n")
    sys.stdout.flush()
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main()
