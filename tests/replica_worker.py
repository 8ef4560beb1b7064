"""One rank of the replica bookkeeping test (run by tests/test_replicas_gloo.py
under torch.distributed.run with the gloo backend, on the CPU)."""
import json
import os
import sys

import numpy as np
import torch
import torch.distributed as dist

sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
import bench  # noqa: E402
from quantized_moe_decode_luce_gb300 import workloads as W  # noqa: E402
from quantized_moe_decode_luce_gb300.replicas import job_throughput  # noqa: E402


def main(out_dir):
    dist.init_process_group("gloo")
    rank, world = dist.get_rank(), dist.get_world_size()
    # rank r "took" 10 (r + 1) ms for 7 units
    value, ms = job_throughput(10.0 * (rank + 1), 7, world, torch.device("cpu"))
    wl = W.Workload("tiny_stack", T=1, H=256, I=256, E=8, k=2, shared=True, clamp=0.0, seed=3,
                    logits="zipf", bias_std=0.1, layers=2, steps=2)
    xs, lg, biases, vocab = bench.draw_inputs(wl, 2, rank)
    digest = [float(np.float64(xs).sum()), float(np.float64(lg).sum()), float(np.float64(vocab[:, :, :64]).sum())]
    json.dump({"rank": rank, "world": world, "value": value, "ms": ms, "digest": digest},
              open(os.path.join(out_dir, f"rank{rank}.json"), "w"))
    dist.barrier()
    dist.destroy_process_group()


if __name__ == "__main__":
    main(sys.argv[1])
