"""Run one benchmark workload's launch a few times, for a profiler.

    python -m gqa_kv_cache_mla_gb300.profile_case --workload mla_decode --launches 3

Builds the seeded workload, uploads it and calls its entry point
``--warmup`` + ``--launches`` times on the current stream, with no timing and
no cache flushing of its own (the profiler controls caches), then checks the
error word.  Device memory stays small (the workload's buffers only).
"""
import argparse
import sys

import torch

from . import device as D
from . import workloads as W


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", choices=sorted(W.REGISTRY), default="mla_decode")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--warmup", type=int, default=2)
    ap.add_argument("--seed", type=int, default=2)
    a = ap.parse_args()
    builder, _, desc = W.REGISTRY[a.workload]
    w = builder(a.seed)
    d = D.for_workload(w, device="cuda", guard=False)
    for _ in range(a.warmup + a.launches):
        d.run()
    torch.cuda.synchronize()
    assert d.flags() == 0
    print("%s: %d launches (%s), units=%d" % (a.workload, a.warmup + a.launches, desc, w.T))
    return 0


if __name__ == "__main__":
    sys.exit(main())
