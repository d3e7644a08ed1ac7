"""Writes other_ranks_sumsq.json: the other ranks' share of the global
gradient sum of squares for the rank-local Llama-3-8B workload.

DeepSpeed ZeRO stages 1-2 walkthrough, 6 step 2: the global gradient norm is
the square root of the sum, all-reduced over the ranks, of each rank's sum
of squares of its reduced gradient shard.  The rank-local workload updates
rank 1's shard only, so the step takes the other ranks' part of that sum as
an input (extra_sumsq).  This script generates it from data: for every other
rank r in 0, 2, 3 and every source rank j in 0..3, the staged slice of rank
r's shard (2,007,565,312 elements) is drawn like rank 1's own slices --
N(0, 5e-4) in fp32, in chunks of 2^26, rounded to bf16 by torch -- from a CPU
torch.Generator seeded 100 + 4 r + j, so the value can be regenerated
without a GPU.  The oracle reduces the four slices of each rank (rank-order
fp32 sum, one division, rounding to bf16) and sums the squares exactly
(orc_reduce_stats, accumulators merged), once.  Only the oracle does
arithmetic here; the draws come from the shared seeded generators.

    python tests/golden/make_other_ranks_sumsq.py   (about 5 minutes on 8 cores)
"""
from __future__ import annotations

import concurrent.futures as cf
import json
import os
import platform
import sys
import time

import numpy as np
import torch

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
sys.path.insert(0, ROOT)

import oracle as orc          # noqa: E402
import workloads as W         # noqa: E402

OUT = os.path.join(HERE, "other_ranks_sumsq.json")
SHARD = 2_007_565_312
ND = 4
OTHER = (0, 2, 3)
STD = 5e-4
CHUNK = W.CHUNK               # the draw chunk of workloads.fill_normal_


def seed(r: int, j: int) -> int:
    return 100 + 4 * r + j


def rank_sumsq(r: int, pool: cf.ThreadPoolExecutor):
    """Exact sum of squares and overflow flag of rank r's reduced shard."""
    gens = [W.generator(seed(r, j), "cpu") for j in range(ND)]
    futs = []
    for c0 in range(0, SHARD, CHUNK):
        n = min(CHUNK, SHARD - c0)
        sl = []
        for g in gens:                      # each generator continues chunk after chunk, as fill_normal_ draws
            x = torch.empty(n, dtype=torch.bfloat16)
            W.fill_normal_(x, STD, g)
            sl.append(x.view(torch.int16).numpy().view(np.uint16))

        def work(sl=sl, n=n):
            acc = orc.ExactAccumulator()
            return acc, orc.reduce_stats(sl, 2, 0, n, acc)
        futs.append(pool.submit(work))
    total = orc.ExactAccumulator()
    ovf = 0
    for f in futs:
        a, o = f.result()
        total.merge(a)
        ovf |= o
    return total, ovf


def main():
    t0 = time.time()
    cores = len(os.sched_getaffinity(0))
    torch.set_num_threads(cores)
    total = orc.ExactAccumulator()
    per = {}
    with cf.ThreadPoolExecutor(max(1, cores - 1)) as pool:
        for r in OTHER:
            acc, ovf = rank_sumsq(r, pool)
            assert ovf == 0, f"rank {r}: non-finite reduced gradient"
            per[str(r)] = acc.value()
            total.merge(acc)
            print(f"rank {r}: {per[str(r)]!r} ({time.time() - t0:.0f} s)", flush=True)
    rec = {"llama3-8b-nd4-r1": {
        "value": total.value(),
        "per_rank": per,
        "ranks": list(OTHER), "n_d": ND, "shard_numel": SHARD,
        "recipe": "slice j of rank r: N(0, 5e-4) drawn in fp32 by a CPU torch.Generator seeded 100 + 4 r + j, "
                  "in chunks of 2^26 elements, rounded to bf16 by torch; the 4 slices of each rank reduced and "
                  "squared by the oracle (orc_reduce_stats), all ranks summed exactly and rounded once",
        "source": "DeepSpeed ZeRO stages 1-2 walkthrough, section 6 step 2 (the global norm all-reduces the "
                  "per-shard sums of squares)",
        "script": "tests/golden/make_other_ranks_sumsq.py",
        "made_with": {"torch": torch.__version__, "machine": platform.machine(), "seconds": round(time.time() - t0)},
    }}
    json.dump(rec, open(OUT, "w"), indent=1)
    print(json.dumps(rec, indent=1))


if __name__ == "__main__":
    main()
