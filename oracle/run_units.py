"""Run the oracle's decode step over a share of (batch, kv-head) units, in a
process of its own, for the CPU baseline of the benchmark.

TEST INFRASTRUCTURE, NOT PRODUCT CODE.  It adds no arithmetic: each unit is
one call of decode.decode_step on that unit's inputs, exactly as the
single-process baseline runs it.  The benchmark starts one such process per
host core (so the oracle runs on every core at once, one unit at a time per
core), each with its own share of the units, and adds up their rates.

    python -m oracle.run_units FILE WORKER NWORKERS BUDGET_S

FILE is an .npz written by the benchmark: for unit i the arrays u{i}_q,
u{i}_k, u{i}_v, u{i}_pt, u{i}_lens (and u{i}_ks, u{i}_vs, u{i}_proj when
present), plus the step parameters under `params`.  The process takes units
WORKER, WORKER + NWORKERS, ... and runs them round-robin until BUDGET_S
seconds of wall time have passed, then prints one JSON line: units done,
wall seconds, CPU seconds.
"""

from __future__ import annotations

import json
import sys
import time

import numpy as np

from . import decode


def main(argv):
    path, worker, nworkers, budget = argv[0], int(argv[1]), int(argv[2]), float(argv[3])
    z = np.load(path)
    page_size, n_sel, n_sink, n_recent, head_dim = (int(x) for x in z["params"][:5])
    selector = ["quest", "sketch", "all"][int(z["params"][5])]
    prm = decode.StepParams(page_size, n_sel, n_sink, n_recent, selector, head_dim)
    n_units = int(z["params"][6])
    mine = []
    for i in range(worker, n_units, nworkers):
        get = lambda k: z[f"u{i}_{k}"] if f"u{i}_{k}" in z.files else None
        mine.append(decode.StepInputs(get("q"), get("k"), get("v"), get("ks"), get("vs"),
                                      get("pt"), get("lens"), get("proj")))
    done, t0, c0 = 0, time.perf_counter(), time.process_time()
    while mine and time.perf_counter() - t0 < budget:
        decode.decode_step(mine[done % len(mine)], prm, units=[(0, 0)])
        done += 1
    print(json.dumps({"units": done, "wall": time.perf_counter() - t0,
                      "cpu": time.process_time() - c0}), flush=True)


if __name__ == "__main__":
    main(sys.argv[1:])
