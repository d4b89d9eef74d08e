"""Timing of the fp64 oracle on the host cores, for the benchmark's CPU baseline.

TEST INFRASTRUCTURE ONLY: the cpu_baseline leg of bench.py runs this module (in fresh
worker processes, one per core, started with ``python -m oracle.cpu_timing``); nothing in
the library's product path imports it.  It times the oracle as it stands -- the forward
(target-excluded log-sum-exp, softplus loss) and the gradient rows of ce_oracle -- on a
random sample of the workload's rows, drawn by the same seeded generator as the GPU
inputs; the drawing of each row is included in the time.

    python -m oracle.cpu_timing '<problem json>' WORKER WORKERS BUDGET_S

prints one JSON line: {"rows": n, "start": t0, "stop": t1} (wall-clock seconds).
"""
from __future__ import annotations

import json
import os
import sys
import time

import numpy as np


def sample_order(T: int) -> np.ndarray:
    """The benchmark's row sample: one fixed random permutation of the rows."""
    return np.random.default_rng(123).permutation(T)


def time_rows(problem, worker: int, workers: int, budget_s: float, block: int = 64) -> dict:
    """Forward and gradient of the oracle on worker's share of the sampled rows (every
    workers-th block of `block` rows of the permutation) until budget_s has passed."""
    from oracle import ce_oracle as O
    N = int(np.sum(problem.labels != problem.ignore_index))
    order = sample_order(problem.T)
    nblocks = -(-problem.T // block)
    done = 0
    t0 = time.time()
    b = worker
    while time.time() - t0 < budget_s:
        rows = np.sort(order[(b % nblocks) * block: (b % nblocks) * block + block])
        z = O.widen(problem.rows(rows), problem.dtype)
        fwd = O.ce_rows(z, problem.labels[rows])
        O.ce_grad_rows(z, problem.labels[rows], fwd, O.row_scale(fwd["valid"], "sum", 1.0 / N))
        done += len(rows)
        b += workers
    return {"rows": done, "start": t0, "stop": time.time()}


def main(argv):
    import gen
    spec = json.loads(argv[0])
    worker, workers, budget = int(argv[1]), int(argv[2]), float(argv[3])
    problem = gen.CEProblem(**spec)
    print(json.dumps(time_rows(problem, worker, workers, budget)), flush=True)


if __name__ == "__main__":
    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
    main(sys.argv[1:])
