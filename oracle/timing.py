"""Timing harness for the oracle on one host core (test infrastructure only: the bench's CPU
baseline across all host cores runs one of these per core).

``python -m oracle.timing <file.npz>`` runs the oracle's step -- block table, slot mapping,
append, attention (over bf16 pages, or over 8-bit pages with the quantizing append) -- on every
sequence stored in the file, one after another, and prints the seconds it spent in the oracle
as one JSON line.  The file holds, per sequence k, the arrays ``cu_k``, ``ctx_k``, ``pages_k``,
``q_k``, ``kn_k``, ``vn_k``, ``kp_k``, ``vp_k`` (bf16 bit patterns as uint16) and the scalars
``n``, ``kv``, ``bs``, ``mb``, ``scale``, ``causal``.  BLAS runs single-threaded (the caller sets
the thread variables before this module starts), so one process is one core.
"""

import json
import sys
import time

import numpy as np

from . import step


def run_file(path):
    d = np.load(path, allow_pickle=False)
    n = int(d["n"])
    run = step.run_step_fp8 if str(d["kv"]) == "fp8" else step.run_step
    spent = 0.0
    bs, mb, scale, causal = int(d["bs"]), int(d["mb"]), float(d["scale"]), bool(d["causal"])
    for k in range(n):
        a = {name: np.array(d[f"{name}_{k}"]) for name in ("cu", "ctx", "pages", "q", "kn", "vn", "kp", "vp")}
        t = time.perf_counter()
        run(a["cu"], a["ctx"], a["pages"], bs, mb, a["q"], a["kn"], a["vn"], a["kp"], a["vp"], scale, causal,
            pool_pages=a["pages"])
        spent += time.perf_counter() - t
    return {"seconds": spent, "seqs": n}


if __name__ == "__main__":
    print(json.dumps(run_file(sys.argv[1])), flush=True)
