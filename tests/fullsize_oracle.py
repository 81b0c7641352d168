"""Oracle results for the full-size workloads, cached on disk.

TEST INFRASTRUCTURE: calls only the oracle and the workload generators.  For
each of the large CG workloads it stores what the full-size parity tests
compare the GPU path with: the oracle's forward solution x of A x = b and
its adjoint solution lambda of A^T lambda = g (same tolerance,
preconditioner and iteration cap as the benchmark), with their iteration
counts and statuses.  dL/dA = -lambda_i x_j is formed from these by
``oracle.grad_A`` when a test needs it (it is as large as the matrix).

The forward and adjoint solves are independent (the adjoint solve does not
read x), so they run as separate processes.  Results go to
``build/oracle_fullsize/<workload>_<key>.npz`` (git-ignored), where the key
hashes the oracle's source, the workload's arrays and the solve options, so a
changed oracle or input is never served from an old file.

    python tests/fullsize_oracle.py [c2 c4 c5]   # compute what is missing
"""
from __future__ import annotations

import hashlib
import json
import multiprocessing as mp
import os
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

CACHE_DIR = os.path.join(ROOT, "build", "oracle_fullsize")
NAMES = ("c2", "c4", "c5")
MAX_ITER = 200000   # the benchmark's cap


def _opts(w):
    return dict(tol=w.tol, pc=w.pc, eps=w.eps if w.pc == "spai" else 0.0, max_iter=MAX_ITER)


def key_of(w) -> str:
    h = hashlib.sha256()
    with open(os.path.join(ROOT, "oracle", "oracle.c"), "rb") as f:
        h.update(f.read())
    for a in (w.A.row_ptr, w.A.col_idx, w.A.vals, w.b, w.g):
        h.update(np.ascontiguousarray(a).tobytes())
    h.update(json.dumps(_opts(w), sort_keys=True).encode())
    return h.hexdigest()[:16]


def path_of(name: str, key: str, part: str) -> str:
    return os.path.join(CACHE_DIR, f"{name}_{key}_{part}.npz")


def _solve(name: str, part: str) -> str:
    """One oracle solve of a full-size workload (run in its own process):
    part "fwd" solves A x = b, part "adj" solves A^T lambda = g."""
    import oracle
    from workloads import build
    w = build(name)
    key = key_of(w)
    out = path_of(name, key, part)
    if os.path.exists(out):
        return out
    o = _opts(w)
    t0 = time.perf_counter()
    if part == "fwd":
        v, inf = oracle.pcg(w.A, w.b, o["tol"], max_iter=o["max_iter"], pc=o["pc"], eps=o["eps"])
    else:
        v, _, inf = oracle.adjoint(w.A, None, w.g, o["tol"], max_iter=o["max_iter"], pc=o["pc"],
                                   eps=o["eps"], with_dA=False)
    inf = dict(inf, seconds=time.perf_counter() - t0)
    os.makedirs(CACHE_DIR, exist_ok=True)
    tmp = out + f".tmp{os.getpid()}.npz"
    np.savez(tmp, v=v, info=json.dumps(inf))
    os.replace(tmp, out)
    return out


def load(name: str, key: str):
    """(x, fwd_info, lambda, adj_info) from the cache, or None."""
    pf, pa = path_of(name, key, "fwd"), path_of(name, key, "adj")
    if not (os.path.exists(pf) and os.path.exists(pa)):
        return None
    f, a = np.load(pf), np.load(pa)
    return f["v"], json.loads(str(f["info"])), a["v"], json.loads(str(a["info"]))


def start(names=NAMES, workers=None):
    """Start the missing solves in a pool of fresh (spawned) processes and
    return (pool, async results); nothing is started when all are cached.
    Spawned, not forked: the caller may already hold a CUDA context."""
    jobs = [(n, p) for n in names for p in ("fwd", "adj")]
    ctx = mp.get_context("spawn")
    pool = ctx.Pool(processes=workers or len(jobs))
    return pool, [pool.apply_async(_solve, j) for j in jobs]


def main(argv):
    names = tuple(argv) or NAMES
    t0 = time.perf_counter()
    pool, res = start(names)
    for r in res:
        print(r.get(), flush=True)
    pool.close()
    pool.join()
    print(f"done in {time.perf_counter() - t0:.0f} s")


if __name__ == "__main__":
    main(sys.argv[1:])
