"""The benchmark's algorithmic byte model and method dispatch (CPU only):
the per-iteration and per-launch byte counts equal the stated formulas
(values and indices of a shared pattern counted once, 8-byte working
vectors), and each workload is timed on the oracle's solver for its own
method."""
import numpy as np

import bench
from workloads import build


def _mat(w, s):
    A = w.A
    return s * A.nnz * A.batch + 4 * A.nnz + 4 * (A.n + 1)


def test_cg_and_jacobi_models():
    w = build("c4", N=12)                       # CG, fp64
    bm = bench.byte_model(w)
    n = w.A.n
    assert bm["per_iteration"] == 12 * w.A.nnz + 4 * (n + 1) + 11 * 8 * n
    assert bm["product_per_launch"] == 12 * w.A.nnz + 4 * (n + 1) + 16 * n
    w = build("c2", N=20)                       # Jacobi-PCG, fp64
    assert bench.byte_model(w)["per_iteration"] == _mat(w, 8) + 13 * 8 * w.A.n
    w = build("c3", N=16, batch=3)              # batched fp32 values, 8-byte working vectors
    bm = bench.byte_model(w)
    assert bm["per_iteration"] == _mat(w, 4) + 13 * 8 * w.A.n * 3
    assert bm["spmv_dot_per_launch"] == _mat(w, 4) + 2 * 4 * w.A.n * 3


def test_bicgstab_model():
    w = build("cd3", N=10)
    bm = bench.byte_model(w)
    n, nnz = w.A.n, w.A.nnz
    mat = 12 * nnz + 4 * (n + 1)
    assert bench.method_of(w) == "bicgstab"
    assert bm["per_iteration"] == 2 * mat + 19 * 8 * n
    assert bm["product_per_launch"] == mat + 3 * 8 * n
    assert bench.metric_of(w) == bench.METRIC_BICG
    assert bench.metric_of(build("c1", N=8)) == bench.METRIC


def test_full_size_models_match_the_stated_figures():
    # c4 at 128^3: 367.9 MB per CG iteration, 216.9 MB per product launch
    w = build("c4")
    bm = bench.byte_model(w)
    assert round(bm["per_iteration"] / 1e6, 1) == 367.9
    assert round(bm["product_per_launch"] / 1e6, 1) == 216.9


def test_oracle_dispatch_follows_the_method():
    w = build("cd3", N=8)
    x, info = bench.oracle_solve(w, w.A, w.b, 10000)
    assert info["status"] == "ok"
    D = w.A.dense()
    assert np.linalg.norm(D @ x - w.b) <= 2 * w.tol * np.linalg.norm(w.b)
    assert np.abs(D - D.T).max() > 0.1          # nonsymmetric: CG would not apply
    w = build("c1", N=8)
    x, info = bench.oracle_solve(w, w.A, w.b, 10000)
    assert info["status"] == "ok"


def test_reference_arm_prints_one_contract_line():
    """`bench.py --impl reference` (the oracle on the host) prints one JSON
    line with the contract's keys; c1 keeps it to a few seconds."""
    import json
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    out = subprocess.run([sys.executable, os.path.join(root, "bench.py"), "--impl", "reference", "--config", "c1",
                          "--steps", "1", "--warmup", "0"], capture_output=True, text=True, timeout=300, cwd=root)
    assert out.returncode == 0, out.stderr
    lines = [l for l in out.stdout.splitlines() if l.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better",
                "scaling", "vs_baseline", "dtype", "data", "config", "impl", "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["value"] > 0 and d["higher_is_better"] is True
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] == 1
    assert d["cpu_baseline"]["host"]["available_cores"] >= 1
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["value"] == d["value"]
    # the same config keys as the main arm's line (bench.config_of)
    for key in ("workload", "n", "nnz", "batch", "pc", "tol", "poll_k", "step", "l2"):
        assert key in d["config"], key
    assert d["config"]["workload"].startswith("c1:")


def test_l2_rule_follows_the_working_set():
    """A workload whose iteration touches more than L2 (126 MiB) is timed
    with no flush; one that fits (the 64x64 Poisson grid, and the
    profiler-capture sizes) gets an L2 flush before every timed step."""
    for name, kw, resident in (("c1", {}, True), ("c2", {}, False), ("c4", {"N": 24}, True)):
        w = build(name, **kw)
        bm = bench.byte_model(w, bench.nnzg_of(w))
        assert bench.l2_resident(bm) == resident, name
        assert bench.l2_rule(bm).startswith("L2 flushed" if resident else "inputs larger than L2"), name
