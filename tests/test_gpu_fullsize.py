"""Parity at the workloads' full sizes (the five CG workloads and the
BiCGStab workload cd3), in the launch configuration the benchmark times (same
options, poll interval 32, forward solve then adjoint).

The large CG workloads c2, c4 and c5 are compared with the oracle's own
full-size solves (computed once by tests/fullsize_oracle.py and cached, or in
spawned processes started at the beginning of the session): x and lambda
within 1e-6 relative, dL/dA against the oracle's -lambda_i x_j on the pattern
within 1e-6 relative, forward and adjoint iteration counts within 2%.
Besides, the checks that hold at any size and outputs the oracle computes
one by one:
  * SpMV: 2000 sampled rows against the oracle's row sums of those rows;
  * solve: status, and the true residual ||b - A x|| / ||b|| <= tol
    recomputed on the host in fp64 from the returned x (scipy, not the GPU);
    the 64x64 Poisson problem and two systems of the 64-system batch are also
    solved by the oracle and compared element by element;
  * adjoint: g.x = lambda.b and sum_k A_k dL/dA_k = -g.x (fp64 on the host),
    the adjoint's own true residual ||g - A^T lambda||, and sampled dL/dA
    entries exactly equal to -lambda_i x_j of the returned vectors.
BiCGStab's Jacobi form iterates on the column-scaled system and confirms
its stop on b - A x of the returned x."""
import numpy as np
import pytest
import scipy.sparse as sp
import torch

import oracle
from workloads import build
from workloads.matrices import CSR

import fullsize_oracle
from gpu_util import make, rel

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

BENCH_KW = dict(max_iter=200000, poll_k=32)


def _system(A, s):
    v = A.vals if A.vals.ndim == 1 else A.vals[s]
    return sp.csr_matrix((v.astype(np.float64), A.col_idx, A.row_ptr), shape=(A.n, A.n))


def _true_rel(A, s, b, x, transpose=False):
    M = _system(A, s)
    if transpose:
        M = M.T.tocsr()
    b = b.astype(np.float64)
    return float(np.linalg.norm(b - M @ x.astype(np.float64)) / np.linalg.norm(b))


_cache = {}


def _workload(name):
    if name not in _cache:
        _cache.clear()
        _cache[name] = build(name)
    return _cache[name]


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5", "cd3"])
def test_fullsize_spmv_sampled_rows(cuda_device, name):
    w = _workload(name)
    A = w.A
    M = make(A)
    g = np.random.default_rng(3)
    shape = (A.n,) if A.vals.ndim == 1 else (A.vals.shape[0], A.n)
    x = g.standard_normal(shape).astype(A.vals.dtype)
    y = M.matvec(torch.from_numpy(x).to(cuda_device)).cpu().numpy()
    rows = np.sort(g.choice(A.n, size=min(2000, A.n), replace=False))
    lo, hi = A.row_ptr[rows], A.row_ptr[rows + 1]
    sub_rp = np.zeros(rows.size + 1, np.int32)
    sub_rp[1:] = np.cumsum(hi - lo)
    idx = np.concatenate([np.arange(a, b) for a, b in zip(lo, hi)])
    for s in range(1 if A.vals.ndim == 1 else min(3, A.vals.shape[0])):
        v = A.vals if A.vals.ndim == 1 else A.vals[s]
        xs = (x if x.ndim == 1 else x[s]).astype(np.float64)
        ys = y if y.ndim == 1 else y[s]
        # the oracle's SpMV on the sampled rows (a CSR of those rows that
        # addresses the full-length vector)
        sub = CSR(rows.size, sub_rp, A.col_idx[idx], v[idx])
        y_o = oracle.spmv(sub, xs)
        scale = oracle.spmv(CSR(rows.size, sub_rp, A.col_idx[idx], np.abs(v[idx])), np.abs(xs))
        tol = 1e-12 if A.vals.dtype == np.float64 else 1e-5
        assert np.all(np.abs(ys[rows].astype(np.float64) - y_o) <= tol * np.maximum(scale, 1e-300))


@pytest.mark.parametrize("name", ["c1", "c2", "c3", "c4", "c5", "cd3"])
def test_fullsize_solve_and_adjoint(cuda_device, name):
    w = _workload(name)
    A = w.A
    M = make(A)
    b = torch.from_numpy(w.b).to(cuda_device)
    g = torch.from_numpy(w.g).to(cuda_device)
    method = w.info.get("method", "cg")
    kw = dict(tol=w.tol, pc=w.pc, eps=w.eps if w.pc == "spai" else 1e-3, method=method, **BENCH_KW)
    x, info = M.solve(b, **kw)
    dldb, dlda, ainfo = M.adjoint(x, g, **kw)
    xh, lb, la = x.cpu().numpy(), dldb.cpu().numpy(), dlda.cpu().numpy()
    nsys = 1 if A.vals.ndim == 1 else A.vals.shape[0]
    X = xh.reshape(nsys, A.n)
    L = lb.reshape(nsys, A.n)
    DA = la.reshape(nsys, A.nnz)
    B = w.b.reshape(nsys, A.n)
    G = w.g.reshape(nsys, A.n)
    rows = A.rows()
    pick = np.random.default_rng(7).choice(A.nnz, size=min(5000, A.nnz), replace=False)
    for s in range(nsys):
        assert info[s].status == "ok" and ainfo[s].status == "ok"
        # true residuals recomputed on the host in fp64
        tr = _true_rel(A, s, B[s], X[s])
        assert tr <= w.tol
        assert abs(tr - info[s].rel_res_true) <= 1e-3 * w.tol
        assert _true_rel(A, s, G[s], L[s], transpose=True) <= w.tol
        # adjoint identities
        gx = float(G[s].astype(np.float64) @ X[s].astype(np.float64))
        lbb = float(L[s].astype(np.float64) @ B[s].astype(np.float64))
        v = A.vals if A.vals.ndim == 1 else A.vals[s]
        sad = float(v.astype(np.float64) @ DA[s].astype(np.float64))
        # |g.x - lambda.b| <= ||lambda|| ||b - A x|| + ||x|| ||g - A lambda|| (both residuals <= tol)
        nrm = lambda a: float(np.linalg.norm(a.astype(np.float64)))
        bound = 10 * w.tol * (nrm(L[s]) * nrm(B[s]) + nrm(X[s]) * nrm(G[s]))
        assert abs(gx - lbb) <= bound
        assert abs(sad + gx) <= bound
        exact = (-L[s][rows[pick]].astype(np.float64) * X[s][A.col_idx[pick]].astype(np.float64))
        assert np.array_equal(DA[s][pick], exact.astype(DA.dtype))


def test_fullsize_c1_matches_oracle(cuda_device):
    w = _workload("c1")
    M = make(w.A)
    x, info = M.solve(torch.from_numpy(w.b).to(cuda_device), tol=w.tol, pc=w.pc, **BENCH_KW)
    xo, io = oracle.pcg(w.A, w.b, w.tol, pc=w.pc)
    assert abs(info[0].iters - io["iters"]) <= max(1, int(0.02 * io["iters"]))
    assert rel(x.cpu().numpy(), xo) <= 1e-6


def test_fullsize_c3_two_systems_match_oracle(cuda_device):
    w = _workload("c3")
    M = make(w.A)
    x, info = M.solve(torch.from_numpy(w.b).to(cuda_device), tol=w.tol, pc=w.pc, **BENCH_KW)
    xh = x.cpu().numpy()
    for s in (0, 37):
        A1 = CSR(w.A.n, w.A.row_ptr, w.A.col_idx, w.A.vals[s])
        xo, io = oracle.pcg(A1, w.b[s], w.tol, pc="jacobi", f32=True)
        assert abs(info[s].iters - io["iters"]) <= max(1, int(0.02 * io["iters"]))
        assert rel(xh[s], xo) <= 1e-6


def _oracle_results(name, w):
    """The oracle's full-size (x, info, lambda, info) for workload `name`:
    from the cache, else from the solves the session started (conftest), else
    computed here in spawned processes."""
    key = fullsize_oracle.key_of(w)
    got = fullsize_oracle.load(name, key)
    if got is None:
        pending = getattr(fullsize_oracle, "PENDING", None)
        if pending is None:
            pool, pending = fullsize_oracle.start((name,))
        for r in pending:
            r.get(timeout=3600)
        got = fullsize_oracle.load(name, key)
    assert got is not None, f"oracle results for {name} missing"
    return got


@pytest.mark.parametrize("name", ["c2", "c4", "c5"])
def test_fullsize_matches_oracle(cuda_device, name):
    """x, iterations, lambda and dL/dA against the oracle at full size, in
    the benchmark's launch configuration."""
    w = _workload(name)
    A = w.A
    M = make(A)
    kw = dict(tol=w.tol, pc=w.pc, eps=w.eps if w.pc == "spai" else 1e-3, **BENCH_KW)
    x, info = M.solve(torch.from_numpy(w.b).to(cuda_device), **kw)
    lam, dA, ainfo = M.adjoint(x, torch.from_numpy(w.g).to(cuda_device), **kw)
    xo, fo, lo, ao = _oracle_results(name, w)
    assert fo["status"] == "ok" and ao["status"] == "ok"
    assert info[0].status == "ok" and ainfo[0].status == "ok"
    assert abs(info[0].iters - fo["iters"]) <= max(1, int(0.02 * fo["iters"])), (info[0].iters, fo["iters"])
    assert abs(ainfo[0].iters - ao["iters"]) <= max(1, int(0.02 * ao["iters"])), (ainfo[0].iters, ao["iters"])
    xh = x.cpu().numpy()
    lh = lam.cpu().numpy()
    ex, el = rel(xh, xo), rel(lh, lo)
    assert ex <= 1e-6, ex
    assert el <= 1e-6, el
    del lam, x
    dAo = oracle.grad_A(A, lo, xo)
    ed = rel(dA.cpu().numpy(), dAo)
    assert ed <= 1e-6, ed
