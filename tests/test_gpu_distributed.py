"""The row-partitioned PCG on one GPU: P partitions held in one process
(LocalComm: halo exchange by device gathers, inner products summed over the
partitions), each partition's arithmetic in the library's kernels
(LibraryLocal: sla_spmv_dot, sla_cg_local_update / _direction, sla_grad_A,
a handle on the local transpose).  x, iterations, lambda and dL/dA against
the oracle; A^T v through H^T against the oracle's product with the
explicit transpose."""
import numpy as np
import pytest
import torch

import oracle
from workloads import build
from workloads.matrices import CSR

from gpu_util import random_csr, rel

pytestmark = pytest.mark.gpu


def _transpose(A):
    rows = A.rows()
    order = np.lexsort((rows, A.col_idx))
    rp = np.zeros(A.n + 1, dtype=np.int32)
    rp[1:] = np.cumsum(np.bincount(A.col_idx, minlength=A.n))
    return CSR(A.n, rp, rows[order].astype(np.int32), A.vals[order])


CASES = [
    ("c2", {"N": 64}, "jacobi", 1e-10),
    ("c4", {"N": 20}, "none", 1e-10),
    ("c5", {"npoints": 8000}, "jacobi", 1e-10),
]


@pytest.mark.parametrize("parts", [1, 3, 4])
@pytest.mark.parametrize("cfg,kw,pc,tol", CASES, ids=[c[0] + "-" + c[2] for c in CASES])
def test_partitioned_solve_and_adjoint_match_the_oracle(cuda_device, parts, cfg, kw, pc, tol):
    from sparse_iterative_linear_csr_b300 import distributed as D
    w = build(cfg, **kw)
    A = w.A
    P = D.partition(A.row_ptr, A.col_idx, parts)
    comm = D.LocalComm(P, cuda_device)
    locs = [D.LibraryLocal(pt, A.vals, cuda_device) for pt in P]
    b = [torch.from_numpy(w.b[pt.r0:pt.r1].copy()).to(cuda_device) for pt in P]
    g = [torch.from_numpy(w.g[pt.r0:pt.r1].copy()).to(cuda_device) for pt in P]
    x, info = D.pcg(comm, locs, b, tol=tol, pc=pc)
    lam, dA, ainfo = D.adjoint(comm, locs, x, g, tol=tol, pc=pc)
    xg = np.concatenate([t.cpu().numpy() for t in x])
    lg = np.concatenate([t.cpu().numpy() for t in lam])
    dAg = np.zeros(A.nnz)
    for pt, d in zip(P, dA):
        dAg[pt.src] = d.cpu().numpy()
    xo, io = oracle.pcg(A, w.b, tol, pc=pc)
    lo, _, ao = oracle.adjoint(A, xo, w.g, tol, pc=pc)
    assert info.status == "ok" and info.rel_res_true <= tol
    assert abs(info.iters - io["iters"]) <= max(1, int(0.02 * io["iters"])), (info.iters, io["iters"])
    assert abs(ainfo.iters - ao["iters"]) <= max(1, int(0.02 * ao["iters"]))
    assert rel(xg, xo) <= 1e-6
    assert rel(lg, lo) <= 1e-6
    assert rel(dAg, oracle.grad_A(A, lo, xo)) <= 1e-6
    v = np.random.default_rng(3).standard_normal(A.n)
    yt = D.matvec_t(comm, locs, [torch.from_numpy(v[pt.r0:pt.r1].copy()).to(cuda_device) for pt in P])
    ytg = np.concatenate([t.cpu().numpy() for t in yt])
    At = _transpose(A)
    scale = oracle.spmv(CSR(A.n, At.row_ptr, At.col_idx, np.abs(At.vals)), np.abs(v))
    assert np.all(np.abs(ytg - oracle.spmv(At, v)) <= 1e-12 * np.maximum(scale, 1e-300))


def test_partitioned_transpose_of_a_nonsymmetric_matrix(cuda_device):
    """H^T sums every halo contribution at its owner: A^T v for a random
    nonsymmetric pattern over 5 partitions."""
    from sparse_iterative_linear_csr_b300 import distributed as D
    A = random_csr(3000, 7, seed=12)
    P = D.partition(A.row_ptr, A.col_idx, 5)
    comm = D.LocalComm(P, cuda_device)
    locs = [D.LibraryLocal(pt, A.vals, cuda_device) for pt in P]
    v = np.random.default_rng(8).standard_normal(A.n)
    yt = D.matvec_t(comm, locs, [torch.from_numpy(v[pt.r0:pt.r1].copy()).to(cuda_device) for pt in P])
    ytg = np.concatenate([t.cpu().numpy() for t in yt])
    At = _transpose(A)
    scale = oracle.spmv(CSR(A.n, At.row_ptr, At.col_idx, np.abs(At.vals)), np.abs(v))
    assert np.all(np.abs(ytg - oracle.spmv(At, v)) <= 1e-12 * np.maximum(scale, 1e-300))
