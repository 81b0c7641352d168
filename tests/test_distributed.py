"""The row-partitioned PCG (torch-sla §3 distributed paragraphs, §3.3
distributed CG and its H^T adjoint paragraph): the partition and exchange
plan, and the partitioned solve, adjoint and transposed product run as
world-size 2 and 4 gloo ranks on the host, against the oracle.

No GPU here: each rank's local arithmetic is a plain fp64 CPU stand-in
(`CpuLocal`, test infrastructure) with the interface of the library-backed
`LibraryLocal`; the partitioning, the halo exchange (H), its transpose (H^T)
and the all-reduced CG loop are the package's own code.  The same loop on
the GPU with the library's kernels is in tests/test_gpu_distributed.py."""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from workloads import build
from workloads.matrices import CSR

from gpu_util import random_csr, rel

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


class CpuLocal:
    """A partition's arithmetic in plain fp64 on the host (torch CPU)."""

    def __init__(self, part, values):
        self.part = part
        v = np.asarray(values, dtype=np.float64)[part.src]
        n = part.nloc
        rows = np.repeat(np.arange(n), np.diff(part.rp))
        self.rows = torch.from_numpy(rows)
        self.cols = torch.from_numpy(part.ci.astype(np.int64))
        self.v = torch.from_numpy(v)
        d = np.ones(part.nown)
        have = part.diag_entry >= 0
        d[have] = v[part.diag_entry[have]]
        self.has_diag = bool(have.all())
        self.dinv = torch.from_numpy(1.0 / d)

    def zeros(self, n=None):
        return torch.zeros(self.part.nloc if n is None else n, dtype=torch.float64)

    def matvec(self, x):
        return torch.zeros(self.part.nloc, dtype=torch.float64).index_add_(0, self.rows, self.v * x[self.cols])

    def matvec_dot(self, p):
        q = self.matvec(p)
        return q, (p @ q).reshape(1)

    def matvec_t(self, v):
        return torch.zeros(self.part.nloc, dtype=torch.float64).index_add_(0, self.cols, self.v * v[self.rows])

    def update(self, alpha, p, q, x, r, z, jacobi):
        n = self.part.nown
        x += alpha * p[:n]
        r -= alpha * q[:n]
        z.copy_(r * self.dinv if jacobi else r)
        return torch.stack([r @ r, r @ z])

    def direction(self, beta, z, p):
        n = self.part.nown
        p[:n] = z + beta * p[:n]

    def residual2(self, x_ext, b):
        d = b - self.matvec(x_ext)[:self.part.nown]
        return (d @ d).reshape(1)

    def dot(self, a, b):
        return (a @ b).reshape(1)

    def grad_A(self, lam, x):
        return -lam[self.rows] * x[self.cols]


def _cases():
    return {
        "c2_jacobi": (build("c2", N=40).A, "jacobi", 1e-10),
        "c4_none": (build("c4", N=12).A, "none", 1e-10),
        "spd_jacobi": (random_csr(500, 6, seed=4, spd=True), "jacobi", 1e-11),
    }


def test_partition_covers_the_matrix_and_reproduces_the_product():
    """Every row in exactly one block; the local matrices with exchanged
    halos give A x row by row (numpy reference), and the halos are exactly
    the columns each block reads outside itself."""
    from sparse_iterative_linear_csr_b300 import distributed as D
    A = build("c5", npoints=3000).A
    x = np.random.default_rng(2).standard_normal(A.n)
    y = oracle.spmv(A, x)
    for P in (1, 2, 3, 7):
        parts = D.partition(A.row_ptr, A.col_idx, P)
        assert parts[0].r0 == 0 and parts[-1].r1 == A.n
        assert all(parts[i].r1 == parts[i + 1].r0 for i in range(P - 1))
        plan = D.exchange_plan(parts)
        ext = []
        for pt in parts:
            e = np.zeros(pt.nloc)
            e[:pt.nown] = x[pt.r0:pt.r1]
            ext.append(e)
        for (p, q), (idx, slots) in plan.items():
            ext[q][parts[q].nown + slots] = ext[p][idx]
        for pt, e in zip(parts, ext):
            k0, k1 = A.row_ptr[pt.r0], A.row_ptr[pt.r1]
            cols = A.col_idx[k0:k1]
            assert np.array_equal(pt.halo, np.unique(cols[(cols < pt.r0) | (cols >= pt.r1)]))
            assert np.array_equal(np.sort(pt.src), np.arange(k0, k1))
            loc = CSR(pt.nloc, pt.rp, pt.ci, A.vals[pt.src])
            yl = oracle.spmv(loc, e)
            assert np.allclose(yl[:pt.nown], y[pt.r0:pt.r1], rtol=1e-13, atol=1e-13)
            assert np.all(yl[pt.nown:] == 0.0)


def test_row_blocks_balance_entries():
    from sparse_iterative_linear_csr_b300 import distributed as D
    A = random_csr(1000, 8, seed=9)
    b = D.row_blocks(A.row_ptr, 4)
    per = np.diff(A.row_ptr[b])
    assert per.max() <= A.nnz / 4 + 40
    with pytest.raises(ValueError):
        D.row_blocks(A.row_ptr, 0)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, out):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    from sparse_iterative_linear_csr_b300 import distributed as D
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        res = {}
        for name, (A, pc, tol) in _cases().items():
            parts = D.partition(A.row_ptr, A.col_idx, world)
            comm = D.DistComm(parts, rank, torch.device("cpu"))
            pt = parts[rank]
            loc = [CpuLocal(pt, A.vals)]
            g = np.random.default_rng(7)
            b = g.standard_normal(A.n)
            gv = g.standard_normal(A.n)
            x, info = D.pcg(comm, loc, [torch.from_numpy(b[pt.r0:pt.r1].copy())], tol=tol, pc=pc)
            lam, dA, ainfo = D.adjoint(comm, loc, x, [torch.from_numpy(gv[pt.r0:pt.r1].copy())], tol=tol, pc=pc)
            v = g.standard_normal(A.n)
            yt = D.matvec_t(comm, loc, [torch.from_numpy(v[pt.r0:pt.r1].copy())])
            res[name] = (pt.r0, pt.r1, x[0].numpy(), info, lam[0].numpy(), pt.src, dA[0].numpy(),
                         yt[0].numpy(), b, gv, v)
        out[rank] = res
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_partitioned_solve_adjoint_and_transpose_on_gloo_ranks(world):
    """x, iterations, lambda and dL/dA of the partitioned solve against the
    oracle; A^T v through the local transposes and H^T against numpy."""
    port = _free_port()
    mgr = mp.Manager()
    out = mgr.dict()
    mp.start_processes(_rank, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    for name, (A, pc, tol) in _cases().items():
        ranks = [out[r][name] for r in range(world)]
        b, gv, v = ranks[0][8], ranks[0][9], ranks[0][10]
        x = np.zeros(A.n)
        lam = np.zeros(A.n)
        dA = np.zeros(A.nnz)
        yt = np.zeros(A.n)
        for r0, r1, xr, info, lr, src, dr, ytr, *_ in ranks:
            x[r0:r1] = xr
            lam[r0:r1] = lr
            dA[src] = dr
            yt[r0:r1] = ytr
            assert info.status == "ok" and info.rel_res_true <= tol
        xo, io = oracle.pcg(A, b, tol, pc=pc)
        lo, dAo, ao = oracle.adjoint(A, xo, gv, tol, pc=pc)
        its = ranks[0][3].iters
        assert all(rk[3].iters == its for rk in ranks)     # every rank saw the same scalars
        assert abs(its - io["iters"]) <= max(1, int(0.02 * io["iters"])), (name, its, io["iters"])
        assert rel(x, xo) <= 1e-6, name
        assert rel(lam, lo) <= 1e-6, name
        assert rel(dA, oracle.grad_A(A, lo, xo)) <= 1e-6, name
        At = CSR(A.n, *_transpose(A))
        assert np.allclose(yt, oracle.spmv(At, v), rtol=1e-12, atol=1e-12), name


def _transpose(A):
    rows = A.rows()
    order = np.lexsort((rows, A.col_idx))
    rp = np.zeros(A.n + 1, dtype=np.int32)
    rp[1:] = np.cumsum(np.bincount(A.col_idx, minlength=A.n))
    return rp, rows[order].astype(np.int32), A.vals[order]
