"""Row-partitioned preconditioned CG and its adjoint (torch-sla, arXiv
2601.13994: §3, the distributed paragraphs -- contiguous row blocks, each
with the halo of columns it reads from other blocks; §3.3, distributed CG --
a halo exchange before every product and all-reduced inner products; the
adjoint paragraph -- the transpose of the halo exchange sums each halo
copy's contribution back at its owner, and dL/dA is assembled locally on the
owned non-zeros).

A partition owns rows [r0, r1) of A.  Its local matrix is square, of size
nloc = nown + nhalo: the owned rows with every column renumbered -- an owned
column j to j - r0, a halo column to nown + (its position in the sorted halo
set) -- and nhalo empty rows, so a local product of the extended vector
[x_own; x_halo] gives the owned rows of A x (and zeros in the halo rows).
The exchange plan lists, for every pair of partitions, which owned entries
one sends and where the other keeps them.

Communication (`LocalComm`: every partition in one process on one device,
the halo copies done by device gathers; `DistComm`: one partition per rank
of a torch.distributed process group, point-to-point sends of the halo
entries and an all-reduce of the inner products) is separate from the local
arithmetic (`LibraryLocal`: the partition's products, CG updates and matrix
gradient run in the library's kernels).  The CG loop (`pcg`) follows the
oracle's order of steps and stopping tests, so on one partition it is the
library's CG, rounded in another order.  Preconditioners: none or Jacobi
(both local).
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass, field

import numpy as np
import torch

from . import CSRMatrix, _check, _lib_handle, _ptr, _stream


# ----------------------------------------------------------------- partition
@dataclass
class Part:
    """One partition: owned rows [r0, r1), the halo (global column indices,
    ascending), the square local CSR (rp, ci) and the global entry of every
    local entry (src), so values and gradients map between the two."""
    index: int
    r0: int
    r1: int
    halo: np.ndarray
    rp: np.ndarray
    ci: np.ndarray
    src: np.ndarray
    diag_entry: np.ndarray = field(default=None)   # local entry of each owned row's diagonal, -1 if none

    @property
    def nown(self) -> int:
        return self.r1 - self.r0

    @property
    def nloc(self) -> int:
        return self.nown + len(self.halo)


def row_blocks(row_ptr: np.ndarray, nparts: int) -> np.ndarray:
    """Boundaries r_0 = 0 < ... < r_P = n of contiguous row blocks holding
    about nnz / P stored entries each (every block at least one row)."""
    n = len(row_ptr) - 1
    if not 1 <= nparts <= n:
        raise ValueError("need 1 <= parts <= n")
    nnz = int(row_ptr[-1])
    b = [0]
    for k in range(1, nparts):
        r = int(np.searchsorted(row_ptr, k * nnz / nparts, side="left"))
        r = min(max(r, b[-1] + 1), n - (nparts - k))
        b.append(r)
    b.append(n)
    return np.asarray(b, dtype=np.int64)


def partition(row_ptr: np.ndarray, col_idx: np.ndarray, nparts: int) -> list[Part]:
    """Split a CSR pattern into nparts contiguous row blocks with halos."""
    row_ptr = np.asarray(row_ptr, dtype=np.int64)
    col_idx = np.asarray(col_idx, dtype=np.int64)
    bounds = row_blocks(row_ptr, nparts)
    parts = []
    for p in range(nparts):
        r0, r1 = int(bounds[p]), int(bounds[p + 1])
        k0, k1 = int(row_ptr[r0]), int(row_ptr[r1])
        cols = col_idx[k0:k1]
        outside = (cols < r0) | (cols >= r1)
        halo = np.unique(cols[outside])
        nown = r1 - r0
        loc = np.where(outside, nown + np.searchsorted(halo, cols), cols - r0)
        rows = np.repeat(np.arange(nown), np.diff(row_ptr[r0:r1 + 1]))
        order = np.lexsort((loc, rows))        # columns ascending within each row
        ci = loc[order].astype(np.int32)
        src = (k0 + order).astype(np.int64)
        rp = np.zeros(nown + len(halo) + 1, dtype=np.int32)
        rp[1:nown + 1] = np.cumsum(np.diff(row_ptr[r0:r1 + 1]))
        rp[nown + 1:] = rp[nown]
        rws = rows[order]
        diag = np.full(nown, -1, dtype=np.int64)
        on = ci == rws
        diag[rws[on]] = np.nonzero(on)[0]
        parts.append(Part(p, r0, r1, halo, rp, ci, src, diag))
    return parts


def owner_of(bounds: np.ndarray, cols: np.ndarray) -> np.ndarray:
    return np.searchsorted(bounds, cols, side="right") - 1


def exchange_plan(parts: list[Part]) -> dict:
    """plan[(p, q)] = (owned local indices of p that q needs, their slots in
    q's halo), for every pair with something to send."""
    bounds = np.asarray([parts[0].r0] + [pt.r1 for pt in parts], dtype=np.int64)
    plan = {}
    for q, pq in enumerate(parts):
        if len(pq.halo) == 0:
            continue
        own = owner_of(bounds, pq.halo)
        for p in np.unique(own):
            slots = np.nonzero(own == p)[0]
            plan[(int(p), q)] = ((pq.halo[slots] - parts[p].r0).astype(np.int64), slots.astype(np.int64))
    return plan


# ----------------------------------------------------------------- communication
class LocalComm:
    """Every partition in this process (one device): the halo exchange is a
    gather from the owner's entries into the receiver's halo slots."""

    def __init__(self, parts: list[Part], device):
        self.parts = parts
        self.held = list(range(len(parts)))
        self.plan = {k: (torch.from_numpy(a).to(device), torch.from_numpy(b).to(device))
                     for k, (a, b) in exchange_plan(parts).items()}

    def exchange(self, vecs):
        """H: fill every partition's halo slots from the owners' entries."""
        for (p, q), (idx, slots) in self.plan.items():
            vecs[q][self.parts[q].nown + slots] = vecs[p][idx]

    def reduce_halo(self, vecs):
        """H^T: add every halo slot's value into its owner's entry, then
        clear the halo slots (the owners hold the sums)."""
        for (p, q), (idx, slots) in self.plan.items():
            vecs[p].index_add_(0, idx, vecs[q][self.parts[q].nown + slots])
        for q, pq in enumerate(self.parts):
            vecs[q][pq.nown:] = 0

    def allreduce(self, vals):
        """Sum over the partitions of per-partition tensors (in partition order)."""
        tot = vals[0].clone()
        for v in vals[1:]:
            tot += v
        return tot


class DistComm:
    """One partition per rank of the default torch.distributed group
    (gloo on the host, NCCL on GPUs): point-to-point halo sends and an
    all-reduce of the inner products."""

    def __init__(self, parts: list[Part], rank: int, device):
        import torch.distributed as dist
        self.dist = dist
        self.parts = parts
        self.rank = rank
        self.held = [rank]
        self.device = device
        plan = exchange_plan(parts)
        self.send = {q: torch.from_numpy(a).to(device) for (p, q), (a, _) in plan.items() if p == rank}
        self.recv = {p: torch.from_numpy(b).to(device) for (p, q), (_, b) in plan.items() if q == rank}

    def _swap(self, outgoing: dict, incoming_sizes: dict, dtype):
        reqs, bufs = [], {}
        for p, n in sorted(incoming_sizes.items()):
            bufs[p] = torch.empty(n, dtype=dtype, device=self.device)
            reqs.append(self.dist.irecv(bufs[p], src=p))
        for q, t in sorted(outgoing.items()):
            reqs.append(self.dist.isend(t.contiguous(), dst=q))
        for r in reqs:
            r.wait()
        return bufs

    def exchange(self, vecs):
        v = vecs[0]
        nown = self.parts[self.rank].nown
        bufs = self._swap({q: v[idx] for q, idx in self.send.items()},
                          {p: len(s) for p, s in self.recv.items()}, v.dtype)
        for p, slots in self.recv.items():
            v[nown + slots] = bufs[p]

    def reduce_halo(self, vecs):
        v = vecs[0]
        nown = self.parts[self.rank].nown
        bufs = self._swap({p: v[nown + slots] for p, slots in self.recv.items()},
                          {q: len(idx) for q, idx in self.send.items()}, v.dtype)
        for q, idx in self.send.items():
            v.index_add_(0, idx, bufs[q])
        v[nown:] = 0

    def allreduce(self, vals):
        t = vals[0].clone()
        self.dist.all_reduce(t)
        return t


# ----------------------------------------------------------------- local arithmetic
class LibraryLocal:
    """A partition's arithmetic on the GPU, in the library's kernels: the
    local product fused with p.q (sla_spmv_dot), the CG updates of the owned
    entries (sla_cg_local_update / sla_cg_local_direction), the transposed
    product (a handle on the local transpose) and the matrix gradient
    (sla_grad_A)."""

    def __init__(self, part: Part, values: np.ndarray, device):
        self.part = part
        self.device = device
        v = np.ascontiguousarray(np.asarray(values, dtype=np.float64)[part.src])
        self.vals = torch.from_numpy(v).to(device)
        rp = torch.from_numpy(part.rp).to(device)
        ci = torch.from_numpy(part.ci).to(device)
        self.M = CSRMatrix(rp, ci, self.vals, reorder=False)
        # the local transpose (rows of the halo columns hold the contributions
        # to other partitions' entries)
        n = part.nloc
        rows = np.repeat(np.arange(n), np.diff(part.rp))
        order = np.lexsort((rows, part.ci))
        trp = np.zeros(n + 1, dtype=np.int32)
        trp[1:] = np.cumsum(np.bincount(part.ci, minlength=n))
        self._trp = torch.from_numpy(trp).to(device)
        self._tci = torch.from_numpy(rows[order].astype(np.int32)).to(device)
        self._tv = torch.from_numpy(np.ascontiguousarray(v[order])).to(device)
        self.MT = CSRMatrix(self._trp, self._tci, self._tv, reorder=False)
        d = np.ones(part.nown)
        have = part.diag_entry >= 0
        d[have] = v[part.diag_entry[have]]
        self.has_diag = bool(have.all())
        self.dinv = torch.from_numpy(1.0 / d).to(device)
        need = C.c_longlong(0)
        _check(_lib_handle().sla_cg_local_work(part.nown, C.byref(need)))
        self.work = torch.empty(max(int(need.value), 2), dtype=torch.float64, device=device)
        self.dots = torch.zeros(2, dtype=torch.float64, device=device)

    def zeros(self, n=None):
        return torch.zeros(self.part.nloc if n is None else n, dtype=torch.float64, device=self.device)

    def matvec_dot(self, p_ext):
        q, d = self.M.matvec_dot(p_ext)
        return q, d.reshape(1)

    def matvec(self, x_ext):
        return self.M.matvec(x_ext)

    def matvec_t(self, v_ext):
        return self.MT.matvec(v_ext)

    def update(self, alpha, p_ext, q_ext, x, r, z, jacobi):
        n = self.part.nown
        _check(_lib_handle().sla_cg_local_update(n, float(alpha), _ptr(p_ext), _ptr(q_ext),
                                                 _ptr(self.dinv) if jacobi else None, _ptr(x), _ptr(r), _ptr(z),
                                                 _ptr(self.dots), _ptr(self.work), self.work.numel(), _stream()))
        return self.dots.clone()

    def direction(self, beta, z, p_ext):
        _check(_lib_handle().sla_cg_local_direction(self.part.nown, float(beta), _ptr(z), _ptr(p_ext), _stream()))

    def residual2(self, x_ext, b):
        """||b - A x||^2 over the owned rows (this partition's share)."""
        from .eigen import GRAM_DIAG, gram, update
        q = self.matvec(x_ext)[:self.part.nown].reshape(1, -1)
        d = update(torch.full((1, 1), -1.0, dtype=torch.float64, device=self.device), q, b.reshape(1, -1))
        return gram(d, mode=GRAM_DIAG).reshape(1)

    def dot(self, a, b):
        from .eigen import gram
        return gram(a.reshape(1, -1), b.reshape(1, -1)).reshape(1)

    def grad_A(self, lam_ext, x_ext):
        out = torch.empty_like(self.vals)
        _check(_lib_handle().sla_grad_A(self.M._h, _ptr(lam_ext), _ptr(x_ext), _ptr(out), _stream()))
        return out


# ----------------------------------------------------------------- solver
@dataclass
class PartInfo:
    iters: int
    status: str
    rel_res_recursive: float
    rel_res_true: float


def pcg(comm, locs, b_own, tol=1e-8, max_iter=10000, pc="none"):
    """Solve A x = b by preconditioned CG over the partitions held in this
    process (comm.held, with their local arithmetic `locs` and owned
    right-hand sides `b_own`), in the oracle's order of steps: the
    recursive-residual test right after the r update, confirmed on the true
    residual of x; z = M^-1 r, beta and the new direction at the top of the
    next iteration; q = A p after a halo exchange of p, alpha = rho / p.q.
    Returns (owned parts of x, PartInfo); the same on every rank."""
    if pc not in ("none", "jacobi"):
        raise ValueError("the partitioned solve takes pc 'none' or 'jacobi'")
    jac = pc == "jacobi"
    if jac and not all(L.has_diag for L in locs):
        raise ValueError("Jacobi needs every diagonal entry stored")
    P = len(locs)
    x = [L.zeros(L.part.nown) for L in locs]
    r = [b.clone() for b in b_own]
    z = [L.zeros(L.part.nown) for L in locs]
    p = [L.zeros() for L in locs]
    q = [L.zeros() for L in locs]
    bb = float(comm.allreduce([L.dot(b, b) for L, b in zip(locs, b_own)]).item())
    if bb == 0.0:
        return x, PartInfo(0, "ok", 0.0, 0.0)
    d0 = comm.allreduce([locs[i].update(0.0, p[i], q[i], x[i], r[i], z[i], jac) for i in range(P)])
    gamma, rho = float(d0[0].item()), float(d0[1].item())
    rho_next = rho
    for i in range(P):
        locs[i].direction(0.0, z[i], p[i])
    tol2bb = tol * tol * bb
    k, status, tr2 = 0, "ok", None

    def true_res2():
        xe = []
        for i in range(P):
            v = locs[i].zeros()
            v[:locs[i].part.nown] = x[i]
            xe.append(v)
        comm.exchange(xe)
        return float(comm.allreduce([locs[i].residual2(xe[i], b_own[i]) for i in range(P)]).item())

    while True:
        if not np.isfinite(gamma):
            status = "breakdown"
            break
        if gamma <= tol2bb:
            tr2 = true_res2()
            if tr2 <= tol2bb:
                status = "ok"
                break
        if k >= max_iter:
            status = "not_converged"
            break
        if k > 0:
            rho_new = rho_next
            if not (rho_new > 0.0) or not np.isfinite(rho_new):
                status = "breakdown"
                break
            beta = rho_new / rho
            rho = rho_new
            for i in range(P):
                locs[i].direction(beta, z[i], p[i])
        comm.exchange(p)
        parts = []
        for i in range(P):
            q[i], dl = locs[i].matvec_dot(p[i])
            parts.append(dl)
        delta = float(comm.allreduce(parts).item())
        if not (delta > 0.0) or not np.isfinite(delta):
            status = "breakdown"
            break
        alpha = rho / delta
        d = comm.allreduce([locs[i].update(alpha, p[i], q[i], x[i], r[i], z[i], jac) for i in range(P)])
        gamma, rho_next = float(d[0].item()), float(d[1].item())
        k += 1
    if tr2 is None or status != "ok":
        tr2 = true_res2()
    return x, PartInfo(k, status, float(np.sqrt(max(gamma, 0.0) / bb)), float(np.sqrt(tr2 / bb)))


def adjoint(comm, locs, x_own, g_own, tol=1e-8, max_iter=10000, pc="none"):
    """Adjoint of x = A^-1 b for a symmetric A (CG): lambda solves
    A lambda = g with the same partitioned solve; dL/db = lambda and
    dL/dA_k = -lambda_row(k) x_col(k) on every partition's owned entries,
    with x's halo exchanged first.  Returns (owned parts of lambda, local
    dL/dA of every held partition in local entry order, PartInfo)."""
    lam, info = pcg(comm, locs, g_own, tol=tol, max_iter=max_iter, pc=pc)
    xe, le = [], []
    for i, L in enumerate(locs):
        v = L.zeros()
        v[:L.part.nown] = x_own[i]
        xe.append(v)
        w = L.zeros()
        w[:L.part.nown] = lam[i]
        le.append(w)
    comm.exchange(xe)
    return lam, [L.grad_A(le[i], xe[i]) for i, L in enumerate(locs)], info


def matvec_t(comm, locs, v_own):
    """y = A^T v over the partitions: each computes its local transposed
    product of [v_own; 0], and the halo rows' contributions are summed at
    their owners (H^T)."""
    ys = []
    for i, L in enumerate(locs):
        e = L.zeros()
        e[:L.part.nown] = v_own[i]
        ys.append(L.matvec_t(e))
    comm.reduce_halo(ys)
    return [y[:L.part.nown] for y, L in zip(ys, locs)]
