"""Helpers shared by the GPU tests: move a workloads.CSR to the device and
compare results with the oracle."""
import numpy as np
import torch

from workloads.matrices import CSR


def to_device(A: CSR, device="cuda:0"):
    rp = torch.from_numpy(np.ascontiguousarray(A.row_ptr)).to(device)
    ci = torch.from_numpy(np.ascontiguousarray(A.col_idx)).to(device)
    v = torch.from_numpy(np.ascontiguousarray(A.vals)).to(device)
    return rp, ci, v


def make(A: CSR, device="cuda:0", validate=True, **opts):
    from sparse_iterative_linear_csr_b300 import CSRMatrix
    rp, ci, v = to_device(A, device)
    return CSRMatrix(rp, ci, v, validate=validate, **opts)


def rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    nb = np.linalg.norm(b)
    return np.linalg.norm(a - b) / (nb if nb > 0 else 1.0)


def random_csr(n, nnz_per_row, seed, dtype=np.float64, spd=False, empty_rows=0):
    """Random pattern with ascending columns; spd=True gives a symmetric,
    strictly diagonally dominant matrix."""
    g = np.random.default_rng(seed)
    rows, cols = [], []
    for i in range(n):
        k = min(n, max(0, int(g.poisson(nnz_per_row))))
        c = np.unique(g.integers(0, n, size=k))
        rows.append(np.full(c.size, i))
        cols.append(c)
    r = np.concatenate(rows) if rows else np.zeros(0, np.int64)
    c = np.concatenate(cols) if cols else np.zeros(0, np.int64)
    if spd:
        r, c = np.concatenate([r, c, np.arange(n)]), np.concatenate([c, r, np.arange(n)])
    key = np.unique(r.astype(np.int64) * n + c)
    r, c = key // n, key % n
    if empty_rows:
        drop = np.isin(r, g.choice(n, size=empty_rows, replace=False))
        r, c = r[~drop], c[~drop]
    v = g.standard_normal(r.size)
    if spd:
        v = -np.abs(v)
        off = r != c
        # symmetric values: take the value of (min, max)
        a = np.minimum(r, c) * n + np.maximum(r, c)
        uniq, inv = np.unique(a, return_inverse=True)
        vs = -np.abs(g.standard_normal(uniq.size))
        v = vs[inv]
        v[~off] = 0.0
        rowsum = np.bincount(r, weights=np.abs(v), minlength=n)
        v[~off] = rowsum[r[~off]] + 1.0
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(r, minlength=n), out=rp[1:])
    return CSR(n, rp.astype(np.int32), c.astype(np.int32), v.astype(dtype))
