"""Sparse SPD test matrices in CSR form (int32 indices, columns ascending).

These are the inputs of the solver, not part of it: grid Laplacians, a
variable-coefficient diffusion operator and a k-nearest-neighbour graph
Laplacian.  The matrices follow the problem statements of the torch-sla paper
(§4, Figure 2: "five-point stencil and homogeneous Dirichlet boundary", the
N = n_grid^2 interior-unknown convention) and the learned-SPAI page (graph
Laplacians of point clouds as SPD systems).

Conventions
-----------
* Unknowns are the interior grid points, numbered lexicographically
  i = ix + N*iy (+ N*N*iz).  Neighbours outside the grid are dropped
  (homogeneous Dirichlet).
* The constant-coefficient stencil is unscaled: diagonal 2d, off-diagonals -1.
* Variable coefficients live on cells; the coefficient of the face between
  cells i and j is the harmonic mean 2 k_i k_j / (k_i + k_j).  A face on the
  Dirichlet boundary takes k_i (the harmonic mean of k_i with itself).  Row i
  holds A_ii = sum of its four face coefficients and A_ij = -k_face.  With
  k == 1 this is exactly the constant-coefficient matrix.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class CSR:
    n: int
    row_ptr: np.ndarray          # int32 [n + 1]
    col_idx: np.ndarray          # int32 [nnz]
    vals: np.ndarray             # float64 or float32, [nnz] or [batch, nnz]
    meta: dict = field(default_factory=dict)

    @property
    def nnz(self) -> int:
        return int(self.row_ptr[-1])

    @property
    def batch(self) -> int:
        return 1 if self.vals.ndim == 1 else int(self.vals.shape[0])

    def rows(self) -> np.ndarray:
        """Row index of every stored entry (int64 [nnz])."""
        return np.repeat(np.arange(self.n, dtype=np.int64), np.diff(self.row_ptr))

    def dense(self, system: int = 0) -> np.ndarray:
        v = self.vals if self.vals.ndim == 1 else self.vals[system]
        d = np.zeros((self.n, self.n), dtype=np.float64)
        d[self.rows(), self.col_idx.astype(np.int64)] = v
        return d


def _from_masked_stencil(n: int, cols: np.ndarray, vals: np.ndarray,
                         valid: np.ndarray) -> tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Rows are the first axis of (n, s) arrays whose columns are already in
    ascending column order; keep the valid entries in row-major order."""
    counts = valid.sum(axis=1)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    col_idx = cols[valid].astype(np.int32)
    v = vals[..., valid] if vals.ndim == 3 else vals[valid]
    return row_ptr.astype(np.int32), col_idx, v


def _grid_offsets(dims: tuple[int, ...]) -> list[tuple[int, int]]:
    """(axis, +-1) neighbour offsets sorted by the resulting column offset."""
    strides = [int(np.prod(dims[:a])) for a in range(len(dims))]
    offs = []
    for a in range(len(dims)):
        offs.append((strides[a], a, -1))
        offs.append((strides[a], a, +1))
    offs.sort(key=lambda t: t[0] * t[2])
    return [(a, s) for (_, a, s) in offs]


def poisson_grid(dims: tuple[int, ...]) -> CSR:
    """Constant-coefficient (2d+1)-point Dirichlet Laplacian on an interior grid."""
    d = len(dims)
    n = int(np.prod(dims))
    idx = np.arange(n, dtype=np.int64)
    coords = np.unravel_index(idx, dims[::-1])[::-1]   # coords[a] = index along axis a
    strides = [int(np.prod(dims[:a])) for a in range(d)]
    offs = _grid_offsets(dims)
    lower = [(a, s) for (a, s) in offs if s * strides[a] < 0]
    upper = [(a, s) for (a, s) in offs if s * strides[a] > 0]
    cols, vals, valid = [], [], []
    for (a, s) in lower:
        cols.append(idx + s * strides[a]); vals.append(np.full(n, -1.0))
        valid.append(coords[a] + s >= 0)
    cols.append(idx); vals.append(np.full(n, 2.0 * d)); valid.append(np.ones(n, bool))
    for (a, s) in upper:
        cols.append(idx + s * strides[a]); vals.append(np.full(n, -1.0))
        valid.append(coords[a] + s < dims[a])
    rp, ci, v = _from_masked_stencil(n, np.stack(cols, 1), np.stack(vals, 1), np.stack(valid, 1))
    return CSR(n, rp, ci, v, meta={"kind": "poisson", "dims": tuple(dims)})


def diffusion2d(N: int, k_cell: np.ndarray) -> CSR:
    """Variable-coefficient five-point diffusion on an N x N interior grid.

    k_cell has shape [N*N] (one system) or [batch, N*N] (one coefficient field
    per system, all on the same pattern)."""
    k = np.atleast_2d(np.asarray(k_cell, dtype=np.float64))
    B, n = k.shape
    assert n == N * N
    idx = np.arange(n, dtype=np.int64)
    ix, iy = idx % N, idx // N

    def face(j_idx, ok):
        kj = k[:, np.where(ok, j_idx, idx)]
        interior = 2.0 * k * kj / (k + kj)
        return np.where(ok[None, :], interior, k)   # boundary face: k_i

    nb = [(-N, iy > 0), (-1, ix > 0), (1, ix < N - 1), (N, iy < N - 1)]
    faces = [face(idx + o, ok) for (o, ok) in nb]
    diag = faces[0] + faces[1] + faces[2] + faces[3]
    cols = np.stack([idx - N, idx - 1, idx, idx + 1, idx + N], 1)
    valid = np.stack([nb[0][1], nb[1][1], np.ones(n, bool), nb[2][1], nb[3][1]], 1)
    vals = np.stack([-faces[0], -faces[1], diag, -faces[2], -faces[3]], 2)  # [B, n, 5]
    counts = valid.sum(axis=1)
    row_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=row_ptr[1:])
    col_idx = cols[valid].astype(np.int32)
    v = np.ascontiguousarray(vals[:, valid])        # [B, nnz], row-major order
    if np.asarray(k_cell).ndim == 1:
        v = np.ascontiguousarray(v[0])
    return CSR(n, row_ptr.astype(np.int32), col_idx, v,
               meta={"kind": "diffusion2d", "dims": (N, N)})


def knn_graph_laplacian(points: np.ndarray, k: int, shift: float, workers: int = -1) -> CSR:
    """A = L + shift*I for the weighted kNN graph of a point cloud.

    Edges: the union of the directed k-nearest-neighbour relations (self
    excluded), so the pattern is symmetric.  h = mean of the n*k directed
    neighbour distances; w_ij = exp(-d_ij^2 / h^2); L = D_w - W."""
    from scipy.spatial import cKDTree

    n = points.shape[0]
    tree = cKDTree(points)
    dist, nbr = tree.query(points, k=k + 1, workers=workers)
    # drop self (column 0 holds the point itself for distinct points)
    self_first = nbr[:, 0] == np.arange(n)
    if not self_first.all():
        raise ValueError("duplicate points in the cloud")
    dist, nbr = dist[:, 1:], nbr[:, 1:]
    h = float(dist.mean())
    src = np.repeat(np.arange(n, dtype=np.int64), k)
    dst = nbr.reshape(-1).astype(np.int64)
    # undirected edge keys min*n + max, deduplicated by sort + adjacent compare
    key = np.sort(np.minimum(src, dst) * n + np.maximum(src, dst))
    keep = np.ones(key.shape[0], dtype=bool)
    keep[1:] = key[1:] != key[:-1]
    key = key[keep]
    a, b = key // n, key % n
    # both orientations, sorted by (row, col)
    both = np.sort(np.concatenate([a * n + b, b * n + a]))
    rows, cols = both // n, both % n
    diff = points[rows] - points[cols]
    d2 = diff[:, 0] * diff[:, 0] + diff[:, 1] * diff[:, 1] + diff[:, 2] * diff[:, 2]
    w = np.exp(-d2 / (h * h))
    counts = np.bincount(rows, minlength=n)
    off_ptr = np.zeros(n + 1, dtype=np.int64)
    np.cumsum(counts, out=off_ptr[1:])
    wsum = np.add.reduceat(w, off_ptr[:-1]) if len(w) else np.zeros(n)
    wsum[counts == 0] = 0.0
    diag = wsum + shift
    # insert the diagonal at its sorted position in each row
    n_lower = np.bincount(rows[cols < rows], minlength=n)
    row_ptr = off_ptr + np.arange(n + 1, dtype=np.int64)
    nnz = int(row_ptr[-1])
    col_idx = np.empty(nnz, dtype=np.int64)
    vals = np.empty(nnz, dtype=np.float64)
    diag_pos = row_ptr[:-1] + n_lower
    is_diag = np.zeros(nnz, dtype=bool)
    is_diag[diag_pos] = True
    col_idx[is_diag] = np.arange(n)
    vals[is_diag] = diag
    col_idx[~is_diag] = cols
    vals[~is_diag] = -w
    return CSR(n, row_ptr.astype(np.int32), col_idx.astype(np.int32), vals,
               meta={"kind": "knn", "k": k, "h": h, "shift": shift})


def convection_diffusion(dims: tuple[int, ...], wind) -> CSR:
    """Nonsymmetric (2d+1)-point convection-diffusion operator on an interior
    grid: the unscaled Dirichlet Laplacian plus first-order upwind convection.

    wind[a] is the scaled velocity h * beta_a along axis a, a scalar or an
    array [n] (one value per unknown).  Along axis a the upwind neighbour
    (the one at -1 for wind >= 0, at +1 for wind < 0) gets -1 - |wind_a|, the
    other neighbour -1, and the diagonal 2d + sum_a |wind_a|.  Rows are
    weakly diagonally dominant with strict dominance next to the boundary,
    so A is a nonsingular M-matrix; wind = 0 gives poisson_grid exactly."""
    d = len(dims)
    n = int(np.prod(dims))
    idx = np.arange(n, dtype=np.int64)
    coords = np.unravel_index(idx, dims[::-1])[::-1]
    strides = [int(np.prod(dims[:a])) for a in range(d)]
    w = [np.broadcast_to(np.asarray(wind[a], dtype=np.float64), (n,)) for a in range(d)]
    offs = _grid_offsets(dims)
    cols, vals, valid = [], [], []

    def entry(a, s):
        upwind = np.where(w[a] >= 0.0, s < 0, s > 0)
        return np.where(upwind, -1.0 - np.abs(w[a]), -1.0)

    lower = [(a, s) for (a, s) in offs if s * strides[a] < 0]
    upper = [(a, s) for (a, s) in offs if s * strides[a] > 0]
    for (a, s) in lower:
        cols.append(idx + s * strides[a]); vals.append(entry(a, s)); valid.append(coords[a] + s >= 0)
    cols.append(idx); vals.append(2.0 * d + sum(np.abs(wa) for wa in w)); valid.append(np.ones(n, bool))
    for (a, s) in upper:
        cols.append(idx + s * strides[a]); vals.append(entry(a, s)); valid.append(coords[a] + s < dims[a])
    rp, ci, v = _from_masked_stencil(n, np.stack(cols, 1), np.stack(vals, 1), np.stack(valid, 1))
    return CSR(n, rp, ci, np.ascontiguousarray(v), meta={"kind": "convdiff", "dims": tuple(dims)})


def rotating_wind(dims: tuple[int, int], peclet: float) -> tuple[np.ndarray, np.ndarray]:
    """Scaled velocity (h beta_x, h beta_y) of the solid-body rotation about
    the centre of an N x M grid, |h beta| up to `peclet` at the corners' mid
    edges: beta = (-(y - 1/2), x - 1/2) * 2 peclet."""
    Nx, Ny = dims
    n = Nx * Ny
    idx = np.arange(n, dtype=np.int64)
    x = (idx % Nx + 1.0) / (Nx + 1.0)
    y = (idx // Nx + 1.0) / (Ny + 1.0)
    return -(y - 0.5) * 2.0 * peclet, (x - 0.5) * 2.0 * peclet
