"""The five synthetic workloads (and scaled-down versions of each).

Each workload is a CSR matrix plus right-hand side(s) and, where a backward
pass is timed, an upstream gradient g.  Seeds: workload c uses seed 1000 + c.
Streams: 1 = b (or the manufactured x*), 2 = cell coefficients, 3 = points,
4 = relabelling permutation, 5 = upstream gradient g.

  c1  2D 5-point Poisson, 64 x 64 interior grid, fp64; x* ~ U(-1,1), b = A x*;
      plain CG to relative residual 1e-10.
  c2  2D 5-point variable-coefficient diffusion, 1024 x 1024; k = exp(N(0,1))
      per cell; b ~ N(0,1); fp64 Jacobi-PCG to 1e-8.
  c3  64 systems on one 256 x 256 pattern; per-system k = exp(0.5 N(0,1));
      fp32 values; b ~ U(-1,1); Jacobi-PCG to 1e-5 per system.
  c4  3D 7-point Poisson, 128^3, fp64; b ~ N(0,1); CG to 1e-8, then the
      adjoint with g ~ N(0,1).
  c5  kNN graph Laplacian of 4M uniform points in the unit cube, k = 12,
      union-symmetrised, weights exp(-d^2/h^2), A = L + 1e-3 I, points relabelled
      by a seeded permutation, fp64; b ~ N(0,1); factored-SPAI PCG
      (M^-1 = G G^T + 1e-3 I) to 1e-8.
  cd3 3D upwind convection-diffusion, 128^3, fp64 (nonsymmetric): the 7-point
      Laplacian plus first-order upwind convection by a solid-body rotation
      about the z axis (scaled speed up to 2 at the side midpoints) and a
      constant 0.5 along z; b ~ N(0,1); Jacobi-BiCGStab to 1e-8, then the
      adjoint (A^T lambda = g) with g ~ N(0,1).  Seed 1006.

`scale` shrinks a workload for tests the oracle finishes in seconds: the grid
side (or point count) is replaced while the recipe is kept.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import rng
from .matrices import CSR, convection_diffusion, diffusion2d, knn_graph_laplacian, poisson_grid


@dataclass
class Workload:
    name: str
    A: CSR
    b: np.ndarray                 # [n] or [batch, n], same dtype as A.vals
    dtype: str                    # "f64" | "f32"
    pc: str                       # "none" | "jacobi" | "spai"
    tol: float
    eps: float = 0.0
    g: np.ndarray | None = None   # upstream gradient for the adjoint
    x_star: np.ndarray | None = None
    info: dict = field(default_factory=dict)


def c1(N: int = 64) -> Workload:
    seed = 1001
    A = poisson_grid((N, N))
    x_star = rng.uniform_pm1(seed, 1, A.n)
    b = _csr_matvec_f64(A, x_star)
    g = rng.normal(seed, 5, A.n)
    return Workload("c1", A, b, "f64", "none", 1e-10, g=g, x_star=x_star,
                    info={"grid": (N, N)})


def c2(N: int = 1024) -> Workload:
    seed = 1002
    n = N * N
    kc = np.exp(rng.normal(seed, 2, n))
    A = diffusion2d(N, kc)
    b = rng.normal(seed, 1, n)
    g = rng.normal(seed, 5, n)
    return Workload("c2", A, b, "f64", "jacobi", 1e-8, g=g, info={"grid": (N, N)})


def c3(N: int = 256, batch: int = 64) -> Workload:
    seed = 1003
    n = N * N
    kc = np.exp(0.5 * rng.normal(seed, 2, batch * n)).reshape(batch, n)
    A = diffusion2d(N, kc)
    A.vals = np.ascontiguousarray(A.vals, dtype=np.float32)
    b = rng.uniform_pm1(seed, 1, batch * n).reshape(batch, n).astype(np.float32)
    g = rng.normal(seed, 5, batch * n).reshape(batch, n).astype(np.float32)
    return Workload("c3", A, b, "f32", "jacobi", 1e-5, g=g,
                    info={"grid": (N, N), "batch": batch})


def c4(N: int = 128) -> Workload:
    seed = 1004
    A = poisson_grid((N, N, N))
    b = rng.normal(seed, 1, A.n)
    g = rng.normal(seed, 5, A.n)
    return Workload("c4", A, b, "f64", "none", 1e-8, g=g, info={"grid": (N, N, N)})


def c5(npoints: int = 4 * 1024 * 1024, k: int = 12) -> Workload:
    seed = 1005
    u = rng.uniform(seed, 3, 3 * npoints).reshape(npoints, 3)
    perm = rng.permutation(seed, 4, npoints)
    pts = np.ascontiguousarray(u[perm])
    A = knn_graph_laplacian(pts, k, 1e-3)
    b = rng.normal(seed, 1, A.n)
    g = rng.normal(seed, 5, A.n)
    return Workload("c5", A, b, "f64", "spai", 1e-8, eps=1e-3, g=g,
                    info={"points": npoints, "k": k})


def cd3(N: int = 128, peclet: float = 2.0) -> Workload:
    seed = 1006
    n = N * N * N
    idx = np.arange(n, dtype=np.int64)
    x = (idx % N + 1.0) / (N + 1.0)
    y = ((idx // N) % N + 1.0) / (N + 1.0)
    wind = (-(y - 0.5) * 2.0 * peclet, (x - 0.5) * 2.0 * peclet, 0.5)
    A = convection_diffusion((N, N, N), wind)
    b = rng.normal(seed, 1, n)
    g = rng.normal(seed, 5, n)
    return Workload("cd3", A, b, "f64", "jacobi", 1e-8, g=g,
                    info={"grid": (N, N, N), "peclet": peclet, "method": "bicgstab"})


def _csr_matvec_f64(A: CSR, x: np.ndarray) -> np.ndarray:
    """b = A x*, used only to manufacture the right-hand side of c1.  Summed
    with numpy (np.add.reduceat), which is neither the oracle nor the GPU code."""
    prod = A.vals * x[A.col_idx]
    return np.add.reduceat(prod, A.row_ptr[:-1].astype(np.int64))


BUILDERS = {"c1": c1, "c2": c2, "c3": c3, "c4": c4, "c5": c5, "cd3": cd3}

# Full sizes of each workload (the shapes the benchmark and the
# full-size parity tests use) and small shapes the oracle solves in seconds.
FULL = {"c1": {}, "c2": {}, "c3": {}, "c4": {}, "c5": {}, "cd3": {}}
SMALL = {"c1": {"N": 64}, "c2": {"N": 96}, "c3": {"N": 48, "batch": 5},
         "c4": {"N": 24}, "c5": {"npoints": 20000}, "cd3": {"N": 24}}


def build(name: str, **kw) -> Workload:
    return BUILDERS[name](**kw)
