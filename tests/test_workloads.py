"""Pins on the seeded input generators (no GPU)."""
import numpy as np
import pytest

from workloads import build, rng
from workloads.matrices import diffusion2d, poisson_grid


def _symmetric(A, system=0):
    v = A.vals if A.vals.ndim == 1 else A.vals[system]
    rows = A.rows()
    cols = A.col_idx.astype(np.int64)
    fwd = dict(zip(zip(rows.tolist(), cols.tolist()), v.tolist()))
    return all(fwd.get((j, i)) == val for (i, j), val in fwd.items())


def _sorted_cols(A):
    for i in range(A.n):
        c = A.col_idx[A.row_ptr[i]:A.row_ptr[i + 1]]
        if np.any(np.diff(c) <= 0):
            return False
    return True


def test_splitmix64_known_values():
    # SplitMix64 with state 0: the first outputs of the reference generator
    # (Steele, Lea, Flood 2014) are 0xE220A8397B1DCDAF, 0x6E789E6AA1B965F4.
    z = np.array([0x9E3779B97F4A7C15, 0x3C6EF372FE94F82A], dtype=np.uint64)
    out = rng._mix(z)
    assert int(out[0]) == 0xE220A8397B1DCDAF
    assert int(out[1]) == 0x6E789E6AA1B965F4


def test_rng_is_counter_based_and_in_range():
    a = rng.uniform(7, 1, 1000)
    b = rng.uniform(7, 1, 500, offset=500)
    assert np.array_equal(a[500:], b)
    assert a.min() >= 0.0 and a.max() < 1.0
    n = rng.normal(7, 2, 200000)
    assert abs(n.mean()) < 0.01 and abs(n.std() - 1.0) < 0.01
    p = rng.permutation(7, 4, 1000)
    assert np.array_equal(np.sort(p), np.arange(1000))


@pytest.mark.parametrize("dims,nnz", [((64, 64), 20224), ((1024, 1024), 5238784),
                                      ((256, 256), 326656), ((128, 128, 128), 14581760)])
def test_grid_nnz_counts(dims, nnz):
    # interior (2d+1)-point stencil: nnz = (2d+1) n - 2 * (boundary faces)
    A = poisson_grid(dims)
    assert A.nnz == nnz
    assert A.row_ptr.dtype == np.int32 and A.col_idx.dtype == np.int32


def test_poisson_structure_small():
    for dims in [(7,), (5, 6), (3, 4, 5)]:
        A = poisson_grid(dims)
        assert _symmetric(A) and _sorted_cols(A)
        D = A.dense()
        assert np.all(np.diag(D) == 2 * len(dims))
        assert np.all(np.linalg.eigvalsh(D) > 0)


def test_diffusion_reduces_to_poisson_at_unit_coefficient():
    A1 = diffusion2d(9, np.ones(81))
    A0 = poisson_grid((9, 9))
    assert np.array_equal(A1.row_ptr, A0.row_ptr)
    assert np.array_equal(A1.col_idx, A0.col_idx)
    assert np.array_equal(A1.vals, A0.vals)


def test_diffusion_harmonic_faces():
    k = np.array([1.0, 3.0, 1.0, 1.0])  # 2x2 grid, cells 0..3
    A = diffusion2d(2, k)
    D = A.dense()
    # face between cells 0 and 1: 2*1*3/(1+3) = 1.5
    assert D[0, 1] == -1.5 and D[1, 0] == -1.5
    # cell 1 diagonal: faces to 0 (1.5), to 3 (2*3*1/4 = 1.5), two boundary faces k=3
    assert D[1, 1] == 1.5 + 1.5 + 3.0 + 3.0
    assert _symmetric(A)


def test_workload_c3_batch_pattern_shared():
    w = build("c3", N=16, batch=3)
    assert w.A.vals.shape == (3, w.A.nnz) and w.A.vals.dtype == np.float32
    assert w.b.shape == (3, 256) and w.b.dtype == np.float32
    for s in range(3):
        assert _symmetric(w.A, s)


def test_knn_laplacian_small():
    w = build("c5", npoints=3000)
    A = w.A
    assert _symmetric(A) and _sorted_cols(A)
    lens = np.diff(A.row_ptr)
    assert lens.min() >= 13          # 12 neighbours + diagonal at least
    D = A.dense()
    off = D - np.diag(np.diag(D))
    # L + 1e-3 I: diagonal = sum of weights + shift, off-diagonals negative
    assert np.all(off <= 0)
    np.testing.assert_allclose(np.diag(D), -off.sum(axis=1) + 1e-3, rtol=1e-13)
    assert np.linalg.eigvalsh(D).min() > 0


# ---------------------------------------------------------------- convection-diffusion (BiCGStab inputs)
def test_convection_diffusion_reduces_to_poisson_without_wind():
    from workloads.matrices import convection_diffusion
    for dims in ((7, 5), (4, 3, 5)):
        A = convection_diffusion(dims, (0.0,) * len(dims))
        P = poisson_grid(dims)
        assert np.array_equal(A.row_ptr, P.row_ptr) and np.array_equal(A.col_idx, P.col_idx)
        assert np.array_equal(A.vals, P.vals)


def test_convection_diffusion_upwinding():
    """Constant wind (+w along x, -u along y): the upstream neighbour gets
    -1 - |wind|, the downstream one -1, the diagonal 2d + sum |wind|; rows
    away from the boundary sum to zero and the matrix is nonsymmetric."""
    from workloads.matrices import convection_diffusion
    N, w, u = 6, 0.75, 0.4
    A = convection_diffusion((N, N), (w, -u))
    D = A.dense()
    i = 2 + N * 2                               # interior unknown (x = 2, y = 2)
    assert D[i, i] == 4.0 + w + u
    assert D[i, i - 1] == -1.0 - w and D[i, i + 1] == -1.0    # x: wind from -x
    assert D[i, i + N] == -1.0 - u and D[i, i - N] == -1.0    # y: wind from +y
    interior = [x + N * y for y in range(1, N - 1) for x in range(1, N - 1)]
    assert np.allclose(D[interior].sum(axis=1), 0.0)
    assert np.all(D.sum(axis=1) >= -1e-15)                   # weakly diagonally dominant rows
    assert np.abs(D - D.T).max() > 0.1


def test_workload_cd3_recipe():
    from workloads import build
    w = build("cd3", N=10)
    n = 1000
    assert w.A.n == n and w.A.nnz == 7 * n - 6 * 100       # 7-point pattern, Dirichlet faces dropped
    assert w.pc == "jacobi" and w.tol == 1e-8 and w.info["method"] == "bicgstab"
    w2 = build("cd3", N=10)
    assert np.array_equal(w.A.vals, w2.A.vals) and np.array_equal(w.b, w2.b)   # seeded
    D = w.A.dense()
    assert np.all(np.diag(D) > 0) and np.abs(D - D.T).max() > 0.1
