"""Pins of the fp64 BiCGStab oracle and its general (transpose) adjoint
against facts fixed outside it: dense LU solves of nonsymmetric systems,
manufactured solutions, the two defining conditions of one BiCGStab step
(the Petrov-Galerkin condition that fixes alpha and the local residual
minimisation that fixes omega), exact one-step convergence on diagonal
systems, finite differences of the loss and the adjoint identities.  No GPU."""
import numpy as np
import pytest
import scipy.linalg

import oracle
from workloads import rng
from workloads.matrices import CSR, convection_diffusion, poisson_grid, rotating_wind


def _csr(D):
    n = D.shape[0]
    rows, cols = np.nonzero(D)
    rp = np.zeros(n + 1, np.int32)
    np.cumsum(np.bincount(rows, minlength=n), out=rp[1:])
    return CSR(n, rp, cols.astype(np.int32), D[rows, cols].astype(np.float64))


def _systems():
    yield "constant wind 2d", convection_diffusion((7, 6), (0.8, -0.4))
    yield "rotating wind 2d", convection_diffusion((9, 8), rotating_wind((9, 8), 3.0))
    yield "strong wind 3d", convection_diffusion((4, 5, 3), (2.5, 0.0, -1.5))


SYSTEMS = list(_systems())


def _rhs(n, stream):
    return rng.normal(11, stream, n)


@pytest.mark.parametrize("pc", ["none", "jacobi"])
@pytest.mark.parametrize("name,A", SYSTEMS, ids=[s[0] for s in SYSTEMS])
def test_matches_dense_lu(name, A, pc):
    D = A.dense()
    assert np.abs(D - D.T).max() > 0.1          # genuinely nonsymmetric
    b = _rhs(A.n, 1)
    xs = scipy.linalg.lu_solve(scipy.linalg.lu_factor(D), b)
    tol = 1e-12
    x, info = oracle.bicgstab(A, b, tol, pc=pc)
    assert info["status"] == "ok"
    assert info["rel_res_true"] <= tol
    kappa = np.linalg.cond(D)
    assert np.linalg.norm(x - xs) / np.linalg.norm(xs) <= 2 * kappa * tol
    # the product of the method is independent of M up to the tolerance
    x2, _ = oracle.bicgstab(A, b, tol, pc="jacobi" if pc == "none" else "none")
    assert np.linalg.norm(x - x2) / np.linalg.norm(xs) <= 4 * kappa * tol


def test_manufactured_solution():
    A = convection_diffusion((12, 10), rotating_wind((12, 10), 5.0))
    xs = rng.uniform_pm1(3, 0, A.n)
    b = A.dense() @ xs
    x, info = oracle.bicgstab(A, b, 1e-13, pc="jacobi")
    assert info["status"] == "ok"
    assert np.abs(x - xs).max() <= 1e-10
    # a warm start at the solution stops before the first product
    x0, info0 = oracle.bicgstab(A, b, 1e-10, pc="jacobi", x0=x)
    assert info0["iters"] == 0 and np.array_equal(x0, x)


@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_first_step_satisfies_its_defining_conditions(pc):
    """After one step x1 = x0 + alpha p^ + omega s^ with p^ = M^-1 r0,
    s = r0 - alpha A p^, s^ = M^-1 s: alpha makes s orthogonal to the shadow
    residual r^ = r0, and omega minimises ||s - omega A s^|| (a 1-column
    least-squares problem, solved here by LAPACK)."""
    A = convection_diffusion((6, 5), (1.2, 0.6))
    D = A.dense()
    b = _rhs(A.n, 2)
    Minv = np.diag(1.0 / np.diag(D)) if pc == "jacobi" else np.eye(A.n)
    ph = Minv @ b
    Ap = D @ ph
    alpha = np.linalg.solve(np.array([[b @ Ap]]), np.array([b @ b]))[0]   # r^ . s = 0
    s = b - alpha * Ap
    sh = Minv @ s
    omega = np.linalg.lstsq((D @ sh)[:, None], s, rcond=None)[0][0]
    x_expect = alpha * ph + omega * sh
    x1, info = oracle.bicgstab(A, b, 1e-14, max_iter=1, pc=pc)
    assert info["status"] == "not_converged" and info["iters"] == 1
    np.testing.assert_allclose(x1, x_expect, rtol=1e-12, atol=1e-14 * np.abs(x_expect).max())
    # the recursive residual after the step is the true one
    assert abs(info["rel_res_recursive"] - info["rel_res_true"]) <= 1e-12


def test_diagonal_system_converges_in_one_step_with_jacobi():
    d = 1.0 + rng.uniform(5, 0, 40) * 9.0
    A = _csr(np.diag(d))
    b = _rhs(40, 3)
    x, info = oracle.bicgstab(A, b, 1e-14, pc="jacobi")
    assert info["status"] == "ok" and info["iters"] == 1
    np.testing.assert_allclose(x, b / d, rtol=1e-15)


def test_spd_system_matches_cg_solution():
    A = poisson_grid((9, 7))
    b = _rhs(A.n, 4)
    xb, ib = oracle.bicgstab(A, b, 1e-12, pc="jacobi")
    xc, ic = oracle.pcg(A, b, 1e-12, pc="jacobi")
    assert ib["status"] == ic["status"] == "ok"
    assert np.linalg.norm(xb - xc) / np.linalg.norm(xc) <= 1e-9


def test_status_codes():
    A = convection_diffusion((5, 5), (0.5, 0.5))
    b = _rhs(A.n, 5)
    x, info = oracle.bicgstab(A, np.zeros(A.n), 1e-10)
    assert info["status"] == "ok" and info["iters"] == 0 and not x.any()
    _, info = oracle.bicgstab(A, b, 1e-10, max_iter=0)
    assert info["status"] == "not_converged" and info["iters"] == 0
    _, info = oracle.bicgstab(A, b, 1e-14, max_iter=3)
    assert info["status"] == "not_converged" and info["iters"] == 3
    # r^ . A r0 = 0 on the first step: a rotation by 90 degrees
    R = _csr(np.array([[0.0, 1.0], [-1.0, 0.0]]))
    _, info = oracle.bicgstab(R, np.array([1.0, 0.0]), 1e-10)
    assert info["status"] == "breakdown"
    # Jacobi needs every diagonal entry stored
    _, info = oracle.bicgstab(R, np.array([1.0, 0.0]), 1e-10, pc="jacobi")
    assert info["status"] == "invalid"
    with pytest.raises(ValueError):
        oracle.bicgstab(A, b, 1e-10, pc="spai")


def _loss_grad(D, b, c):
    """L(x) = c . x + 0.5 ||x||^2 at x = D^-1 b; returns (L, dL/dx)."""
    x = scipy.linalg.lu_solve(scipy.linalg.lu_factor(D), b)
    return c @ x + 0.5 * x @ x, c + x


@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_adjoint_matches_finite_differences(pc):
    A = convection_diffusion((5, 4), (1.5, -0.7))
    D = A.dense()
    b = _rhs(A.n, 6)
    c = _rhs(A.n, 7)
    x, _ = oracle.bicgstab(A, b, 1e-14, pc=pc)
    _, g = _loss_grad(D, b, c)
    dldb, dlda, info = oracle.bicgstab_adjoint(A, x, g, 1e-14, pc=pc)
    assert info["status"] == "ok"
    # the adjoint solves the transposed system, not A itself
    lam = scipy.linalg.lu_solve(scipy.linalg.lu_factor(D.T), g)
    np.testing.assert_allclose(dldb, lam, rtol=1e-9, atol=1e-12)
    assert np.abs(lam - scipy.linalg.lu_solve(scipy.linalg.lu_factor(D), g)).max() > 1e-3
    h = 1e-6
    for i in range(A.n):
        e = np.zeros(A.n); e[i] = h
        fd = (_loss_grad(D, b + e, c)[0] - _loss_grad(D, b - e, c)[0]) / (2 * h)
        assert abs(fd - dldb[i]) <= 1e-7 * max(1.0, abs(fd))
    rows = A.rows()
    for k in range(A.nnz):
        E = np.zeros_like(D); E[rows[k], A.col_idx[k]] = h
        fd = (_loss_grad(D + E, b, c)[0] - _loss_grad(D - E, b, c)[0]) / (2 * h)
        assert abs(fd - dlda[k]) <= 1e-7 * max(1.0, abs(fd))


def test_adjoint_identities():
    A = convection_diffusion((10, 9), rotating_wind((10, 9), 4.0))
    b = _rhs(A.n, 8)
    g = _rhs(A.n, 9)
    tol = 1e-13
    x, _ = oracle.bicgstab(A, b, tol, pc="jacobi")
    dldb, dlda, info = oracle.bicgstab_adjoint(A, x, g, tol, pc="jacobi")
    assert info["status"] == "ok" and info["rel_res_true"] <= tol
    scale = np.linalg.norm(g) * np.linalg.norm(x)
    assert abs(g @ x - dldb @ b) <= 1e-9 * scale                  # g^T x = lambda^T b
    assert abs((A.vals * dlda).sum() + g @ x) <= 1e-9 * scale     # sum A . dL/dA = -g^T x



def test_three_distinct_eigenvalues_terminate_in_three_steps():
    """For a diagonalisable A with m distinct eigenvalues the BiCG residual
    polynomial annihilates r0 after m steps, so BiCGStab (whose residual is
    that polynomial times the stabilising one) is at the rounding level after
    m = 3 iterations.  Pins the recurrence for p (beta and the omega term):
    any other combination loses the bi-orthogonality this rests on."""
    n = 30
    S = np.eye(n) + 0.3 * rng.uniform_pm1(13, 0, n * n).reshape(n, n) / np.sqrt(n)
    lam = np.array([1.0, 2.0, 5.0])[np.arange(n) % 3]
    T = S @ np.diag(lam) @ np.linalg.inv(S)
    A = _csr(T)
    b = _rhs(n, 10)
    x, info = oracle.bicgstab(A, b, 1e-11)
    assert info["status"] == "ok" and info["iters"] <= 3
    xs = np.linalg.solve(T, b)
    assert np.linalg.norm(x - xs) / np.linalg.norm(xs) <= 1e-9


def test_batched_systems_are_solved_independently():
    """A batch on one pattern (values [batch][nnz]) gives each system's own
    solution, as the single-system calls do."""
    dims = (6, 5)
    mats = [convection_diffusion(dims, w) for w in ((0.5, 0.2), (-1.0, 0.7), rotating_wind(dims, 2.0))]
    A = CSR(mats[0].n, mats[0].row_ptr, mats[0].col_idx, np.stack([m.vals for m in mats]))
    b = np.stack([_rhs(A.n, 20 + s) for s in range(3)])
    x, infos = oracle.bicgstab(A, b, 1e-12, pc="jacobi")
    for s, M in enumerate(mats):
        xs, inf = oracle.bicgstab(M, b[s], 1e-12, pc="jacobi")
        assert np.array_equal(x[s], xs) and infos[s] == inf
        assert np.linalg.norm(M.dense() @ x[s] - b[s]) <= 1e-11 * np.linalg.norm(b[s])
