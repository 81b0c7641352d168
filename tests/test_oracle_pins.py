"""Pins of the fp64 CPU oracle against facts fixed outside it: closed-form
eigenpairs of the Dirichlet Laplacian, dense LU, manufactured solutions, exact
CG termination on few-eigenvalue right-hand sides, the classical CG iteration
bound, a hand-derived preconditioner example, finite differences and the
adjoint identities.  No GPU."""
import math
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.linalg

import oracle
from workloads import build
from workloads.matrices import CSR, diffusion2d, poisson_grid

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ---------------------------------------------------------------- helpers
def laplacian_eig(dims, modes):
    """Closed-form eigenpair of the unscaled Dirichlet Laplacian on an interior
    grid: v(i) = prod_a sin(j_a pi (i_a+1)/(N_a+1)),
    lambda = sum_a 4 sin^2(j_a pi / (2 (N_a+1)))."""
    n = int(np.prod(dims))
    idx = np.arange(n)
    coords = np.unravel_index(idx, dims[::-1])[::-1]
    v = np.ones(n)
    lam = 0.0
    for a, (N, j) in enumerate(zip(dims, modes)):
        m = (j * (coords[a] + 1)) % (2 * (N + 1))       # exact integer argument reduction
        v *= np.sin(np.pi * m / (N + 1))
        lam += 4.0 * np.sin(j * np.pi / (2 * (N + 1))) ** 2
    return v, lam


def dense_solve(A, b, system=0):
    D = A.dense(system)
    lu = scipy.linalg.lu_factor(D)
    return scipy.linalg.lu_solve(lu, b)


def cond2(A, system=0):
    ev = np.linalg.eigvalsh(A.dense(system))
    return ev[-1] / ev[0]


def random_csr(n, density, rng_, sym=False, spd=False):
    D = (rng_.random((n, n)) < density) * rng_.standard_normal((n, n))
    if sym or spd:
        D = np.triu(D) + np.triu(D, 1).T
    if spd:
        D = D - np.diag(np.diag(D))
        D = D + np.diag(np.abs(D).sum(1) + 1.0)
    rows, cols = np.nonzero(D)
    rp = np.zeros(n + 1, dtype=np.int32)
    np.cumsum(np.bincount(rows, minlength=n), out=rp[1:])
    return CSR(n, rp, cols.astype(np.int32), D[rows, cols].astype(np.float64))


# ---------------------------------------------------------------- SpMV
@pytest.mark.parametrize("dims,modes", [((17,), (3,)), ((12, 9), (2, 5)), ((6, 7, 5), (1, 3, 2)),
                                        ((64, 64), (1, 1)), ((64, 64), (64, 64))])
def test_spmv_laplacian_eigenvectors(dims, modes):
    A = poisson_grid(dims)
    v, lam = laplacian_eig(dims, modes)
    y = oracle.spmv(A, v)
    # rounding bound of a row sum: a few ulps of ||A||_inf * max|v| (= 4d max|v|)
    atol = 8 * np.finfo(float).eps * 4 * len(dims) * np.abs(v).max()
    np.testing.assert_allclose(y, lam * v, rtol=0, atol=atol)
    # and the eigenvalue is recovered to that same precision
    assert abs((v @ y) / (v @ v) - lam) <= atol


def test_spmv_brute_force_dense():
    g = np.random.default_rng(0)
    for n in (1, 2, 7, 40):
        A = random_csr(n, 0.3, g)
        x = g.standard_normal(n)
        np.testing.assert_allclose(oracle.spmv(A, x), A.dense() @ x, rtol=1e-13, atol=1e-13)


def test_spmv_empty_rows():
    A = CSR(3, np.array([0, 0, 2, 2], np.int32), np.array([0, 2], np.int32), np.array([2.0, -1.0]))
    y = oracle.spmv(A, np.array([1.0, 5.0, 3.0]))
    assert y.tolist() == [0.0, -1.0, 0.0]


# ---------------------------------------------------------------- CG / PCG
@pytest.mark.parametrize("maker,pc", [
    (lambda: poisson_grid((10, 12)), "none"),
    (lambda: poisson_grid((10, 12)), "jacobi"),
    (lambda: build("c2", N=12).A, "jacobi"),
    (lambda: build("c5", npoints=160).A, "spai"),
    (lambda: build("c5", npoints=160).A, "jacobi"),
    (lambda: random_csr(150, 0.05, np.random.default_rng(3), spd=True), "spai"),
])
def test_pcg_matches_dense_lu(maker, pc):
    A = maker()
    b = np.random.default_rng(1).standard_normal(A.n)
    tol = 1e-10
    x, info = oracle.pcg(A, b, tol, pc=pc, eps=1e-3)
    assert info["status"] == "ok"
    assert info["rel_res_true"] <= tol
    x_lu = dense_solve(A, b)
    err = np.linalg.norm(x - x_lu) / np.linalg.norm(x_lu)
    assert err <= cond2(A) * tol


def test_pcg_manufactured_solution_c1():
    w = build("c1")
    x, info = oracle.pcg(w.A, w.b, w.tol, pc=w.pc)
    N = 64
    kappa = 1.0 / math.tan(math.pi / (2 * (N + 1))) ** 2   # closed form lambda_max / lambda_min
    assert abs(kappa - 1711.7) < 0.5
    assert info["status"] == "ok" and info["rel_res_true"] <= w.tol
    err = np.linalg.norm(x - w.x_star) / np.linalg.norm(w.x_star)
    assert err <= kappa * w.tol
    # classical bound: iterations <= ceil(sqrt(kappa)/2 * ln(2/tol))
    assert info["iters"] <= math.ceil(0.5 * math.sqrt(kappa) * math.log(2 / w.tol))


@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_pcg_eigenvector_rhs_one_iteration(pc):
    dims = (64, 64)
    A = poisson_grid(dims)
    v, lam = laplacian_eig(dims, (3, 7))
    x, info = oracle.pcg(A, v, 1e-12, pc=pc)
    assert info["iters"] == 1
    np.testing.assert_allclose(x, v / lam, rtol=0, atol=1e-12 * np.abs(v / lam).max())


def test_pcg_three_eigenvalues_terminates_in_three():
    dims = (30, 30)
    A = poisson_grid(dims)
    b = sum(laplacian_eig(dims, m)[0] for m in [(1, 1), (2, 5), (9, 4)])
    x, info = oracle.pcg(A, b, 1e-11)
    assert info["status"] == "ok" and info["iters"] <= 3


def test_jacobi_on_constant_diagonal_equals_plain_cg():
    w = build("c1")
    x0, i0 = oracle.pcg(w.A, w.b, 1e-10, pc="none")
    x1, i1 = oracle.pcg(w.A, w.b, 1e-10, pc="jacobi")
    assert i0["iters"] == i1["iters"]
    np.testing.assert_allclose(x1, x0, rtol=0, atol=1e-12)


def test_jacobi_is_exact_inverse_on_diagonal_matrix():
    # M^-1 = D^-1 = A^-1 for a diagonal A: one iteration; plain CG needs one
    # iteration per distinct eigenvalue.
    n = 40
    d = np.arange(1, n + 1, dtype=np.float64) ** 1.5
    A = CSR(n, np.arange(n + 1, dtype=np.int32), np.arange(n, dtype=np.int32), d)
    b = np.random.default_rng(6).standard_normal(n)
    x, info = oracle.pcg(A, b, 1e-12, pc="jacobi")
    assert info["iters"] == 1
    np.testing.assert_allclose(x, b / d, rtol=1e-14)
    x, info = oracle.pcg(A, b, 1e-12, pc="none")
    assert info["iters"] > 10


def test_zero_rhs_and_status_codes():
    A = poisson_grid((8, 8))
    x, info = oracle.pcg(A, np.zeros(64), 1e-8)
    assert info["iters"] == 0 and info["status"] == "ok" and not x.any()
    x, info = oracle.pcg(A, np.ones(64), 1e-12, max_iter=2)
    assert info["status"] == "not_converged" and info["iters"] == 2
    b = np.ones(64)
    b[5] = np.nan
    assert oracle.pcg(A, b, 1e-8)[1]["status"] == "breakdown"
    # indefinite matrix: p.Ap <= 0 shows up
    D = CSR(2, np.array([0, 1, 2], np.int32), np.array([0, 1], np.int32), np.array([1.0, -1.0]))
    assert oracle.pcg(D, np.array([1.0, 1.0]), 1e-8)[1]["status"] == "breakdown"


def test_initial_guess():
    A = poisson_grid((20, 20))
    b = np.random.default_rng(5).standard_normal(400)
    x_lu = dense_solve(A, b)
    x, info = oracle.pcg(A, b, 1e-10, x0=x_lu)
    assert info["iters"] <= 1
    x, info = oracle.pcg(A, b, 1e-10, x0=np.ones(400))
    assert info["status"] == "ok" and info["rel_res_true"] <= 1e-10


# ---------------------------------------------------------------- SPAI preconditioner
def _load_golden():
    A_e, M_e, eps = [], [], None
    for line in open(os.path.join(GOLDEN, "spai_3x3.txt")):
        if line.startswith("#") or not line.strip():
            continue
        t = line.split()
        if t[0] == "A":
            A_e.append((int(t[1]), int(t[2]), float(t[3])))
        elif t[0] == "eps":
            eps = float(t[1])
        elif t[0] == "M":
            M_e.append((int(t[1]), int(t[2]), Fraction(int(t[3]), int(t[4]))))
    n = 3
    D = np.zeros((n, n))
    for i, j, v in A_e:
        D[i, j] = v
    rows, cols = np.nonzero(D)
    rp = np.zeros(n + 1, np.int32)
    np.cumsum(np.bincount(rows, minlength=n), out=rp[1:])
    A = CSR(n, rp, cols.astype(np.int32), D[rows, cols])
    Mx = np.zeros((n, n))
    for i, j, f in M_e:
        Mx[i, j] = float(f)
    return A, eps, Mx


def test_spai_hand_derived_example():
    A, eps, M_expected = _load_golden()
    M = np.stack([oracle.spai_apply(A, e, eps) for e in np.eye(3)], axis=1)
    np.testing.assert_allclose(M, M_expected, rtol=1e-15, atol=1e-16)


def test_spai_diagonal_matrix_is_jacobi_plus_eps():
    d = np.array([2.0, 5.0, 0.25, 9.0])
    A = CSR(4, np.arange(5, dtype=np.int32), np.arange(4, dtype=np.int32), d)
    r = np.array([1.0, -2.0, 3.0, 0.5])
    np.testing.assert_allclose(oracle.spai_apply(A, r, 0.01), r / d + 0.01 * r, rtol=1e-15)


def test_spai_operator_is_spd():
    w = build("c5", npoints=120)
    n = w.A.n
    M = np.stack([oracle.spai_apply(w.A, e, 1e-3) for e in np.eye(n)], axis=1)
    np.testing.assert_allclose(M, M.T, rtol=0, atol=1e-15 * np.abs(M).max())
    assert np.linalg.eigvalsh(M).min() > 0


def test_spai_factor_pattern_is_lower_triangle():
    w = build("c5", npoints=500)
    grp, gci, gv = oracle.spai_factor(w.A)
    assert grp[-1] == (w.A.nnz + w.A.n) // 2
    rows = np.repeat(np.arange(w.A.n), np.diff(grp))
    assert np.all(gci <= rows)
    diag = gci == rows
    assert np.all(gv[diag] > 0) and np.all(gv[~diag] >= 0)   # -A_ij > 0 for a Laplacian


# ---------------------------------------------------------------- adjoint
def _loss(A, b, g, tol=1e-14):
    x, _ = oracle.pcg(A, b, tol)
    return float(g @ x)


def test_adjoint_db_central_differences():
    A = build("c2", N=6).A
    g_ = np.random.default_rng(2)
    b = g_.standard_normal(A.n)
    g = g_.standard_normal(A.n)
    x, _ = oracle.pcg(A, b, 1e-14)
    dldb, dlda, info = oracle.adjoint(A, x, g, 1e-14)
    h = 1e-4
    for i in [0, 7, 17, 35]:
        e = np.zeros(A.n); e[i] = h
        fd = (_loss(A, b + e, g) - _loss(A, b - e, g)) / (2 * h)
        assert abs(fd - dldb[i]) <= 1e-8 * max(1.0, abs(fd))


def test_adjoint_dA_central_differences():
    # perturbing one stored entry alone makes A nonsymmetric: use dense LU
    A = build("c2", N=5).A
    g_ = np.random.default_rng(4)
    b = g_.standard_normal(A.n)
    g = g_.standard_normal(A.n)
    x, _ = oracle.pcg(A, b, 1e-14)
    dldb, dlda, _ = oracle.adjoint(A, x, g, 1e-14)
    rows = A.rows()
    D = A.dense()
    h = 1e-5
    for k in [0, 3, 11, 40, A.nnz - 1]:
        i, j = rows[k], A.col_idx[k]
        Dp = D.copy(); Dp[i, j] += h
        Dm = D.copy(); Dm[i, j] -= h
        fd = (g @ np.linalg.solve(Dp, b) - g @ np.linalg.solve(Dm, b)) / (2 * h)
        assert abs(fd - dlda[k]) <= 1e-7 * max(1.0, abs(fd))


@pytest.mark.parametrize("pc", ["none", "jacobi", "spai"])
def test_adjoint_identities(pc):
    w = build("c5", npoints=2000)
    A = w.A
    x, _ = oracle.pcg(A, w.b, 1e-12, pc=pc, eps=1e-3)
    dldb, dlda, info = oracle.adjoint(A, x, w.g, 1e-12, pc=pc, eps=1e-3)
    assert info["status"] == "ok"
    gx = float(w.g @ x)
    # g^T x = lambda^T b  and  sum_k A_k dL/dA_k = -g^T x
    assert abs(float(dldb @ w.b) - gx) <= 1e-9 * abs(gx)
    assert abs(float(A.vals @ dlda) + gx) <= 1e-9 * abs(gx)


def test_adjoint_matches_autograd_through_dense_lu():
    """Gradients of L = g^T A^-1 b from torch autograd through a dense LU
    solve (torch.linalg.solve) equal the oracle's adjoint on the 64 x 64
    Poisson problem of torch-sla §4, Figure 2."""
    import torch
    w = build("c1")
    A = w.A
    rows = torch.from_numpy(A.rows())
    cols = torch.from_numpy(A.col_idx.astype(np.int64))
    vals = torch.tensor(A.vals, dtype=torch.float64, requires_grad=True)
    b = torch.tensor(np.random.default_rng(9).standard_normal(A.n), requires_grad=True)
    g = torch.from_numpy(np.random.default_rng(10).standard_normal(A.n))
    D = torch.zeros(A.n, A.n, dtype=torch.float64).index_put((rows, cols), vals)
    x = torch.linalg.solve(D, b)
    loss = g @ x
    loss.backward()
    xo, _ = oracle.pcg(A, b.detach().numpy(), 1e-14)
    dldb, dlda, _ = oracle.adjoint(A, xo, g.numpy(), 1e-14)
    assert abs(loss.item() - float(g.numpy() @ xo)) <= 1e-12 * abs(loss.item())
    np.testing.assert_allclose(dldb, b.grad.numpy(), rtol=0, atol=1e-10 * np.abs(dldb).max())
    np.testing.assert_allclose(dlda, vals.grad.numpy(), rtol=0, atol=1e-10 * np.abs(dlda).max())


def test_unrolled_autograd_cg_loss_agrees():
    """The naive path of torch-sla §4, Figure 2 (autograd through every CG
    iteration) reaches the same loss value as the oracle solve."""
    import torch
    w = build("c1")
    A = w.A
    rows = torch.from_numpy(A.rows())
    cols = torch.from_numpy(A.col_idx.astype(np.int64))
    vals = torch.tensor(A.vals, dtype=torch.float64, requires_grad=True)
    b = torch.tensor(np.random.default_rng(9).standard_normal(A.n), requires_grad=True)
    g = torch.from_numpy(np.random.default_rng(10).standard_normal(A.n))

    def matvec(v):
        return torch.zeros(A.n, dtype=torch.float64).index_add(0, rows, vals * v[cols])

    x = torch.zeros(A.n, dtype=torch.float64)
    r = b.clone()
    p = r.clone()
    rr = r @ r
    bb = (b @ b).item()
    for _ in range(1000):
        q = matvec(p)
        a = rr / (p @ q)
        x = x + a * p
        r = r - a * q
        rr_new = r @ r
        if rr_new.item() <= 1e-24 * bb:
            break
        p = r + (rr_new / rr) * p
        rr = rr_new
    loss = g @ x
    loss.backward()
    xo, _ = oracle.pcg(A, b.detach().numpy(), 1e-14)
    assert abs(loss.item() - float(g.numpy() @ xo)) <= 1e-10 * abs(loss.item())
    assert b.grad is not None and vals.grad is not None


# ---------------------------------------------------------------- fp32 storage mode
def test_f32_mode_solution_and_residual():
    w = build("c3", N=24, batch=2)
    x, infos = oracle.pcg(w.A, w.b, w.tol, pc="jacobi")
    for s in range(2):
        assert infos[s]["status"] == "ok"
        assert infos[s]["rel_res_true"] <= w.tol
        xs = x[s]
        assert np.array_equal(xs, xs.astype(np.float32).astype(np.float64))  # fp32 values
        x_lu = dense_solve(w.A, w.b[s].astype(np.float64), s)
        err = np.linalg.norm(xs - x_lu) / np.linalg.norm(x_lu)
        assert err <= cond2(w.A, s) * w.tol
        x64, i64 = oracle.pcg(CSR(w.A.n, w.A.row_ptr, w.A.col_idx, w.A.vals[s].astype(np.float64)),
                              w.b[s].astype(np.float64), w.tol, pc="jacobi", f32=False)
        assert abs(infos[s]["iters"] - i64["iters"]) <= max(2, 0.05 * i64["iters"])


def _f32_cases():
    """fp32-representable systems: the c3 recipe at a small size (two
    systems) and a random diagonally dominant SPD matrix, with fp32 b and g."""
    w = build("c3", N=24, batch=2)
    cases = [(CSR(w.A.n, w.A.row_ptr, w.A.col_idx, w.A.vals[s]), w.b[s], w.g[s], w.tol, "jacobi")
             for s in range(2)]
    g = np.random.default_rng(21)
    R = random_csr(120, 0.05, g, spd=True)
    R32 = CSR(R.n, R.row_ptr, R.col_idx, R.vals.astype(np.float32))
    cases.append((R32, g.standard_normal(R.n).astype(np.float32),
                  g.standard_normal(R.n).astype(np.float32), 1e-5, "none"))
    return cases


@pytest.mark.parametrize("case", range(3))
def test_f32_mode_is_the_fp64_recurrence_rounded_on_return(case):
    """The reading of "fp32 values": the matrix, b and the returned x (and
    lambda, dL/dA) are fp32, while the CG recurrence itself runs in fp64.  So
    on fp32-representable A and b the fp32 mode must take exactly the fp64
    mode's iterations and return exactly float32 of the fp64 mode's x; the
    adjoint likewise returns float32 of the fp64 lambda and dL/dA formed from
    those fp32 vectors, rounded once.  A reading that rounds the working
    vectors (r, p, q, z) to fp32 changes the iterates and fails this."""
    A32, b, gv, tol, pc = _f32_cases()[case]
    A64 = CSR(A32.n, A32.row_ptr, A32.col_idx, A32.vals.astype(np.float64))
    x32, i32 = oracle.pcg(A32, b, tol, pc=pc, f32=True)
    x64, i64 = oracle.pcg(A64, b.astype(np.float64), tol, pc=pc, f32=False)
    assert i32["status"] == i64["status"] == "ok"
    assert i32["iters"] == i64["iters"]
    assert np.array_equal(x32, x64.astype(np.float32).astype(np.float64))
    l32, d32, a32 = oracle.adjoint(A32, x32, gv, tol, pc=pc, f32=True)
    l64, _, a64 = oracle.adjoint(A64, x64, gv.astype(np.float64), tol, pc=pc, f32=False)
    assert a32["iters"] == a64["iters"]
    assert np.array_equal(l32, l64.astype(np.float32).astype(np.float64))
    rows = A32.rows()
    # the product of two fp32 values is exact in fp64; one rounding to fp32
    exact = (-l32[rows] * x32[A32.col_idx]).astype(np.float32).astype(np.float64)
    assert np.array_equal(d32, exact)


def test_grad_A_is_the_stored_pattern_outer_product():
    """oracle.grad_A: dL/dA_k = -lambda_row(k) x_col(k), by brute force over
    a dense outer product restricted to the pattern."""
    g = np.random.default_rng(5)
    A = random_csr(40, 0.2, g)
    lam, x = g.standard_normal(A.n), g.standard_normal(A.n)
    D = -np.outer(lam, x)
    rows = A.rows()
    assert np.array_equal(oracle.grad_A(A, lam, x), D[rows, A.col_idx])
