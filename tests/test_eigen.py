"""eigsh (torch-sla §3 sparse tensor types) by LOBPCG on the library's block
product: eigenvalues against closed forms (grid Laplacians) and the dense
oracle, eigenvectors by their residuals, eigenvalue gradients by finite
differences of the oracle; the block product against the oracle's SpMV."""
import numpy as np
import pytest
import torch

import oracle
from workloads.matrices import CSR, poisson_grid

from gpu_util import make, random_csr, rel


def laplacian_eigs(dims):
    """All eigenvalues of the unscaled Dirichlet grid Laplacian (closed form):
    sums over the axes of 2 - 2 cos(j pi / (N + 1)), j = 1..N."""
    axes = [2.0 - 2.0 * np.cos(np.arange(1, N + 1) * np.pi / (N + 1)) for N in dims]
    tot = axes[0]
    for a in axes[1:]:
        tot = (tot[:, None] + a[None, :]).ravel()
    return np.sort(tot)


@pytest.mark.parametrize("dims", [(30,), (9, 11), (5, 6, 7)])
def test_dense_oracle_matches_the_closed_form(dims):
    A = poisson_grid(dims)
    w, V = oracle.eigsh_dense(A, 6)
    assert np.allclose(w, laplacian_eigs(dims)[:6], rtol=1e-12, atol=1e-12)
    D = np.zeros((A.n, A.n))
    D[A.rows(), A.col_idx] = A.vals
    assert np.allclose(D @ V.T, V.T * w, atol=1e-10)
    wl, _ = oracle.eigsh_dense(A, 3, largest=True)
    assert np.allclose(wl, laplacian_eigs(dims)[::-1][:3], rtol=1e-12)


@pytest.mark.gpu
def test_spmm_matches_the_oracle_per_column(cuda_device):
    from sparse_iterative_linear_csr_b300.eigen import spmm
    A = random_csr(700, 7, seed=5)
    M = make(A)
    X = np.random.default_rng(1).standard_normal((5, A.n))
    Y = spmm(M, torch.from_numpy(X).to(cuda_device)).cpu().numpy()
    for j in range(5):
        y_o = oracle.spmv(A, X[j])
        scale = oracle.spmv(CSR(A.n, A.row_ptr, A.col_idx, np.abs(A.vals)), np.abs(X[j]))
        assert np.all(np.abs(Y[j] - y_o) <= 1e-12 * np.maximum(scale, 1e-300))


@pytest.mark.gpu
@pytest.mark.parametrize("dims,k", [((40, 40), 6), ((12, 12, 12), 5), ((200,), 4)])
def test_lobpcg_grid_laplacians_against_closed_form(cuda_device, dims, k):
    from sparse_iterative_linear_csr_b300.eigen import lobpcg
    A = poisson_grid(dims)
    M = make(A)
    theta, V, info = lobpcg(M, k, tol=1e-9, max_iter=5000)
    assert info.converged, info
    assert np.allclose(theta.cpu().numpy(), laplacian_eigs(dims)[:k], rtol=1e-9)
    V = V.cpu().numpy()
    for j in range(k):
        r = oracle.spmv(A, V[j]) - theta[j].item() * V[j]
        assert np.linalg.norm(r) <= 1e-8 * abs(theta[j].item())


@pytest.mark.gpu
@pytest.mark.parametrize("largest", [False, True])
def test_lobpcg_random_spd_against_dense_oracle(cuda_device, largest):
    from sparse_iterative_linear_csr_b300.eigen import lobpcg
    A = random_csr(300, 6, seed=11, spd=True)
    M = make(A)
    theta, V, info = lobpcg(M, 4, largest=largest, tol=1e-10, max_iter=5000)
    w, Vo = oracle.eigsh_dense(A, 4, largest=largest)
    assert info.converged
    assert np.allclose(theta.cpu().numpy(), w, rtol=1e-9)
    # eigenvectors agree up to sign (the spectrum of this matrix is simple)
    Vg = V.cpu().numpy()
    for j in range(4):
        assert min(rel(Vg[j], Vo[j]), rel(-Vg[j], Vo[j])) <= 1e-6


@pytest.mark.gpu
def test_eigenvalue_gradient_against_finite_differences(cuda_device):
    """d theta_j / d A_k = v_j[row] v_j[col]; checked on symmetric pairs of
    entries (A_ij and A_ji moved together keep the matrix symmetric)."""
    from sparse_iterative_linear_csr_b300.eigen import eigsh
    A = random_csr(120, 5, seed=3, spd=True)
    M = make(A)
    vals = M.values.clone().requires_grad_(True)
    theta = eigsh(M, vals, 3, tol=1e-12, max_iter=10000)
    weights = torch.tensor([1.0, -0.5, 2.0], dtype=torch.float64, device=cuda_device)
    (theta * weights).sum().backward()
    g = vals.grad.cpu().numpy()
    rows = A.rows()
    key = {(int(r), int(c)): k for k, (r, c) in enumerate(zip(rows, A.col_idx))}
    h = 1e-6
    picks = [k for k in range(A.nnz) if rows[k] < A.col_idx[k]][:6] + [k for k in range(A.nnz) if rows[k] == A.col_idx[k]][:3]
    for k in picks:
        i, j = int(rows[k]), int(A.col_idx[k])
        ks = [k] if i == j else [k, key[(j, i)]]
        def L(delta):
            v = A.vals.copy()
            v[ks] += delta
            w, _ = oracle.eigsh_dense(CSR(A.n, A.row_ptr, A.col_idx, v), 3)
            return float(w @ np.array([1.0, -0.5, 2.0]))
        fd = (L(h) - L(-h)) / (2 * h)
        assert abs(fd - g[ks].sum()) <= 1e-6 * max(1.0, abs(fd))


@pytest.mark.gpu
@pytest.mark.parametrize("ka,kb,n", [(1, 1, 1), (5, 7, 1000), (12, 36, 33333), (64, 64, 257), (36, 36, 100000)])
def test_block_gram_and_update_match_numpy(cuda_device, ka, kb, n):
    """The library's block kernels against numpy's fp64 products: G = A B^T
    (full, upper triangle mirrored for one block and for two, diagonal) and
    Y = C^T S + Yin, in place too; ragged column counts exercise the staged
    chunks' tails."""
    from sparse_iterative_linear_csr_b300.eigen import GRAM_DIAG, GRAM_UPPER, gram, update
    g = np.random.default_rng(ka * 1000 + kb)
    A = g.standard_normal((ka, n))
    B = g.standard_normal((kb, n))
    Ad = torch.from_numpy(A).to(cuda_device)
    Bd = torch.from_numpy(B).to(cuda_device)
    scale = np.sqrt(n)
    G = gram(Ad, Bd).cpu().numpy()
    assert np.abs(G - A @ B.T).max() <= 1e-12 * scale * 10
    Gs = gram(Ad).cpu().numpy()
    assert np.array_equal(Gs, Gs.T) and np.abs(Gs - A @ A.T).max() <= 1e-12 * scale * 10
    d = gram(Ad, mode=GRAM_DIAG).cpu().numpy()
    assert np.abs(d - (A * A).sum(1)).max() <= 1e-12 * scale * 10
    if ka == kb:
        Gu = gram(Ad, Bd, mode=GRAM_UPPER).cpu().numpy()
        full = A @ B.T
        iu = np.triu_indices(ka)
        assert np.array_equal(Gu, Gu.T)
        assert np.abs(Gu[iu] - full[iu]).max() <= 1e-12 * scale * 10
    Cm = g.standard_normal((kb, ka))
    Y = update(torch.from_numpy(Cm).to(cuda_device), Bd).cpu().numpy()
    assert np.abs(Y - Cm.T @ B).max() <= 1e-12 * kb
    Y2 = Ad.clone()
    update(torch.from_numpy(Cm).to(cuda_device), Bd, Y2, out=Y2)
    assert np.abs(Y2.cpu().numpy() - (A + Cm.T @ B)).max() <= 1e-12 * kb


@pytest.mark.gpu
def test_block_kernels_reject_bad_sizes(cuda_device):
    import ctypes as C
    from sparse_iterative_linear_csr_b300 import _lib
    lib = _lib.load()
    need = C.c_longlong(0)
    assert lib.sla_block_gram_work(65, 1, 0, 10, C.byref(need)) == _lib.SLA_ERR_INVALID
    assert lib.sla_block_gram_work(3, 4, 1, 10, C.byref(need)) == _lib.SLA_ERR_INVALID
    assert lib.sla_block_gram_work(3, 3, 7, 10, C.byref(need)) == _lib.SLA_ERR_INVALID
    assert lib.sla_block_gram_work(3, 4, 3, 10, C.byref(need)) == _lib.SLA_ERR_INVALID
    assert lib.sla_block_update(0, 3, 10, None, None, None, None, None) == _lib.SLA_ERR_INVALID
