"""GPU parity of BiCGStab and its transpose adjoint (fp64) against the CPU
oracle on the same seeded nonsymmetric systems, through the C ABI.

Tolerances as for CG: ||x - x_oracle|| / ||x_oracle|| <= 1e-6, iteration
count within 2% of the oracle's (at least +-1), and the true residual of the
returned x at most tol.  Right Jacobi preconditioning runs on the GPU as the
column-scaled matrix A D^-1 (rounded differently from the oracle's D^-1 p);
its stopping check measures ||b - A x|| on the unscaled values for the
x = y / d it returns, so the reported true residual is at most tol."""
import numpy as np
import pytest
import torch

import oracle
from workloads import build, rng
from workloads.matrices import CSR, convection_diffusion, poisson_grid, rotating_wind

from gpu_util import make, random_csr, rel

pytestmark = pytest.mark.gpu



def _iters_ok(a, b):
    return abs(a - b) <= max(1, int(0.02 * b))


def _nonsym_random(n, seed):
    """Random pattern with a dominant diagonal: nonsymmetric, nonsingular."""
    A = random_csr(n, 6, seed=seed)
    rows = A.rows()
    # add the diagonal where it is missing, then make it dominant
    have = np.zeros(n, bool)
    have[rows[A.col_idx == rows]] = True
    r = np.concatenate([rows, np.flatnonzero(~have)])
    c = np.concatenate([A.col_idx.astype(np.int64), np.flatnonzero(~have)])
    v = np.concatenate([A.vals, np.zeros((~have).sum())])
    order = np.lexsort((c, r))
    r, c, v = r[order], c[order], v[order]
    off = r != c
    rowsum = np.bincount(r, weights=np.abs(v) * off, minlength=n)
    v[~off] = rowsum[r[~off]] * 1.2 + 0.5
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(r, minlength=n), out=rp[1:])
    return CSR(n, rp.astype(np.int32), c.astype(np.int32), v)


def _cases():
    yield "convdiff2d_rot_96", convection_diffusion((96, 96), rotating_wind((96, 96), 3.0))
    yield "convdiff3d_25_odd", convection_diffusion((25, 25, 25), (1.0, -0.5, 0.3))
    yield "cd3_24", build("cd3", N=24).A
    yield "random_2001", _nonsym_random(2001, 5)
    yield "random_1", _nonsym_random(1, 6)
    yield "random_2", _nonsym_random(2, 7)


CASES = list(_cases())


# grid patterns whose BiCGStab products take the sliced form by default
SLICED = ("convdiff2d_rot_96", "convdiff3d_25_odd", "cd3_24")


@pytest.mark.parametrize("staged", [False, True], ids=["default", "staged"])
@pytest.mark.parametrize("pc", ["none", "jacobi"])
@pytest.mark.parametrize("name,A", CASES, ids=[c[0] for c in CASES])
def test_bicgstab_parity(cuda_device, name, A, pc, staged):
    tol = 1e-10
    b = rng.normal(21, 1, A.n)
    M = make(A, staged=staged)
    x, info = M.solve(torch.from_numpy(b).to(cuda_device), tol=tol, max_iter=20000, pc=pc, method="bicgstab")
    form = M.layout_of("B")[0]
    if staged:
        assert form in (0, 1, 2), form
    elif name in SLICED:
        assert form in (6, 7), form
    xo, io = oracle.bicgstab(A, b, tol, max_iter=20000, pc=pc)
    assert io["status"] == "ok"
    assert info[0].status == "ok", info[0]
    assert _iters_ok(info[0].iters, io["iters"]), (info[0].iters, io["iters"])
    assert rel(x.cpu().numpy(), xo) <= 1e-6
    assert info[0].rel_res_true <= tol
    assert abs(oracle.rel_residual(A, b, x.cpu().numpy()) - info[0].rel_res_true) <= 1e-3 * tol


def test_bicgstab_batch_with_a_zero_rhs(cuda_device):
    """Three systems on one pattern (different winds), one with b = 0: the
    frozen system returns x = 0 after 0 iterations while the others run."""
    dims = (40, 30)
    winds = [(0.5, 0.25), rotating_wind(dims, 2.0), (-1.5, 1.0)]
    mats = [convection_diffusion(dims, w) for w in winds]
    A = CSR(mats[0].n, mats[0].row_ptr, mats[0].col_idx, np.stack([m.vals for m in mats]))
    b = rng.normal(22, 1, 3 * A.n).reshape(3, A.n)
    b[1] = 0.0
    M = make(A)
    for pc in ("none", "jacobi"):
        x, info = M.solve(torch.from_numpy(b).to(cuda_device), tol=1e-9, max_iter=5000, pc=pc, method="bicgstab")
        xo, io = oracle.bicgstab(A, b, 1e-9, max_iter=5000, pc=pc)
        xh = x.cpu().numpy()
        for s in range(3):
            assert info[s].status == io[s]["status"] == "ok"
            assert _iters_ok(info[s].iters, io[s]["iters"])
            assert rel(xh[s], xo[s]) <= 1e-6
        assert info[1].iters == 0 and not xh[1].any()


def _skewed_nonsym(n, seed):
    """Nonsymmetric, strictly diagonally dominant by rows: every 32nd row
    holds 40 random columns within 500 of the diagonal, the others 2, plus
    the diagonal (every 32-row group of A holds one row far longer than the
    rest; the rows of A^T are even)."""
    g = np.random.default_rng(seed)
    lens = np.full(n, 2)
    lens[::32] = 40
    r = np.repeat(np.arange(n), lens)
    c = np.clip(r + g.integers(-500, 501, size=r.size), 0, n - 1)
    key = np.unique(r.astype(np.int64) * n + c)
    r, c = key // n, key % n
    off = r != c
    r = np.concatenate([r[off], np.arange(n)])
    c = np.concatenate([c[off], np.arange(n)])
    v = np.concatenate([g.standard_normal(r.size - n), np.zeros(n)])
    v[-n:] = np.bincount(r[:-n], weights=np.abs(v[:-n]), minlength=n) * 1.2 + 0.5
    order = np.lexsort((c, r))
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(np.bincount(r, minlength=n))
    return CSR(n, rp, c[order].astype(np.int32), v[order])


@pytest.mark.parametrize("split", [None, True, False], ids=["auto", "split", "rows"])
def test_bicgstab_split_group_sums(cuda_device, split):
    """BiCGStab (right Jacobi) and its transpose adjoint on staged products
    of a pattern whose 32-row groups each hold one row far longer than the
    rest: by default A's groups are summed split over the lanes (the
    lane-per-row walk costs 3.2 times the split one) and A^T's are not
    (1.3); forced either way.  x, lambda and dL/dA against the oracle."""
    A = _skewed_nonsym(20000, 5)
    tol = 1e-10
    gen = np.random.default_rng(31)
    bh, gh = gen.standard_normal(A.n), gen.standard_normal(A.n)
    M = make(A, reorder=False, staged=True, split=split)
    x, info = M.solve(torch.from_numpy(bh).to(cuda_device), tol=tol, max_iter=20000, pc="jacobi", method="bicgstab")
    form, _, sp = M.layout_of("B")
    assert form in (1, 2) and sp == (split is not False), (form, sp)
    xo, io = oracle.bicgstab(A, bh, tol, max_iter=20000, pc="jacobi")
    xh = x.cpu().numpy()
    assert info[0].status == io["status"] == "ok"
    assert _iters_ok(info[0].iters, io["iters"]), (info[0].iters, io["iters"])
    assert rel(xh, xo) <= 1e-6
    assert info[0].rel_res_true <= tol
    dldb, dlda, ai = M.adjoint(x, torch.from_numpy(gh).to(cuda_device), tol=tol, max_iter=20000, pc="jacobi",
                               method="bicgstab")
    form, _, sp = M.layout_of("BT")
    assert form in (1, 2) and sp == bool(split), (form, sp)
    lb_o, la_o, ao = oracle.bicgstab_adjoint(A, xh, gh, tol, max_iter=20000, pc="jacobi")
    lb, la = dldb.cpu().numpy(), dlda.cpu().numpy()
    assert ai[0].status == ao["status"] == "ok"
    assert _iters_ok(ai[0].iters, ao["iters"]), (ai[0].iters, ao["iters"])
    assert rel(lb, lb_o) <= 1e-6 and rel(la, la_o) <= 1e-6
    assert np.array_equal(la, -lb[A.rows()] * xh[A.col_idx])


@pytest.mark.parametrize("staged", [False, True], ids=["default", "staged"])
@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_bicgstab_adjoint_parity(cuda_device, pc, staged):
    w = build("cd3", N=24)
    M = make(w.A, staged=staged)
    b = torch.from_numpy(w.b).to(cuda_device)
    g = torch.from_numpy(w.g).to(cuda_device)
    tol = 1e-10
    x, _ = M.solve(b, tol=tol, max_iter=20000, pc=pc, method="bicgstab")
    dldb, dlda, info = M.adjoint(x, g, tol=tol, max_iter=20000, pc=pc, method="bicgstab")
    assert (M.layout_of("BT")[0] in (0, 1, 2)) == staged
    xh = x.cpu().numpy()
    lb_o, la_o, io = oracle.bicgstab_adjoint(w.A, xh, w.g, tol, max_iter=20000, pc=pc)
    lb, la = dldb.cpu().numpy(), dlda.cpu().numpy()
    assert info[0].status == io["status"] == "ok"
    assert _iters_ok(info[0].iters, io["iters"])
    assert rel(lb, lb_o) <= 1e-6
    assert rel(la, la_o) <= 1e-6
    exact = -lb[w.A.rows()] * xh[w.A.col_idx]
    assert np.array_equal(la, exact)
    # the transpose matters: the CG-style adjoint (A itself) is far off
    lam_wrong, _ = oracle.bicgstab(w.A, w.g, tol, pc=pc)
    assert rel(lam_wrong, lb_o) > 1e-3
    # identities: g.x = lambda.b, sum A . dL/dA = -g.x
    scale = np.linalg.norm(w.g) * np.linalg.norm(xh)
    assert abs(w.g @ xh - lb @ w.b) <= 1e-7 * scale
    assert abs((w.A.vals * la).sum() + w.g @ xh) <= 1e-7 * scale


def test_bicgstab_adjoint_after_value_update(cuda_device):
    """The transposed values follow update_values (the pattern is kept)."""
    dims = (32, 32)
    A1 = convection_diffusion(dims, (1.0, 0.5))
    A2 = convection_diffusion(dims, rotating_wind(dims, 2.5))
    M = make(A1)
    b = rng.normal(23, 1, A1.n)
    g = rng.normal(23, 2, A1.n)
    tb, tg = torch.from_numpy(b).to(cuda_device), torch.from_numpy(g).to(cuda_device)
    for A in (A1, A2):
        M.update_values(torch.from_numpy(A.vals).to(cuda_device))
        x, _ = M.solve(tb, tol=1e-10, method="bicgstab", pc="jacobi")
        lb, la, info = M.adjoint(x, tg, tol=1e-10, method="bicgstab", pc="jacobi")
        lb_o, la_o, _ = oracle.bicgstab_adjoint(A, x.cpu().numpy(), g, 1e-10, pc="jacobi")
        assert info[0].status == "ok"
        assert rel(lb.cpu().numpy(), lb_o) <= 1e-6
        assert rel(la.cpu().numpy(), la_o) <= 1e-6


def test_bicgstab_autograd(cuda_device):
    from sparse_iterative_linear_csr_b300 import solve
    w = build("cd3", N=16)
    M = make(w.A)
    vals = M.values.clone().requires_grad_(True)
    b = torch.from_numpy(w.b).to(cuda_device).requires_grad_(True)
    g = torch.from_numpy(w.g).to(cuda_device)
    x = solve(M, vals, b, tol=1e-12, pc="jacobi", max_iter=20000, method="bicgstab")
    (x * g).sum().backward()
    xo, _ = oracle.bicgstab(w.A, w.b, 1e-12, pc="jacobi")
    lb_o, la_o, _ = oracle.bicgstab_adjoint(w.A, xo, w.g, 1e-12, pc="jacobi")
    assert rel(x.detach().cpu().numpy(), xo) <= 1e-9
    assert rel(b.grad.cpu().numpy(), lb_o) <= 1e-9
    assert rel(vals.grad.cpu().numpy(), la_o) <= 1e-9


@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_bicgstab_warm_start(cuda_device, pc):
    A = convection_diffusion((50, 50), rotating_wind((50, 50), 2.0))
    b = rng.normal(24, 1, A.n)
    M = make(A)
    tb = torch.from_numpy(b).to(cuda_device)
    x1, i1 = M.solve(tb, tol=1e-4, pc=pc, method="bicgstab")
    x2, i2 = M.solve(tb, tol=1e-10, pc=pc, method="bicgstab", x0=x1)
    xo, io = oracle.bicgstab(A, b, 1e-10, pc=pc, x0=x1.cpu().numpy())
    assert i2[0].status == "ok" and _iters_ok(i2[0].iters, io["iters"])
    assert rel(x2.cpu().numpy(), xo) <= 1e-6
    # a warm start that already meets the tolerance stops before any product
    x3, i3 = M.solve(tb, tol=1e-4, pc=pc, method="bicgstab", x0=x2)
    assert i3[0].iters == 0 and i3[0].status == "ok"
    assert rel(x3.cpu().numpy(), x2.cpu().numpy()) <= 1e-15


def test_bicgstab_iteration_cap_matches_oracle_iterates(cuda_device):
    A = convection_diffusion((30, 20), (1.0, -0.7))
    b = rng.normal(25, 1, A.n)
    M = make(A)
    tb = torch.from_numpy(b).to(cuda_device)
    for pc in ("none", "jacobi"):
        for cap in (0, 1, 3):
            x, info = M.solve(tb, tol=1e-14, max_iter=cap, pc=pc, method="bicgstab")
            xo, io = oracle.bicgstab(A, b, 1e-14, max_iter=cap, pc=pc)
            assert info[0].status == io["status"] == "not_converged"
            assert info[0].iters == io["iters"] == cap
            assert rel(x.cpu().numpy(), xo) <= 1e-12


def test_bicgstab_breakdown_and_invalid(cuda_device):
    from sparse_iterative_linear_csr_b300 import SLAError
    R = CSR(2, np.array([0, 1, 2], np.int32), np.array([1, 0], np.int32), np.array([1.0, -1.0]))
    M = make(R)
    x, info = M.solve(torch.tensor([1.0, 0.0], dtype=torch.float64, device=cuda_device), tol=1e-10,
                      method="bicgstab")
    assert info[0].status == "breakdown" == oracle.bicgstab(R, np.array([1.0, 0.0]), 1e-10)[1]["status"]
    with pytest.raises(SLAError):      # Jacobi without a stored diagonal
        M.solve(torch.tensor([1.0, 0.0], dtype=torch.float64, device=cuda_device), pc="jacobi",
                method="bicgstab")
    A = convection_diffusion((8, 8), (1.0, 1.0))
    M = make(A)
    tb = torch.ones(A.n, dtype=torch.float64, device=cuda_device)
    for which in ("B", "BT", "G", "GT"):   # not built before their first solve
        with pytest.raises(SLAError):
            M.layout_of(which)
    with pytest.raises(SLAError):      # SPAI is for SPD systems
        M.solve(tb, pc="spai", method="bicgstab")
    x, _ = M.solve(tb, method="bicgstab")
    M.adjoint(x, tb, method="bicgstab")
    assert M.layout_of("B")[0] in (0, 1, 2, 5, 6, 7) and M.layout_of("BT")[0] in (0, 1, 2, 5, 6, 7)
    A32 = CSR(A.n, A.row_ptr, A.col_idx, A.vals.astype(np.float32))
    M32 = make(A32)
    with pytest.raises(SLAError):      # fp64 only
        M32.solve(tb.float(), method="bicgstab")


def test_bicgstab_on_spd_matches_cg(cuda_device):
    A = poisson_grid((60, 50))
    b = rng.normal(26, 1, A.n)
    M = make(A)
    tb = torch.from_numpy(b).to(cuda_device)
    xb, ib = M.solve(tb, tol=1e-11, pc="jacobi", method="bicgstab")
    xc, ic = M.solve(tb, tol=1e-11, pc="jacobi")
    assert ib[0].status == ic[0].status == "ok"
    assert rel(xb.cpu().numpy(), xc.cpu().numpy()) <= 1e-8


@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_bicgstab_reordered_parity(cuda_device, pc):
    """A scattered labelling of a convection-diffusion grid: the handle
    iterates on the reverse Cuthill-McKee ordering, the oracle on the
    caller's; solution and adjoint agree."""
    dims = (80, 70)
    A0 = convection_diffusion(dims, rotating_wind(dims, 2.0))
    perm = rng.permutation(27, 0, A0.n)        # new label of old unknown i: inv[i]
    inv = np.empty_like(perm)
    inv[perm] = np.arange(A0.n)
    D_rows = A0.rows()
    r, c = inv[D_rows], inv[A0.col_idx]
    order = np.lexsort((c, r))
    rp = np.zeros(A0.n + 1, np.int64)
    np.cumsum(np.bincount(r, minlength=A0.n), out=rp[1:])
    A = CSR(A0.n, rp.astype(np.int32), c[order].astype(np.int32), A0.vals[order])
    b = rng.normal(27, 1, A.n)
    g = rng.normal(27, 2, A.n)
    M = make(A, reorder=True)
    assert M.layout()[2]
    x, info = M.solve(torch.from_numpy(b).to(cuda_device), tol=1e-10, pc=pc, method="bicgstab")
    xo, io = oracle.bicgstab(A, b, 1e-10, pc=pc)
    assert info[0].status == "ok" and _iters_ok(info[0].iters, io["iters"])
    assert rel(x.cpu().numpy(), xo) <= 1e-6
    lb, la, ia = M.adjoint(x, torch.from_numpy(g).to(cuda_device), tol=1e-10, pc=pc, method="bicgstab")
    lb_o, la_o, _ = oracle.bicgstab_adjoint(A, x.cpu().numpy(), g, 1e-10, pc=pc)
    assert ia[0].status == "ok"
    assert rel(lb.cpu().numpy(), lb_o) <= 1e-6
    assert rel(la.cpu().numpy(), la_o) <= 1e-6
