"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle
on the same seeded inputs, element by element, at sizes the oracle finishes
in seconds (many warp groups and CTAs and a ragged tail), plus edge cases.

Every product test runs with the default form (by the row lengths the
sliced, the direct thread-per-row or a warp-staged form), the warp-staged forms (staged=True), the warp pipeline
(pipeline=True), the producer/consumer form (producer_consumer=True), the
sliced form (sliced=True), the last three wherever they apply, and the
warp-staged forms with every staged group summed split over the lanes
(staged=True, split=True); the solve tests run with one kernel per step in
a CUDA graph (the default) and with the persistent iteration kernel
(fused=True), each with every product form.

Tolerances: SpMV relative error <= 1e-12 (fp64) and <= 1e-5 (fp32);
||x - x_oracle|| / ||x_oracle|| <= 1e-6; iteration count within 2% of the
oracle's (at least +-1); true residual of the returned x <= tol."""
import numpy as np
import pytest
import torch

import oracle
from workloads import build
from workloads.matrices import CSR, poisson_grid

from gpu_util import make, random_csr, rel

pytestmark = pytest.mark.gpu

SPMV_TOL = {np.float64: 1e-12, np.float32: 1e-5}


def _iters_ok(a, b):
    return abs(a - b) <= max(1, int(0.02 * b))


def _spmv_cases():
    yield "poisson1d_5000", poisson_grid((5000,))
    yield "poisson2d_64", poisson_grid((64, 64))
    yield "poisson3d_24", poisson_grid((24, 24, 24))
    yield "diffusion_96", build("c2", N=96).A
    yield "knn_3000", build("c5", npoints=3000).A
    for n in (1, 2, 31, 33, 257, 1000):
        yield f"random_{n}", random_csr(n, 6, seed=n)
    yield "empty_rows", random_csr(500, 4, seed=7, empty_rows=40)
    # one row far longer than a staging tile, plus short rows around it
    n = 12001
    cols = [np.arange(n)] + [np.array([i]) for i in range(1, n)]
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum([c.size for c in cols])
    g = np.random.default_rng(3)
    yield "dense_row", CSR(n, rp, np.concatenate(cols).astype(np.int32), g.standard_normal(int(rp[-1])))


FORMS = {"default": {}, "staged": {"staged": True}, "pipe": {"pipeline": True},
         "pc": {"producer_consumer": True}, "sliced": {"sliced": True},
         "split": {"staged": True, "split": True}}
# patterns whose sliced copy pads by at most 15% (the sliced form applies)
SLICED = ("poisson2d_64", "poisson3d_24", "diffusion_96", "knn_3000")
PIPE = pytest.mark.parametrize("mode", list(FORMS))
MODES = pytest.mark.parametrize("mode,fused", [(m, f) for f in (False, True) for m in FORMS],
                                ids=[f"{m}-{'fused' if f else 'steps'}" for f in (False, True) for m in FORMS])


@PIPE
@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("name,A", list(_spmv_cases()), ids=lambda v: v if isinstance(v, str) else "")
def test_spmv_parity(cuda_device, name, A, dtype, mode):
    A = CSR(A.n, A.row_ptr, A.col_idx, A.vals.astype(dtype))
    x = np.random.default_rng(11).standard_normal(A.n).astype(dtype)
    M = make(A, **FORMS[mode])
    form = M.layout()[0]
    if mode in ("staged", "split") or name == "dense_row":   # the dense row fits no bulk-copy form, nor the direct one
        assert form in (0, 1, 2)
        if mode == "split" and form in (1, 2) and name != "dense_row":
            assert M.layout_of("A")[2]
    elif mode == "default" and name == "knn_3000":   # long rows: the sliced form
        assert form == 6, form
    elif mode == "default" and name == "poisson3d_24":   # 7-point rows: the sliced form for short rows
        assert form == 7, form
    elif mode == "default" and name in ("poisson2d_64", "diffusion_96"):   # 5-point rows: the short-row sliced form
        assert form == 7, form
    elif mode == "default" and name == "poisson1d_5000":   # 3-point rows: the direct form
        assert form == 5, form
    elif mode == "pipe" and name != "knn_3000":   # groups of 32 short rows fit the warp pipeline
        assert form == 3, form
    elif mode == "pc":
        assert form == 4, form
    elif mode == "sliced" and name in SLICED:
        assert form in (6, 7), form
    xd = torch.from_numpy(x).to(cuda_device)
    y = M.matvec(xd).cpu().numpy()
    y_o = oracle.spmv(A, x.astype(np.float64))
    scale = oracle.spmv(CSR(A.n, A.row_ptr, A.col_idx, np.abs(A.vals)), np.abs(x.astype(np.float64)))
    tol = SPMV_TOL[dtype]
    assert np.all(np.abs(y - y_o) <= tol * np.maximum(scale, 1e-300) + (0 if dtype == np.float64 else 1e-30))
    yd, dot = M.matvec_dot(xd)
    assert np.array_equal(yd.cpu().numpy(), y)
    d_o = float(x.astype(np.float64) @ y.astype(np.float64))
    assert abs(dot.item() - d_o) <= 1e-12 * max(1.0, float(np.abs(x) @ np.abs(y)))


@PIPE
def test_spmv_batched(cuda_device, mode):
    w = build("c3", N=40, batch=3)
    M = make(w.A, **FORMS[mode])
    x = torch.from_numpy(w.b).to(cuda_device)
    y = M.matvec(x).cpu().numpy()
    for s in range(3):
        y_o = oracle.spmv(w.A, w.b[s].astype(np.float64), system=s)
        assert rel(y[s], y_o) <= 1e-6
    _, dots = M.matvec_dot(x)
    for s in range(3):
        assert abs(dots[s].item() - float(w.b[s].astype(np.float64) @ y[s].astype(np.float64))) <= 1e-9


SOLVE_CASES = [
    ("c1", {}, "none"),
    ("c2", {"N": 96}, "jacobi"),
    ("c3", {"N": 48, "batch": 5}, "jacobi"),
    ("c4", {"N": 24}, "none"),
    ("c5", {"npoints": 20000}, "spai"),
    ("c5", {"npoints": 20000}, "jacobi"),
    ("c2", {"N": 64}, "spai"),
    ("c3", {"N": 32, "batch": 3}, "spai"),
]


@MODES
@pytest.mark.parametrize("cfg,kw,pc", SOLVE_CASES, ids=[f"{c}-{p}-{k}" for c, k, p in SOLVE_CASES])
def test_pcg_parity(cuda_device, cfg, kw, pc, mode, fused):
    w = build(cfg, **kw)
    M = make(w.A, fused=fused, **FORMS[mode])
    b = torch.from_numpy(w.b).to(cuda_device)
    x, info = M.solve(b, tol=w.tol, max_iter=20000, pc=pc, eps=1e-3, poll_k=16)
    x = x.cpu().numpy()
    xo, io = oracle.pcg(w.A, w.b, w.tol, max_iter=20000, pc=pc, eps=1e-3)
    bs = w.b
    if M.batch == 1 and w.A.vals.ndim == 1:
        x, xo, io, bs = x[None], xo[None], [io], w.b[None]
    for s in range(len(info)):
        assert info[s].status == "ok" and io[s]["status"] == "ok"
        assert _iters_ok(info[s].iters, io[s]["iters"]), (info[s].iters, io[s]["iters"])
        assert rel(x[s], xo[s]) <= 1e-6
        assert info[s].rel_res_true <= w.tol
        # the reported true residual is the residual of the returned x
        assert abs(oracle.rel_residual(w.A, bs[s], x[s], system=s) - info[s].rel_res_true) <= 1e-3 * w.tol


ADJ_CASES = [("c4", {"N": 24}, "none"), ("c2", {"N": 64}, "jacobi"), ("c5", {"npoints": 20000}, "spai"),
             ("c3", {"N": 32, "batch": 3}, "jacobi")]


@MODES
@pytest.mark.parametrize("cfg,kw,pc", ADJ_CASES, ids=[f"{c}-{p}" for c, k, p in ADJ_CASES])
def test_adjoint_parity(cuda_device, cfg, kw, pc, mode, fused):
    w = build(cfg, **kw)
    M = make(w.A, fused=fused, **FORMS[mode])
    b = torch.from_numpy(w.b).to(cuda_device)
    g = torch.from_numpy(w.g).to(cuda_device)
    x, _ = M.solve(b, tol=w.tol, max_iter=20000, pc=pc)
    dldb, dlda, info = M.adjoint(x, g, tol=w.tol, max_iter=20000, pc=pc)
    xh = x.cpu().numpy()
    lb_o, la_o, io = oracle.adjoint(w.A, xh, w.g, w.tol, max_iter=20000, pc=pc, eps=1e-3)
    lb, la = dldb.cpu().numpy(), dlda.cpu().numpy()
    if lb.ndim == 1:
        lb, la, lb_o, la_o, io = lb[None], la[None], lb_o[None], la_o[None], [io]
    for s in range(lb.shape[0]):
        assert info[s].status == "ok" and _iters_ok(info[s].iters, io[s]["iters"])
        assert rel(lb[s], lb_o[s]) <= 1e-6
        assert rel(la[s], la_o[s]) <= 1e-6
        # dA is exactly -lambda_i x_j of the returned lambda and x
        rows = w.A.rows()
        exact = (-lb[s][rows].astype(np.float64) * xh[s if xh.ndim == 2 else slice(None)][w.A.col_idx]
                 .astype(np.float64)).astype(la.dtype)
        assert np.array_equal(la[s], exact)


def test_autograd_wrapper(cuda_device):
    from sparse_iterative_linear_csr_b300 import solve
    w = build("c2", N=48)
    M = make(w.A)
    vals = M.values.clone().requires_grad_(True)
    b = torch.from_numpy(w.b).to(cuda_device).requires_grad_(True)
    g = torch.from_numpy(w.g).to(cuda_device)
    x = solve(M, vals, b, tol=1e-12, pc="jacobi", max_iter=20000)
    (x * g).sum().backward()
    xo, _ = oracle.pcg(w.A, w.b, 1e-12, pc="jacobi")
    lb_o, la_o, _ = oracle.adjoint(w.A, xo, w.g, 1e-12, pc="jacobi")
    assert rel(x.detach().cpu().numpy(), xo) <= 1e-9
    assert rel(b.grad.cpu().numpy(), lb_o) <= 1e-9
    assert rel(vals.grad.cpu().numpy(), la_o) <= 1e-9


# ------------------------------------------------------------------ edge cases
def test_zero_rhs(cuda_device):
    w = build("c1")
    M = make(w.A)
    x, info = M.solve(torch.zeros(w.A.n, dtype=torch.float64, device=cuda_device), tol=1e-8)
    assert info[0].iters == 0 and info[0].status == "ok" and not x.abs().sum().item()
    # also with an initial guess
    x, info = M.solve(torch.zeros(w.A.n, dtype=torch.float64, device=cuda_device), tol=1e-8,
                      x0=torch.ones(w.A.n, dtype=torch.float64, device=cuda_device))
    assert info[0].iters == 0 and not x.abs().sum().item()


FUSED = pytest.mark.parametrize("fused", [True, False], ids=["fused", "steps"])


@FUSED
@pytest.mark.parametrize("max_iter", [0, 1, 2, 37])
def test_max_iter_reached(cuda_device, max_iter, fused):
    w = build("c2", N=40)
    M = make(w.A, fused=fused)
    b = torch.from_numpy(w.b).to(cuda_device)
    x, info = M.solve(b, tol=1e-12, max_iter=max_iter, pc="jacobi", poll_k=8)
    xo, io = oracle.pcg(w.A, w.b, 1e-12, max_iter=max_iter, pc="jacobi")
    assert info[0].status == "not_converged" == io["status"]
    assert info[0].iters == io["iters"] == max_iter
    assert rel(x.cpu().numpy(), xo) <= 1e-9


@FUSED
def test_breakdown_nan_and_indefinite(cuda_device, fused):
    w = build("c1")
    M = make(w.A, fused=fused)
    b = torch.from_numpy(w.b).to(cuda_device).clone()
    b[17] = float("nan")
    _, info = M.solve(b, tol=1e-8)
    assert info[0].status == "breakdown"
    D = CSR(3, np.array([0, 1, 2, 3], np.int32), np.array([0, 1, 2], np.int32), np.array([1.0, -1.0, 2.0]))
    M2 = make(D, fused=fused)
    _, info = M2.solve(torch.ones(3, dtype=torch.float64, device=cuda_device), tol=1e-8)
    assert info[0].status == "breakdown" == oracle.pcg(D, np.ones(3), 1e-8)[1]["status"]


@FUSED
def test_initial_guess_parity(cuda_device, fused):
    w = build("c2", N=64)
    M = make(w.A, fused=fused)
    b = torch.from_numpy(w.b).to(cuda_device)
    x0 = np.random.default_rng(1).standard_normal(w.A.n)
    x, info = M.solve(b, tol=1e-9, pc="jacobi", x0=torch.from_numpy(x0).to(cuda_device))
    xo, io = oracle.pcg(w.A, w.b, 1e-9, pc="jacobi", x0=x0)
    assert _iters_ok(info[0].iters, io["iters"]) and rel(x.cpu().numpy(), xo) <= 1e-6


def test_invalid_inputs_rejected(cuda_device):
    from sparse_iterative_linear_csr_b300 import CSRMatrix, SLAError
    dev = cuda_device
    rp = torch.tensor([0, 2, 1, 3], dtype=torch.int32, device=dev)       # decreasing row_ptr
    ci = torch.tensor([0, 1, 2], dtype=torch.int32, device=dev)
    v = torch.ones(3, dtype=torch.float64, device=dev)
    with pytest.raises(SLAError, match="row_ptr"):
        CSRMatrix(rp, ci, v)
    rp = torch.tensor([0, 2, 3, 3], dtype=torch.int32, device=dev)
    with pytest.raises(SLAError, match="ascending"):
        CSRMatrix(rp, torch.tensor([1, 0, 2], dtype=torch.int32, device=dev), v)
    with pytest.raises(SLAError, match="range"):
        CSRMatrix(rp, torch.tensor([0, 5, 2], dtype=torch.int32, device=dev), v)
    # missing diagonal: fine for plain CG set-up, rejected for Jacobi / SPAI
    M = CSRMatrix(torch.tensor([0, 1, 2], dtype=torch.int32, device=dev),
                  torch.tensor([1, 0], dtype=torch.int32, device=dev), torch.ones(2, dtype=torch.float64,
                                                                                  device=dev))
    b = torch.ones(2, dtype=torch.float64, device=dev)
    for pc in ("jacobi", "spai"):
        with pytest.raises(SLAError, match="diagonal"):
            M.solve(b, pc=pc)
    with pytest.raises(SLAError, match="tol"):
        M.solve(b, tol=0.0)


def test_spai_rejects_unsymmetric_pattern(cuda_device):
    from sparse_iterative_linear_csr_b300 import SLAError
    A = CSR(3, np.array([0, 2, 3, 4], np.int32), np.array([0, 2, 1, 2], np.int32), np.array([2.0, -1, 2, 2]))
    M = make(A)
    with pytest.raises(SLAError, match="symmetric"):
        M.solve(torch.ones(3, dtype=torch.float64, device=cuda_device), pc="spai")


@FUSED
def test_timeout_reports_and_keeps_iterate(cuda_device, fused):
    w = build("c4", N=48)
    M = make(w.A, fused=fused)
    b = torch.from_numpy(w.b).to(cuda_device)
    x, info = M.solve(b, tol=1e-14, max_iter=100000, poll_k=1, timeout_s=1e-4)
    assert info[0].status in ("timeout", "ok")
    assert info[0].status == "timeout" and info[0].iters < 100000
    assert np.isfinite(x.cpu().numpy()).all()


@pytest.mark.parametrize("pc", ["spai", "jacobi"])
def test_repeat_solves_are_deterministic(cuda_device, pc):
    w = build("c5", npoints=20000)
    M = make(w.A)
    b = torch.from_numpy(w.b).to(cuda_device)
    x1, i1 = M.solve(b, tol=1e-8, pc=pc)
    x2, i2 = M.solve(b, tol=1e-8, pc=pc, poll_k=7)
    assert i1[0].iters == i2[0].iters and torch.equal(x1, x2)


@pytest.mark.parametrize("staged", [False, True], ids=["sliced", "staged"])
def test_update_values(cuda_device, staged):
    """New values at a new address after a solve (the CUDA graphs that read
    the caller's values are rebuilt: the staged form's; the sliced copy's
    are refreshed in place): the next solve follows the new matrix."""
    w = build("c2", N=48)
    M = make(w.A, staged=staged)
    assert (M.layout()[0] in (0, 1, 2)) == staged
    b = torch.from_numpy(w.b).to(cuda_device)
    for pc in ("jacobi", "spai"):        # graphs captured on the first values
        M.solve(b, tol=1e-10, pc=pc)
    v2 = M.values * 2.0
    M.update_values(v2)
    A2 = CSR(w.A.n, w.A.row_ptr, w.A.col_idx, w.A.vals * 2.0)
    for pc in ("jacobi", "spai"):
        x, info = M.solve(b, tol=1e-10, pc=pc)
        xo, io = oracle.pcg(A2, w.b, 1e-10, pc=pc, eps=1e-3)
        assert _iters_ok(info[0].iters, io["iters"]) and rel(x.cpu().numpy(), xo) <= 1e-6, pc


@pytest.mark.parametrize("pc", ["none", "jacobi"])
def test_batch_with_a_frozen_system(cuda_device, pc):
    """A batch of 8 fp32 systems on one 5-point grid (the short-row sliced
    form).  System 3 has b = 0 and freezes at the start while the others
    iterate; every system's x and iteration count against the oracle, and
    its reported true residual."""
    w = build("c3", N=40, batch=8)
    b = w.b.copy()
    b[3] = 0.0
    M = make(w.A)
    assert M.layout()[0] in (6, 7)
    x, info = M.solve(torch.from_numpy(b).to(cuda_device), tol=w.tol, max_iter=20000, pc=pc, poll_k=16)
    xo, io = oracle.pcg(w.A, b, w.tol, max_iter=20000, pc=pc)
    xh = x.cpu().numpy()
    assert info[3].iters == 0 and not xh[3].any()
    for s in range(8):
        assert info[s].status == "ok" and io[s]["status"] == "ok"
        assert _iters_ok(info[s].iters, io[s]["iters"]), (s, info[s].iters, io[s]["iters"])
        assert rel(xh[s], xo[s]) <= 1e-6
        assert info[s].rel_res_true <= w.tol


def test_sliced_windows_batched(cuda_device):
    """Three systems on one kNN pattern (rows sorted by length within
    256-row windows, so the sliced products run a warp per window): the
    product, the fused product and dot, the Jacobi-PCG solve and BiCGStab
    per system against the oracle.  BiCGStab's iteration count on this
    symmetric problem moves with the rounding order (system 0: oracle 132,
    sliced 133, staged 142 iterations, measured), so for it x, the status
    and the true residual are checked, not the count."""
    A1 = build("c5", npoints=5000).A
    scale = np.array([1.0, 1.25, 1.5])
    A = CSR(A1.n, A1.row_ptr, A1.col_idx, np.stack([A1.vals * s for s in scale]))
    M = make(A)
    assert M.layout()[0] == 6
    g = np.random.default_rng(17)
    x = g.standard_normal((3, A.n))
    xd = torch.from_numpy(x).to(cuda_device)
    y = M.matvec(xd).cpu().numpy()
    yd, dots = M.matvec_dot(xd)
    assert np.array_equal(yd.cpu().numpy(), y)
    for s in range(3):
        yo = oracle.spmv(A, x[s], system=s)
        ref = oracle.spmv(CSR(A.n, A.row_ptr, A.col_idx, np.abs(A.vals[s])), np.abs(x[s]))
        assert np.all(np.abs(y[s] - yo) <= 1e-12 * ref)
        assert abs(dots[s].item() - float(x[s] @ y[s])) <= 1e-12 * float(np.abs(x[s]) @ np.abs(y[s]))
    b = g.standard_normal((3, A.n))
    bd = torch.from_numpy(b).to(cuda_device)
    for method in ("cg", "bicgstab"):
        xs, info = M.solve(bd, tol=1e-10, max_iter=5000, pc="jacobi", method=method)
        xo, io = (oracle.pcg if method == "cg" else oracle.bicgstab)(A, b, 1e-10, max_iter=5000, pc="jacobi")
        for s in range(3):
            assert info[s].status == "ok" and info[s].rel_res_true <= 1e-10, (method, s)
            if method == "cg":
                assert _iters_ok(info[s].iters, io[s]["iters"]), (method, s)
            assert rel(xs[s].cpu().numpy(), xo[s]) <= 1e-6
    assert M.layout_of("B")[0] == 6


def test_matrix_without_entries(cuda_device):
    """A pattern with no stored entries (nnz = 0, every row empty): the
    product and p.Ap are zero, and CG returns x = 0 as the oracle does --
    after 0 iterations with status ok for b = 0, and with status breakdown
    (p.Ap = 0 at the first step) otherwise."""
    n = 1000
    A = CSR(n, np.zeros(n + 1, np.int32), np.zeros(0, np.int32), np.zeros(0))
    M = make(A)
    assert M.layout()[0] == 5
    x = torch.from_numpy(np.random.default_rng(2).standard_normal(n)).to(cuda_device)
    assert not M.matvec(x).cpu().numpy().any()
    y, dot = M.matvec_dot(x)
    assert not y.cpu().numpy().any() and dot.item() == 0.0
    for b in (np.zeros(n), np.random.default_rng(3).standard_normal(n)):
        xs, info = M.solve(torch.from_numpy(b).to(cuda_device), tol=1e-8, max_iter=100)
        xo, io = oracle.pcg(A, b, 1e-8, max_iter=100, pc="none")
        assert (info[0].status, info[0].iters) == (io["status"], io["iters"]), (info[0], io)
        assert not xs.cpu().numpy().any()


def _window_pattern(n, lo, hi, seed):
    """Rows of lo..hi random columns, 2% of them empty, plus an empty block
    of 100 rows inside the third 256-row window and 7 empty rows at the end."""
    g = np.random.default_rng(seed)
    lens = g.integers(lo, hi + 1, n)
    lens[g.random(n) < 0.02] = 0
    lens[512:612] = 0
    lens[-7:] = 0
    rp = np.zeros(n + 1, np.int64)
    rp[1:] = np.cumsum(lens)
    ci = np.concatenate([np.sort(g.choice(n, size=k, replace=False)) for k in lens])
    return CSR(n, rp.astype(np.int32), ci.astype(np.int32), g.standard_normal(int(rp[-1])))


def _slice_widths(lens, window):
    """Widths of the 32-row slices with the rows in their own order and with
    the rows of every window sorted by decreasing length."""
    n = lens.size
    ns = (n + 31) // 32

    def widths(v):
        return np.concatenate([v, np.zeros(ns * 32 - n, v.dtype)]).reshape(ns, 32).max(1)
    return widths(lens), widths(np.concatenate([np.sort(lens[w:w + window])[::-1] for w in range(0, n, window)]))


@pytest.mark.parametrize("dtype", [np.float64, np.float32])
@pytest.mark.parametrize("sliced", [False, True], ids=["default", "sliced"])
@pytest.mark.parametrize("lo,hi,form", [(12, 18, 6), (5, 7, 7)], ids=["long", "short"])
def test_sliced_windows_with_empty_rows(cuda_device, lo, hi, form, sliced, dtype):
    """The sliced products on rows sorted by length within 256-row windows
    (a warp per window, its sums written in row order) where windows hold
    empty rows, whole slices of them, and the last window and slice are
    ragged (3001 rows): y = A x and p.Ap against the oracle."""
    A = _window_pattern(3001, lo, hi, seed=lo)
    lens = np.diff(A.row_ptr.astype(np.int64))
    w_rows, w_sorted = _slice_widths(lens, 256)
    pad_rows, pad_sorted = 32 * int(w_rows.sum()), 32 * int(w_sorted.sum())
    # the layout these rows get: sorted within 256-row windows (sorting pads
    # less, and at most 6% over nnz at the smallest window), within the
    # sliced form's padding limit, with whole slices of empty rows
    assert pad_sorted <= 1.06 * A.nnz < pad_rows and pad_rows > 1.02 * A.nnz
    assert (w_sorted == 0).sum() >= 3
    A = CSR(A.n, A.row_ptr, A.col_idx, A.vals.astype(dtype))
    M = make(A, reorder=False, sliced=sliced)
    assert M.layout()[0] == form, M.layout()
    x = np.random.default_rng(23).standard_normal(A.n).astype(dtype)
    xd = torch.from_numpy(x).to(cuda_device)
    y = M.matvec(xd).cpu().numpy()
    y_o = oracle.spmv(A, x.astype(np.float64))
    scale = oracle.spmv(CSR(A.n, A.row_ptr, A.col_idx, np.abs(A.vals)), np.abs(x.astype(np.float64)))
    assert np.all(np.abs(y - y_o) <= SPMV_TOL[dtype] * np.maximum(scale, 1e-300) + (0 if dtype == np.float64 else 1e-30))
    assert np.all(y[lens == 0] == 0)
    yd, dot = M.matvec_dot(xd)
    assert np.array_equal(yd.cpu().numpy(), y)
    d_o = float(x.astype(np.float64) @ y.astype(np.float64))
    assert abs(dot.item() - d_o) <= 1e-12 * max(1.0, float(np.abs(x) @ np.abs(y)))


@pytest.mark.parametrize("reorder,sliced", [(False, False), (True, False), (False, True), (True, True)])
def test_spai_follows_update_values(cuda_device, reorder, sliced):
    """After a SPAI solve, new values (a symmetric scaling D A D, same
    pattern) give the SPAI factor of the new matrix: the handle keeps G's
    pattern, permutation and layout and recomputes only its values (also
    for a reordered handle and for sliced factors)."""
    w = build("c5", npoints=6000)
    A = w.A
    M = make(A, reorder=reorder, sliced=sliced)
    assert M.layout()[2] == reorder
    b = torch.from_numpy(w.b).to(cuda_device)
    x1, i1 = M.solve(b, tol=1e-10, pc="spai", eps=1e-3)
    xo1, io1 = oracle.pcg(A, w.b, 1e-10, pc="spai", eps=1e-3)
    assert _iters_ok(i1[0].iters, io1["iters"]) and rel(x1.cpu().numpy(), xo1) <= 1e-6
    d = 0.5 + np.random.default_rng(4).random(A.n)
    v2 = A.vals * d[A.rows()] * d[A.col_idx]
    A2 = CSR(A.n, A.row_ptr, A.col_idx, v2)
    M.update_values(torch.from_numpy(v2).to(cuda_device))
    x2, i2 = M.solve(b, tol=1e-10, pc="spai", eps=1e-3)
    xo2, io2 = oracle.pcg(A2, w.b, 1e-10, pc="spai", eps=1e-3)
    assert i2[0].status == "ok" and _iters_ok(i2[0].iters, io2["iters"])
    assert rel(x2.cpu().numpy(), xo2) <= 1e-6
    lam, dA, ai = M.adjoint(x2, torch.from_numpy(w.g).to(cuda_device), tol=1e-10, pc="spai", eps=1e-3)
    lo, dAo, ao = oracle.adjoint(A2, x2.cpu().numpy(), w.g, 1e-10, pc="spai", eps=1e-3)
    assert _iters_ok(ai[0].iters, ao["iters"]) and rel(lam.cpu().numpy(), lo) <= 1e-6


@pytest.mark.parametrize("cfg", ["c5", "c3"])
def test_spai_batch_follows_update_values(cuda_device, cfg):
    """Three systems on one pattern with SPAI (the kNN Laplacian in fp64,
    the 2D grid in fp32): after new values for every system (D_s A_s D_s,
    a different scaling per system) each system's factor is that of its new
    matrix -- the positions of G^T's values in A found at the first fill
    serve all systems and every later fill -- so every solve matches the
    oracle's on the new values."""
    g = np.random.default_rng(9)
    if cfg == "c5":
        A1 = build("c5", npoints=4000).A
        A = CSR(A1.n, A1.row_ptr, A1.col_idx, np.stack([A1.vals * s for s in (1.0, 1.5, 0.75)]))
        b, tol = g.standard_normal((3, A.n)), 1e-10
    else:
        w = build("c3", N=32, batch=3)
        A, b, tol = w.A, w.b, w.tol
    bd = torch.from_numpy(b).to(cuda_device)
    M = make(A)

    def check(Ak):
        x, info = M.solve(bd, tol=tol, max_iter=20000, pc="spai", eps=1e-3)
        xo, io = oracle.pcg(Ak, b, tol, max_iter=20000, pc="spai", eps=1e-3)
        for s in range(3):
            assert info[s].status == "ok" and io[s]["status"] == "ok"
            assert _iters_ok(info[s].iters, io[s]["iters"]), (s, info[s].iters, io[s]["iters"])
            assert rel(x[s].cpu().numpy(), xo[s]) <= 1e-6
            assert info[s].rel_res_true <= tol
    check(A)
    r = A.rows()
    v2 = np.stack([A.vals[s] * d[r] * d[A.col_idx] for s, d in enumerate(0.5 + g.random((3, A.n)))])
    A2 = CSR(A.n, A.row_ptr, A.col_idx, v2.astype(A.vals.dtype))
    M.update_values(torch.from_numpy(A2.vals).to(cuda_device))
    check(A2)


def _walk_costs(rp):
    """Warp-wide fp64 steps of a staged product over 32-row groups, summed:
    one lane per row (the longest row of every group) and with the group's
    entries split into 32 runs of C = ceil(cnt / 32) entries rounded up to
    odd, plus the rounds joining the pieces of cut rows."""
    rp = np.asarray(rp, dtype=np.int64)
    n = rp.size - 1
    row = split = 0
    for r0 in range(0, n, 32):
        r1 = min(r0 + 32, n)
        lo, hi = rp[r0:r1] - rp[r0], rp[r0 + 1:r1 + 1] - rp[r0]
        cnt = int(hi[-1])
        if cnt == 0:
            continue
        C = ((cnt + 31) // 32) | 1
        ne = hi > lo
        row += int((hi - lo).max())
        split += C + int(((hi[ne] - 1) // C - lo[ne] // C).max())
    return row, split


def _lower_and_transpose(A):
    rows = A.rows()
    keep = A.col_idx <= rows
    r, c = rows[keep], A.col_idx[keep]
    rp_g = np.zeros(A.n + 1, np.int64)
    rp_g[1:] = np.cumsum(np.bincount(r, minlength=A.n))
    rp_t = np.zeros(A.n + 1, np.int64)
    rp_t[1:] = np.cumsum(np.bincount(c, minlength=A.n))
    return rp_g, rp_t


def _skewed_spd(n, seed):
    """Symmetric, strictly diagonally dominant matrix: every 32nd row holds
    40 random columns of its own within 500 of the diagonal, the others 2,
    each mirrored (so every 32-row group holds a few rows far longer than
    the rest, and fits one lane per row)."""
    g = np.random.default_rng(seed)
    lens = np.full(n, 2)
    lens[::32] = 40
    r = np.repeat(np.arange(n), lens)
    c = np.clip(r + g.integers(-500, 501, size=r.size), 0, n - 1)
    r, c = np.concatenate([r, c]), np.concatenate([c, r])
    off = r != c
    key = np.unique(np.minimum(r[off], c[off]).astype(np.int64) * n + np.maximum(r[off], c[off]))
    lo, hi = key // n, key % n
    v = -(0.1 + g.random(key.size))
    r = np.concatenate([lo, hi, np.arange(n)])
    c = np.concatenate([hi, lo, np.arange(n)])
    v = np.concatenate([v, v, np.zeros(n)])
    v[-n:] = np.bincount(r[:-n], weights=np.abs(v[:-n]), minlength=n) + 1.0
    order = np.lexsort((c, r))
    rp = np.zeros(n + 1, np.int32)
    rp[1:] = np.cumsum(np.bincount(r, minlength=n))
    return CSR(n, rp, c[order].astype(np.int32), v[order])


SPLIT_CASES = [("knn_20000", lambda: build("c5", npoints=20000).A), ("skewed_20000", lambda: _skewed_spd(20000, 5))]


@pytest.mark.parametrize("name,mk", SPLIT_CASES, ids=[c[0] for c in SPLIT_CASES])
def test_split_sums_follow_the_walk_cost(cuda_device, name, mk):
    """The staged product splits its groups' entries over the lanes exactly
    when the lane-per-row walk would cost at least 1.8 times the split one
    (warp-wide fp64 steps summed over the matrix), recomputed here from the
    patterns of A, G = tril(A) and G^T (caller order): on the skewed
    pattern all three split, on the kNN Laplacian (row lengths too even)
    none does.  By default and forced either way, the SPAI solve, the
    adjoint and the product match the oracle."""
    A = mk()
    rp_g, rp_t = _lower_and_transpose(A)
    gen = np.random.default_rng(21)
    bh, gh = gen.standard_normal(A.n), gen.standard_normal(A.n)
    b = torch.from_numpy(bh).to(cuda_device)
    g = torch.from_numpy(gh).to(cuda_device)
    xo, io = oracle.pcg(A, bh, 1e-10, pc="spai", eps=1e-3)
    lo_, _, ao = oracle.adjoint(A, xo, gh, 1e-10, pc="spai", eps=1e-3)
    for split in (None, True, False):
        M = make(A, reorder=False, staged=True, split=split)
        x, info = M.solve(b, tol=1e-10, pc="spai", eps=1e-3)
        for which, rp in (("A", A.row_ptr), ("G", rp_g), ("GT", rp_t)):
            form, _, sp = M.layout_of(which)
            assert form in (1, 2), (which, form)
            row, cut = _walk_costs(rp)
            want = {None: row >= 1.8 * cut, True: True, False: False}[split]
            assert sp == want, (which, split, row, cut, sp)
            if split is None:
                assert sp == (name == "skewed_20000"), (which, row, cut)
        assert info[0].status == "ok" and _iters_ok(info[0].iters, io["iters"]), (info[0].iters, io["iters"])
        assert rel(x.cpu().numpy(), xo) <= 1e-6
        lam, dA, ai = M.adjoint(x, g, tol=1e-10, pc="spai", eps=1e-3)
        assert _iters_ok(ai[0].iters, ao["iters"]) and rel(lam.cpu().numpy(), lo_) <= 1e-6
        assert rel(dA.cpu().numpy(), oracle.grad_A(A, lo_, xo)) <= 1e-6
        y = M.matvec(b).cpu().numpy()
        scale = oracle.spmv(CSR(A.n, A.row_ptr, A.col_idx, np.abs(A.vals)), np.abs(bh))
        assert np.all(np.abs(y - oracle.spmv(A, bh)) <= 1e-12 * scale)


@FUSED
def test_launch_count_advances(cuda_device, fused):
    """Kernel-per-step solves launch three kernels per iteration; the
    persistent kernel one per poll interval (plus set-up and the final pass)."""
    from sparse_iterative_linear_csr_b300 import launch_count
    w = build("c1")
    M = make(w.A, fused=fused)
    c0 = launch_count()
    _, info = M.solve(torch.from_numpy(w.b).to(cuda_device), tol=1e-10, poll_k=16)
    it = info[0].iters
    if fused:
        assert c0 + it // 16 + 2 <= launch_count() <= c0 + it // 16 + 8
    else:
        assert launch_count() >= c0 + 3 * it


@pytest.mark.parametrize("form,opt", [(3, "pipeline"), (4, "producer_consumer")])
def test_unaligned_values_leave_the_pipeline(cuda_device, form, opt):
    """Values at an 8-byte offset cannot be bulk-copied: the handle falls
    back to the default form, and returns to the bulk-copy form once
    aligned values are swapped in; products agree with the oracle."""
    A = poisson_grid((40, 40))
    from gpu_util import to_device
    from sparse_iterative_linear_csr_b300 import CSRMatrix
    rp, ci, v = to_device(A, cuda_device)
    buf = torch.zeros(A.nnz + 1, dtype=torch.float64, device=cuda_device)
    off = buf[1:]
    off.copy_(v)
    assert off.data_ptr() % 16 == 8
    x = np.random.default_rng(5).standard_normal(A.n)
    xd = torch.from_numpy(x).to(cuda_device)
    y_o = oracle.spmv(A, x)
    M = CSRMatrix(rp, ci, off, **{opt: True})
    assert M.layout()[0] in (0, 1, 2, 5)
    assert rel(M.matvec(xd).cpu().numpy(), y_o) <= 1e-13
    M.update_values(v)
    assert M.layout()[0] == form
    assert rel(M.matvec(xd).cpu().numpy(), y_o) <= 1e-13
    M.update_values(off)
    assert M.layout()[0] in (0, 1, 2, 5)
    xs, info = M.solve(torch.from_numpy(y_o).to(cuda_device), tol=1e-10, pc="jacobi")
    assert info[0].status == "ok" and rel(xs.cpu().numpy(), x) <= 1e-6


def test_product_time_records_live_launches(cuda_device):
    """With time_product the solve times one product kernel per graph
    launch; the per-launch time is positive and far below the solve time."""
    w = build("c2", N=96)
    from gpu_util import to_device
    from sparse_iterative_linear_csr_b300 import CSRMatrix
    rp, ci, v = to_device(w.A, cuda_device)
    M = CSRMatrix(rp, ci, v, time_product=True)
    b = torch.from_numpy(w.b).to(cuda_device)
    assert M.product_time() == (0.0, 0)
    _, info = M.solve(b, tol=w.tol, pc="jacobi", poll_k=8)
    ms, n = M.product_time(reset=False)
    assert n >= info[0].iters // 8 - 2 and ms > 0.0
    assert M.product_time(reset=True)[1] == n and M.product_time() == (0.0, 0)
    plain = CSRMatrix(rp, ci, v)
    plain.solve(b, tol=w.tol, pc="jacobi", poll_k=8)
    assert plain.product_time() == (0.0, 0)


# --------------------------------------------------------------- reordering
REORDER_CASES = [
    ("c2", {"N": 64}, "jacobi"),
    ("c5", {"npoints": 20000}, "spai"),
    ("c5", {"npoints": 20000}, "jacobi"),
    ("c3", {"N": 32, "batch": 3}, "jacobi"),
    ("c1", {}, "none"),
]


@pytest.mark.parametrize("fused", [False, True], ids=["steps", "fused"])
@pytest.mark.parametrize("cfg,kw,pc", REORDER_CASES, ids=[f"{c}-{p}" for c, k, p in REORDER_CASES])
def test_reordered_solve_and_adjoint_parity(cuda_device, cfg, kw, pc, fused):
    """Iterating on P A P^T (reverse Cuthill-McKee) solves the caller's
    system: x, iterations and the adjoint match the oracle on A itself."""
    w = build(cfg, **kw)
    M = make(w.A, reorder=True, fused=fused)
    assert M.layout()[2]
    b = torch.from_numpy(w.b).to(cuda_device)
    g = torch.from_numpy(w.g).to(cuda_device)
    x, info = M.solve(b, tol=w.tol, max_iter=20000, pc=pc, eps=1e-3, poll_k=16)
    xh = x.cpu().numpy()
    xo, io = oracle.pcg(w.A, w.b, w.tol, max_iter=20000, pc=pc, eps=1e-3)
    X, XO, IO = (xh, xo, io) if M.batch > 1 or w.A.vals.ndim == 2 else (xh[None], xo[None], [io])
    bs = w.b if w.b.ndim == 2 else w.b[None]
    for s in range(len(info)):
        assert info[s].status == "ok" and _iters_ok(info[s].iters, IO[s]["iters"]), (info[s].iters, IO[s]["iters"])
        assert rel(X[s], XO[s]) <= 1e-6
        assert abs(oracle.rel_residual(w.A, bs[s], X[s], system=s) - info[s].rel_res_true) <= 1e-3 * w.tol
    lb, la, ainfo = M.adjoint(x, g, tol=w.tol, max_iter=20000, pc=pc, eps=1e-3)
    lb_o, la_o, aio = oracle.adjoint(w.A, xh, w.g, w.tol, max_iter=20000, pc=pc, eps=1e-3)
    lb, la = lb.cpu().numpy(), la.cpu().numpy()
    if lb.ndim == 1:
        lb, la, lb_o, la_o, aio = lb[None], la[None], lb_o[None], la_o[None], [aio]
    for s in range(lb.shape[0]):
        assert ainfo[s].status == "ok" and _iters_ok(ainfo[s].iters, aio[s]["iters"])
        assert rel(lb[s], lb_o[s]) <= 1e-6 and rel(la[s], la_o[s]) <= 1e-6


def test_scattered_pattern_is_reordered(cuda_device):
    """A grid relabelled at random is detected as scattered and reordered;
    the solve still matches the oracle, the SpMV API still works on A, and
    an initial guess and new values pass through the permutation."""
    base = poisson_grid((400, 400))
    n = base.n
    perm = np.random.default_rng(4).permutation(n)
    inv = np.empty(n, np.int64)
    inv[perm] = np.arange(n)
    rows = base.rows()
    r2, c2 = inv[rows], inv[base.col_idx]
    order = np.lexsort((c2, r2))
    rp = np.zeros(n + 1, np.int64)
    np.cumsum(np.bincount(r2, minlength=n), out=rp[1:])
    A = CSR(n, rp.astype(np.int32), c2[order].astype(np.int32), base.vals[order])
    M = make(A)
    assert M.layout()[2], "a randomly relabelled grid should be reordered"
    assert not make(A, reorder=False).layout()[2]
    x_true = np.random.default_rng(2).standard_normal(n)
    b = oracle.spmv(A, x_true)
    bt = torch.from_numpy(b).to(cuda_device)
    assert rel(M.matvec(torch.from_numpy(x_true).to(cuda_device)).cpu().numpy(), b) <= 1e-13
    x, info = M.solve(bt, tol=1e-9, pc="jacobi", max_iter=20000)
    xo, io = oracle.pcg(A, b, 1e-9, pc="jacobi", max_iter=20000)
    assert info[0].status == "ok" and _iters_ok(info[0].iters, io["iters"])
    assert rel(x.cpu().numpy(), xo) <= 1e-6
    x0 = np.random.default_rng(3).standard_normal(n)
    x1, i1 = M.solve(bt, tol=1e-9, pc="jacobi", max_iter=20000, x0=torch.from_numpy(x0).to(cuda_device))
    xo1, io1 = oracle.pcg(A, b, 1e-9, pc="jacobi", max_iter=20000, x0=x0)
    assert _iters_ok(i1[0].iters, io1["iters"]) and rel(x1.cpu().numpy(), xo1) <= 1e-6
    M.update_values(M.values * 3.0)
    A3 = CSR(n, A.row_ptr, A.col_idx, A.vals * 3.0)
    x3, i3 = M.solve(bt, tol=1e-9, pc="jacobi", max_iter=20000)
    xo3, io3 = oracle.pcg(A3, b, 1e-9, pc="jacobi", max_iter=20000)
    assert _iters_ok(i3[0].iters, io3["iters"]) and rel(x3.cpu().numpy(), xo3) <= 1e-6


@pytest.mark.parametrize("which,what", [(0, b"bulk copy"), (1, b"grid barrier")])
def test_device_wait_gives_up_and_reports(cuda_device, which, what):
    """A device wait that never ends (an mbarrier nothing arrives at; a grid
    barrier one CTA never reaches) gives up after its limit (5 ms here),
    records where, and lets the kernel return: the call returns
    SLA_ERR_CUDA with the location, and the device stays usable."""
    import ctypes as C
    from sparse_iterative_linear_csr_b300 import _lib
    lib = _lib.load()
    stream = C.c_void_p(torch.cuda.current_stream().cuda_stream)
    assert lib.sla_wait_selftest(which, 0.005, stream) == _lib.SLA_ERR_CUDA
    msg = lib.sla_last_error()
    assert b"gave up" in msg and what in msg, msg
    assert lib.sla_wait_selftest(2, 0.005, stream) == _lib.SLA_ERR_INVALID
    w = build("c1", N=16)
    M = make(w.A)
    x, info = M.solve(torch.from_numpy(w.b).to(cuda_device), tol=1e-10)
    xo, _ = oracle.pcg(w.A, w.b, 1e-10)
    assert info[0].status == "ok" and rel(x.cpu().numpy(), xo) <= 1e-6
