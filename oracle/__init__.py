"""Python entry to the plain fp64 C oracle (oracle.c).

TEST INFRASTRUCTURE ONLY.  The product library never imports this package;
only the tests, the smoke check and the benchmark's CPU-baseline leg do.  The
oracle shares no code with the CUDA library: it is built from oracle.c alone
with gcc (no fused multiply-add) the first time it is needed, or by
``build_oracle()``.

Every function takes the CSR arrays of a workloads.CSR (int32 row_ptr /
col_idx; values fp64 or fp32 -- fp32 values are widened exactly) and returns
numpy arrays.  Batched systems are solved one by one on the shared pattern.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

PC = {"none": 0, "jacobi": 1, "spai": 2}
STATUS = {0: "ok", 1: "not_converged", 2: "breakdown", 3: "invalid"}

_dp = C.POINTER(C.c_double)
_ip = C.POINTER(C.c_int)


def build_oracle(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so next to it."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-ffp-contract=off", "-fno-fast-math",
                               "-shared", "-fPIC", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = C.CDLL(build_oracle())
            lib.oracle_spmv.argtypes = [C.c_int, _ip, _ip, _dp, _dp, _dp]
            lib.oracle_spmv.restype = None
            lib.oracle_spai_nnz.argtypes = [C.c_int, _ip, _ip]
            lib.oracle_spai_nnz.restype = C.c_longlong
            lib.oracle_spai_factor.argtypes = [C.c_int, _ip, _ip, _dp, _ip, _ip, _dp]
            lib.oracle_spai_factor.restype = C.c_int
            lib.oracle_spai_apply.argtypes = [C.c_int, _ip, _ip, _dp, C.c_double, C.c_int,
                                              _dp, _dp, _dp]
            lib.oracle_spai_apply.restype = None
            lib.oracle_pcg.argtypes = [C.c_int, _ip, _ip, _dp, _dp, _dp, C.c_double, C.c_int,
                                       C.c_int, C.c_double, C.c_int, C.c_int, _ip, _dp, _dp]
            lib.oracle_pcg.restype = C.c_int
            lib.oracle_adjoint.argtypes = [C.c_int, _ip, _ip, _dp, _dp, _dp, C.c_double,
                                           C.c_int, C.c_int, C.c_double, C.c_int, _dp, _dp,
                                           _ip, _dp, _dp]
            lib.oracle_adjoint.restype = C.c_int
            lib.oracle_grad_A.argtypes = [C.c_int, _ip, _ip, _dp, _dp, C.c_int, _dp]
            lib.oracle_grad_A.restype = None
            lib.oracle_rel_residual.argtypes = [C.c_int, _ip, _ip, _dp, _dp, _dp]
            lib.oracle_rel_residual.restype = C.c_double
            lib.oracle_bicgstab.argtypes = [C.c_int, _ip, _ip, _dp, _dp, _dp, C.c_double, C.c_int,
                                            C.c_int, C.c_int, _ip, _dp, _dp]
            lib.oracle_bicgstab.restype = C.c_int
            lib.oracle_bicgstab_adjoint.argtypes = [C.c_int, _ip, _ip, _dp, _dp, _dp, C.c_double,
                                                    C.c_int, C.c_int, _dp, _dp, _ip, _dp, _dp]
            lib.oracle_bicgstab_adjoint.restype = C.c_int
            _lib = lib
    return _lib


def _i(a):
    a = np.ascontiguousarray(a, dtype=np.int32)
    return a, a.ctypes.data_as(_ip)


def _d(a):
    a = np.ascontiguousarray(a, dtype=np.float64)
    return a, a.ctypes.data_as(_dp)


def _system_vals(A, s):
    v = A.vals if A.vals.ndim == 1 else A.vals[s]
    return v


def spmv(A, x, system: int = 0) -> np.ndarray:
    """y = A x in fp64 (row sums in stored order)."""
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, system))
    xx, xp = _d(x)
    y = np.empty(A.n, dtype=np.float64)
    lib.oracle_spmv(A.n, rpp, cip, vp, xp, y.ctypes.data_as(_dp))
    return y


def spai_factor(A, system: int = 0):
    """G on the pattern of tril(A): returns (row_ptr, col_idx, vals)."""
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, system))
    ng = lib.oracle_spai_nnz(A.n, rpp, cip)
    grp = np.empty(A.n + 1, dtype=np.int32)
    gci = np.empty(max(ng, 1), dtype=np.int32)
    gv = np.empty(max(ng, 1), dtype=np.float64)
    st = lib.oracle_spai_factor(A.n, rpp, cip, vp, grp.ctypes.data_as(_ip),
                                gci.ctypes.data_as(_ip), gv.ctypes.data_as(_dp))
    if st != 0:
        raise ValueError("SPAI factor needs a positive diagonal")
    return grp, gci[:ng], gv[:ng]


def spai_apply(A, r, eps: float, f32: bool = False, system: int = 0) -> np.ndarray:
    """z = G (G^T r) + eps r for the closed-form G of A."""
    lib = _load()
    grp, gci, gv = spai_factor(A, system)
    grp, grpp = _i(grp)
    gci, gcip = _i(gci)
    gv, gvp = _d(gv)
    rr, rp_ = _d(r)
    t = np.empty(A.n, dtype=np.float64)
    z = np.empty(A.n, dtype=np.float64)
    lib.oracle_spai_apply(A.n, grpp, gcip, gvp, float(eps), int(f32), rp_,
                          t.ctypes.data_as(_dp), z.ctypes.data_as(_dp))
    return z


def _solve_one(A, s, b, tol, max_iter, pc, eps, f32, x0):
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, s))
    bb, bp = _d(b)
    x = np.zeros(A.n, dtype=np.float64) if x0 is None else np.array(x0, dtype=np.float64)
    it = C.c_int(0)
    rr = C.c_double(0)
    rt = C.c_double(0)
    st = lib.oracle_pcg(A.n, rpp, cip, vp, bp, x.ctypes.data_as(_dp), float(tol), int(max_iter),
                        PC[pc], float(eps), int(f32), int(x0 is not None), C.byref(it),
                        C.byref(rr), C.byref(rt))
    return x, dict(iters=it.value, rel_res_recursive=rr.value, rel_res_true=rt.value,
                   status=STATUS[st])


def pcg(A, b, tol, max_iter=100000, pc="none", eps=0.0, f32=None, x0=None):
    """Solve A x = b (batched over the first axis of b when A is batched).

    Returns (x, info) for one system or (x[batch, n], [info, ...]) for a batch.
    f32 defaults to "A.vals is float32"."""
    if f32 is None:
        f32 = A.vals.dtype == np.float32
    if A.vals.ndim == 1:
        return _solve_one(A, 0, b, tol, max_iter, pc, eps, f32, x0)
    xs, infos = [], []
    for s in range(A.vals.shape[0]):
        x, inf = _solve_one(A, s, b[s], tol, max_iter, pc, eps, f32,
                            None if x0 is None else x0[s])
        xs.append(x)
        infos.append(inf)
    return np.stack(xs), infos


def _adjoint_one(A, s, x, g, tol, max_iter, pc, eps, f32, with_dA=True):
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, s))
    gg, gp = _d(g)
    if with_dA:
        xx, xp = _d(x)
        dlda = np.zeros(A.nnz, dtype=np.float64)
        dp = dlda.ctypes.data_as(_dp)
    else:
        xp = dlda = dp = None
    dldb = np.zeros(A.n, dtype=np.float64)
    it = C.c_int(0)
    rr = C.c_double(0)
    rt = C.c_double(0)
    st = lib.oracle_adjoint(A.n, rpp, cip, vp, xp, gp, float(tol), int(max_iter), PC[pc],
                            float(eps), int(f32), dldb.ctypes.data_as(_dp),
                            dp, C.byref(it), C.byref(rr), C.byref(rt))
    return dldb, dlda, dict(iters=it.value, rel_res_recursive=rr.value,
                            rel_res_true=rt.value, status=STATUS[st])


def adjoint(A, x, g, tol, max_iter=100000, pc="none", eps=0.0, f32=None, with_dA=True):
    """(dL/db, dL/dA on the pattern, info) for upstream gradient g = dL/dx.
    with_dA=False solves for lambda only (x is not read; dL/dA is None)."""
    if f32 is None:
        f32 = A.vals.dtype == np.float32
    if A.vals.ndim == 1:
        return _adjoint_one(A, 0, x, g, tol, max_iter, pc, eps, f32, with_dA)
    out = [_adjoint_one(A, s, None if x is None else x[s], g[s], tol, max_iter, pc, eps, f32, with_dA)
           for s in range(A.vals.shape[0])]
    return (np.stack([o[0] for o in out]),
            np.stack([o[1] for o in out]) if with_dA else None,
            [o[2] for o in out])


def grad_A(A, lam, x, f32=None, system: int = 0) -> np.ndarray:
    """dL/dA_k = -lambda_row(k) x_col(k) on the stored pattern (rounded to
    fp32 in fp32 mode), for one system."""
    if f32 is None:
        f32 = A.vals.dtype == np.float32
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    ll, lp = _d(lam)
    xx, xp = _d(x)
    out = np.empty(max(A.nnz, 1), dtype=np.float64)
    lib.oracle_grad_A(A.n, rpp, cip, lp, xp, int(f32), out.ctypes.data_as(_dp))
    return out[:A.nnz]


def _bicgstab_one(A, s, b, tol, max_iter, pc, x0):
    if pc not in ("none", "jacobi"):
        raise ValueError("BiCGStab takes pc 'none' or 'jacobi'")
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, s))
    bb, bp = _d(b)
    x = np.zeros(A.n, dtype=np.float64) if x0 is None else np.array(x0, dtype=np.float64)
    it = C.c_int(0)
    rr = C.c_double(0)
    rt = C.c_double(0)
    st = lib.oracle_bicgstab(A.n, rpp, cip, vp, bp, x.ctypes.data_as(_dp), float(tol), int(max_iter),
                             PC[pc], int(x0 is not None), C.byref(it), C.byref(rr), C.byref(rt))
    return x, dict(iters=it.value, rel_res_recursive=rr.value, rel_res_true=rt.value,
                   status=STATUS[st])


def bicgstab(A, b, tol, max_iter=100000, pc="none", x0=None):
    """Solve a general (nonsymmetric) A x = b by right-preconditioned
    BiCGStab in fp64; batched like pcg."""
    if A.vals.ndim == 1:
        return _bicgstab_one(A, 0, b, tol, max_iter, pc, x0)
    out = [_bicgstab_one(A, s, b[s], tol, max_iter, pc, None if x0 is None else x0[s])
           for s in range(A.vals.shape[0])]
    return np.stack([o[0] for o in out]), [o[1] for o in out]


def _bicgstab_adjoint_one(A, s, x, g, tol, max_iter, pc):
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, s))
    xx, xp = _d(x)
    gg, gp = _d(g)
    dldb = np.zeros(A.n, dtype=np.float64)
    dlda = np.zeros(A.nnz, dtype=np.float64)
    it = C.c_int(0)
    rr = C.c_double(0)
    rt = C.c_double(0)
    st = lib.oracle_bicgstab_adjoint(A.n, rpp, cip, vp, xp, gp, float(tol), int(max_iter), PC[pc],
                                     dldb.ctypes.data_as(_dp), dlda.ctypes.data_as(_dp),
                                     C.byref(it), C.byref(rr), C.byref(rt))
    return dldb, dlda, dict(iters=it.value, rel_res_recursive=rr.value,
                            rel_res_true=rt.value, status=STATUS[st])


def bicgstab_adjoint(A, x, g, tol, max_iter=100000, pc="none"):
    """(dL/db, dL/dA on the pattern, info) for a general A: A^T lambda = g
    solved by BiCGStab on the explicit transpose."""
    if A.vals.ndim == 1:
        return _bicgstab_adjoint_one(A, 0, x, g, tol, max_iter, pc)
    out = [_bicgstab_adjoint_one(A, s, x[s], g[s], tol, max_iter, pc)
           for s in range(A.vals.shape[0])]
    return (np.stack([o[0] for o in out]), np.stack([o[1] for o in out]),
            [o[2] for o in out])


def rel_residual(A, b, x, system: int = 0) -> float:
    lib = _load()
    rp, rpp = _i(A.row_ptr)
    ci, cip = _i(A.col_idx)
    v, vp = _d(_system_vals(A, system))
    bb, bp = _d(b)
    xx, xp = _d(x)
    return lib.oracle_rel_residual(A.n, rpp, cip, vp, bp, xp)


def eigsh_dense(A, k, largest=False, system: int = 0):
    """The k smallest (largest) eigenpairs of the symmetric matrix A, by the
    plain definition: a dense symmetric eigendecomposition (LAPACK through
    numpy.linalg.eigh) of the matrix the CSR arrays describe.  Returns
    (eigenvalues ascending [k] (descending when largest), eigenvectors [k, n])."""
    n = A.n
    D = np.zeros((n, n))
    rows = np.repeat(np.arange(n), np.diff(A.row_ptr))
    D[rows, A.col_idx] = _system_vals(A, system)
    w, V = np.linalg.eigh((D + D.T) / 2)
    if largest:
        w, V = w[::-1], V[:, ::-1]
    return w[:k].copy(), V[:, :k].T.copy()
