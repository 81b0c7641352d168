"""B300 (sm_103a) preconditioned conjugate gradient on CSR matrices, with the
adjoint backward pass.

Python face of libsla.so: it only marshals torch CUDA tensors (device memory
and the current stream) into the C ABI of include/sla.h; every step of the
solve runs in the library's kernels.

    A = CSRMatrix(row_ptr, col_idx, values)          # int32, int32, fp64/fp32 (CUDA)
    x, info = A.solve(b, tol=1e-8, pc="jacobi")
    y = A.matvec(x)
    x = solve(A, values, b, tol=1e-8)               # differentiable in values and b

A batch of systems on one pattern: values [batch, nnz], b [batch, n].
Follows torch-sla (arXiv 2601.13994): §3 (SparseTensor with a shared-pattern
batch, .matvec / .solve, autograd wrapper stashing (A, x) and running one
adjoint solve in backward) and §3.3 (the adjoint gradient -lambda_i x_j on the
stored non-zeros).
"""
from __future__ import annotations

import ctypes as C
from dataclasses import dataclass

import torch

from . import _lib
from ._lib import PC, STATUS_NAMES

__all__ = ["CSRMatrix", "SLAError", "SolveInfo", "solve", "launch_count"]


class SLAError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status
        self.status_name = STATUS_NAMES.get(status, str(status))


@dataclass
class SolveInfo:
    iters: int
    rel_res_recursive: float
    rel_res_true: float
    status: str


def _lib_handle():
    return _lib.load()


def _check(st: int, allow=()):
    if st != _lib.SLA_OK and st not in allow:
        raise SLAError(st, _lib_handle().sla_last_error().decode())
    return st


def _stream(stream=None) -> C.c_void_p:
    s = torch.cuda.current_stream() if stream is None else stream
    return C.c_void_p(s.cuda_stream)


def _ptr(t: torch.Tensor) -> C.c_void_p:
    return C.c_void_p(t.data_ptr())


def launch_count() -> int:
    """Kernels libsla has launched in this process (graph nodes included)."""
    return int(_lib_handle().sla_launch_count())


def _method(method: str, cg: str, bicgstab: str):
    if method not in ("cg", "bicgstab"):
        raise ValueError(f"method must be 'cg' or 'bicgstab', not {method!r}")
    return getattr(_lib_handle(), cg if method == "cg" else bicgstab)


class CSRMatrix:
    """A CSR matrix (or a batch of matrices sharing one pattern) on the GPU.

    row_ptr: int32 [n+1], col_idx: int32 [nnz] (ascending per row), values:
    float64 or float32 [nnz] or [batch, nnz]; all CUDA tensors, kept alive by
    this object.  validate=True checks the structure on the device;
    pipeline=True uses the warp-pipeline product where it applies;
    fused=True runs CG / Jacobi-PCG as the persistent iteration kernel
    instead of a CUDA graph of one kernel per step; time_product=True
    records the live duration of one product kernel per graph launch
    (product_time); producer_consumer=True uses the producer/consumer
    product where it applies; reorder=True / False forces / forbids
    iterating on a reverse Cuthill-McKee reordering (default: reorder
    scattered patterns); staged=True keeps the warp-staged product forms
    where the direct (thread-per-row) or the sliced form would be the
    default, for every matrix of the solves;
    sliced=True uses the sliced product form (a handle-owned copy of the
    iteration matrix and of the SPAI factors in 32-row slices) where it
    applies; split=True / False forces / forbids summing the staged groups
    with their entries split evenly over the lanes (default: chosen per
    matrix from its row lengths)."""

    def __init__(self, row_ptr: torch.Tensor, col_idx: torch.Tensor, values: torch.Tensor,
                 validate: bool = True, pipeline: bool = False, fused: bool = False,
                 time_product: bool = False, producer_consumer: bool = False, reorder: bool | None = None,
                 staged: bool = False, sliced: bool = False, split: bool | None = None, stream=None):
        lib = _lib_handle()
        for t, name in ((row_ptr, "row_ptr"), (col_idx, "col_idx"), (values, "values")):
            if not t.is_cuda:
                raise ValueError(f"{name} must be a CUDA tensor")
            if not t.is_contiguous():
                raise ValueError(f"{name} must be contiguous")
        if row_ptr.dtype != torch.int32 or col_idx.dtype != torch.int32:
            raise ValueError("row_ptr and col_idx must be int32")
        if values.dtype not in (torch.float64, torch.float32):
            raise ValueError("values must be float64 or float32")
        self.n = row_ptr.numel() - 1
        self.nnz = col_idx.numel()
        self.batch = 1 if values.dim() == 1 else values.shape[0]
        if values.shape[-1] != self.nnz:
            raise ValueError("values must have nnz entries per system")
        self.dtype = values.dtype
        self.row_ptr, self.col_idx, self.values = row_ptr, col_idx, values
        self._h = C.c_void_p()
        dt = _lib.SLA_F64 if values.dtype == torch.float64 else _lib.SLA_F32
        _check(lib.sla_csr_create(self.n, self.nnz, self.batch, dt, _ptr(row_ptr), _ptr(col_idx),
                                  _ptr(values), (_lib.SLA_VALIDATE if validate else 0) |
                                  (_lib.SLA_WARP_PIPELINE if pipeline else 0) |
                                  (_lib.SLA_PERSISTENT if fused else 0) |
                                  (_lib.SLA_TIME_PRODUCT if time_product else 0) |
                                  (_lib.SLA_PRODUCER_CONSUMER if producer_consumer else 0) |
                                  (_lib.SLA_STAGED if staged else 0) |
                                  (_lib.SLA_SLICED if sliced else 0) |
                                  ({None: 0, True: _lib.SLA_SPLIT_ROWS, False: _lib.SLA_ROW_WALK}[split]) |
                                  ({None: 0, True: _lib.SLA_REORDER, False: _lib.SLA_NO_REORDER}[reorder]),
                                  _stream(stream),
                                  C.byref(self._h)))

    # -------------------------------------------------------------- lifetime
    def close(self):
        if getattr(self, "_h", None) and self._h.value:
            _lib_handle().sla_csr_destroy(self._h)
            self._h = C.c_void_p()

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def __enter__(self):
        return self

    def __exit__(self, *a):
        self.close()

    # -------------------------------------------------------------- helpers
    def _vec_shape(self):
        return (self.n,) if self.batch == 1 and self.values.dim() == 1 else (self.batch, self.n)

    def _check_vec(self, v: torch.Tensor, name: str):
        if not v.is_cuda or v.dtype != self.dtype or not v.is_contiguous():
            raise ValueError(f"{name} must be a contiguous CUDA tensor of dtype {self.dtype}")
        if v.numel() != self.batch * self.n:
            raise ValueError(f"{name} must have batch*n = {self.batch * self.n} entries")

    @staticmethod
    def _opts(tol, max_iter, pc, eps, poll_k, use_x0, timeout_s):
        if pc not in PC:
            raise ValueError(f"pc must be one of {sorted(PC)}")
        return _lib.PcgOpts(float(tol), int(max_iter), PC[pc], float(eps), int(poll_k), int(use_x0),
                            float(timeout_s))

    def _infos(self, arr):
        return [SolveInfo(a.iters, a.rel_res_recursive, a.rel_res_true, STATUS_NAMES[a.status]) for a in arr]

    # -------------------------------------------------------------- API
    def product_time(self, reset: bool = True) -> tuple[float, int]:
        """(summed ms, launches timed) of the live product kernel (time_product=True)."""
        ms, n = C.c_double(), C.c_longlong()
        _check(_lib_handle().sla_product_time(self._h, C.byref(ms), C.byref(n), int(reset)))
        return ms.value, n.value

    def layout(self) -> tuple[int, int, bool]:
        """(product form 0..5, CTAs per system, reordered) of the matrix the solves iterate on."""
        f, g, r = C.c_int(), C.c_int(), C.c_int()
        _check(_lib_handle().sla_csr_layout(self._h, C.byref(f), C.byref(g), C.byref(r)))
        return f.value, g.value, bool(r.value)

    def layout_of(self, which: str = "A") -> tuple[int, int, bool]:
        """(product form, CTAs per system, split group sums) of the iteration
        matrix ("A"); after a SPAI solve of the factor "G" or "GT"; after a
        BiCGStab solve of its matrix "B", after its adjoint of "BT"."""
        f, g, b = C.c_int(), C.c_int(), C.c_int()
        _check(_lib_handle().sla_csr_layout_of(self._h, {"A": 0, "G": 1, "GT": 2, "B": 3, "BT": 4}[which],
                                               C.byref(f), C.byref(g), C.byref(b)))
        return f.value, g.value, bool(b.value)

    def update_values(self, values: torch.Tensor, stream=None):
        if values.dtype != self.dtype or values.numel() != self.batch * self.nnz or not values.is_cuda:
            raise ValueError("values must match the handle's dtype and size")
        values = values.contiguous()
        _check(_lib_handle().sla_csr_update_values(self._h, _ptr(values), _stream(stream)))
        self.values = values

    def matvec(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        """y = A x (torch-sla §3, .matvec)."""
        self._check_vec(x, "x")
        y = torch.empty_like(x)
        _check(_lib_handle().sla_spmv(self._h, _ptr(x), _ptr(y), _stream(stream)))
        return y

    def matvec_dot(self, x: torch.Tensor, stream=None):
        """(y = A x, x.y per system) from the fused SpMV + inner-product kernel."""
        self._check_vec(x, "x")
        y = torch.empty_like(x)
        d = torch.empty(self.batch, dtype=torch.float64, device=x.device)
        _check(_lib_handle().sla_spmv_dot(self._h, _ptr(x), _ptr(y), _ptr(d), _stream(stream)))
        return y, d

    def solve(self, b: torch.Tensor, tol: float = 1e-8, max_iter: int = 10000, pc: str = "none",
              eps: float = 1e-3, poll_k: int = 32, x0: torch.Tensor | None = None,
              timeout_s: float = 0.0, raise_on_fail: bool = False, method: str = "cg", stream=None):
        """Solve A x = b; returns (x, [SolveInfo per system]).  method "cg":
        preconditioned CG (symmetric positive definite A); "bicgstab":
        BiCGStab for a general A (fp64; pc "none" or "jacobi")."""
        self._check_vec(b, "b")
        if x0 is not None:
            self._check_vec(x0, "x0")
            x = x0.clone()
        else:
            x = torch.empty_like(b)
        o = self._opts(tol, max_iter, pc, eps, poll_k, x0 is not None, timeout_s)
        info = (_lib.SolveInfo * self.batch)()
        fn = _method(method, "sla_pcg_solve", "sla_bicgstab_solve")
        st = fn(self._h, _ptr(b), _ptr(x), C.byref(o), info, _stream(stream))
        _check(st, allow=() if raise_on_fail else (_lib.SLA_ERR_NOT_CONVERGED, _lib.SLA_ERR_BREAKDOWN,
                                                   _lib.SLA_ERR_TIMEOUT))
        return x, self._infos(info)

    def adjoint(self, x: torch.Tensor, g: torch.Tensor, tol: float = 1e-8, max_iter: int = 10000,
                pc: str = "none", eps: float = 1e-3, poll_k: int = 32, want_dA: bool = True,
                timeout_s: float = 0.0, method: str = "cg", stream=None):
        """(dL/db, dL/dA on the pattern or None, [SolveInfo]) for g = dL/dx.
        method "bicgstab" solves A^T lambda = g on an explicit transpose."""
        self._check_vec(x, "x")
        self._check_vec(g, "g")
        dldb = torch.empty_like(g)
        dlda = torch.empty_like(self.values) if want_dA else None
        o = self._opts(tol, max_iter, pc, eps, poll_k, False, timeout_s)
        info = (_lib.SolveInfo * self.batch)()
        fn = _method(method, "sla_adjoint", "sla_bicgstab_adjoint")
        st = fn(self._h, _ptr(x), _ptr(g), C.byref(o), _ptr(dldb), _ptr(dlda) if dlda is not None else None, info,
                _stream(stream))
        _check(st, allow=(_lib.SLA_ERR_NOT_CONVERGED, _lib.SLA_ERR_BREAKDOWN, _lib.SLA_ERR_TIMEOUT))
        return dldb, dlda, self._infos(info)


class _Solve(torch.autograd.Function):
    @staticmethod
    def forward(ctx, values, b, A, kw):
        if values.data_ptr() != A.values.data_ptr():
            A.update_values(values)
        x, info = A.solve(b.contiguous(), **kw)
        ctx.A, ctx.kw = A, kw
        ctx.save_for_backward(x)
        ctx.info = info
        return x

    @staticmethod
    def backward(ctx, gx):
        (x,) = ctx.saved_tensors
        kw = {k: v for k, v in ctx.kw.items()
              if k in ("tol", "max_iter", "pc", "eps", "poll_k", "timeout_s", "method")}
        dldb, dlda, _ = ctx.A.adjoint(x, gx.contiguous(), want_dA=ctx.needs_input_grad[0], **kw)
        return (dlda if ctx.needs_input_grad[0] else None,
                dldb if ctx.needs_input_grad[1] else None, None, None)


def solve(A: CSRMatrix, values: torch.Tensor, b: torch.Tensor, **kw) -> torch.Tensor:
    """x = A(values)^-1 b, differentiable with respect to values and b: the
    backward pass is one adjoint solve (A^T lambda = dL/dx) plus
    dL/dA_ij = -lambda_i x_j on the stored entries.  method="bicgstab"
    (keyword) serves a nonsymmetric A, forward and adjoint."""
    return _Solve.apply(values, b, A, kw)
