"""The allocation-free fused SpMV + dot entry point (sla_spmv_dot_static),
called through the C ABI, against the handle-based sla_spmv_dot on the same
inputs, twice in a row (the shared device scratch keeps the previous call's
contents).  It serves callers that cannot let the library allocate device
memory: programs that own all device memory through their own allocator,
and latency-critical loops where cudaMalloc / cudaFree would synchronise the
device.  Collected last on purpose."""
import ctypes as C

import numpy as np
import pytest
import torch

from workloads import build
from workloads.matrices import CSR

from gpu_util import make, random_csr

pytestmark = pytest.mark.gpu


def _static_call(lib, M, x, y, dot, stream):
    from sparse_iterative_linear_csr_b300 import _lib
    dt = _lib.SLA_F64 if M.dtype == torch.float64 else _lib.SLA_F32
    return lib.sla_spmv_dot_static(M.n, M.nnz, M.batch, dt, C.c_void_p(M.row_ptr.data_ptr()),
                                   C.c_void_p(M.col_idx.data_ptr()), C.c_void_p(M.values.data_ptr()),
                                   C.c_void_p(x.data_ptr()), C.c_void_p(y.data_ptr()),
                                   C.c_void_p(dot.data_ptr()), C.c_void_p(stream.cuda_stream))


def _cases():
    yield "diffusion_96_f64", build("c2", N=96).A
    yield "poisson3d_20_f64", build("c4", N=20).A
    yield "knn_4000_f64", build("c5", npoints=4000).A
    yield "empty_rows_f64", random_csr(700, 5, seed=2, empty_rows=30)
    yield "batch3_f32", build("c3", N=40, batch=3).A
    A = build("c2", N=50).A
    yield "diffusion_50_f32", CSR(A.n, A.row_ptr, A.col_idx, A.vals.astype(np.float32))


@pytest.mark.parametrize("name,A", list(_cases()), ids=lambda v: v if isinstance(v, str) else "")
def test_static_matches_handle_entry_point(cuda_device, name, A):
    from sparse_iterative_linear_csr_b300 import _lib
    lib = _lib.load()
    M = make(A)
    g = np.random.default_rng(5)
    shape = (A.n,) if A.vals.ndim == 1 else (A.vals.shape[0], A.n)
    x = torch.from_numpy(g.standard_normal(shape).astype(A.vals.dtype)).to(cuda_device)
    y_ref, dot_ref = M.matvec_dot(x)
    stream = torch.cuda.current_stream()
    tol = 1e-12 if A.vals.dtype == np.float64 else 1e-5
    for _ in range(2):   # two calls in a row on the shared scratch
        y = torch.full_like(x, float("nan"))
        dot = torch.full((M.batch,), float("nan"), dtype=torch.float64, device=cuda_device)
        st = _static_call(lib, M, x, y, dot, stream)
        assert st == _lib.SLA_OK, lib.sla_last_error()
        torch.cuda.synchronize()
        yr, yd = y_ref.cpu().numpy().astype(np.float64), y.cpu().numpy().astype(np.float64)
        scale = np.abs(yr).max() if yr.size else 1.0
        assert np.all(np.abs(yd - yr) <= tol * max(scale, 1e-300))
        dr, dd = dot_ref.cpu().numpy(), dot.cpu().numpy()
        assert np.all(np.abs(dd - dr) <= 1e-12 * np.maximum(np.abs(dr), 1.0))


def test_static_rejects_batch_beyond_maximum(cuda_device):
    from sparse_iterative_linear_csr_b300 import _lib
    lib = _lib.load()
    A = build("c2", N=8).A
    M = make(A)
    x = torch.zeros(65 * A.n, dtype=torch.float64, device=cuda_device)
    y = torch.zeros_like(x)
    dot = torch.zeros(65, dtype=torch.float64, device=cuda_device)
    dt = _lib.SLA_F64
    st = lib.sla_spmv_dot_static(A.n, A.nnz, 65, dt, C.c_void_p(M.row_ptr.data_ptr()),
                                 C.c_void_p(M.col_idx.data_ptr()), C.c_void_p(M.values.data_ptr()),
                                 C.c_void_p(x.data_ptr()), C.c_void_p(y.data_ptr()), C.c_void_p(dot.data_ptr()),
                                 C.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == _lib.SLA_ERR_INVALID
    assert b"batch" in lib.sla_last_error()
