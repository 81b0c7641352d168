"""ctypes declarations of the C ABI in include/sla.h (argument marshalling only).

Loading fails loudly when libsla.so is missing: there is no CPU fallback."""
from __future__ import annotations

import ctypes as C
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libsla.so")

SLA_OK, SLA_ERR_INVALID, SLA_ERR_CUDA, SLA_ERR_NOMEM, SLA_ERR_NOT_CONVERGED, SLA_ERR_BREAKDOWN, \
    SLA_ERR_TIMEOUT, SLA_ERR_UNSUPPORTED = range(8)
STATUS_NAMES = {SLA_OK: "ok", SLA_ERR_INVALID: "invalid", SLA_ERR_CUDA: "cuda", SLA_ERR_NOMEM: "nomem",
                SLA_ERR_NOT_CONVERGED: "not_converged", SLA_ERR_BREAKDOWN: "breakdown",
                SLA_ERR_TIMEOUT: "timeout", SLA_ERR_UNSUPPORTED: "unsupported"}
SLA_F64, SLA_F32 = 0, 1
PC = {"none": 0, "jacobi": 1, "spai": 2}
SLA_VALIDATE = 1
SLA_WARP_PIPELINE = 2
SLA_PERSISTENT = 4
SLA_TIME_PRODUCT = 8
SLA_PRODUCER_CONSUMER = 16
SLA_REORDER = 32
SLA_NO_REORDER = 64
SLA_STAGED = 128
SLA_SLICED = 256
SLA_SPLIT_ROWS = 512
SLA_ROW_WALK = 1024

# every function the header declares
EXPORTS = ["sla_pcg_opts_default", "sla_csr_create", "sla_csr_update_values", "sla_spmv", "sla_spmv_dot",
           "sla_pcg_solve", "sla_adjoint", "sla_csr_destroy", "sla_last_error", "sla_launch_count",
           "sla_spmv_dot_static", "sla_csr_layout", "sla_csr_layout_of", "sla_product_time", "sla_spmm", "sla_bicgstab_solve",
           "sla_bicgstab_adjoint", "sla_fp64_fma_rate", "sla_wait_selftest", "sla_block_gram_work", "sla_block_gram",
           "sla_block_update", "sla_grad_A", "sla_cg_local_work", "sla_cg_local_update", "sla_cg_local_direction"]


class PcgOpts(C.Structure):
    _fields_ = [("tol", C.c_double), ("max_iter", C.c_int), ("pc", C.c_int), ("eps", C.c_double),
                ("poll_k", C.c_int), ("use_x0", C.c_int), ("timeout_s", C.c_double)]


class SolveInfo(C.Structure):
    _fields_ = [("iters", C.c_int), ("rel_res_recursive", C.c_double), ("rel_res_true", C.c_double),
                ("status", C.c_int)]


_vp = C.c_void_p
_lib = None


def load(path: str = LIB_PATH) -> C.CDLL:
    """Load libsla.so (built by sparse_iterative_linear_csr_b300.build)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with "
                           "`python -m sparse_iterative_linear_csr_b300.build` (no CPU fallback exists)")
    lib = C.CDLL(path)
    lib.sla_pcg_opts_default.argtypes = [C.POINTER(PcgOpts)]
    lib.sla_pcg_opts_default.restype = None
    lib.sla_csr_create.argtypes = [C.c_int, C.c_longlong, C.c_int, C.c_int, _vp, _vp, _vp, C.c_uint, _vp,
                                   C.POINTER(_vp)]
    lib.sla_csr_update_values.argtypes = [_vp, _vp, _vp]
    lib.sla_csr_layout.argtypes = [_vp, C.POINTER(C.c_int), C.POINTER(C.c_int), C.POINTER(C.c_int)]
    lib.sla_csr_layout_of.argtypes = [_vp, C.c_int, C.POINTER(C.c_int), C.POINTER(C.c_int), C.POINTER(C.c_int)]
    lib.sla_product_time.argtypes = [_vp, C.POINTER(C.c_double), C.POINTER(C.c_longlong), C.c_int]
    lib.sla_spmv.argtypes = [_vp, _vp, _vp, _vp]
    lib.sla_spmm.argtypes = [_vp, _vp, _vp, C.c_int, _vp]
    lib.sla_spmv_dot.argtypes = [_vp, _vp, _vp, _vp, _vp]
    lib.sla_pcg_solve.argtypes = [_vp, _vp, _vp, C.POINTER(PcgOpts), C.POINTER(SolveInfo), _vp]
    lib.sla_adjoint.argtypes = [_vp, _vp, _vp, C.POINTER(PcgOpts), _vp, _vp, C.POINTER(SolveInfo), _vp]
    lib.sla_bicgstab_solve.argtypes = [_vp, _vp, _vp, C.POINTER(PcgOpts), C.POINTER(SolveInfo), _vp]
    lib.sla_bicgstab_adjoint.argtypes = [_vp, _vp, _vp, C.POINTER(PcgOpts), _vp, _vp, C.POINTER(SolveInfo),
                                         _vp]
    lib.sla_csr_destroy.argtypes = [_vp]
    lib.sla_last_error.argtypes = []
    lib.sla_last_error.restype = C.c_char_p
    # allocation-free fused SpMV + dot (no handle; fixed device scratch)
    lib.sla_spmv_dot_static.argtypes = [C.c_int, C.c_longlong, C.c_int, C.c_int, _vp, _vp, _vp, _vp, _vp, _vp,
                                        _vp]
    lib.sla_spmv_dot_static.restype = C.c_int
    lib.sla_fp64_fma_rate.argtypes = [C.POINTER(C.c_double), _vp]
    lib.sla_fp64_fma_rate.restype = C.c_int
    lib.sla_wait_selftest.argtypes = [C.c_int, C.c_double, _vp]
    lib.sla_wait_selftest.restype = C.c_int
    lib.sla_block_gram_work.argtypes = [C.c_int, C.c_int, C.c_int, C.c_longlong, C.POINTER(C.c_longlong)]
    lib.sla_block_gram_work.restype = C.c_int
    lib.sla_block_gram.argtypes = [C.c_int, C.c_int, C.c_longlong, _vp, _vp, C.c_int, _vp, _vp, C.c_longlong, _vp]
    lib.sla_block_gram.restype = C.c_int
    lib.sla_block_update.argtypes = [C.c_int, C.c_int, C.c_longlong, _vp, _vp, _vp, _vp, _vp]
    lib.sla_block_update.restype = C.c_int
    lib.sla_grad_A.argtypes = [_vp, _vp, _vp, _vp, _vp]
    lib.sla_grad_A.restype = C.c_int
    lib.sla_cg_local_work.argtypes = [C.c_int, C.POINTER(C.c_longlong)]
    lib.sla_cg_local_work.restype = C.c_int
    lib.sla_cg_local_update.argtypes = [C.c_int, C.c_double, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, C.c_longlong, _vp]
    lib.sla_cg_local_update.restype = C.c_int
    lib.sla_cg_local_direction.argtypes = [C.c_int, C.c_double, _vp, _vp, _vp]
    lib.sla_cg_local_direction.restype = C.c_int
    lib.sla_launch_count.argtypes = []
    lib.sla_launch_count.restype = C.c_ulonglong
    for f in ["sla_csr_create", "sla_csr_update_values", "sla_csr_layout", "sla_csr_layout_of", "sla_product_time", "sla_spmm", "sla_spmv", "sla_spmv_dot", "sla_pcg_solve",
              "sla_adjoint", "sla_bicgstab_solve", "sla_bicgstab_adjoint", "sla_csr_destroy"]:
        getattr(lib, f).restype = C.c_int
    _lib = lib
    return lib
