"""The C-ABI library builds for sm_103a, loads without a GPU and exports
every function include/sla.h declares.  No compute call is made here."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "sla.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_iterative_linear_csr_b300 import build, _lib
    build.build()
    return _lib.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sla_[A-Za-z0-9_]+)\s*\(", text)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for f in ["sla_csr_create", "sla_spmv", "sla_pcg_solve", "sla_adjoint", "sla_csr_destroy",
              "sla_last_error"]:
        assert f in names


def test_every_declared_symbol_is_exported(lib):
    from sparse_iterative_linear_csr_b300 import _lib
    names = declared_functions()
    assert sorted(_lib.EXPORTS) == names
    for f in names:
        assert hasattr(lib, f), f


def test_host_only_calls(lib):
    from sparse_iterative_linear_csr_b300 import _lib
    o = _lib.PcgOpts()
    lib.sla_pcg_opts_default(C.byref(o))
    assert o.tol == 1e-8 and o.max_iter == 10000 and o.poll_k == 32 and o.pc == 0
    # argument checks fail before any CUDA call
    h = C.c_void_p()
    st = lib.sla_csr_create(0, 0, 1, 0, None, None, None, 0, None, C.byref(h))
    assert st == _lib.SLA_ERR_INVALID
    assert b"n must be" in lib.sla_last_error()
    assert lib.sla_pcg_solve(None, None, None, C.byref(o), None, None) == _lib.SLA_ERR_INVALID
    assert lib.sla_csr_destroy(None) == _lib.SLA_ERR_INVALID
    f, g, sp = C.c_int(-1), C.c_int(-1), C.c_int(-1)
    for fn, args in ((lib.sla_csr_layout_of, (None, 0, C.byref(f), C.byref(g), C.byref(sp))),
                     (lib.sla_csr_layout, (None, C.byref(f), C.byref(g), C.byref(sp))),
                     (lib.sla_csr_update_values, (None, None, None))):
        assert fn(*args) == _lib.SLA_ERR_INVALID
        assert b"null handle" in lib.sla_last_error()
    assert (f.value, g.value, sp.value) == (-1, -1, -1)


def test_struct_layouts_match_header():
    from sparse_iterative_linear_csr_b300 import _lib
    assert C.sizeof(_lib.PcgOpts) == 40
    assert _lib.PcgOpts.timeout_s.offset == 32
    assert C.sizeof(_lib.SolveInfo) == 32
    assert _lib.SolveInfo.status.offset == 24


def test_no_oracle_in_product_package():
    pkg = os.path.join(ROOT, "sparse_iterative_linear_csr_b300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
                assert "oracle.c" not in src, f


@pytest.mark.parametrize("case", ["n0", "nnz_neg", "null_x", "null_dot", "null_rowptr", "batch_big",
                                  "dtype"])
def test_static_entry_rejects_bad_arguments_without_launching(lib, case):
    """sla_spmv_dot_static checks its arguments before any CUDA call: each
    bad argument returns SLA_ERR_INVALID and launches nothing."""
    from sparse_iterative_linear_csr_b300 import _lib
    p = C.c_void_p(16)   # never dereferenced: the checks fail first
    args = dict(n=4, nnz=4, batch=1, dt=0, rp=p, ci=p, v=p, x=p, y=p, dot=p)
    if case == "n0":
        args["n"] = 0
    elif case == "nnz_neg":
        args["nnz"] = -1
    elif case == "null_x":
        args["x"] = None
    elif case == "null_dot":
        args["dot"] = None
    elif case == "null_rowptr":
        args["rp"] = None
    elif case == "batch_big":
        args["batch"] = 65
    else:
        args["dt"] = 7
    before = lib.sla_launch_count()
    st = lib.sla_spmv_dot_static(args["n"], args["nnz"], args["batch"], args["dt"], args["rp"], args["ci"],
                                 args["v"], args["x"], args["y"], args["dot"], None)
    assert st == _lib.SLA_ERR_INVALID
    assert lib.sla_last_error()
    assert lib.sla_launch_count() == before


def test_fp64_probe_rejects_null_output(lib):
    from sparse_iterative_linear_csr_b300 import _lib
    assert lib.sla_fp64_fma_rate(None, None) == _lib.SLA_ERR_INVALID
