"""Seeded synthetic inputs shared by the oracle tests, the GPU tests and the
benchmark.  This package builds matrices and vectors only; it holds none of
the solver's arithmetic (no CG, no preconditioner, no adjoint)."""
from .configs import BUILDERS, FULL, SMALL, Workload, build  # noqa: F401
from .matrices import CSR  # noqa: F401
