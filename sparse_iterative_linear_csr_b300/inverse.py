"""Differentiable inverse problem through the solver: recover a conductivity
field from the solution it produces.

torch-sla (arXiv 2601.13994), §4, Figure 3: a conductivity field kappa* in
[0.5, 1.5] is recovered with Adam from the observed solution u_obs of the
diffusion problem it defines, the gradient of the misfit coming from one
adjoint solve per step (§3.2: dL/dA_ij = -lambda_i u_j on the pattern, which
autograd carries back to kappa through the operator's assembly).

Here the operator is the five-point variable-coefficient diffusion of the
benchmark workloads (interior unknowns on an N x N grid, homogeneous
Dirichlet boundary): an interior face between cells i and j has coefficient
2 k_i k_j / (k_i + k_j), a boundary face k_i, A_ii is the sum of the four face
coefficients and A_ij = -k_face.  `assemble` builds the CSR values from the
cell field with torch operations, so autograd differentiates the assembly;
the solve and its adjoint are the library's kernels (CSRMatrix via the C
ABI).  kappa = 0.5 + sigmoid(theta) keeps the field inside (0.5, 1.5).
The solution is observed for several sources at once (a batch of systems
on the shared pattern): with one source the conductivity is barely
determined wherever the solution's gradient vanishes.

    python -m sparse_iterative_linear_csr_b300.inverse [--N 64] [--steps 300]
"""
from __future__ import annotations

import argparse
import json
import math
import time

import torch

from . import CSRMatrix, solve

def five_point_pattern(N: int, device="cpu"):
    """CSR pattern (int32 row_ptr [n+1], col_idx [nnz]) of the five-point
    operator on the N x N interior grid, lexicographic order, and the
    [n, 5] mask of the slots present in each row (slots in ascending column
    order: south i - N, west i - 1, diagonal, east i + 1, north i + N)."""
    n = N * N
    idx = torch.arange(n, device=device)
    ix, iy = idx % N, idx // N
    mask = torch.stack([iy > 0, ix > 0, torch.ones_like(ix, dtype=torch.bool), ix < N - 1, iy < N - 1], 1)
    cols = torch.stack([idx - N, idx - 1, idx, idx + 1, idx + N], 1)
    counts = mask.sum(1)
    row_ptr = torch.zeros(n + 1, dtype=torch.int64, device=device)
    row_ptr[1:] = torch.cumsum(counts, 0)
    return row_ptr.to(torch.int32), cols[mask].to(torch.int32), mask


def assemble(kappa: torch.Tensor, mask: torch.Tensor) -> torch.Tensor:
    """CSR values of the harmonic-mean five-point operator for the cell
    field kappa [N, N] (differentiable), in the order of five_point_pattern."""
    k = kappa
    hx = 2.0 * k[:, :-1] * k[:, 1:] / (k[:, :-1] + k[:, 1:])   # face between (y, x) and (y, x + 1)
    hy = 2.0 * k[:-1, :] * k[1:, :] / (k[:-1, :] + k[1:, :])   # face between (y, x) and (y + 1, x)
    west = torch.cat([k[:, :1], hx], 1)      # boundary face on the left uses k itself
    east = torch.cat([hx, k[:, -1:]], 1)
    south = torch.cat([k[:1, :], hy], 0)
    north = torch.cat([hy, k[-1:, :]], 0)
    diag = west + east + south + north
    slots = torch.stack([-south, -west, diag, -east, -north], 2).reshape(-1, 5)
    return slots[mask]


def reference_field(N: int, device="cpu", dtype=torch.float64) -> torch.Tensor:
    """A smooth ground-truth conductivity in [0.5, 1.5]."""
    t = (torch.arange(N, device=device, dtype=dtype) + 0.5) / N
    y, x = torch.meshgrid(t, t, indexing="ij")
    f = torch.sin(2 * math.pi * x) * torch.cos(3 * math.pi * y) + 0.5 * torch.sin(5 * math.pi * x * y)
    f = f / f.abs().max()
    return 1.0 + 0.5 * f


def sources(N: int, count: int = 4, device="cpu", dtype=torch.float64) -> torch.Tensor:
    """`count` smooth right-hand sides [count, N*N]: a constant and
    products of sines of increasing frequency."""
    t = (torch.arange(N, device=device, dtype=dtype) + 0.5) / N
    y, x = torch.meshgrid(t, t, indexing="ij")
    fs = [torch.ones_like(x)]
    for j in range(1, count):
        fs.append(torch.sin(math.pi * (j + 1) * x) * torch.cos(math.pi * j * y) + 0.25)
    return torch.stack(fs).reshape(count, N * N).contiguous()


def misfit(u: torch.Tensor, u_obs: torch.Tensor) -> torch.Tensor:
    return ((u - u_obs) ** 2).sum() / (u_obs ** 2).sum()


def recover(N: int = 64, steps: int = 300, lr: float = 0.05, tol: float = 1e-10, pc: str = "jacobi",
            n_sources: int = 4, device="cuda", log_every: int = 0) -> dict:
    """Recover reference_field(N) from u_obs[s] = A(kappa*)^-1 f_s for the
    sources f_s of `sources` by Adam on theta, kappa = 0.5 + sigmoid(theta),
    starting from kappa = 1.  One step is one batched solve and one batched
    adjoint on the library."""
    dev = torch.device(device)
    rp, ci, mask = five_point_pattern(N, dev)
    k_true = reference_field(N, dev)
    B = n_sources
    v_true = assemble(k_true, mask).expand(B, -1).contiguous()
    A = CSRMatrix(rp, ci, v_true.clone())
    f = sources(N, B, dev)
    kw = dict(tol=tol, pc=pc, max_iter=100000)
    with torch.no_grad():
        u_obs = solve(A, v_true, f, **kw)
    k_err0 = float(torch.linalg.norm(1.0 - k_true) / torch.linalg.norm(k_true))
    theta = torch.zeros(N, N, dtype=torch.float64, device=dev, requires_grad=True)
    opt = torch.optim.Adam([theta], lr=lr)
    history = []
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    for it in range(steps):
        opt.zero_grad()
        kappa = 0.5 + torch.sigmoid(theta)
        u = solve(A, assemble(kappa, mask).expand(B, -1).contiguous(), f, **kw)
        loss = misfit(u, u_obs)
        loss.backward()
        opt.step()
        if log_every and (it % log_every == 0 or it == steps - 1):
            history.append((it, loss.item()))
    torch.cuda.synchronize(dev)
    wall = time.perf_counter() - t0
    with torch.no_grad():
        kappa = 0.5 + torch.sigmoid(theta)
        u = solve(A, assemble(kappa, mask).expand(B, -1).contiguous(), f, **kw)
        return {
            "N": N, "sources": B, "steps": steps, "ms_per_step": 1e3 * wall / max(steps, 1),
            "kappa_rel_err_initial": k_err0,
            "kappa_rel_err": float(torch.linalg.norm(kappa - k_true) / torch.linalg.norm(k_true)),
            "u_rel_err": float(torch.linalg.norm(u - u_obs) / torch.linalg.norm(u_obs)),
            "kappa_range": [float(kappa.min()), float(kappa.max())],
            "loss_history": history,
        }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--N", type=int, default=64)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--lr", type=float, default=0.05)
    ap.add_argument("--tol", type=float, default=1e-10)
    ap.add_argument("--sources", type=int, default=4)
    args = ap.parse_args()
    out = recover(args.N, args.steps, args.lr, args.tol, n_sources=args.sources, log_every=max(1, args.steps // 10))
    print(json.dumps(out))


if __name__ == "__main__":
    main()
