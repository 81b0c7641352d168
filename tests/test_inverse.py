"""The differentiable inverse problem (torch-sla §4, Figure 3) built on the
solver: the torch assembly of the operator, the chain rule from the misfit
to the conductivity, and (on the GPU) the library's adjoint path."""
import numpy as np
import pytest
import torch

import oracle
from workloads.matrices import CSR, diffusion2d
from sparse_iterative_linear_csr_b300 import inverse as inv


@pytest.mark.parametrize("N", [1, 2, 5, 9])
def test_assembly_matches_the_workload_generator(N):
    """assemble() gives exactly the values of the benchmark's diffusion
    recipe (itself pinned to the Poisson matrix at k = 1)."""
    k = np.exp(np.random.default_rng(N).standard_normal(N * N))
    ref = diffusion2d(N, k)
    rp, ci, mask = inv.five_point_pattern(N)
    assert np.array_equal(rp.numpy(), ref.row_ptr) and np.array_equal(ci.numpy(), ref.col_idx)
    vals = inv.assemble(torch.from_numpy(k).reshape(N, N), mask).numpy()
    assert np.allclose(vals, ref.vals, rtol=1e-15, atol=0)


def _dense_loss(kappa, mask, rp, ci, f, u_obs):
    """Misfit with a dense LU solve (torch) on the assembled matrix."""
    n = f.numel()
    vals = inv.assemble(kappa, mask)
    rows = torch.repeat_interleave(torch.arange(n), (rp[1:] - rp[:-1]).long())
    A = torch.zeros(n, n, dtype=torch.float64).index_put((rows, ci.long()), vals)
    return inv.misfit(torch.linalg.solve(A, f), u_obs)


def test_gradient_chain_against_oracle_finite_differences():
    """dL/dkappa by autograd through a dense solve agrees with central
    differences of the misfit computed with the oracle's PCG: pins the
    assembly derivative and the chain to the conductivity."""
    N = 5
    rp, ci, mask = inv.five_point_pattern(N)
    f = torch.ones(N * N, dtype=torch.float64)
    k_true = inv.reference_field(N)
    A0 = CSR(N * N, rp.numpy(), ci.numpy(), inv.assemble(k_true, mask).numpy())
    u_obs = torch.from_numpy(oracle.pcg(A0, f.numpy(), 1e-14, pc="jacobi", max_iter=1000)[0])
    kappa = (k_true * 0.7 + 0.3).clone().requires_grad_(True)
    _dense_loss(kappa, mask, rp, ci, f, u_obs).backward()

    def L(kap):
        A = CSR(N * N, rp.numpy(), ci.numpy(), inv.assemble(kap, mask).numpy())
        u = oracle.pcg(A, f.numpy(), 1e-14, pc="jacobi", max_iter=1000)[0]
        return float(inv.misfit(torch.from_numpy(u), u_obs))

    h = 1e-6
    for (i, j) in [(0, 0), (2, 3), (4, 1), (1, 4)]:
        e = torch.zeros(N, N, dtype=torch.float64)
        e[i, j] = h
        fd = (L(kappa.detach() + e) - L(kappa.detach() - e)) / (2 * h)
        assert abs(fd - kappa.grad[i, j].item()) <= 1e-6 * max(1.0, abs(fd))


@pytest.mark.gpu
def test_gradient_through_the_library_matches_dense(cuda_device):
    """The library's solve + adjoint (dL/dA on the pattern, chained by
    autograd) gives the same dL/dkappa as the dense reference."""
    from sparse_iterative_linear_csr_b300 import CSRMatrix, solve
    N = 12
    rp, ci, mask = inv.five_point_pattern(N)
    f = torch.ones(N * N, dtype=torch.float64)
    k_true = inv.reference_field(N)
    v_true = inv.assemble(k_true, mask)
    A_true = CSR(N * N, rp.numpy(), ci.numpy(), v_true.numpy())
    u_obs = torch.from_numpy(oracle.pcg(A_true, f.numpy(), 1e-14, pc="jacobi", max_iter=5000)[0])
    kappa = (k_true * 0.6 + 0.4).clone().requires_grad_(True)
    _dense_loss(kappa, mask, rp, ci, f, u_obs).backward()
    g_ref = kappa.grad.clone()

    dev = cuda_device
    rpd, cid, maskd = rp.to(dev), ci.to(dev), mask.to(dev)
    M = CSRMatrix(rpd, cid, v_true.to(dev).contiguous())
    kd = kappa.detach().to(dev).requires_grad_(True)
    u = solve(M, inv.assemble(kd, maskd).contiguous(), f.to(dev), tol=1e-13, pc="jacobi", max_iter=5000)
    inv.misfit(u, u_obs.to(dev)).backward()
    g = kd.grad.cpu()
    assert torch.linalg.norm(g - g_ref) <= 1e-6 * torch.linalg.norm(g_ref)


@pytest.mark.gpu
def test_recovery_reduces_the_misfit(cuda_device):
    out = inv.recover(N=24, steps=300, lr=0.05, device=cuda_device, log_every=299)
    first, last = out["loss_history"][0][1], out["loss_history"][-1][1]
    assert last < 1e-3 * first
    assert out["kappa_rel_err"] < 0.25 * out["kappa_rel_err_initial"]
    assert 0.5 < out["kappa_range"][0] and out["kappa_range"][1] < 1.5
