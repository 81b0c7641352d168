#!/usr/bin/env python
"""Benchmark: preconditioned CG + adjoint on one B300, one JSON line.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config c5] [--also c4] [--impl ours|reference]

A step is one pass of the whole hot path on the workload: the forward PCG
solve A x = b and the backward pass (adjoint solve A^T lambda = g, dL/db,
dL/dA on the pattern).  The headline metric is PCG iterations per second
(forward + adjoint iterations / wall time on the device), with the
per-iteration HBM traffic of the algorithmic byte model, the fused SpMV + dot
kernel's achieved bandwidth, and the solve time.

Default workload (N = 1): the largest single-GPU configuration, the kNN
graph Laplacian of 4M points (k = 12, union-symmetrised, relabelled), fp64,
SPAI-PCG (M^-1 = G G^T + 1e-3 I) to 1e-8, b, g ~ N(0,1); the 3D 7-point
Poisson problem on 128^3 (CG to 1e-8) is measured after it and reported under
"secondary" (--also).  Other workloads: --config c1..c5, cd3.  Under
torchrun every rank solves its own replica (no data-path collective); value
= iterations of all ranks / max-over-ranks time.
`--impl reference` times the plain CPU oracle on the host cores instead.

`--config cd3` measures BiCGStab instead: a nonsymmetric 3D
convection-diffusion system, forward solve plus the adjoint solve on the
explicit transpose, reported as BiCGStab iterations per second.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

DESCR = {
    "c1": "2D 5-point Poisson 64x64 Dirichlet (n=4096, nnz=20224), fp64, CG to 1e-10, b = A x*",
    "c2": "2D 5-point variable-coefficient diffusion 1024x1024 (n=1048576, nnz=5238784), "
          "k=exp(N(0,1)) harmonic faces, fp64, Jacobi-PCG to 1e-8, b,g ~ N(0,1)",
    "c3": "64 systems on one 256x256 5-point pattern, k=exp(0.5 N(0,1)), fp32 values, "
          "Jacobi-PCG to 1e-5 per system, b ~ U(-1,1)",
    "c4": "3D 7-point Poisson 128^3 (n=2097152, nnz=14581760), fp64, CG to 1e-8, b,g ~ N(0,1)",
    "c5": "kNN graph Laplacian, 4M points in the unit cube, k=12 union, A = L + 1e-3 I, relabelled, fp64, "
          "SPAI-PCG (G G^T + 1e-3 I) to 1e-8",
    "cd3": "3D 7-point upwind convection-diffusion 128^3 (n=2097152, nnz=14581760), rotating wind about z "
           "(scaled speed <= 2) + 0.5 along z, fp64, nonsymmetric, Jacobi-BiCGStab to 1e-8, b,g ~ N(0,1)",
}
MAX_ITER = 200000
# full sizes (grid side / point count) of the workloads
FULL_SIZE = {"c1": (64, 64), "c2": (1024, 1024), "c3": (256, 256), "c4": (128, 128, 128),
             "cd3": (128, 128, 128), "c5_points": 4 * 1024 * 1024}
METRIC = "PCG iterations/s (forward + adjoint); HBM GB/s per iteration (fraction of B300 peak); solve ms"
METRIC_BICG = ("BiCGStab iterations/s (forward + transpose adjoint); HBM GB/s per iteration "
               "(fraction of B300 peak); solve ms")


def method_of(w):
    return w.info.get("method", "cg")


def metric_of(w):
    return METRIC_BICG if method_of(w) == "bicgstab" else METRIC


def oracle_solve(w, A, b, max_iter):
    """The oracle's solver for the workload's method (test infrastructure,
    used only by the CPU legs)."""
    import oracle
    if method_of(w) == "bicgstab":
        return oracle.bicgstab(A, b, w.tol, max_iter=max_iter, pc=w.pc)
    return oracle.pcg(A, b, w.tol, max_iter=max_iter, pc=w.pc, eps=w.eps)
L2_BYTES = 126 * 1024 * 1024
NOMINAL_HBM_GBS = 8000.0


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except Exception:
        return 6400.0, "fallback"


def byte_model(w, nnzg=None):
    """Algorithmic bytes: per CG iteration, per fused SpMV + dot launch, and
    for the dL/dA pass.  Indices int32; s = value bytes; col_idx/row_ptr of a
    shared-pattern batch counted once."""
    A = w.A
    n, nnz, B = A.n, A.nnz, A.batch
    s = 4 if w.dtype == "f32" else 8   # matrix values and caller vectors
    v = 8                              # working vectors of the recurrence (fp64 or fp32 pairs)
    rp = 4 * (n + 1)
    if method_of(w) == "bicgstab":
        # BiCGStab: two products (values, columns, row pointers, the source
        # vector gathered once) and 19 vector passes: v = A p (p, r^ read, v
        # written), s = r - alpha v (3), t = A s (s, t), the x/r update (x, p,
        # s, t, r^ read; x, r written) and the direction update (r, p, v
        # read; p written).
        mat = s * nnz * B + 4 * nnz + rp
        return {"per_iteration": 2 * mat + 19 * v * n * B,
                "spmv_dot_per_launch": mat + 2 * s * n * B,
                "product_per_launch": mat + 3 * v * n * B,
                "grad_A": 4 * nnz + rp + s * nnz * B + 2 * s * n * B}
    # The per-iteration model is fixed in advance for the three-kernel
    # schedule (product: p read once, q written; x/r update: x, r, p, q
    # [, dinv] read, x, r written; p update: r, p [, dinv] read, p written),
    # 11 vector passes for CG and 13 for Jacobi; SPAI: 128 n.  It does not
    # follow the kernels' own schedule, so gains show as time.
    if w.pc == "spai":
        it = 12 * nnz + 24 * nnzg + 3 * rp + 128 * n
    elif w.pc == "jacobi":
        it = (s * nnz * B + 4 * nnz + rp + 13 * v * n * B)
    else:
        it = (s * nnz * B + 4 * nnz + rp + 11 * v * n * B)
    spmv = s * nnz * B + 4 * nnz + rp + 2 * s * n * B
    # the CG product kernel: values, columns, row pointers, p gathered once
    # and q written at the working precision (8 bytes)
    product = s * nnz * B + 4 * nnz + rp + 2 * v * n * B
    grad = (4 * nnz + rp + s * nnz * B + 2 * s * n * B)
    return {"per_iteration": it, "spmv_dot_per_launch": spmv, "product_per_launch": product, "grad_A": grad}


def kernel_source_hash():
    """Hash of the device code of the iteration kernels (a recorded DRAM
    traffic figure is reported only while these sources are unchanged)."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "sparse_iterative_linear_csr_b300", "csrc")
    for f in ("common.cuh", "df.cuh", "kernels.cuh", "bicgstab.cuh"):
        with open(os.path.join(d, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(config, kernel, src_hash):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources (profiles/traffic.tsv)."""
    p = os.path.join(ROOT, "profiles", "traffic.tsv")
    if not os.path.exists(p):
        return None
    for line in open(p):
        if line.startswith("#") or not line.strip():
            continue
        f = line.rstrip("\n").split("\t")
        if len(f) >= 4 and f[0] == config and f[1] == kernel and f[2] == src_hash:
            return float(f[3])
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, bus_id=None):
        self.proc = None
        self.bus_id = bus_id

    def start(self):
        cmd = ["nvidia-smi", "--query-gpu=" + self.FIELDS, "--format=csv,noheader,nounits", "-lms", "100"]
        if self.bus_id:
            cmd += ["-i", self.bus_id]
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        time.sleep(0.15)
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except Exception:
            self.proc.kill()
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx.append(float(f[2]))
            except ValueError:
                continue
            for nm, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def bus_id_of(dev):
    try:
        import torch
        p = torch.cuda.get_device_properties(dev)
        return "%08X:%02X:%02X.0" % (p.pci_domain_id, p.pci_bus_id, p.pci_device_id)
    except Exception:
        return None


def host_cpu():
    """Model name of the host's cores and the number the process may use."""
    model = "unknown"
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.startswith("model name"):
                    model = line.split(":", 1)[1].strip()
                    break
    except OSError:
        pass
    try:
        avail = len(os.sched_getaffinity(0))
    except AttributeError:
        avail = os.cpu_count() or 1
    return {"model": model, "available_cores": avail}


def _single_system(w):
    A = w.A
    b = w.b if w.b.ndim == 1 else w.b[0]
    if A.vals.ndim == 2:
        from workloads.matrices import CSR
        A = CSR(A.n, A.row_ptr, A.col_idx, A.vals[0])
    return A, b


def oracle_calibrate(w, budget_s):
    """Iterations of the oracle's forward solve that take about budget_s
    seconds on one host core beyond the solve's own set-up (the time per
    iteration from a 1- and a 3-iteration solve)."""
    A, b = _single_system(w)
    t = []
    for k in (1, 3):
        t0 = time.perf_counter()
        oracle_solve(w, A, b, k)
        t.append(time.perf_counter() - t0)
    per_it = max((t[1] - t[0]) / 2.0, 1e-6)
    return int(max(2, min(MAX_ITER, budget_s / per_it)))


def oracle_calls(w, cap, calls):
    """The oracle as it stands, single-threaded: `calls` forward solves of at
    most `cap` iterations each (first system of a batch).  Returns the
    iterations and seconds of every call and the host core it ran on."""
    A, b = _single_system(w)
    out = []
    for _ in range(calls):
        t0 = time.perf_counter()
        _, inf = oracle_solve(w, A, b, cap)
        out.append((int(inf["iters"]), time.perf_counter() - t0))
    try:
        cpu = os.sched_getcpu()
    except AttributeError:
        cpu = None
    return out, cpu


def oracle_summary(w, calls, cpu_id, what):
    its = sum(c[0] for c in calls)
    dt = sum(c[1] for c in calls)
    name = "BiCGStab" if method_of(w) == "bicgstab" else "PCG"
    return {"value": its / dt, "unit": "iterations/s", "cores": 1, "kind": "oracle",
            "sample": f"{what}: {len(calls)} call(s) of the oracle's forward {name} solve (system 0), "
                      f"{calls[0][0]} iterations each, {its} iterations in {dt:.1f} s, "
                      f"single-threaded fp64 C oracle",
            "per_call_iterations_per_s": [round(c[0] / c[1], 2) for c in calls],
            "host_cpu_id": cpu_id, "host": host_cpu()}


# Both oracle legs time the same thing: calls of the forward solve capped
# at ORACLE_CALL_S seconds of iterations each.
ORACLE_CALL_S = 4.0


def cpu_sample(w, calls=3):
    """cpu_baseline of the main line: the oracle timed on the host cores."""
    cap = oracle_calibrate(w, ORACLE_CALL_S)
    res, cpu = oracle_calls(w, cap, calls)
    return oracle_summary(w, res, cpu, "bounded sample")


def layouts_of(M, pc):
    """Product form, CTAs per system and split group sums of the iteration
    matrix and, under SPAI, of G and G^T (as the handle chose them)."""
    out = {}
    for which in (("A", "G", "GT") if pc == "spai" else ("A",)):
        f, g, sp = M.layout_of(which)
        out[which] = {"form": f, "ctas": g, "split": sp}
    return out


def config_of(name, w, poll_k, bm):
    """The `config` object, the same for both arms."""
    method = method_of(w)
    scaled = w.info.get("grid") != FULL_SIZE.get(name, w.info.get("grid")) or \
        w.info.get("points") != FULL_SIZE.get(name + "_points", w.info.get("points"))
    tag = " (SCALED DOWN: a profiler-capture size, not the workload)" if scaled else ""
    return {"workload": f"{name}: {DESCR[name]}{tag}", "n": w.A.n, "nnz": w.A.nnz, "batch": w.A.batch,
            "pc": w.pc, "tol": w.tol, "poll_k": poll_k,
            "step": ("forward BiCGStab solve + adjoint BiCGStab solve on the explicit A^T + dL/dA pass"
                     if method == "bicgstab" else "forward PCG solve + adjoint solve + dL/dA pass"),
            "l2": l2_rule(bm)}


def l2_resident(bm):
    """A step's working set (the bytes one iteration touches) fits in L2."""
    return bm["per_iteration"] <= L2_BYTES


def l2_rule(bm):
    """How the timed steps treat L2: inputs larger than L2, or an L2 flush
    before every timed step (steps then timed one by one, the flush outside
    their events)."""
    mb, l2 = bm["per_iteration"] / 1e6, L2_BYTES / 2**20
    if not l2_resident(bm):
        return f"inputs larger than L2: {mb:.1f} MB touched per iteration vs {l2:.0f} MiB L2; no flush"
    return (f"L2 flushed before every timed step (a {2 * l2:.0f} MiB write outside the step's CUDA events; "
            f"steps timed one by one): {mb:.1f} MB touched per iteration vs {l2:.0f} MiB L2, so the "
            f"iterations within a step run from L2")


def size_override(args, name):
    """Smaller versions of a workload (same recipe) for profiler captures
    that must hold only a few GB on the device: --grid N (grid side of
    c1-c4, cd3), --points P (c5)."""
    if name == "c5" and args.points:
        return {"npoints": args.points}
    if name != "c5" and args.grid:
        return {"N": args.grid}
    return {}


def nnzg_of(w):
    return (w.A.nnz + w.A.n) // 2 if w.pc == "spai" else None


def run_reference(args, w, rank):
    if rank != 0:
        return
    cap = oracle_calibrate(w, ORACLE_CALL_S)
    if args.warmup > 0:
        oracle_calls(w, max(2, cap // 4), args.warmup)
    t0 = time.perf_counter()
    res, cpu = oracle_calls(w, cap, args.steps)
    dt = time.perf_counter() - t0
    its = sum(c[0] for c in res)
    v = its / dt
    bm = byte_model(w, nnzg_of(w))
    line = {"metric": metric_of(w), "value": v, "unit": "iterations/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1000 * dt / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "f64" if w.dtype == "f64" else "f32", "data": "synthetic", "impl": "reference",
            "config": config_of(args.config, w, args.poll_k, bm),
            "cpu_baseline": oracle_summary(w, res, cpu, "one step = one call"),
            "e2e": {"value": v, "unit": "iterations/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    line["cpu_baseline"]["value"] = v
    print(json.dumps(line), flush=True)


def aggregate(ms, iters, world, device):
    """Whole-job view of a timed region run by every rank: the slowest rank's
    time and the iterations of all ranks (identity for one rank)."""
    if world <= 1:
        return ms, iters
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], device=device, dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    it = torch.tensor([iters], device=device, dtype=torch.float64)
    dist.all_reduce(it, op=dist.ReduceOp.SUM)
    return t.item(), int(it.item())


def measure(args, name, dev, world, rank, stream, lib, with_cpu, e2e_steps, fma_rate):
    """Time `args.steps` steps of workload `name` (after `args.warmup`) and
    return the fields of its JSON line."""
    import torch
    import sparse_iterative_linear_csr_b300 as sla
    from workloads import build

    w = build(name, **size_override(args, name))
    A = w.A
    rp = torch.from_numpy(A.row_ptr).to(dev)
    ci = torch.from_numpy(A.col_idx).to(dev)
    vals = torch.from_numpy(A.vals).to(dev)
    b = torch.from_numpy(w.b).to(dev)
    g = torch.from_numpy(w.g).to(dev)
    M = sla.CSRMatrix(rp, ci, vals, pipeline=args.warp_pipeline, fused=args.persistent, time_product=True,
                      producer_consumer=args.producer_consumer, staged=args.staged, sliced=args.sliced)
    method = method_of(w)
    kw = dict(tol=w.tol, max_iter=MAX_ITER, pc=w.pc, eps=w.eps if w.pc == "spai" else 1e-3,
              poll_k=args.poll_k, method=method)

    def step():
        x, inf = M.solve(b, **kw)
        dldb, dlda, ainf = M.adjoint(x, g, **kw)
        return x, inf, ainf

    for _ in range(max(args.warmup, 0)):
        x, inf, ainf = step()
    bad = [i.status for i in inf + ainf if i.status != "ok"]
    if bad:
        raise SystemExit(f"{name}: solve did not converge: {bad}")

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    bm = byte_model(w, nnzg_of(w))
    # a working set that fits in L2: every timed step starts from a flushed
    # L2 (a write of twice its size between steps, outside their events)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device=dev) if l2_resident(bm) else None
    sampler = ClockSampler(bus_id_of(dev))
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    marks = []
    iters = 0
    l0 = sla.launch_count()
    M.product_time(reset=True)
    barrier()
    sampler.start()
    e0.record(stream)
    t_wall = time.perf_counter()
    for k in range(args.steps):
        if flush is not None:
            flush.fill_(k)
            marks.append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
            marks[-1][0].record(stream)
        x, inf, ainf = step()
        if flush is not None:
            marks[-1][1].record(stream)
        iters += sum(i.iters for i in inf) + sum(i.iters for i in ainf)
    e1.record(stream)
    barrier()
    t_wall = time.perf_counter() - t_wall
    clocks = sampler.stop()
    launches = sla.launch_count() - l0
    prod_ms, prod_n = M.product_time(reset=True)
    region_ms = sum(a.elapsed_time(b) for a, b in marks) if marks else e0.elapsed_time(e1)
    ms, iters_all = aggregate(region_ms, iters, world, dev)
    value = iters_all / (ms / 1000.0)

    # forward solve time alone (one extra timed solve, same configuration)
    f0 = torch.cuda.Event(enable_timing=True)
    f1 = torch.cuda.Event(enable_timing=True)
    f0.record(stream)
    _, finf = M.solve(b, **kw)
    f1.record(stream)
    torch.cuda.synchronize()
    fwd_ms = f0.elapsed_time(f1)

    # dominant kernel: the product kernel (CG: q = A p fused with p.q;
    # BiCGStab: v = A p fused with r^.v), timed live inside the timed region
    # (CUDA events the solve records on its stream around the first product
    # kernel of every graph launch); with the persistent iteration kernel
    # there is no separate product launch, so the fused SpMV + dot API kernel
    # is timed alone on the same operands.
    if prod_n > 0:
        kern_ms = prod_ms / prod_n
        kern_bytes = bm["product_per_launch"]
        if method == "bicgstab":
            kern_desc = (f"k_bicg_v (BiCGStab product v = A p fused with r^.v), live in the timed solves: "
                         f"{prod_n} launches timed with CUDA events on the solve stream")
            kern_name = "k_bicg_v"
        else:
            kern_desc = (f"k_spmv_iter (CG product q = A p fused with p.q), live in the timed solves: "
                         f"{prod_n} launches timed with CUDA events on the solve stream")
            kern_name = "k_spmv_iter"
    else:
        import ctypes as C
        xin = x.contiguous()
        yout = torch.empty_like(xin)
        dout = torch.empty(A.batch, dtype=torch.float64, device=dev)
        cargs = (M._h, C.c_void_p(xin.data_ptr()), C.c_void_p(yout.data_ptr()), C.c_void_p(dout.data_ptr()),
                 C.c_void_p(stream.cuda_stream))
        for _ in range(5):
            lib.sla_spmv_dot(*cargs)
        reps = 50
        k0 = torch.cuda.Event(enable_timing=True)
        k1 = torch.cuda.Event(enable_timing=True)
        k0.record(stream)
        for _ in range(reps):
            lib.sla_spmv_dot(*cargs)
        k1.record(stream)
        torch.cuda.synchronize()
        kern_ms = k0.elapsed_time(k1) / reps
        kern_bytes = bm["spmv_dot_per_launch"]
        kern_desc = "k_spmv (SpMV fused with x.Ax), timed alone on the step's matrix"
        kern_name = "k_spmv"
    peak, peak_kind = peaks()
    achieved = kern_bytes / (kern_ms * 1e-3) / 1e9
    src = kernel_source_hash()
    traffic = recorded_traffic(name, kern_name, src)
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "traffic": traffic, "peak_kind": peak_kind,
            "kernel": kern_desc, "algorithmic_bytes_per_launch": kern_bytes, "ms_per_launch": kern_ms,
            "frac_of_nominal_8tbs": achieved / NOMINAL_HBM_GBS}
    # The fp64 roof: one fp64 FMA per stored entry plus one per row for the
    # fused dot (fp64 systems; fp32 systems run double-float arithmetic on
    # the fp32 pipe), against the fp64 FMA rate measured on this GPU.
    hbm_us = kern_bytes / (peak * 1e9) * 1e6
    if w.dtype == "f64" and fma_rate:
        fma = (A.nnz + A.n) * A.batch
        fp64_us = fma / fma_rate * 1e6
        roof["fp64"] = {"fma_per_launch": fma, "fma_rate_per_s": fma_rate,
                        "rate_method": "sla_fp64_fma_rate: independent fp64 FMA chains on every SM, CUDA events, "
                                       "best of 3 launches",
                        "time_us_at_rate": fp64_us, "achieved_fma_per_s": fma / (kern_ms * 1e-3),
                        "frac": fma / (kern_ms * 1e-3) / fma_rate}
        bind = "fp64" if fp64_us > hbm_us else "hbm"
        roof["binding_roof"] = {"bound": bind, "time_us": max(hbm_us, fp64_us),
                                "frac": max(hbm_us, fp64_us) / (kern_ms * 1e3)}
    else:
        roof["binding_roof"] = {"bound": "hbm", "time_us": hbm_us, "frac": hbm_us / (kern_ms * 1e3)}

    # bytes of one system's iteration (a batched iteration moves B of them)
    per_it_gbs = bm["per_iteration"] / A.batch * iters / (ms * 1e-3) / 1e9
    out = {
        "value": value, "ms_per_step": ms / args.steps, "dtype": w.dtype,
        "config": config_of(name, w, args.poll_k, bm),
        "iterations_per_step": iters // max(args.steps, 1),
        "forward_iterations": finf[0].iters, "solve_ms": fwd_ms,
        "hbm_gbs_per_iteration": per_it_gbs,
        "hbm_frac_per_iteration": {"of_measured": per_it_gbs / peak, "of_nominal_8tbs": per_it_gbs / NOMINAL_HBM_GBS},
        "bytes_per_iteration_model": bm["per_iteration"],
        "roofline": roof, "gpu_launches": int(launches), "clocks": clocks,
        "wall_s_timed": t_wall, "kernel_src": src, "product_form": M.layout()[0],
        "product_ctas_per_system": M.layout()[1], "metric": metric_of(w),
        "layouts": layouts_of(M, w.pc),
    }
    if w.dtype == "f32":
        # the working vectors are 8-byte double-float slots; the same
        # iteration counted with 4-byte working vectors (fp32 storage)
        n, nnz, B = A.n, A.nnz, A.batch
        it4 = 4 * nnz * B + 4 * nnz + 4 * (n + 1) + 13 * 4 * n * B
        out["hbm_frac_per_iteration"]["of_measured_4byte_vectors"] = (
            it4 / A.batch * iters / (ms * 1e-3) / 1e9) / peak

    if e2e_steps > 0:
        # end to end through the public API with host buffers: every step
        # copies its inputs (values, b, g) in from pinned memory and its
        # results (x, dL/db, dL/dA) out into pinned memory, all inside the
        # timed region.  The copies run on their own streams into and out of
        # double buffers: step k+1's inputs go in while step k computes, and
        # step k's results come out while step k+1 computes (a solve returns
        # once it has finished, so only the first upload and the last
        # download are not overlapped).
        h_vals = vals.cpu().pin_memory()
        h_b = b.cpu().pin_memory()
        h_g = g.cpu().pin_memory()
        d_in = [(torch.empty_like(vals), torch.empty_like(b), torch.empty_like(g)) for _ in range(2)]
        o_out = [(torch.empty_like(h_b).pin_memory(), torch.empty_like(h_b).pin_memory(),
                  torch.empty_like(h_vals).pin_memory()) for _ in range(2)]
        h2d = h_vals.numel() * h_vals.element_size() + 2 * h_b.numel() * h_b.element_size()
        d2h = 2 * h_b.numel() * h_b.element_size() + h_vals.numel() * h_vals.element_size()
        up_s, down_s = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        comp_s = torch.cuda.current_stream(dev)

        def upload(k):
            dv, dbk, dgk = d_in[k % 2]
            with torch.cuda.stream(up_s):
                dv.copy_(h_vals, non_blocking=True)
                dbk.copy_(h_b, non_blocking=True)
                dgk.copy_(h_g, non_blocking=True)
                ev = torch.cuda.Event()
                ev.record(up_s)
            return ev

        barrier()
        t0 = time.perf_counter()
        e2e_iters = 0
        ev_next = upload(0)
        for k in range(e2e_steps):
            ev_in = ev_next
            if k + 1 < e2e_steps:   # into the other buffers (step k-1 has finished with them)
                ev_next = upload(k + 1)
            comp_s.wait_event(ev_in)
            dv, dbk, dgk = d_in[k % 2]
            M.update_values(dv)
            xx, i1 = M.solve(dbk, **kw)
            lb, la, i2 = M.adjoint(xx, dgk, **kw)
            ox, olb, ola = o_out[k % 2]
            down_s.wait_stream(comp_s)
            with torch.cuda.stream(down_s):
                ox.copy_(xx, non_blocking=True)
                olb.copy_(lb, non_blocking=True)
                ola.copy_(la, non_blocking=True)
            # the results' memory is reused only once their copies are done
            # (downloads into one host buffer are ordered on down_s)
            for t_ in (xx, lb, la):
                t_.record_stream(down_s)
            del xx, lb, la
            e2e_iters += sum(i.iters for i in i1) + sum(i.iters for i in i2)
        torch.cuda.synchronize()
        e2e_ms, e2e_iters_all = aggregate((time.perf_counter() - t0) * 1000.0, e2e_iters, world, dev)
        out["e2e"] = {"value": e2e_iters_all / (e2e_ms / 1000.0), "unit": "iterations/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h}
        M.update_values(vals)

    out["cpu_baseline"] = cpu_sample(w) if (rank == 0 and with_cpu) else None
    M.close()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--config", default="c5", choices=sorted(DESCR))
    ap.add_argument("--also", default=None,
                    help="comma-separated workloads measured after the main one and reported under "
                         "'secondary' (default: c4 when the main workload is c5; 'none' for none)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--poll-k", type=int, default=32)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=4)
    ap.add_argument("--warp-pipeline", action="store_true",
                    help="use the warp-pipeline product where it applies")
    ap.add_argument("--producer-consumer", action="store_true",
                    help="use the producer/consumer product where it applies")
    ap.add_argument("--staged", action="store_true",
                    help="keep the warp-staged product forms where the direct form would be the default")
    ap.add_argument("--grid", type=int, default=0,
                    help="grid side of a smaller c1-c4/cd3 (profiler captures; the line is then not the workload's)")
    ap.add_argument("--points", type=int, default=0,
                    help="point count of a smaller c5 (profiler captures; the line is then not the workload's)")
    ap.add_argument("--sliced", action="store_true",
                    help="use the sliced product form where it applies")
    ap.add_argument("--persistent", action="store_true",
                    help="CG / Jacobi-PCG as the persistent iteration kernel (not a graph of kernels)")
    args = ap.parse_args()

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        from workloads import build
        run_reference(args, build(args.config), rank)
        return

    import ctypes as C
    import torch
    import sparse_iterative_linear_csr_b300 as sla

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    stream = torch.cuda.current_stream()
    lib = sla._lib.load()
    rate = C.c_double(0.0)
    st = lib.sla_fp64_fma_rate(C.byref(rate), C.c_void_p(stream.cuda_stream))
    fma_rate = rate.value if st == 0 else None

    main_line = measure(args, args.config, dev, world, rank, stream, lib, not args.no_cpu_baseline,
                        args.e2e_steps, fma_rate)
    also = args.also if args.also is not None else ("c4" if args.config == "c5" else "none")
    secondary = {}
    for name in [a for a in also.split(",") if a and a != "none"]:
        sec = measure(args, name, dev, world, rank, stream, lib, False, 0, fma_rate)
        secondary[name] = {k: sec[k] for k in ("value", "ms_per_step", "config", "iterations_per_step",
                                               "forward_iterations", "solve_ms", "hbm_gbs_per_iteration",
                                               "hbm_frac_per_iteration", "roofline", "clocks",
                                               "product_form", "gpu_launches")}
        secondary[name]["unit"] = "iterations/s"

    if rank == 0:
        m = main_line
        line = {
            "metric": m["metric"], "value": m["value"], "unit": "iterations/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": m["ms_per_step"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": m["dtype"],
            "data": "synthetic", "config": m["config"],
            "iterations_per_step": m["iterations_per_step"], "forward_iterations": m["forward_iterations"],
            "solve_ms": m["solve_ms"], "hbm_gbs_per_iteration": m["hbm_gbs_per_iteration"],
            "hbm_frac_per_iteration": m["hbm_frac_per_iteration"],
            "bytes_per_iteration_model": m["bytes_per_iteration_model"], "roofline": m["roofline"],
            "e2e": m.get("e2e"), "gpu_launches": m["gpu_launches"], "clocks": m["clocks"],
            "cpu_baseline": m["cpu_baseline"], "wall_s_timed": m["wall_s_timed"], "kernel_src": m["kernel_src"],
            "product_form": m["product_form"], "product_ctas_per_system": m["product_ctas_per_system"],
            "layouts": m["layouts"], "fp64_fma_rate_per_s": fma_rate,
        }
        if secondary:
            line["secondary"] = secondary
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
