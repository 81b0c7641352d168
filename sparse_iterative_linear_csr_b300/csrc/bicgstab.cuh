// bicgstab.cuh -- BiCGStab for general (nonsymmetric) CSR systems, fp64.
//
// The method is van der Vorst's stabilised bi-conjugate gradient (SIAM J.
// Sci. Stat. Comput. 13(2), 1992), in the right-preconditioned form of
// Barrett et al., "Templates for the Solution of Linear Systems", §2.3.8,
// with the shadow residual r^ = r0 -- the nonsymmetric Krylov solver that
// torch-sla's native iterative backend offers beside CG (torch-sla, §3
// backends paragraph).  Right Jacobi preconditioning is applied as a column scaling
// of the stored values, A^ = A D^-1 (D = diag(A)), built once per solve: the
// iteration runs unpreconditioned on A^ y = b and returns x = D^-1 y, which
// is the right-preconditioned iteration with p^ = D^-1 p and s^ = D^-1 s
// folded into the products (the residual b - A x = b - A^ y is the same up
// to rounding; the stopping test is confirmed on b - A x itself).
//
// One iteration is five kernels, captured in a CUDA graph like the CG step:
//   k_bicg_v:  v = A^ p, sigma = r^.v  (+ the true-residual check) -> alpha
//   k_bicg_s:  s = r - alpha v        (in place over r)
//   k_bicg_t:  t = A^ s, t.t, t.s     -> omega
//   k_bicg_xr: y += alpha p + omega s, r = s - omega t, r.r, r^.r -> beta
//   k_bicg_p:  p = r + beta (p - omega v)
// Vector traffic per iteration: 17 n-vectors (2 + 3 + 1 + 7 + 4) besides the
// two products.  The scalar logic keeps the oracle's order of tests.
#pragma once

#include "kernels.cuh"

namespace sla {

// ----------------------------------------------------------------- scalar logic
// (thread 0 of the last CTA of one system, on its State)

// After rho0 = r^.r0 of the set-up (r^ = p = r0).
__device__ __forceinline__ void bicg_start(State* s, Ctrl* c, double rho) {
    s->omega = 1.0;
    s->alpha = 1.0;
    s->beta = 0.0;
    s->phase = 1;
    if (rho == 0.0 || !finite(rho)) {
        if (s->check) s->rho_bad = 1;   // decided by the pending true-residual check
        else freeze(s, c, ST_BREAKDOWN);
        return;
    }
    s->rho = rho;
}

// After sigma = r^.v (and, when the recursive residual had met the
// tolerance, the true residual of the current iterate).
__device__ __forceinline__ void bicg_after_v(State* s, Ctrl* c, double sigma, bool checked, double tr2) {
    if (checked) {
        s->tr2 = tr2;
        if (tr2 <= s->tol2bb) { freeze(s, c, ST_OK); return; }
        s->check = 0;
        if (s->iter >= s->max_iter) { freeze(s, c, ST_NOT_CONVERGED); return; }
        if (s->rho_bad) { freeze(s, c, ST_BREAKDOWN); return; }
    }
    s->delta = sigma;
    if (sigma == 0.0 || !finite(sigma)) { freeze(s, c, ST_BREAKDOWN); return; }
    s->alpha = s->rho / sigma;
}

// After t.t and t.s: omega minimises ||s - omega t|| (0 when t = 0).
__device__ __forceinline__ void bicg_after_t(State* s, Ctrl* c, double tt, double ts) {
    const double w = tt > 0.0 ? ts / tt : 0.0;
    s->omega = w;
    if (!finite(w)) freeze(s, c, ST_BREAKDOWN);
}

// After the x / r update: gamma = r.r, rho' = r^.r.  The tests run in the
// order of the loop head: the residual test (a pending true-residual check
// when it passes), omega = 0 with the test failed, the iteration cap, then
// rho'.
__device__ __forceinline__ void bicg_after_update(State* s, Ctrl* c, double gamma, double rho_new) {
    s->gamma = gamma;
    s->iter += 1;
    if (!finite(gamma)) { freeze(s, c, ST_BREAKDOWN); return; }
    s->check = (gamma <= s->tol2bb);
    if (!s->check) {
        if (s->omega == 0.0) { freeze(s, c, ST_BREAKDOWN); return; }
        if (s->iter >= s->max_iter) { freeze(s, c, ST_NOT_CONVERGED); return; }
    }
    if (rho_new == 0.0 || !finite(rho_new)) {
        if (s->check) { s->rho_bad = 1; s->beta = 0.0; return; }
        freeze(s, c, ST_BREAKDOWN);
        return;
    }
    s->beta = (rho_new / s->rho) * (s->alpha / s->omega);
    s->rho = rho_new;
}

// ----------------------------------------------------------------- vector access
// W consecutive fp64 entries (W = 2: one 16-byte access; needs n even).
template <int W> struct Vd { double e[W]; };

template <int W>
__device__ __forceinline__ Vd<W> vld(const double* p, int i) {
    Vd<W> o;
    if constexpr (W == 2) {
        const double2 t = ld_vec(reinterpret_cast<const double2*>(p) + i);
        o.e[0] = t.x;
        o.e[1] = t.y;
    } else {
        o.e[0] = ld_vec(p + i);
    }
    return o;
}
// a vector read for the last time in the iteration
template <int W>
__device__ __forceinline__ Vd<W> vld_last(const double* p, int i) {
    Vd<W> o;
    if constexpr (W == 2) {
        const double2 t = ld_vec_last(reinterpret_cast<const double2*>(p) + i);
        o.e[0] = t.x;
        o.e[1] = t.y;
    } else {
        o.e[0] = ld_vec_last(p + i);
    }
    return o;
}
template <int W>
__device__ __forceinline__ void vst(double* p, int i, const Vd<W>& v) {
    if constexpr (W == 2) st_vec(reinterpret_cast<double2*>(p) + i, make_double2(v.e[0], v.e[1]));
    else st_vec(p + i, v.e[0]);
}

#define BICG_LOOP(W) for (int i = blockIdx.x * NT + threadIdx.x; i < S.n / (W); i += gridDim.x * NT)

// ----------------------------------------------------------------- kernels
// Set-up after r0: r^ = r0, p = r0, rho0 = r^.r0.
template <int W>
__global__ void __launch_bounds__(NT) k_bicg_dir(Sys S, const double* __restrict__ r, double* __restrict__ rh,
                                                 double* __restrict__ p) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[RED_DOUBLES];
    r += vo; rh += vo; p += vo;
    double rho = 0.0;
    BICG_LOOP(W) {
        const Vd<W> ri = vld<W>(r, i);
        vst<W>(rh, i, ri);
        vst<W>(p, i, ri);
#pragma unroll
        for (int e = 0; e < W; ++e) rho = fma(ri.e[e], ri.e[e], rho);
    }
    double v[1] = {rho}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) bicg_start(st, S.ctl, tot[0]);
}

// x_c = y_c / d_c: the iterate of the column-scaled iteration mapped back,
// divided exactly as the returned x is (k_bicg_scale).
struct GatherUnscaled {
    const double* y;
    const double* d;
    __device__ __forceinline__ double operator()(int c) const { return ld_nc(y + c) / ld_nc(d + c); }
};
// ||b - A0 x||^2 over this CTA's rows with x = y / d (A0: the unscaled
// values): the true residual of the x the solve returns.  Out of line for
// the staged forms, like residual_staged.
template <int FORM>
__device__ __noinline__ double residual_unscaled_staged(const Mat& A, const double* __restrict__ a0,
                                                        const double* y, const double* d,
                                                        const double* __restrict__ b, double* dsm) {
    double tr2 = 0.0;
    spmv_rows<double, double>(A, a0, GatherUnscaled{y, d}, [&](int i) { return b[i]; },
                              [&](int, double s, double bi) { sq_acc(tr2, resid(bi, s)); }, dsm);
    return tr2;
}
template <int FORM>
__device__ __forceinline__ double residual_unscaled(const Mat& A, const double* __restrict__ a0, const double* y,
                                                    const double* d, const double* __restrict__ b, double* dsm) {
    if constexpr (FORM == 5 || sliced_form(FORM)) {   // on the CSR arrays (a0 is CSR-ordered)
        double tr2 = 0.0;
        spmv_direct<double, double>(A, a0, GatherUnscaled{y, d}, [&](int i) { return b[i]; },
                                    [&](int, double s, double bi) { sq_acc(tr2, resid(bi, s)); });
        return tr2;
    } else {
        return residual_unscaled_staged<FORM>(A, a0, y, d, b, dsm);
    }
}

// v = A p, sigma = r^.v; with `check` set, the true residual first:
// ||b - A y||^2, or with right Jacobi (dsc != nullptr, the iteration on the
// column-scaled A D^-1) ||b - A0 x||^2 of the x = y / d the solve returns,
// on the unscaled values a0, so the stopping test holds for that x.
template <int FORM>
__global__ void __launch_bounds__(NT, (ProductCtas<double, FORM>::value))
    k_bicg_v(Mat A, Sys S, const double* __restrict__ av, const double* __restrict__ p, double* __restrict__ v,
             const double* __restrict__ rh, const double* __restrict__ y, const double* __restrict__ b,
             const double* __restrict__ a0, const double* __restrict__ dsc) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    av += val_offset<FORM>(A, sys, S.nnz); p += vo; v += vo; rh += vo; y += vo; b += vo;
    const bool check = ld_cg(&st->check) != 0;
    double tr2 = 0.0, sigma = 0.0;
    if (check) {
        if (dsc) tr2 = residual_unscaled<FORM>(A, a0 + ao, y, dsc + vo, b, dsm);
        else tr2 = residual_pass<double, FORM>(A, av, y, b, dsm);
    }
    spmv_vec<double, FORM, double, double>(A, av, p, [&](int i) { return ld_vec(rh + i); },
                                           [&](int i, double s, double rhi) {
                                               st_vec(v + i, s);
                                               sigma = fma(rhi, s, sigma);
                                           },
                                           dsm);
    double vals[2] = {sigma, tr2}, tot[2];
    if (grid_sum<2>(vals, part, cnt, tot, red) && threadIdx.x == 0)
        bicg_after_v(st, S.ctl, tot[0], check, tot[1]);
}

// s = r - alpha v, written over r.
template <int W>
__global__ void __launch_bounds__(NT) k_bicg_s(Sys S, double* __restrict__ r, const double* __restrict__ v) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    r += vo; v += vo;
    const double alpha = ld_cg(&st->alpha);
    BICG_LOOP(W) {
        Vd<W> ri = vld<W>(r, i);
        const Vd<W> vi = vld<W>(v, i);
#pragma unroll
        for (int e = 0; e < W; ++e) ri.e[e] = fma(-alpha, vi.e[e], ri.e[e]);
        vst<W>(r, i, ri);
    }
}

// t = A s, t.t and t.s -> omega.
template <int FORM>
__global__ void __launch_bounds__(NT, (ProductCtas<double, FORM>::value))
    k_bicg_t(Mat A, Sys S, const double* __restrict__ av, const double* __restrict__ s, double* __restrict__ t) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    av += val_offset<FORM>(A, sys, S.nnz); s += vo; t += vo;
    double tt = 0.0, ts = 0.0;
    spmv_vec<double, FORM, double, double>(A, av, s, [&](int i) { return ld_vec(s + i); },
                                           [&](int i, double q, double si) {
                                               st_vec(t + i, q);
                                               tt = fma(q, q, tt);
                                               ts = fma(q, si, ts);
                                           },
                                           dsm);
    double vals[2] = {tt, ts}, tot[2];
    if (grid_sum<2>(vals, part, cnt, tot, red) && threadIdx.x == 0) bicg_after_t(st, S.ctl, tot[0], tot[1]);
}

// y += alpha p + omega s; r = s - omega t (r holds s on entry); gamma = r.r,
// rho' = r^.r.
template <int W>
__global__ void __launch_bounds__(NT) k_bicg_xr(Sys S, double* __restrict__ y, const double* __restrict__ p,
                                                double* __restrict__ r, const double* __restrict__ t,
                                                const double* __restrict__ rh) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[RED_DOUBLES];
    y += vo; p += vo; r += vo; t += vo; rh += vo;
    const double alpha = ld_cg(&st->alpha), omega = ld_cg(&st->omega);
    double g = 0.0, rho = 0.0;
    BICG_LOOP(W) {
        Vd<W> yi = vld<W>(y, i), si = vld<W>(r, i);
        const Vd<W> pi = vld<W>(p, i), ti = vld_last<W>(t, i), hi = vld<W>(rh, i);
#pragma unroll
        for (int e = 0; e < W; ++e) {
            yi.e[e] = fma(omega, si.e[e], fma(alpha, pi.e[e], yi.e[e]));
            const double rn = fma(-omega, ti.e[e], si.e[e]);
            si.e[e] = rn;
            g = fma(rn, rn, g);
            rho = fma(hi.e[e], rn, rho);
        }
        vst<W>(y, i, yi);
        vst<W>(r, i, si);
    }
    double vals[2] = {g, rho}, tot[2];
    if (grid_sum<2>(vals, part, cnt, tot, red) && threadIdx.x == 0)
        bicg_after_update(st, S.ctl, tot[0], tot[1]);
}

// p = r + beta (p - omega v).
template <int W>
__global__ void __launch_bounds__(NT) k_bicg_p(Sys S, double* __restrict__ p, const double* __restrict__ r,
                                               const double* __restrict__ v) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    p += vo; r += vo; v += vo;
    const double beta = ld_cg(&st->beta), omega = ld_cg(&st->omega);
    BICG_LOOP(W) {
        Vd<W> pi = vld<W>(p, i);
        const Vd<W> ri = vld<W>(r, i), vi = vld_last<W>(v, i);
#pragma unroll
        for (int e = 0; e < W; ++e) pi.e[e] = fma(beta, fma(-omega, vi.e[e], pi.e[e]), ri.e[e]);
        vst<W>(p, i, pi);
    }
}

// x = x * d (MUL) or x / d (division), every system: the change of variable
// y = D x of the column-scaled iteration, and back.
template <bool MUL>
__global__ void __launch_bounds__(NT) k_bicg_scale(Sys S, double* __restrict__ x, const double* __restrict__ d) {
    const size_t vo = (size_t)blockIdx.y * S.n;
    x += vo; d += vo;
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) x[i] = MUL ? x[i] * d[i] : x[i] / d[i];
}

// out[s][k] = in[s][k] / d[s][col(k)]: the values of A D^-1.
__global__ void __launch_bounds__(NT) k_bicg_colscale(long long nnz, int n, const int* __restrict__ ci,
                                                      const double* __restrict__ in, const double* __restrict__ d,
                                                      double* __restrict__ out) {
    const int sys = blockIdx.y;
    in += (size_t)sys * nnz;
    out += (size_t)sys * nnz;
    d += (size_t)sys * n;
    for (long long k = (long long)blockIdx.x * NT + threadIdx.x; k < nnz; k += (long long)gridDim.x * NT)
        out[k] = in[k] / d[ci[k]];
}

#undef BICG_LOOP

}  // namespace sla
