// kernels.cuh -- the PCG iteration, set-up and adjoint kernels.
//
// Batches: blockIdx.y is the system.  All systems share row_ptr / col_idx
// and the row-block partition; values, vectors, solver state, partial sums
// and arrival counters are offset per system.  A converged system's CTAs
// return at once, so frozen systems cost no memory traffic.
//
// SpMV layout: the rows are cut into row blocks of at most MAXR rows whose
// non-zeros fit a TILE-entry shared-memory stage (a row longer than TILE is a
// block of its own).  A CTA streams a block's values and column indices with
// coalesced, evict-first loads, gathers the vector entries they address, and
// stages (value, vector entry) pairs in shared memory; then one thread per
// row forms the row sum with one fp64 fused multiply-add per non-zero.  One
// FMA per non-zero is the least fp64 work an SpMV can do, which matters on a
// part whose fp64 rate is low next to its memory bandwidth.
//
// Grids are persistent in x (CTAs walk row blocks / vector ranges with a
// grid stride).  Inner products are reduced in a fixed order (grid_sum) and
// the last CTA to finish updates that system's scalars on the device, so no
// host round trip sits inside an iteration.
//
// CG step order (torch-sla §3.3, distributed CG; Hestenes-Stiefel order):
//   k_spmv_iter:  q = A p, delta = p.q -> alpha = rho / delta  (and, when the
//                 recursive residual met tol, the true residual of x first)
//   k_update:     x += alpha p, r -= alpha q, gamma = r.r, (Jacobi) rho' = r.z
//   [SPAI]        k_spai_t: t = G^T r ; k_spai_z: z = G t + eps r, rho' = r.z
//   k_pupdate:    p = z + beta p
#pragma once

#include "common.cuh"

namespace sla {

// Per-call addressing of a batch.
struct Sys {
    int n;            // rows (= columns)
    long long nnz;    // stored entries of one system
    State* st;        // [batch]
    Ctrl* ctl;        // one
    unsigned* cnt;    // [batch] arrival counters
    double* part;     // [batch][pstride] partial sums
    int pstride;
};

struct Mat {
    const int* rp;
    const int* ci;
    const int* rbs;   // row-block starts [nblk + 1]
    int nblk;
};

#define SYS_PROLOGUE                                            \
    const int sys = blockIdx.y;                                 \
    State* st = S.st + sys;                                     \
    double* part = S.part + (size_t)sys * S.pstride;            \
    unsigned* cnt = S.cnt + sys;                                \
    const size_t vo = (size_t)sys * S.n;                        \
    const size_t ao = (size_t)sys * S.nnz;                      \
    (void)st; (void)part; (void)cnt; (void)vo; (void)ao;

// ----------------------------------------------------------------- gathers
template <typename T>
struct GatherVec {  // vector entry at the system precision
    const T* v;
    __device__ __forceinline__ double operator()(int c) const { return (double)ld_nc(v + c); }
};
template <typename T>
struct GatherRounded {  // fp64 iterate rounded to the returned precision
    const double* v;
    __device__ __forceinline__ double operator()(int c) const { return rnd<T>(ld_nc(v + c)); }
};

// Walk the row blocks of this CTA.  For every row, epi(row, sum) is called by
// exactly one thread (thread-per-row for normal blocks, thread 0 for a long
// row).  Must be called by all threads of the CTA.
template <typename VT, int TILE, class Gather, class Epi>
__device__ __forceinline__ void spmv_rows(const Mat& A, const VT* __restrict__ av, Gather gather, Epi epi,
                                          double* sa, double* sx, double* red) {
    constexpr int PER = TILE / NT;
    for (int b = blockIdx.x; b < A.nblk; b += gridDim.x) {
        const int r0 = A.rbs[b], r1 = A.rbs[b + 1];
        const int k0 = A.rp[r0], k1 = A.rp[r1];
        const int cnt = k1 - k0;
        if (cnt <= TILE) {
            int c[PER];
            double a[PER], xv[PER];
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int e = threadIdx.x + j * NT;
                if (e < cnt) {
                    c[j] = ld_stream(A.ci + k0 + e);
                    a[j] = (double)ld_stream(av + k0 + e);
                }
            }
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int e = threadIdx.x + j * NT;
                if (e < cnt) xv[j] = gather(c[j]);
            }
#pragma unroll
            for (int j = 0; j < PER; ++j) {
                const int e = threadIdx.x + j * NT;
                if (e < cnt) { sa[e] = a[j]; sx[e] = xv[j]; }
            }
            __syncthreads();
            const int row = r0 + threadIdx.x;
            if (row < r1) {
                const int e0 = A.rp[row] - k0, e1 = A.rp[row + 1] - k0;
                double s = 0.0;
                for (int e = e0; e < e1; ++e) s = fma(sa[e], sx[e], s);
                epi(row, s);
            }
            __syncthreads();
        } else {  // one long row
            double s = 0.0;
            for (int k = k0 + threadIdx.x; k < k1; k += NT)
                s = fma((double)ld_stream(av + k), gather(ld_stream(A.ci + k)), s);
            double v[1] = {s};
            block_sum<1>(v, red);
            if (threadIdx.x == 0) epi(r0, v[0]);
            __syncthreads();
        }
    }
}

// ----------------------------------------------------------------- scalar logic
// All of these run in thread 0 of the last CTA of one system.
__device__ __forceinline__ void freeze(State* s, Ctrl* c, int status) {
    s->status = status;
    s->done = 1;
    __threadfence();
    if (atomicAdd(&c->ndone, 1) + 1 == (int)gridDim.y) c->all_done = 1;
}

// After the p.q reduction (and the optional true-residual check).
__device__ __forceinline__ void after_spmv(State* s, Ctrl* c, double delta, bool checked, double tr2) {
    if (checked) {
        s->tr2 = tr2;
        if (tr2 <= s->tol2bb) { freeze(s, c, ST_OK); return; }
        s->check = 0;
        if (s->iter >= s->max_iter) { freeze(s, c, ST_NOT_CONVERGED); return; }
        if (s->rho_bad) { freeze(s, c, ST_BREAKDOWN); return; }
    }
    s->delta = delta;
    if (!(delta > 0.0) || !finite(delta)) { freeze(s, c, ST_BREAKDOWN); return; }
    s->alpha = s->rho / delta;
    s->iter += 1;
}

// beta from the new r.z (or, in the set-up phase, the first rho).
__device__ __forceinline__ void new_direction(State* s, Ctrl* c, double rho_new) {
    if (!(rho_new > 0.0) || !finite(rho_new)) {
        if (s->check) { s->rho_bad = 1; s->beta = 0.0; s->phase = 1; }
        else freeze(s, c, ST_BREAKDOWN);
        return;
    }
    if (s->phase == 0) { s->rho = rho_new; s->phase = 1; return; }
    s->beta = rho_new / s->rho;
    s->rho = rho_new;
}

// After the x / r update: convergence test on the recursive residual.
__device__ __forceinline__ void after_update(State* s, Ctrl* c, double gamma, bool have_rho,
                                             double rho_new) {
    s->gamma = gamma;
    if (!finite(gamma)) { freeze(s, c, ST_BREAKDOWN); return; }
    s->check = (gamma <= s->tol2bb);
    if (!s->check && s->iter >= s->max_iter) { freeze(s, c, ST_NOT_CONVERGED); return; }
    if (have_rho) new_direction(s, c, rho_new);
}

__device__ __forceinline__ void start_state(State* s, Ctrl* c, double bb, double gamma, double tol,
                                            int max_iter) {
    s->bb = bb;
    s->tol2bb = tol * tol * bb;
    s->gamma = gamma;
    s->iter = 0;
    s->max_iter = max_iter;
    s->status = ST_OK;
    s->done = 0;
    s->check = 0;
    s->rho_bad = 0;
    s->phase = 0;
    s->alpha = s->beta = s->rho = s->delta = s->tr2 = 0.0;
    if (bb == 0.0) { freeze(s, c, ST_OK); return; }   // x = 0 is exact
    if (!finite(gamma)) { freeze(s, c, ST_BREAKDOWN); return; }
    s->check = (gamma <= s->tol2bb);
    if (!s->check && max_iter <= 0) freeze(s, c, ST_NOT_CONVERGED);
}

// ----------------------------------------------------------------- SpMV API
// y = A x, and dot[sys] = x.y when dot != nullptr.
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_spmv(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ x,
                                             T* __restrict__ y, double* dot) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; x += vo; y += vo;
    double acc = 0.0;
    spmv_rows<T, TILE>(A, av, GatherVec<T>{x},
                       [&](int i, double s) {
                           const T yi = (T)s;
                           y[i] = yi;
                           acc = fma((double)x[i], (double)yi, acc);
                       },
                       dsm, dsm + TILE, red);
    if (dot) {
        double v[1] = {acc}, tot[1];
        if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) dot[sys] = tot[0];
    }
}

// ----------------------------------------------------------------- iteration
// q = A p, delta = p.q; with `check` set, ||b - A round(x)||^2 first.
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_spmv_iter(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ p,
                                                  T* __restrict__ q, const double* __restrict__ x,
                                                  const T* __restrict__ b) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; p += vo; q += vo; x += vo; b += vo;
    const bool check = ld_cg(&st->check) != 0;
    double tr2 = 0.0, delta = 0.0;
    if (check) {
        spmv_rows<T, TILE>(A, av, GatherRounded<T>{x},
                           [&](int i, double s) {
                               const double e = (double)b[i] - s;
                               tr2 = fma(e, e, tr2);
                           },
                           dsm, dsm + TILE, red);
    }
    spmv_rows<T, TILE>(A, av, GatherVec<T>{p},
                       [&](int i, double s) {
                           const T qi = (T)s;
                           q[i] = qi;
                           delta = fma((double)p[i], (double)qi, delta);
                       },
                       dsm, dsm + TILE, red);
    double v[2] = {delta, tr2}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0) after_spmv(st, S.ctl, tot[0], check, tot[1]);
}

// x += alpha p; r -= alpha q; gamma = r.r; rho' = r.z (PC 0: z = r, PC 1:
// z = r / A_ii; PC 2: z comes later from the SPAI kernels).
template <typename T, int PC>
__global__ void __launch_bounds__(NT) k_update(Sys S, double* __restrict__ x, T* __restrict__ r,
                                               const T* __restrict__ p, const T* __restrict__ q,
                                               const double* __restrict__ dinv) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[2 * NWARP];
    x += vo; r += vo; p += vo; q += vo;
    if (PC == 1) dinv += vo;
    const double alpha = ld_cg(&st->alpha);
    double g = 0.0, rz = 0.0;
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
        const double pi = (double)ld_stream(p + i);
        const double qi = (double)ld_stream(q + i);
        x[i] = fma(alpha, pi, x[i]);
        const double ri = rnd<T>(fma(-alpha, qi, (double)r[i]));
        r[i] = (T)ri;
        g = fma(ri, ri, g);
        if (PC == 1) rz = fma(ri, rnd<T>(ri * dinv[i]), rz);
    }
    double v[2] = {g, rz}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0)
        after_update(st, S.ctl, tot[0], PC != 2, PC == 0 ? tot[0] : tot[1]);
}

// p = z + beta p   (INIT: p = z)
template <typename T, int PC, bool INIT>
__global__ void __launch_bounds__(NT) k_pupdate(Sys S, T* __restrict__ p, const T* __restrict__ r,
                                                const T* __restrict__ z, const double* __restrict__ dinv) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    p += vo; r += vo;
    if (PC == 1) dinv += vo;
    if (PC == 2) z += vo;
    const double beta = INIT ? 0.0 : ld_cg(&st->beta);
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
        double zi;
        if (PC == 0) zi = (double)r[i];
        else if (PC == 1) zi = rnd<T>((double)r[i] * dinv[i]);
        else zi = (double)z[i];
        p[i] = INIT ? (T)zi : (T)fma(beta, (double)p[i], zi);
    }
}

// SPAI, first product: t = G^T r (explicit transposed CSR of G; G values
// are per system, [batch][nnz(G)]).
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_spai_t(Mat GT, Sys S, long long nnzg, const double* __restrict__ gtv,
                                               const T* __restrict__ r, T* __restrict__ t) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    gtv += (size_t)sys * nnzg; r += vo; t += vo;
    spmv_rows<double, TILE>(GT, gtv, GatherVec<T>{r}, [&](int i, double s) { t[i] = (T)s; }, dsm, dsm + TILE,
                            red);
}

// SPAI, second product: z = G t + eps r, rho' = r.z -> beta (or rho at set-up).
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_spai_z(Mat G, Sys S, long long nnzg, const double* __restrict__ gv,
                                               const T* __restrict__ t, const T* __restrict__ r,
                                               T* __restrict__ z, double eps) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    gv += (size_t)sys * nnzg; t += vo; r += vo; z += vo;
    double rz = 0.0;
    spmv_rows<double, TILE>(G, gv, GatherVec<T>{t},
                            [&](int i, double s) {
                                const double ri = (double)r[i];
                                const double zi = rnd<T>(fma(eps, ri, s));
                                z[i] = (T)zi;
                                rz = fma(ri, zi, rz);
                            },
                            dsm, dsm + TILE, red);
    double v[1] = {rz}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) new_direction(st, S.ctl, tot[0]);
}

// ----------------------------------------------------------------- set-up / final
// x = 0, r = b, b copied into the workspace, bb = b.b.
template <typename T>
__global__ void __launch_bounds__(NT) k_init(Sys S, const T* __restrict__ b_user, T* __restrict__ bw,
                                             double* __restrict__ x, T* __restrict__ r, double tol, int max_iter) {
    SYS_PROLOGUE
    __shared__ double red[2 * NWARP];
    b_user += vo; bw += vo; x += vo; r += vo;
    double bb = 0.0;
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
        const T bi = b_user[i];
        bw[i] = bi;
        r[i] = bi;
        x[i] = 0.0;
        bb = fma((double)bi, (double)bi, bb);
    }
    double v[1] = {bb}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0)
        start_state(st, S.ctl, tot[0], tot[0], tol, max_iter);
}

// With an initial guess: x = x0, r = b - A x0, bb = b.b, gamma = r.r.
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_init_x0(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ b_user,
                                                const T* __restrict__ x0, T* __restrict__ bw,
                                                double* __restrict__ x, T* __restrict__ r, double tol,
                                                int max_iter) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; b_user += vo; x0 += vo; bw += vo; x += vo; r += vo;
    double bb = 0.0, g = 0.0;
    spmv_rows<T, TILE>(A, av, GatherVec<T>{x0},
                       [&](int i, double s) {
                           const T bi = b_user[i];
                           bw[i] = bi;
                           x[i] = (double)x0[i];
                           const double ri = rnd<T>((double)bi - s);
                           r[i] = (T)ri;
                           bb = fma((double)bi, (double)bi, bb);
                           g = fma(ri, ri, g);
                       },
                       dsm, dsm + TILE, red);
    double v[2] = {bb, g}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0)
        start_state(st, S.ctl, tot[0], tot[1], tol, max_iter);
}

// First direction for PC 0 / 1: p = z, rho = r.z.
template <typename T, int PC>
__global__ void __launch_bounds__(NT) k_init_dir(Sys S, T* __restrict__ p, const T* __restrict__ r,
                                                 const double* __restrict__ dinv) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[2 * NWARP];
    p += vo; r += vo;
    if (PC == 1) dinv += vo;
    double rz = 0.0;
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
        const double ri = (double)r[i];
        const double zi = PC == 1 ? rnd<T>(ri * dinv[i]) : ri;
        p[i] = (T)zi;
        rz = fma(ri, zi, rz);
    }
    double v[1] = {rz}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) new_direction(st, S.ctl, tot[0]);
}

struct Stat {
    int iters;
    int status;
    double rel_rec;
    double rel_true;
    int done;
    int pad;
};

// Returned x = round(x_w) (0 when b = 0); true residual of that x; statistics.
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_final(Mat A, Sys S, const T* __restrict__ av, const double* __restrict__ x,
                                              const T* __restrict__ bw, T* __restrict__ x_out, Stat* out) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; x += vo; bw += vo; x_out += vo;
    const bool zero_b = ld_cg(&st->bb) == 0.0;
    double tr2 = 0.0;
    spmv_rows<T, TILE>(A, av, GatherRounded<T>{x},
                       [&](int i, double s) {
                           x_out[i] = zero_b ? (T)0 : (T)x[i];
                           const double e = (double)bw[i] - s;
                           tr2 = fma(e, e, tr2);
                       },
                       dsm, dsm + TILE, red);
    double v[1] = {tr2}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) {
        const double bb = st->bb;
        Stat o;
        o.iters = st->iter;
        o.status = st->status;
        o.rel_rec = bb > 0.0 ? sqrt(st->gamma / bb) : 0.0;
        o.rel_true = bb > 0.0 ? sqrt(tot[0] / bb) : 0.0;
        o.done = st->done;
        o.pad = 0;
        out[sys] = o;
    }
}

// dL/dA_k = -lambda_row(k) * x_col(k) over the pattern (row blocks; the row
// of each staged entry is recorded in shared memory so reads and writes of
// the nnz-sized arrays stream).
template <typename T, int TILE>
__global__ void __launch_bounds__(NT) k_grad_A(Mat A, Sys S, const T* __restrict__ lam, const T* __restrict__ x,
                                               T* __restrict__ dA) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    int* srow = reinterpret_cast<int*>(dsm);
    lam += vo; x += vo; dA += ao;
    for (int b = blockIdx.x; b < A.nblk; b += gridDim.x) {
        const int r0 = A.rbs[b], r1 = A.rbs[b + 1];
        const int k0 = A.rp[r0], k1 = A.rp[r1];
        const int cnt_ = k1 - k0;
        if (cnt_ <= TILE) {
            const int row = r0 + threadIdx.x;
            if (row < r1) {
                const int e0 = A.rp[row] - k0, e1 = A.rp[row + 1] - k0;
                for (int e = e0; e < e1; ++e) srow[e] = row;
            }
            __syncthreads();
            for (int e = threadIdx.x; e < cnt_; e += NT) {
                const int c = ld_stream(A.ci + k0 + e);
                const double li = (double)ld_nc(lam + srow[e]);
                __stcs(dA + k0 + e, (T)(-li * (double)ld_nc(x + c)));
            }
            __syncthreads();
        } else {
            const double li = (double)lam[r0];
            for (int k = k0 + threadIdx.x; k < k1; k += NT)
                __stcs(dA + k, (T)(-li * (double)ld_nc(x + ld_stream(A.ci + k))));
        }
    }
}

}  // namespace sla
