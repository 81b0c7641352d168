// kernels.cuh -- the PCG iteration, set-up and adjoint kernels.
//
// Batches: blockIdx.y is the system.  All systems share row_ptr / col_idx
// and the row-block partition; values, vectors, solver state, partial sums
// and arrival counters are offset per system.  A converged system's CTAs
// return at once, so frozen systems cost no memory traffic.
//
// SpMV layout (spmv_rows): one warp per group of 32 consecutive rows; the
// warp stages its non-zeros in shared memory, then each lane forms its row
// sum with one fp64 fused multiply-add per non-zero.  One FMA per non-zero is
// the least fp64 work an SpMV can do, which matters on a part whose fp64 rate
// is low next to its memory bandwidth.
//
// Grids are persistent in x (warps / CTAs walk row groups / vector ranges
// with a grid stride).  Inner products are reduced in a fixed order (grid_sum) and
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
    int n;            // rows
    int cap;          // staged entries per warp (per 32-row group)
    int async;        // 1: cp.async double-buffered staging (spmv_rows_async)
    int wstride;      // doubles of shared memory per warp (both staging forms)
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

// Rows are taken in groups of 32, one warp per group (grid stride over
// groups).  The warp stages its group's non-zeros -- values streamed with
// coalesced evict-first loads, the vector entries they address gathered
// through the read-only path -- as (value, entry) pairs in its own slice of
// shared memory (`cap` pairs), then each lane sums its own row with one fp64
// FMA per non-zero.  Only __syncwarp orders the two phases, so warps progress
// independently and hide each other's memory latency.  A group with more than
// `cap` non-zeros is summed straight from global memory: rows up to LONG
// entries by their lane, longer rows by the whole warp.
// epi(row, sum) is called once per row of the matrix by the row's lane.
constexpr int STAGE_U = 4;     // entries per lane in flight while staging
constexpr int LONG_ROW = 64;   // longer rows of an unstaged group go warp-wide

template <typename VT, class Gather, class Epi>
__device__ __forceinline__ void spmv_rows(const Mat& A, const VT* __restrict__ av, Gather gather, Epi epi,
                                          double* wsm) {
    const int lane = threadIdx.x & 31;
    const int cap = A.cap;
    double* sa = wsm + (threadIdx.x >> 5) * A.wstride;
    double* sx = sa + cap;
    const int ngroups = (A.n + 31) >> 5;
    const int nwarps = (gridDim.x * NT) >> 5;
    for (int grp = (blockIdx.x * NT + threadIdx.x) >> 5; grp < ngroups; grp += nwarps) {
        const int row = (grp << 5) + lane;
        const int rlo = ld_nc(A.rp + min(row, A.n));
        const int rhi = ld_nc(A.rp + min(row + 1, A.n));
        const int k0 = __shfl_sync(0xffffffffu, rlo, 0);
        const int k1 = __shfl_sync(0xffffffffu, rhi, 31);
        const int cnt = k1 - k0;
        double s = 0.0;
        if (cnt <= cap) {
            for (int base = 0; base < cnt; base += 32 * STAGE_U) {
                int c[STAGE_U];
                double a[STAGE_U], xv[STAGE_U];
#pragma unroll
                for (int j = 0; j < STAGE_U; ++j) {
                    const int e = base + j * 32 + lane;
                    if (e < cnt) {
                        c[j] = ld_stream(A.ci + k0 + e);
                        a[j] = (double)ld_stream(av + k0 + e);
                    }
                }
#pragma unroll
                for (int j = 0; j < STAGE_U; ++j) {
                    const int e = base + j * 32 + lane;
                    if (e < cnt) xv[j] = gather(c[j]);
                }
#pragma unroll
                for (int j = 0; j < STAGE_U; ++j) {
                    const int e = base + j * 32 + lane;
                    if (e < cnt) { sa[e] = a[j]; sx[e] = xv[j]; }
                }
            }
            __syncwarp();
            for (int e = rlo - k0; e < rhi - k0; ++e) s = fma(sa[e], sx[e], s);
            __syncwarp();
        } else {
            if (rhi - rlo <= LONG_ROW)
                for (int k = rlo; k < rhi; ++k) s = fma((double)ld_stream(av + k), gather(ld_stream(A.ci + k)), s);
            unsigned longs = __ballot_sync(0xffffffffu, rhi - rlo > LONG_ROW);
            while (longs) {
                const int src = __ffs(longs) - 1;
                longs &= longs - 1;
                const int a0 = __shfl_sync(0xffffffffu, rlo, src);
                const int a1 = __shfl_sync(0xffffffffu, rhi, src);
                double t = 0.0;
                for (int k = a0 + lane; k < a1; k += 32)
                    t = fma((double)ld_stream(av + k), gather(ld_stream(A.ci + k)), t);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == src) s = t;
            }
        }
        if (row < A.n) epi(row, s);
    }
}

// Pipelined form of spmv_rows for a plain vector gather (v[col] at its stored
// precision).  Each warp double-buffers its groups' values and column
// indices in shared memory with cp.async: the copies of the next group are in
// flight while the warp gathers and sums the current one, so every warp keeps
// ~12 bytes x (entries per group) of streaming traffic outstanding without
// holding registers for it.  The gathered entries go through registers
// (GATHER_U per lane in flight) into the warp's slice, then each lane sums
// its own row with one fp64 FMA per entry.  Shared memory per warp:
// 2*cap*(sizeof(VT) + 4) + 8*cap bytes (async_smem_per_warp).
constexpr int GATHER_U = 8;

template <typename VT>
__host__ __device__ constexpr size_t async_smem_per_warp(int cap) {
    return (size_t)2 * cap * (sizeof(VT) + sizeof(int)) + (size_t)cap * sizeof(double);
}

template <typename VT, typename T, class Epi>
__device__ __forceinline__ void spmv_rows_async(const Mat& A, const VT* __restrict__ av, const T* __restrict__ v,
                                                Epi epi, double* wsm) {
    const int lane = threadIdx.x & 31;
    const int cap = A.cap;
    char* base = reinterpret_cast<char*>(wsm + (threadIdx.x >> 5) * A.wstride);
    VT* sv = reinterpret_cast<VT*>(base);
    int* sc = reinterpret_cast<int*>(base + 2 * cap * sizeof(VT));
    double* sx = reinterpret_cast<double*>(base + 2 * cap * (sizeof(VT) + sizeof(int)));
    const unsigned long long pol = l2_evict_first();
    const int ngroups = (A.n + 31) >> 5;
    const int nwarps = (gridDim.x * NT) >> 5;
    const int g0 = (blockIdx.x * NT + threadIdx.x) >> 5;

    auto issue = [&](int grp, int stage) {
        if (grp < ngroups) {
            const int k0 = ld_nc(A.rp + (grp << 5));
            const int k1 = ld_nc(A.rp + min((grp << 5) + 32, A.n));
            if (k1 - k0 <= cap) {
                VT* dv = sv + stage * cap;
                int* dc = sc + stage * cap;
                for (int e = lane; e < k1 - k0; e += 32) {
                    cp_async<sizeof(VT)>(dv + e, av + k0 + e, pol);
                    cp_async<4>(dc + e, A.ci + k0 + e, pol);
                }
            }
        }
        cp_commit();
    };

    issue(g0, 0);
    int stage = 0;
    for (int grp = g0; grp < ngroups; grp += nwarps, stage ^= 1) {
        issue(grp + nwarps, stage ^ 1);
        const int row = (grp << 5) + lane;
        const int rlo = ld_nc(A.rp + min(row, A.n));
        const int rhi = ld_nc(A.rp + min(row + 1, A.n));
        const int k0 = __shfl_sync(0xffffffffu, rlo, 0);
        const int k1 = __shfl_sync(0xffffffffu, rhi, 31);
        const int cnt = k1 - k0;
        cp_wait<1>();  // this group's values and columns have landed
        __syncwarp();
        double s = 0.0;
        if (cnt <= cap) {
            const VT* cv = sv + stage * cap;
            const int* cc = sc + stage * cap;
            for (int b0 = 0; b0 < cnt; b0 += 32 * GATHER_U) {
                double xv[GATHER_U];
#pragma unroll
                for (int j = 0; j < GATHER_U; ++j) {
                    const int e = b0 + j * 32 + lane;
                    if (e < cnt) xv[j] = (double)ld_nc(v + cc[e]);
                }
#pragma unroll
                for (int j = 0; j < GATHER_U; ++j) {
                    const int e = b0 + j * 32 + lane;
                    if (e < cnt) sx[e] = xv[j];
                }
            }
            __syncwarp();
            for (int e = rlo - k0; e < rhi - k0; ++e) s = fma((double)cv[e], sx[e], s);
        } else {
            if (rhi - rlo <= LONG_ROW)
                for (int k = rlo; k < rhi; ++k) s = fma((double)ld_stream(av + k), (double)ld_nc(v + ld_stream(A.ci + k)), s);
            unsigned longs = __ballot_sync(0xffffffffu, rhi - rlo > LONG_ROW);
            while (longs) {
                const int src = __ffs(longs) - 1;
                longs &= longs - 1;
                const int a0 = __shfl_sync(0xffffffffu, rlo, src);
                const int a1 = __shfl_sync(0xffffffffu, rhi, src);
                double t = 0.0;
                for (int k = a0 + lane; k < a1; k += 32)
                    t = fma((double)ld_stream(av + k), (double)ld_nc(v + ld_stream(A.ci + k)), t);
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
                if (lane == src) s = t;
            }
        }
        __syncwarp();  // this stage and sx are free for reuse
        if (row < A.n) epi(row, s);
    }
    cp_wait<0>();
}

// Product with a plain vector gather: the pipelined form when the matrix was
// set up for it, the single-stage form otherwise.
template <typename VT, typename T, class Epi>
__device__ __forceinline__ void spmv_vec(const Mat& A, const VT* __restrict__ av, const T* __restrict__ v, Epi epi,
                                         double* wsm) {
    if (A.async) spmv_rows_async<VT>(A, av, v, epi, wsm);
    else spmv_rows<VT>(A, av, GatherVec<T>{v}, epi, wsm);
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
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spmv(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ x,
                                             T* __restrict__ y, double* dot) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; x += vo; y += vo;
    double acc = 0.0;
    spmv_vec<T>(A, av, x,
                 [&](int i, double s) {
                     const T yi = (T)s;
                     y[i] = yi;
                     acc = fma((double)x[i], (double)yi, acc);
                 },
                 dsm);
    if (dot) {
        double v[1] = {acc}, tot[1];
        if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) dot[sys] = tot[0];
    }
}

// ----------------------------------------------------------------- iteration
// q = A p, delta = p.q; with `check` set, ||b - A round(x)||^2 first.
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spmv_iter(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ p,
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
        spmv_rows<T>(A, av, GatherRounded<T>{x},
                     [&](int i, double s) {
                         const double e = (double)b[i] - s;
                         tr2 = fma(e, e, tr2);
                     },
                     dsm);
    }
    spmv_vec<T>(A, av, p,
                 [&](int i, double s) {
                     const T qi = (T)s;
                     q[i] = qi;
                     delta = fma((double)p[i], (double)qi, delta);
                 },
                 dsm);
    double v[2] = {delta, tr2}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0) after_spmv(st, S.ctl, tot[0], check, tot[1]);
}

// Pairs of consecutive entries (8/16-byte vector accesses) for the streaming
// kernels; used when n is even, so every system's vectors stay aligned.
template <typename T> struct Pair;
template <> struct Pair<double> { using type = double2; };
template <> struct Pair<float> { using type = float2; };

// x += alpha p; r -= alpha q; gamma = r.r; rho' = r.z (PC 0: z = r, PC 1:
// z = r / A_ii; PC 2: z comes later from the SPAI kernels).
template <typename T, int PC>
__device__ __forceinline__ void update_one(double alpha, double& x, T& r, double p, double q, double dinv,
                                           double& g, double& rz) {
    x = fma(alpha, p, x);
    const double ri = rnd<T>(fma(-alpha, q, (double)r));
    r = (T)ri;
    g = fma(ri, ri, g);
    if (PC == 1) rz = fma(ri, rnd<T>(ri * dinv), rz);
}

template <typename T, int PC, bool PAIRS>
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
    if (PAIRS) {
        // two pairs per thread per trip, all loads issued before any use
        using P2 = typename Pair<T>::type;
        const int n2 = S.n >> 1;
        const int stride = gridDim.x * NT;
        for (int i0 = blockIdx.x * NT + threadIdx.x; i0 < n2; i0 += 2 * stride) {
            P2 p2[2], q2[2], r2[2];
            double2 x2[2], d2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    p2[u] = ld_stream(reinterpret_cast<const P2*>(p) + i);
                    q2[u] = ld_stream(reinterpret_cast<const P2*>(q) + i);
                    x2[u] = reinterpret_cast<const double2*>(x)[i];
                    r2[u] = reinterpret_cast<const P2*>(r)[i];
                    d2[u] = PC == 1 ? ld_stream(reinterpret_cast<const double2*>(dinv) + i) : make_double2(0.0, 0.0);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    update_one<T, PC>(alpha, x2[u].x, r2[u].x, (double)p2[u].x, (double)q2[u].x, d2[u].x, g, rz);
                    update_one<T, PC>(alpha, x2[u].y, r2[u].y, (double)p2[u].y, (double)q2[u].y, d2[u].y, g, rz);
                    reinterpret_cast<double2*>(x)[i] = x2[u];
                    reinterpret_cast<P2*>(r)[i] = r2[u];
                }
            }
        }
    } else {
        for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
            double xi = x[i];
            T ri = r[i];
            update_one<T, PC>(alpha, xi, ri, (double)ld_stream(p + i), (double)ld_stream(q + i),
                              PC == 1 ? dinv[i] : 0.0, g, rz);
            x[i] = xi;
            r[i] = ri;
        }
    }
    double v[2] = {g, rz}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0)
        after_update(st, S.ctl, tot[0], PC != 2, PC == 0 ? tot[0] : tot[1]);
}

// p = z + beta p   (INIT: p = z)
template <typename T, int PC, bool INIT>
__device__ __forceinline__ T pnew(double beta, double p, double r, double dinv, double z) {
    double zi;
    if (PC == 0) zi = r;
    else if (PC == 1) zi = rnd<T>(r * dinv);
    else zi = z;
    return INIT ? (T)zi : (T)fma(beta, p, zi);
}

template <typename T, int PC, bool INIT, bool PAIRS>
__global__ void __launch_bounds__(NT) k_pupdate(Sys S, T* __restrict__ p, const T* __restrict__ r,
                                                const T* __restrict__ z, const double* __restrict__ dinv) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    p += vo; r += vo;
    if (PC == 1) dinv += vo;
    if (PC == 2) z += vo;
    const double beta = INIT ? 0.0 : ld_cg(&st->beta);
    if (PAIRS) {
        using P2 = typename Pair<T>::type;
        const int n2 = S.n >> 1;
        const int stride = gridDim.x * NT;
        for (int i0 = blockIdx.x * NT + threadIdx.x; i0 < n2; i0 += 2 * stride) {
            P2 r2[2], p2[2], z2[2];
            double2 d2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    r2[u] = ld_stream(reinterpret_cast<const P2*>(r) + i);
                    p2[u] = INIT ? P2{} : reinterpret_cast<const P2*>(p)[i];
                    d2[u] = PC == 1 ? ld_stream(reinterpret_cast<const double2*>(dinv) + i) : make_double2(0.0, 0.0);
                    z2[u] = PC == 2 ? ld_stream(reinterpret_cast<const P2*>(z) + i) : P2{};
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    p2[u].x = pnew<T, PC, INIT>(beta, (double)p2[u].x, (double)r2[u].x, d2[u].x, (double)z2[u].x);
                    p2[u].y = pnew<T, PC, INIT>(beta, (double)p2[u].y, (double)r2[u].y, d2[u].y, (double)z2[u].y);
                    reinterpret_cast<P2*>(p)[i] = p2[u];
                }
            }
        }
    } else {
        for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT)
            p[i] = pnew<T, PC, INIT>(beta, INIT ? 0.0 : (double)p[i], (double)r[i], PC == 1 ? dinv[i] : 0.0,
                                     PC == 2 ? (double)z[i] : 0.0);
    }
}

// SPAI, first product: t = G^T r (explicit transposed CSR of G; G values
// are per system, [batch][nnz(G)]).
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spai_t(Mat GT, Sys S, long long nnzg, const double* __restrict__ gtv,
                                               const T* __restrict__ r, T* __restrict__ t) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    gtv += (size_t)sys * nnzg; r += vo; t += vo;
    spmv_vec<double>(GT, gtv, r, [&](int i, double s) { t[i] = (T)s; }, dsm);
}

// SPAI, second product: z = G t + eps r, rho' = r.z -> beta (or rho at set-up).
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spai_z(Mat G, Sys S, long long nnzg, const double* __restrict__ gv,
                                               const T* __restrict__ t, const T* __restrict__ r,
                                               T* __restrict__ z, double eps) {
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    gv += (size_t)sys * nnzg; t += vo; r += vo; z += vo;
    double rz = 0.0;
    spmv_vec<double>(G, gv, t,
                      [&](int i, double s) {
                          const double ri = (double)r[i];
                          const double zi = rnd<T>(fma(eps, ri, s));
                          z[i] = (T)zi;
                          rz = fma(ri, zi, rz);
                      },
                      dsm);
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
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_init_x0(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ b_user,
                                                const T* __restrict__ x0, T* __restrict__ bw,
                                                double* __restrict__ x, T* __restrict__ r, double tol,
                                                int max_iter) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; b_user += vo; x0 += vo; bw += vo; x += vo; r += vo;
    double bb = 0.0, g = 0.0;
    spmv_rows<T>(A, av, GatherVec<T>{x0},
                 [&](int i, double s) {
                     const T bi = b_user[i];
                     bw[i] = bi;
                     x[i] = (double)x0[i];
                     const double ri = rnd<T>((double)bi - s);
                     r[i] = (T)ri;
                     bb = fma((double)bi, (double)bi, bb);
                     g = fma(ri, ri, g);
                 },
                 dsm);
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
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_final(Mat A, Sys S, const T* __restrict__ av, const double* __restrict__ x,
                                              const T* __restrict__ bw, T* __restrict__ x_out, Stat* out) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; x += vo; bw += vo; x_out += vo;
    const bool zero_b = ld_cg(&st->bb) == 0.0;
    double tr2 = 0.0;
    spmv_rows<T>(A, av, GatherRounded<T>{x},
                 [&](int i, double s) {
                     x_out[i] = zero_b ? (T)0 : (T)x[i];
                     const double e = (double)bw[i] - s;
                     tr2 = fma(e, e, tr2);
                 },
                 dsm);
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

// dL/dA_k = -lambda_row(k) * x_col(k) over the pattern.  One warp per group
// of 32 rows: the row of each of the group's entries is recorded in the
// warp's shared-memory slice, then the entries stream (coalesced reads of
// col_idx, coalesced writes of dA).  A group with more than `cap` entries is
// written row by row from its lanes.
template <typename T>
__global__ void __launch_bounds__(NT) k_grad_A(Mat A, Sys S, const T* __restrict__ lam, const T* __restrict__ x,
                                               T* __restrict__ dA) {
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    int* srow = reinterpret_cast<int*>(dsm + (threadIdx.x >> 5) * A.wstride);
    const int lane = threadIdx.x & 31;
    lam += vo; x += vo; dA += ao;
    const int ngroups = (A.n + 31) >> 5;
    const int nwarps = (gridDim.x * NT) >> 5;
    for (int grp = (blockIdx.x * NT + threadIdx.x) >> 5; grp < ngroups; grp += nwarps) {
        const int row = (grp << 5) + lane;
        const int rlo = ld_nc(A.rp + min(row, A.n));
        const int rhi = ld_nc(A.rp + min(row + 1, A.n));
        const int k0 = __shfl_sync(0xffffffffu, rlo, 0);
        const int k1 = __shfl_sync(0xffffffffu, rhi, 31);
        const int cnt_ = k1 - k0;
        if (cnt_ <= A.cap) {
            for (int e = rlo - k0; e < rhi - k0; ++e) srow[e] = row;
            __syncwarp();
            for (int e = lane; e < cnt_; e += 32) {
                const int c = ld_stream(A.ci + k0 + e);
                const double li = (double)ld_nc(lam + srow[e]);
                __stcs(dA + k0 + e, (T)(-li * (double)ld_nc(x + c)));
            }
            __syncwarp();
        } else if (row < A.n) {
            const double li = (double)lam[row];
            for (int k = rlo; k < rhi; ++k) __stcs(dA + k, (T)(-li * (double)ld_nc(x + ld_stream(A.ci + k))));
        }
    }
}

}  // namespace sla
