// kernels.cuh -- the PCG iteration, set-up and adjoint kernels.
//
// Batches: blockIdx.y is the system.  All systems share row_ptr / col_idx;
// values, vectors, solver state, partial sums and arrival counters are
// offset per system.  A converged system's CTAs return at once, so frozen
// systems cost no memory traffic.
//
// Precision (Prec<T>, T = stored vector type):
//  * fp64 systems compute in fp64: one fused multiply-add per stored entry
//    in the SpMV (the least fp64 work an SpMV can do -- B300's fp64 pipe
//    issues at 1/64 of its fp32 rate), fp64 updates and dot products.
//  * fp32 systems store A, b, r, p, q, z, t in fp32 and keep x and the
//    Jacobi reciprocal as double-float pairs (df.cuh).  All element-wise
//    arithmetic is double-float on the fp32 pipe: products of fp32 values
//    are exact and sums carry ~48 bits before each stored vector is rounded
//    to fp32.  Only per-thread totals and the solver scalars use fp64.
//
// SpMV layout (spmv_rows / spmv_rows_async): one warp per group of 32 / L
// consecutive rows (L = 1, 2 or 4 lanes per row, from the row lengths); the
// warp stages its non-zeros in its own shared-memory slice, then the lanes of
// each row sum it.  Grids are persistent in x.
// Inner products are reduced in a fixed order (grid_sum) and the last CTA to
// finish updates that system's scalars on the device, so no host round trip
// sits inside an iteration.
//
// CG step order (torch-sla §3.3, distributed CG; Hestenes-Stiefel order):
//   k_spmv_iter:  q = A p, delta = p.q -> alpha = rho / delta  (and, when the
//                 recursive residual met tol, the true residual of x first)
//   k_update:     x += alpha p, r -= alpha q, gamma = r.r, (Jacobi) rho' = r.z
//   [SPAI]        k_spai_t: t = G^T r ; k_spai_z: z = G t + eps r, rho' = r.z
//   k_pupdate:    p = z + beta p
#pragma once

#include <type_traits>

#include "common.cuh"
#include "df.cuh"

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
    int cap;          // staged entries per warp (per group of 32 / lanes rows)
    int async;        // 0: register staging (spmv_rows); 1 / 2: cp.async staging, value/column
                      //    copies single / double buffered (spmv_rows_async)
    int wstride;      // doubles of shared memory per warp (both staging forms)
    int lanes;        // lanes per row: 1, 2 or 4 (a group holds 32 / lanes rows)
    int lshift;       // log2(lanes)
};

#define SYS_PROLOGUE                                            \
    const int sys = blockIdx.y;                                 \
    State* st = S.st + sys;                                     \
    double* part = S.part + (size_t)sys * S.pstride;            \
    unsigned* cnt = S.cnt + sys;                                \
    const size_t vo = (size_t)sys * S.n;                        \
    const size_t ao = (size_t)sys * S.nnz;                      \
    (void)st; (void)part; (void)cnt; (void)vo; (void)ao;

// ----------------------------------------------------------------- precision
template <typename T> struct Prec;
template <> struct Prec<double> {
    using acc = double;   // row sums and inner products
    using w = double;     // working vectors of the recurrence (r, p, q, z, t)
    using xw = double;    // stored iterate x and Jacobi reciprocal
    using gv = double;    // SPAI factor values
    using sc = double;    // broadcast solver scalars
    static __device__ __forceinline__ acc zero() { return 0.0; }
    static __device__ __forceinline__ double total(acc a) { return a; }
    static __device__ __forceinline__ sc scal(double v) { return v; }
};
template <> struct Prec<float> {
    using acc = DF;
    using w = float2;     // double-float pair in an 8-byte slot
    using xw = float2;
    using gv = float2;
    using sc = DF;
    static __device__ __forceinline__ acc zero() { return DF{0.0f, 0.0f}; }
    static __device__ __forceinline__ double total(acc a) { return df_to_double(a); }
    static __device__ __forceinline__ sc scal(double v) { return df_from_double(v); }
};

// working value <-> accumulator form
__device__ __forceinline__ double ld_w(double v) { return v; }
__device__ __forceinline__ DF ld_w(float2 v) { return DF{v.x, v.y}; }
__device__ __forceinline__ DF ld_w(float v) { return DF{v, 0.0f}; }
__device__ __forceinline__ double to_w(double s) { return s; }
__device__ __forceinline__ float2 to_w(DF s) { return make_float2(s.hi, s.lo); }

// accumulator arithmetic
__device__ __forceinline__ double amul(double a, double b) { return a * b; }
__device__ __forceinline__ DF amul(DF a, DF b) { return df_mul(a, b); }
__device__ __forceinline__ double afma(double a, double b, double c) { return fma(a, b, c); }
__device__ __forceinline__ DF afma(DF a, DF b, DF c) { return df_add(df_mul(a, b), c); }
__device__ __forceinline__ double aneg(double a) { return -a; }
__device__ __forceinline__ DF aneg(DF a) { return df_neg(a); }

// acc += a * v
__device__ __forceinline__ void mac(double& s, double a, double v) { s = fma(a, v, s); }
__device__ __forceinline__ void mac(DF& s, float a, float v) { s = df_fma_ff(a, v, s); }
__device__ __forceinline__ void mac(DF& s, float a, float2 v) { s = df_fma_df(DF{v.x, v.y}, a, s); }
__device__ __forceinline__ void mac(DF& s, float2 g, float2 v) { s = df_add(s, df_mul(DF{g.x, g.y}, DF{v.x, v.y})); }

// stored value nearest to an accumulator
__device__ __forceinline__ double to_store(double s) { return s; }
__device__ __forceinline__ float to_store(DF s) { return df_round(s); }

// x value seen by the true-residual check (the returned precision)
__device__ __forceinline__ double x_out_of(double x) { return x; }
__device__ __forceinline__ float x_out_of(float2 x) { return __fadd_rn(x.x, x.y); }

// ----------------------------------------------------------------- gathers
template <typename T>
struct GatherVec {  // vector entry at the system precision
    const T* v;
    __device__ __forceinline__ T operator()(int c) const { return ld_nc(v + c); }
};
template <typename T>
struct GatherX {    // stored iterate, rounded to the returned precision
    const typename Prec<T>::xw* v;
    __device__ __forceinline__ T operator()(int c) const { return x_out_of(ld_nc(v + c)); }
};

__device__ __forceinline__ double acc_xor(double t, int o) { return __shfl_xor_sync(0xffffffffu, t, o); }
__device__ __forceinline__ DF acc_xor(DF t, int o) {
    return DF{__shfl_xor_sync(0xffffffffu, t.hi, o), __shfl_xor_sync(0xffffffffu, t.lo, o)};
}
__device__ __forceinline__ void acc_add(double& a, double b) { a += b; }
__device__ __forceinline__ void acc_add(DF& a, DF b) { a = df_add(a, b); }

// Rows are taken in groups of R = 32 / L consecutive rows, one warp per group
// (grid stride over groups), L = A.lanes lanes per row chosen from the row
// lengths so that a group's entries fit the warp's stage.  The warp stages
// the group's non-zeros -- values and column indices streamed with
// coalesced evict-first loads, the vector entries they address gathered
// through the read-only path -- in its own slice of shared memory (`cap`
// entries), then the L lanes of each row sum interleaved entries (one fp64
// FMA per entry for fp64 systems) and combine with log2(L) shuffle adds.
// Only __syncwarp orders the phases, so warps progress independently and
// hide each other's memory latency.  A group with more than `cap` non-zeros
// is summed straight from global memory (rows longer than LONG_ROW by the
// whole warp).
// For every row, pre(row) is called early by the row's first lane (its result
// is carried to the epilogue, so that load overlaps the gathers) and
// epi(row, sum, carried) once the sum is complete.
constexpr int STAGE_U = 4;     // entries per lane in flight while staging
constexpr int LONG_ROW = 64;   // longer rows of an unstaged group go warp-wide

// Bounds of this lane's row in group grp (empty past the last row).
__device__ __forceinline__ void row_bounds(const Mat& A, int grp, int& row, int& rlo, int& rhi) {
    const int lane = threadIdx.x & 31;
    const long long r = ((((long long)grp) << 5) + lane) >> A.lshift;
    row = (int)(r < A.n ? r : A.n);
    rlo = ld_nc(A.rp + row);
    rhi = ld_nc(A.rp + min(row + 1, A.n));
}

// Sum of the lanes of each row's segment (every lane of the segment gets it).
template <typename ACC>
__device__ __forceinline__ void segment_sum(ACC& s, int lanes) {
    for (int o = lanes >> 1; o > 0; o >>= 1) acc_add(s, acc_xor(s, o));
}

// Rows of a group that did not fit the stage, summed from global memory.
template <typename T, typename VT, class Gather>
__device__ __forceinline__ typename Prec<T>::acc unstaged_row(const Mat& A, const VT* __restrict__ av,
                                                              Gather gather, int rlo, int rhi) {
    using acc_t = typename Prec<T>::acc;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (A.lanes - 1);
    acc_t s = Prec<T>::zero();
    if (rhi - rlo <= LONG_ROW)
        for (int k = rlo + sub; k < rhi; k += A.lanes) mac(s, ld_stream(av + k), gather(ld_stream(A.ci + k)));
    unsigned longs = __ballot_sync(0xffffffffu, rhi - rlo > LONG_ROW && sub == 0);
    while (longs) {
        const int src = __ffs(longs) - 1;
        longs &= longs - 1;
        const int a0 = __shfl_sync(0xffffffffu, rlo, src);
        const int a1 = __shfl_sync(0xffffffffu, rhi, src);
        acc_t t = Prec<T>::zero();
        for (int k = a0 + lane; k < a1; k += 32) mac(t, ld_stream(av + k), gather(ld_stream(A.ci + k)));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc_add(t, acc_xor(t, o));
        if (lane == src) s = t;
    }
    return s;
}

template <typename T, typename VT, class Gather, class Pre, class Epi>
__device__ __forceinline__ void spmv_rows(const Mat& A, const VT* __restrict__ av, Gather gather, Pre pre,
                                          Epi epi, double* wsm) {
    using acc_t = typename Prec<T>::acc;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (A.lanes - 1);
    const int cap = A.cap;
    using XT = decltype(gather(0));
    char* base = reinterpret_cast<char*>(wsm + (threadIdx.x >> 5) * A.wstride);
    VT* sa = reinterpret_cast<VT*>(base);
    XT* sx = reinterpret_cast<XT*>(base + cap * sizeof(VT));
    const int ngroups = (A.n + (32 >> A.lshift) - 1) >> (5 - A.lshift);
    const int nwarps = (gridDim.x * NT) >> 5;
    for (int grp = (blockIdx.x * NT + threadIdx.x) >> 5; grp < ngroups; grp += nwarps) {
        int row, rlo, rhi;
        row_bounds(A, grp, row, rlo, rhi);
        const bool own = sub == 0 && row < A.n;
        const auto carried = own ? pre(row) : decltype(pre(0)){};
        const int k0 = __shfl_sync(0xffffffffu, rlo, 0);
        const int k1 = __shfl_sync(0xffffffffu, rhi, 31);
        const int cnt = k1 - k0;
        acc_t s = Prec<T>::zero();
        if (cnt <= cap) {
            for (int b0 = 0; b0 < cnt; b0 += 32 * STAGE_U) {
                int c[STAGE_U];
                VT a[STAGE_U];
                XT xv[STAGE_U];
#pragma unroll
                for (int j = 0; j < STAGE_U; ++j) {
                    const int e = b0 + j * 32 + lane;
                    if (e < cnt) {
                        c[j] = ld_stream(A.ci + k0 + e);
                        a[j] = ld_stream(av + k0 + e);
                    }
                }
#pragma unroll
                for (int j = 0; j < STAGE_U; ++j) {
                    const int e = b0 + j * 32 + lane;
                    if (e < cnt) xv[j] = gather(c[j]);
                }
#pragma unroll
                for (int j = 0; j < STAGE_U; ++j) {
                    const int e = b0 + j * 32 + lane;
                    if (e < cnt) { sa[e] = a[j]; sx[e] = xv[j]; }
                }
            }
            __syncwarp();
            for (int e = rlo - k0 + sub; e < rhi - k0; e += A.lanes) mac(s, sa[e], sx[e]);
            __syncwarp();
        } else {
            s = unstaged_row<T>(A, av, gather, rlo, rhi);
        }
        segment_sum(s, A.lanes);
        if (own) epi(row, s, carried);
    }
}

// Asynchronous form of spmv_rows for a plain vector gather.  A group's
// values and column indices are copied into the warp's slice with cp.async
// (L2 evict-first), then the vector entries they address are gathered into
// the slice with cp.async as well (L2 evict-last: the vector is re-read by
// every product), so a warp keeps a whole group of gathers in flight without
// holding a register for any of them.  With A.async == 2 the value/column
// copies are double-buffered: the next group's copies are issued as soon as
// the current group's gathers are, so only the gather latency is exposed per
// group; with A.async == 1 (large groups) they are single-buffered.  For
// matrices whose columns stay near the row (GASYNC false) the gathers go
// through registers instead, GATHER_U per lane in flight: they mostly hit L1,
// which the asynchronous copies serve less well.  Row bounds are loaded one
// group ahead.
// Shared memory per warp: async*cap*(sizeof(VT) + 4) + cap*sizeof(T).
constexpr int GATHER_U = 4;   // register gathers per lane in flight

template <typename VT, typename T>
__host__ __device__ constexpr size_t async_smem_per_warp(int cap, int bufs) {
    return (size_t)bufs * cap * (sizeof(VT) + sizeof(int)) + (size_t)cap * sizeof(T);
}

template <typename T, typename VT, typename XT, bool GASYNC, class Pre, class Epi>
__device__ __forceinline__ void spmv_rows_async(const Mat& A, const VT* __restrict__ av, const XT* __restrict__ v,
                                                Pre pre, Epi epi, double* wsm) {
    using acc_t = typename Prec<T>::acc;
    const int lane = threadIdx.x & 31;
    const int sub = lane & (A.lanes - 1);
    const int cap = A.cap;
    const int bufs = A.async;
    char* base = reinterpret_cast<char*>(wsm + (threadIdx.x >> 5) * A.wstride);
    VT* sv = reinterpret_cast<VT*>(base);
    int* sc = reinterpret_cast<int*>(base + bufs * cap * sizeof(VT));
    XT* sx = reinterpret_cast<XT*>(base + bufs * cap * (sizeof(VT) + sizeof(int)));
    const unsigned long long stream_pol = l2_evict_first();
    const unsigned long long keep_pol = l2_evict_last();
    const int ngroups = (A.n + (32 >> A.lshift) - 1) >> (5 - A.lshift);
    const int nwarps = (gridDim.x * NT) >> 5;
    const int g0 = (blockIdx.x * NT + threadIdx.x) >> 5;

    // copies of a group's values and columns into buffer `b` (k0, k1: its entry range)
    auto issue_vc = [&](int grp, int b, int k0, int k1) {
        if (grp < ngroups && k1 - k0 <= cap) {
            VT* dv = sv + b * cap;
            int* dc = sc + b * cap;
            for (int e = lane; e < k1 - k0; e += 32) {
                cp_async<sizeof(VT)>(dv + e, av + k0 + e, stream_pol);
                cp_async<4>(dc + e, A.ci + k0 + e, stream_pol);
            }
        }
        cp_commit();
    };

    int row, rlo, rhi, nrow, nlo, nhi;
    row_bounds(A, g0, row, rlo, rhi);
    issue_vc(g0, 0, __shfl_sync(0xffffffffu, rlo, 0), __shfl_sync(0xffffffffu, rhi, 31));
    row_bounds(A, g0 + nwarps, nrow, nlo, nhi);
    int b = 0;
    for (int grp = g0; grp < ngroups; grp += nwarps) {
        const bool own = sub == 0 && row < A.n;
        const auto carried = own ? pre(row) : decltype(pre(0)){};
        int frow, flo, fhi;
        row_bounds(A, grp + 2 * nwarps, frow, flo, fhi);
        const int k0 = __shfl_sync(0xffffffffu, rlo, 0);
        const int k1 = __shfl_sync(0xffffffffu, rhi, 31);
        const int cnt = k1 - k0;
        const int nk0 = __shfl_sync(0xffffffffu, nlo, 0);
        const int nk1 = __shfl_sync(0xffffffffu, nhi, 31);
        // With register gathers and two buffers the next group's copies can
        // start before this group's have landed.
        const bool early = bufs == 2 && !GASYNC;
        if (early) {
            issue_vc(grp + nwarps, b ^ 1, nk0, nk1);
            cp_wait<1>();  // this group's values and columns have landed
        } else {
            cp_wait<0>();
        }
        __syncwarp();
        acc_t s = Prec<T>::zero();
        if (cnt <= cap) {
            const int* cc = sc + b * cap;
            if (GASYNC) {
                for (int e = lane; e < cnt; e += 32) cp_async<sizeof(XT)>(sx + e, v + cc[e], keep_pol);
                cp_commit();
                if (bufs == 2) {
                    issue_vc(grp + nwarps, b ^ 1, nk0, nk1);
                    cp_wait<1>();  // gathers done; the next group's copies may still fly
                } else {
                    cp_wait<0>();
                }
            } else {
                for (int b0 = 0; b0 < cnt; b0 += 32 * GATHER_U) {
                    XT xv[GATHER_U];
#pragma unroll
                    for (int j = 0; j < GATHER_U; ++j) {
                        const int e = b0 + j * 32 + lane;
                        if (e < cnt) xv[j] = ld_nc(v + cc[e]);
                    }
#pragma unroll
                    for (int j = 0; j < GATHER_U; ++j) {
                        const int e = b0 + j * 32 + lane;
                        if (e < cnt) sx[e] = xv[j];
                    }
                }
            }
            __syncwarp();
            const VT* cv = sv + b * cap;
            for (int e = rlo - k0 + sub; e < rhi - k0; e += A.lanes) mac(s, cv[e], sx[e]);
        } else {
            if (bufs == 2 && !early) issue_vc(grp + nwarps, b ^ 1, nk0, nk1);
            s = unstaged_row<T>(A, av, GatherVec<XT>{v}, rlo, rhi);
        }
        segment_sum(s, A.lanes);
        __syncwarp();  // buffers free for reuse
        if (bufs == 1) issue_vc(grp + nwarps, 0, nk0, nk1);
        else b ^= 1;
        if (own) epi(row, s, carried);
        row = nrow; rlo = nlo; rhi = nhi;
        nrow = frow; nlo = flo; nhi = fhi;
    }
    cp_wait<0>();
}

// Product with a plain vector gather in one of three compiled forms (the
// host picks one per matrix, so each kernel instantiation carries a single
// path): FORM 0 register staging (spmv_rows); FORM 1 cp.async value/column
// staging with register gathers; FORM 2 cp.async staging and gathers.
template <typename T, int FORM, typename VT, typename XT, class Pre, class Epi>
__device__ __forceinline__ void spmv_vec(const Mat& A, const VT* __restrict__ av, const XT* __restrict__ v, Pre pre,
                                         Epi epi, double* wsm) {
    if constexpr (FORM == 0) spmv_rows<T, VT>(A, av, GatherVec<XT>{v}, pre, epi, wsm);
    else spmv_rows_async<T, VT, XT, FORM == 2>(A, av, v, pre, epi, wsm);
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

// ----------------------------------------------------------------- element-wise arithmetic
// acc += a * b
__device__ __forceinline__ void dot_acc(double& s, double a, double b) { s = fma(a, b, s); }
__device__ __forceinline__ void dot_acc(DF& s, float a, float b) { s = df_fma_ff(a, b, s); }
__device__ __forceinline__ void dot_acc(DF& s, float2 a, float2 b) { s = afma(ld_w(a), ld_w(b), s); }

// b - s for a row sum s
__device__ __forceinline__ double resid(double b, double s) { return b - s; }
__device__ __forceinline__ DF resid(float b, DF s) { return df_add_f(df_neg(s), b); }
__device__ __forceinline__ void sq_acc(double& t, double e) { t = fma(e, e, t); }
__device__ __forceinline__ void sq_acc(DF& t, DF e) { t = df_add(t, df_sqr(e)); }

// One element of the x / r update: x += alpha p; r -= alpha q; g += r^2;
// (Jacobi) rz += r (r dinv).  A = accumulator type, W = working value type.
template <int PC, typename A, typename W, typename XW>
__device__ __forceinline__ void update_one(A alpha, XW& x, W& r, W p, W q, XW dinv, A& g, A& rz) {
    x = to_w(afma(alpha, ld_w(p), ld_w(x)));
    const A rn = afma(aneg(alpha), ld_w(q), ld_w(r));
    r = to_w(rn);
    g = afma(rn, rn, g);
    if (PC == 1) rz = afma(rn, amul(rn, ld_w(dinv)), rz);
}

// -lambda_i x_j, rounded once
__device__ __forceinline__ double neg_prod(double l, double x) { return -l * x; }
__device__ __forceinline__ float neg_prod(float l, float x) { return df_round(two_prod(-l, x)); }

// ----------------------------------------------------------------- SpMV API
// y = A x, and dot[sys] = x.y when dot != nullptr.
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spmv(Mat A, Sys S, const T* __restrict__ av,
                                                            const T* __restrict__ x, T* __restrict__ y, double* dot) {
    using acc_t = typename Prec<T>::acc;
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; x += vo; y += vo;
    acc_t acc = Prec<T>::zero();
    spmv_vec<T, FORM, T, T>(A, av, x, [&](int i) { return x[i]; },
                   [&](int i, acc_t s, T xi) {
                       const T yi = to_store(s);
                       y[i] = yi;
                       dot_acc(acc, xi, yi);
                   },
                   dsm);
    if (dot) {
        double v[1] = {Prec<T>::total(acc)}, tot[1];
        if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) dot[sys] = tot[0];
    }
}

// ----------------------------------------------------------------- iteration
// ||b - A round(x)||^2 over this CTA's rows (the true-residual check).  Kept
// out of line: it runs only when the recursive residual has met the
// tolerance, and inlining it would cost the main product registers.
template <typename T, int FORM>
__device__ __noinline__ typename Prec<T>::acc residual_pass(const Mat& A, const T* __restrict__ av,
                                                            const typename Prec<T>::xw* __restrict__ x,
                                                            const T* __restrict__ b, double* dsm) {
    using acc_t = typename Prec<T>::acc;
    acc_t tr2 = Prec<T>::zero();
    spmv_rows<T, T>(A, av, GatherX<T>{x}, [&](int i) { return b[i]; },
                    [&](int, acc_t s, T bi) { sq_acc(tr2, resid(bi, s)); }, dsm);
    return tr2;
}

// q = A p, delta = p.q; with `check` set, ||b - A round(x)||^2 first.
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, IterMinCtas<T>::value)
    k_spmv_iter(Mat A, Sys S, const T* __restrict__ av, const typename Prec<T>::w* __restrict__ p,
                typename Prec<T>::w* __restrict__ q, const typename Prec<T>::xw* __restrict__ x,
                const T* __restrict__ b) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; p += vo; q += vo; x += vo; b += vo;
    const bool check = ld_cg(&st->check) != 0;
    acc_t tr2 = Prec<T>::zero(), delta = Prec<T>::zero();
    if (check) tr2 = residual_pass<T, FORM>(A, av, x, b, dsm);
    spmv_vec<T, FORM, T, W>(A, av, p, [&](int i) { return p[i]; },
                      [&](int i, acc_t s, W pi) {
                          const W qi = to_w(s);
                          q[i] = qi;
                          dot_acc(delta, pi, qi);
                      },
                      dsm);
    double v[2] = {Prec<T>::total(delta), Prec<T>::total(tr2)}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0) after_spmv(st, S.ctl, tot[0], check, tot[1]);
}

// Pairs of consecutive 8-byte entries (16-byte accesses) for the streaming
// kernels; used when n is even, so every system's vectors stay aligned.
template <typename X> struct XPair;
template <> struct XPair<double> { using type = double2; };
template <> struct XPair<float2> { using type = float4; };

__device__ __forceinline__ void split2(double2 v, double& a, double& b) { a = v.x; b = v.y; }
__device__ __forceinline__ void split2(float4 v, float2& a, float2& b) {
    a = make_float2(v.x, v.y);
    b = make_float2(v.z, v.w);
}
__device__ __forceinline__ double2 join2(double a, double b) { return make_double2(a, b); }
__device__ __forceinline__ float4 join2(float2 a, float2 b) { return make_float4(a.x, a.y, b.x, b.y); }

// x += alpha p; r -= alpha q; gamma = r.r; rho' = r.z (PC 0: z = r, PC 1:
// z = r / A_ii; PC 2: z comes later from the SPAI kernels).
template <typename T, int PC, bool PAIRS>
__global__ void __launch_bounds__(NT) k_update(Sys S, typename Prec<T>::xw* __restrict__ x,
                                               typename Prec<T>::w* __restrict__ r,
                                               const typename Prec<T>::w* __restrict__ p,
                                               const typename Prec<T>::w* __restrict__ q,
                                               const typename Prec<T>::xw* __restrict__ dinv) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    using XW = typename Prec<T>::xw;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[2 * NWARP];
    x += vo; r += vo; p += vo; q += vo;
    if (PC == 1) dinv += vo;
    const acc_t alpha = Prec<T>::scal(ld_cg(&st->alpha));
    acc_t g = Prec<T>::zero(), rz = Prec<T>::zero();
    if (PAIRS) {
        // two pairs per thread per trip, all loads issued before any use
        using P2 = typename XPair<W>::type;
        using X2 = typename XPair<XW>::type;
        const int n2 = S.n >> 1;
        const int stride = gridDim.x * NT;
        for (int i0 = blockIdx.x * NT + threadIdx.x; i0 < n2; i0 += 2 * stride) {
            P2 p2[2], q2[2], r2[2];
            X2 x2[2], d2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    p2[u] = ld_stream(reinterpret_cast<const P2*>(p) + i);
                    q2[u] = ld_stream(reinterpret_cast<const P2*>(q) + i);
                    x2[u] = reinterpret_cast<const X2*>(x)[i];
                    r2[u] = reinterpret_cast<const P2*>(r)[i];
                    if (PC == 1) d2[u] = ld_stream(reinterpret_cast<const X2*>(dinv) + i);
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    XW xa, xb, da{}, db{};
                    W pa, pb, qa, qb, ra, rb;
                    split2(x2[u], xa, xb);
                    split2(p2[u], pa, pb);
                    split2(q2[u], qa, qb);
                    split2(r2[u], ra, rb);
                    if (PC == 1) split2(d2[u], da, db);
                    update_one<PC>(alpha, xa, ra, pa, qa, da, g, rz);
                    update_one<PC>(alpha, xb, rb, pb, qb, db, g, rz);
                    reinterpret_cast<X2*>(x)[i] = join2(xa, xb);
                    reinterpret_cast<P2*>(r)[i] = join2(ra, rb);
                }
            }
        }
    } else {
        for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
            XW xi = x[i];
            W ri = r[i];
            update_one<PC>(alpha, xi, ri, ld_stream(p + i), ld_stream(q + i), PC == 1 ? dinv[i] : XW{}, g, rz);
            x[i] = xi;
            r[i] = ri;
        }
    }
    double v[2] = {Prec<T>::total(g), Prec<T>::total(rz)}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0)
        after_update(st, S.ctl, tot[0], PC != 2, PC == 0 ? tot[0] : tot[1]);
}

// p = z + beta p   (INIT: p = z)
template <int PC, bool INIT, typename A, typename W, typename XW>
__device__ __forceinline__ W pnew(A beta, W p, W r, XW dinv, W z) {
    A zi;
    if (PC == 0) zi = ld_w(r);
    else if (PC == 1) zi = amul(ld_w(r), ld_w(dinv));
    else zi = ld_w(z);
    return INIT ? to_w(zi) : to_w(afma(beta, ld_w(p), zi));
}

template <typename T, int PC, bool INIT, bool PAIRS>
__global__ void __launch_bounds__(NT) k_pupdate(Sys S, typename Prec<T>::w* __restrict__ p,
                                                const typename Prec<T>::w* __restrict__ r,
                                                const typename Prec<T>::w* __restrict__ z,
                                                const typename Prec<T>::xw* __restrict__ dinv) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    using XW = typename Prec<T>::xw;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    p += vo; r += vo;
    if (PC == 1) dinv += vo;
    if (PC == 2) z += vo;
    const acc_t beta = Prec<T>::scal(INIT ? 0.0 : ld_cg(&st->beta));
    if (PAIRS) {
        using P2 = typename XPair<W>::type;
        using X2 = typename XPair<XW>::type;
        const int n2 = S.n >> 1;
        const int stride = gridDim.x * NT;
        for (int i0 = blockIdx.x * NT + threadIdx.x; i0 < n2; i0 += 2 * stride) {
            P2 r2[2], p2[2], z2[2];
            X2 d2[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    r2[u] = ld_stream(reinterpret_cast<const P2*>(r) + i);
                    p2[u] = INIT ? P2{} : reinterpret_cast<const P2*>(p)[i];
                    if (PC == 1) d2[u] = ld_stream(reinterpret_cast<const X2*>(dinv) + i);
                    z2[u] = PC == 2 ? ld_stream(reinterpret_cast<const P2*>(z) + i) : P2{};
                }
            }
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    XW da{}, db{};
                    W ra, rb, pa, pb, za, zb;
                    split2(r2[u], ra, rb);
                    split2(p2[u], pa, pb);
                    split2(z2[u], za, zb);
                    if (PC == 1) split2(d2[u], da, db);
                    reinterpret_cast<P2*>(p)[i] =
                        join2(pnew<PC, INIT>(beta, pa, ra, da, za), pnew<PC, INIT>(beta, pb, rb, db, zb));
                }
            }
        }
    } else {
        for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT)
            p[i] = pnew<PC, INIT>(beta, INIT ? W{} : p[i], r[i], PC == 1 ? dinv[i] : XW{}, PC == 2 ? z[i] : W{});
    }
}

// SPAI, first product: t = G^T r (explicit transposed CSR of G; G values
// are per system, [batch][nnz(G)]).
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spai_t(Mat GT, Sys S, long long nnzg,
                                                              const typename Prec<T>::gv* __restrict__ gtv,
                                                              const typename Prec<T>::w* __restrict__ r,
                                                              typename Prec<T>::w* __restrict__ t) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    gtv += (size_t)sys * nnzg; r += vo; t += vo;
    spmv_vec<T, FORM, typename Prec<T>::gv, W>(GT, gtv, r, [](int) { return W{}; },
                                         [&](int i, acc_t s, W) { t[i] = to_w(s); }, dsm);
}

// SPAI, second product: z = G t + eps r, rho' = r.z -> beta (or rho at set-up).
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS) k_spai_z(Mat G, Sys S, long long nnzg,
                                                              const typename Prec<T>::gv* __restrict__ gv,
                                                              const typename Prec<T>::w* __restrict__ t,
                                                              const typename Prec<T>::w* __restrict__ r,
                                                              typename Prec<T>::w* __restrict__ z, double eps) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    gv += (size_t)sys * nnzg; t += vo; r += vo; z += vo;
    const acc_t e = Prec<T>::scal(eps);
    acc_t rz = Prec<T>::zero();
    spmv_vec<T, FORM, typename Prec<T>::gv, W>(G, gv, t, [&](int i) { return r[i]; },
                                         [&](int i, acc_t s, W ri) {
                                             const W zi = to_w(afma(e, ld_w(ri), s));
                                             z[i] = zi;
                                             dot_acc(rz, ri, zi);
                                         },
                                         dsm);
    double v[1] = {Prec<T>::total(rz)}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) new_direction(st, S.ctl, tot[0]);
}

// ----------------------------------------------------------------- set-up / final
// x = 0, r = b, b copied into the workspace, bb = b.b.
template <typename T>
__global__ void __launch_bounds__(NT) k_init(Sys S, const T* __restrict__ b_user, T* __restrict__ bw,
                                             typename Prec<T>::xw* __restrict__ x, typename Prec<T>::w* __restrict__ r,
                                             double tol, int max_iter) {
    SYS_PROLOGUE
    __shared__ double red[2 * NWARP];
    b_user += vo; bw += vo; x += vo; r += vo;
    typename Prec<T>::acc bb = Prec<T>::zero();
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
        const T bi = b_user[i];
        bw[i] = bi;
        r[i] = to_w(ld_w(bi));
        x[i] = typename Prec<T>::xw{};
        dot_acc(bb, bi, bi);
    }
    double v[1] = {Prec<T>::total(bb)}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0)
        start_state(st, S.ctl, tot[0], tot[0], tol, max_iter);
}

__device__ __forceinline__ double x_from(double v) { return v; }
__device__ __forceinline__ float2 x_from(float v) { return make_float2(v, 0.0f); }

// With an initial guess: x = x0, r = b - A x0, bb = b.b, gamma = r.r.
template <typename T>
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS)
    k_init_x0(Mat A, Sys S, const T* __restrict__ av, const T* __restrict__ b_user, const T* __restrict__ x0,
              T* __restrict__ bw, typename Prec<T>::xw* __restrict__ x, typename Prec<T>::w* __restrict__ r,
              double tol, int max_iter) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; b_user += vo; x0 += vo; bw += vo; x += vo; r += vo;
    acc_t bb = Prec<T>::zero(), g = Prec<T>::zero();
    spmv_rows<T, T>(A, av, GatherVec<T>{x0}, [&](int i) { return b_user[i]; },
                    [&](int i, acc_t s, T bi) {
                        bw[i] = bi;
                        x[i] = x_from(x0[i]);
                        const acc_t ri = resid(bi, s);
                        r[i] = to_w(ri);
                        dot_acc(bb, bi, bi);
                        g = afma(ri, ri, g);
                    },
                    dsm);
    double v[2] = {Prec<T>::total(bb), Prec<T>::total(g)}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0)
        start_state(st, S.ctl, tot[0], tot[1], tol, max_iter);
}

// First direction for PC 0 / 1: p = z, rho = r.z.
template <typename T, int PC>
__global__ void __launch_bounds__(NT) k_init_dir(Sys S, typename Prec<T>::w* __restrict__ p,
                                                 const typename Prec<T>::w* __restrict__ r,
                                                 const typename Prec<T>::xw* __restrict__ dinv) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[2 * NWARP];
    p += vo; r += vo;
    if (PC == 1) dinv += vo;
    acc_t rz = Prec<T>::zero();
    for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
        const W ri = r[i];
        const acc_t zi = PC == 1 ? amul(ld_w(ri), ld_w(dinv[i])) : ld_w(ri);
        p[i] = to_w(zi);
        rz = afma(ld_w(ri), zi, rz);
    }
    double v[1] = {Prec<T>::total(rz)}, tot[1];
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
__global__ void __launch_bounds__(NT, SPMV_MIN_CTAS)
    k_final(Mat A, Sys S, const T* __restrict__ av, const typename Prec<T>::xw* __restrict__ x,
            const T* __restrict__ bw, T* __restrict__ x_out, Stat* out) {
    using acc_t = typename Prec<T>::acc;
    SYS_PROLOGUE
    extern __shared__ double dsm[];
    __shared__ double red[2 * NWARP];
    av += ao; x += vo; bw += vo; x_out += vo;
    const bool zero_b = ld_cg(&st->bb) == 0.0;
    acc_t tr2 = Prec<T>::zero();
    spmv_rows<T, T>(A, av, GatherX<T>{x}, [&](int i) { return bw[i]; },
                    [&](int i, acc_t s, T bi) {
                        x_out[i] = zero_b ? T(0) : x_out_of(x[i]);
                        sq_acc(tr2, resid(bi, s));
                    },
                    dsm);
    double v[1] = {Prec<T>::total(tr2)}, tot[1];
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

// dL/dA_k = -lambda_row(k) * x_col(k) over the pattern.  One warp per row
// group (as in the SpMV): the row of each of the group's entries is recorded in the
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
    const int sub = lane & (A.lanes - 1);
    const int ngroups = (A.n + (32 >> A.lshift) - 1) >> (5 - A.lshift);
    const int nwarps = (gridDim.x * NT) >> 5;
    for (int grp = (blockIdx.x * NT + threadIdx.x) >> 5; grp < ngroups; grp += nwarps) {
        int row, rlo, rhi;
        row_bounds(A, grp, row, rlo, rhi);
        const int k0 = __shfl_sync(0xffffffffu, rlo, 0);
        const int k1 = __shfl_sync(0xffffffffu, rhi, 31);
        const int cnt_ = k1 - k0;
        if (cnt_ <= A.cap) {
            for (int e = rlo - k0 + sub; e < rhi - k0; e += A.lanes) srow[e] = row;
            __syncwarp();
            for (int e = lane; e < cnt_; e += 32) {
                const int c = ld_stream(A.ci + k0 + e);
                __stcs(dA + k0 + e, neg_prod(ld_nc(lam + srow[e]), ld_nc(x + c)));
            }
            __syncwarp();
        } else if (row < A.n) {
            const T li = lam[row];
            for (int k = rlo + sub; k < rhi; k += A.lanes) __stcs(dA + k, neg_prod(li, ld_nc(x + ld_stream(A.ci + k))));
        }
    }
}

}  // namespace sla
