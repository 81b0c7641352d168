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
    long long nnz;    // stored entries of the pattern
    int ccap;         // warp pipeline: entries per stage (multiple of 4)
    int stages;       // warp pipeline: ring stages
    int* err;         // device error bits (Ctrl::err; Ctrl::diag follows at err + 2)
    int direct;       // 1: the layout's kernels run the direct form (no shared-memory staging)
    int bal;          // 1: staged groups (one lane per row, cp.async forms) are summed with the
                      //    entries split evenly over the lanes (balanced_group_sum)
    int swin;         // 1: sliced rows sorted within windows of SLICE_WIN rows, run a warp per
                      //    window with the epilogue in row order (spmv_sliced_win)
    // Sliced form (FORM 6): the rows in slices of 32, each slice stored
    // column by column (entry j of the slice's 32 rows side by side), padded
    // to the slice's longest row.
    const int* sptr;     // [nslices + 1] first entry of every slice (multiples of 32)
    const int* sperm;    // [nslices * 32] row held by every slot (>= n: empty), or nullptr (slot = row)
    const int* scol;     // [sptr[nslices]] column of every sliced entry (padding: a valid column)
    int nslices;
    long long vstride;   // per-system stride of the sliced values
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

// Sums of products of fp32 systems are accumulated compensated (the Dot2
// scheme of Ogita, Rump and Oishi, "Accurate sum and dot product", 2005):
// the pair holds a running fp32 sum and a running fp32 sum of its rounding
// errors (each exact by two-sum) and of the products' low parts, and is
// normalised (acc_norm) once, when the sum is complete -- about 10 fp32
// operations per term instead of a full double-float addition, with an
// accuracy close to that of a sum carried in twice fp32's precision.
__device__ __forceinline__ void acc_push(DF& s, DF p) {
    const DF t = two_sum(s.hi, p.hi);
    s.hi = t.hi;
    s.lo = __fadd_rn(s.lo, __fadd_rn(t.lo, p.lo));
}
__device__ __forceinline__ void acc_norm(double&) {}
__device__ __forceinline__ void acc_norm(DF& s) { s = two_sum(s.hi, s.lo); }
// a * b for double-float a, b: the high parts' product exact, the cross
// terms rounded into its low part (not normalised)
__device__ __forceinline__ DF dprod(DF a, DF b) {
    DF p = two_prod(a.hi, b.hi);
    p.lo = __fmaf_rn(a.hi, b.lo, p.lo);
    p.lo = __fmaf_rn(a.lo, b.hi, p.lo);
    return p;
}
// s += a * b into an accumulator
__device__ __forceinline__ void acc_fma(double& s, double a, double b) { s = fma(a, b, s); }
__device__ __forceinline__ void acc_fma(DF& s, DF a, DF b) { acc_push(s, dprod(a, b)); }

// acc += a * v
__device__ __forceinline__ void mac(double& s, double a, double v) { s = fma(a, v, s); }
__device__ __forceinline__ void mac(DF& s, float a, float v) { acc_push(s, two_prod(a, v)); }
__device__ __forceinline__ void mac(DF& s, float a, float2 v) {
    DF p = two_prod(a, v.x);
    p.lo = __fmaf_rn(a, v.y, p.lo);
    acc_push(s, p);
}
__device__ __forceinline__ void mac(DF& s, float2 g, float2 v) { acc_push(s, dprod(DF{g.x, g.y}, DF{v.x, v.y})); }

// stored value nearest to an accumulator
__device__ __forceinline__ double to_store(double s) { return s; }
__device__ __forceinline__ float to_store(DF s) { return df_round(s); }

// x value seen by the true-residual check (the returned precision)
__device__ __forceinline__ double x_out_of(double x) { return x; }
__device__ __forceinline__ float x_out_of(float2 x) { return __fadd_rn(x.x, x.y); }

// ----------------------------------------------------------------- gathers
// COH: the vector is rewritten during the kernel (the fused iteration), so
// gathers use plain loads instead of the read-only path.
template <typename T, bool COH = false>
__device__ __forceinline__ T ld_gather(const T* p) {
    if constexpr (COH) return ld_coh(p);
    else if constexpr (SLA_L2_KEEP) return ld_pol<true>(p, pol_keep());
    else return ld_nc(p);
}
template <typename T, bool COH = false>
struct GatherVec {  // vector entry at the system precision
    const T* v;
    __device__ __forceinline__ T operator()(int c) const { return ld_gather<T, COH>(v + c); }
};
template <typename T, bool COH = false>
struct GatherX {    // stored iterate, rounded to the returned precision
    const typename Prec<T>::xw* v;
    __device__ __forceinline__ T operator()(int c) const {
        return x_out_of(ld_gather<typename Prec<T>::xw, COH>(v + c));
    }
};

__device__ __forceinline__ double acc_xor(double t, int o) { return __shfl_xor_sync(0xffffffffu, t, o); }
__device__ __forceinline__ DF acc_xor(DF t, int o) {
    return DF{__shfl_xor_sync(0xffffffffu, t.hi, o), __shfl_xor_sync(0xffffffffu, t.lo, o)};
}
__device__ __forceinline__ double acc_from(double t, int src) { return __shfl_sync(0xffffffffu, t, src); }
__device__ __forceinline__ DF acc_from(DF t, int src) {
    return DF{__shfl_sync(0xffffffffu, t.hi, src), __shfl_sync(0xffffffffu, t.lo, src)};
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
    acc_norm(s);
    unsigned longs = __ballot_sync(0xffffffffu, rhi - rlo > LONG_ROW && sub == 0);
    while (longs) {
        const int src = __ffs(longs) - 1;
        longs &= longs - 1;
        const int a0 = __shfl_sync(0xffffffffu, rlo, src);
        const int a1 = __shfl_sync(0xffffffffu, rhi, src);
        acc_t t = Prec<T>::zero();
        for (int k = a0 + lane; k < a1; k += 32) mac(t, ld_stream(av + k), gather(ld_stream(A.ci + k)));
        acc_norm(t);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) acc_add(t, acc_xor(t, o));
        if (lane == src) s = t;
    }
    return s;
}

// Direct form: one thread per row (grid stride over rows).  The thread
// loads its row's values and column indices (evict-first; the warp's rows
// are consecutive, so the lines its loads touch are shared through L1),
// gathers the vector entries they address through the read-only path and
// sums them (one fp64 FMA per entry for fp64 systems).  No shared memory:
// the kernels carrying it are built for high occupancy (many resident warps
// per SM hide the load latency), which on B300 beats staging a warp's rows
// for patterns with short rows.
template <typename T, typename VT, class Gather, class Pre, class Epi>
__device__ __forceinline__ void spmv_direct(const Mat& A, const VT* __restrict__ av, Gather gather, Pre pre,
                                            Epi epi) {
    using acc_t = typename Prec<T>::acc;
    const int stride = gridDim.x * NT;
    for (int row = blockIdx.x * NT + threadIdx.x; row < A.n; row += stride) {
        const int lo = ld_nc(A.rp + row), hi = ld_nc(A.rp + row + 1);
        const auto carried = pre(row);
        acc_t s = Prec<T>::zero();
        for (int k = lo; k < hi; ++k) mac(s, ld_mat(av + k), gather(ld_mat(A.ci + k)));
        acc_norm(s);
        epi(row, s, carried);
    }
}

// Sliced form: one warp per slice of 32 rows (grid stride over slices;
// the 8 warps of a CTA take 8 consecutive slices).  Lane l owns the slice's
// l-th row: its entry j sits at sptr[slice] + 32 j + l, so each value and
// column load of the warp reads 32 consecutive entries (coalesced), and
// every lane of a slice runs the same trip count (the slice's width).  The
// entries go in batches of SLICE_U -- all loads of a batch issued before its
// gathers -- then one at a time.  Padding entries hold the value 0 and a
// valid column.  Rows are summed in stored order (one fp64 FMA per entry
// for fp64 systems).  No shared memory (but see spmv_sliced_win).
// Measured on B300 inside the running iteration (kNN Laplacian; 3D and 2D
// grids): plain batches beat batches predicated on the width, batches of 3
// or 4 software-pipelined (the next batch's values and columns loaded
// before this batch's FMAs), and 3 resident CTAs per SM (kNN product 191 us
// against 204-282 us).  With the window epilogue and both SPAI factors
// sliced (kNN SPAI-PCG, CG iterations/s): batches of 2 / 4 / 5 / 6 / 7 / 8
// 2.01k / 2.04k / 2.12k / 2.13k / 2.08k / 2.09k (the A product 198 / 186 /
// 179 / 179 / 180 / 181 us).
#ifndef SLA_SLICE_U
#define SLA_SLICE_U 6
#endif
#ifndef SLA_SLICE_REST
#define SLA_SLICE_REST 1   // the last w % U entries of a slot as one batch (0: one at a time)
#endif
constexpr int SLICE_U = SLA_SLICE_U;

// Batch of the short-row sliced form (7): measured on the 3D 7-point
// product inside the running iteration, 7 (49.6 us) beat 2, 4, 6 and 8
// (50.0, 51.3, 51.7, 50.8 us).
#ifndef SLA_SLICE_U_SHORT
#define SLA_SLICE_U_SHORT 7
#endif
// K entries j .. j + K - 1 of a slot: all loads of values and columns
// issued before the gathers, then the FMAs in order.
template <int K, typename VT, typename ACC, class Gather>
__device__ __forceinline__ void slice_batch(ACC& s, const VT* v, const int* c, int j, Gather gather) {
    VT a[K];
    int cc[K];
#pragma unroll
    for (int u = 0; u < K; ++u) {
        a[u] = ld_mat(v + (j + u) * 32);
        cc[u] = ld_mat(c + (j + u) * 32);
    }
#pragma unroll
    for (int u = 0; u < K; ++u) mac(s, a[u], gather(cc[u]));
}
// The last w % U entries as one batch of their own size (R < U).
template <int R, typename VT, typename ACC, class Gather>
__device__ __forceinline__ void slice_rest(ACC& s, const VT* v, const int* c, int j, int r, Gather gather) {
    if constexpr (R > 0) {
        if (r == R) slice_batch<R>(s, v, c, j, gather);
        else slice_rest<R - 1>(s, v, c, j, r, gather);
    }
}

// Sum of this lane's slot of slice sl: batches of U entries, then the rest
// as one batch.
template <typename T, typename VT, int U, class Gather>
__device__ __forceinline__ typename Prec<T>::acc slice_sum(const Mat& A, const VT* __restrict__ sv, Gather gather,
                                                          int sl, int lane) {
    using acc_t = typename Prec<T>::acc;
    const int base = ld_nc(A.sptr + sl);
    const int w = (ld_nc(A.sptr + sl + 1) - base) >> 5;
    acc_t s = Prec<T>::zero();
    const VT* v = sv + base + lane;
    const int* c = A.scol + base + lane;
    int j = 0;
    for (; j + U <= w; j += U) slice_batch<U>(s, v, c, j, gather);
#if SLA_SLICE_REST
    slice_rest<U - 1>(s, v, c, j, w - j, gather);
#else
    for (; j < w; ++j) mac(s, ld_mat(v + j * 32), gather(ld_mat(c + j * 32)));
#endif
    acc_norm(s);
    return s;
}

template <typename T, typename VT, int U = SLICE_U, class Gather, class Pre, class Epi>
__device__ __forceinline__ void spmv_sliced(const Mat& A, const VT* __restrict__ sv, Gather gather, Pre pre,
                                            Epi epi) {
    const int lane = threadIdx.x & 31;
    const int nwarps = (gridDim.x * NT) >> 5;
    for (int sl = (blockIdx.x * NT + threadIdx.x) >> 5; sl < A.nslices; sl += nwarps) {
        const int slot = (sl << 5) + lane;
        const int row = A.sperm ? ld_nc(A.sperm + slot) : slot;
        const bool live = row < A.n;
        const auto carried = live ? pre(row) : decltype(pre(0)){};
        const auto s = slice_sum<T, VT, U>(A, sv, gather, sl, lane);
        if (live) epi(row, s, carried);
    }
}

// Sliced form with rows sorted within windows of SLICE_WIN rows (Mat::swin):
// a warp takes whole windows (SLICE_WIN / 32 slices), parks the window's
// slot sums in its shared-memory slice at their rows' places, and then runs
// the epilogue for the window's rows in row order, so the epilogue's vector
// accesses are coalesced instead of following the slot order.
// Shared memory per warp: SLICE_WIN accumulators (wsm, A.wstride doubles).
constexpr int SLICE_WIN = 256;
template <typename T, typename VT, int U = SLICE_U, class Gather, class Pre, class Epi>
__device__ __forceinline__ void spmv_sliced_win(const Mat& A, const VT* __restrict__ sv, Gather gather, Pre pre,
                                                Epi epi, double* wsm) {
    using acc_t = typename Prec<T>::acc;
    using C = decltype(pre(0));
    constexpr int SPW = SLICE_WIN / 32;   // slices per window
    const int lane = threadIdx.x & 31;
    acc_t* sums = reinterpret_cast<acc_t*>(wsm + (threadIdx.x >> 5) * A.wstride);
    const int nwin = (A.nslices + SPW - 1) / SPW;
    const int nwarps = (gridDim.x * NT) >> 5;
    for (int win = (blockIdx.x * NT + threadIdx.x) >> 5; win < nwin; win += nwarps) {
        const int row0 = win * SLICE_WIN;
        const int sl1 = min((win + 1) * SPW, A.nslices);
        for (int sl = win * SPW; sl < sl1; ++sl) {
            const int row = ld_nc(A.sperm + (sl << 5) + lane);
            const auto s = slice_sum<T, VT, U>(A, sv, gather, sl, lane);
            if (row < A.n) sums[row - row0] = s;
        }
        __syncwarp();
        C carried[SPW];
#pragma unroll
        for (int k = 0; k < SPW; ++k) {
            const int row = row0 + k * 32 + lane;
            carried[k] = row < A.n ? pre(row) : C{};
        }
#pragma unroll
        for (int k = 0; k < SPW; ++k) {
            const int row = row0 + k * 32 + lane;
            if (row < A.n) epi(row, sums[k * 32 + lane], carried[k]);
        }
        __syncwarp();   // the sums are read before the next window writes them
    }
}

// Offset of system `sys`'s values: the CSR values ([batch][nnz]) or, for
// the sliced forms, the sliced values ([batch][vstride]).
template <int FORM>
__device__ __forceinline__ size_t val_offset(const Mat& A, int sys, long long nnz) {
    return (size_t)sys * (size_t)(sliced_form(FORM) ? A.vstride : nnz);
}

template <typename T, typename VT, class Gather, class Pre, class Epi>
__device__ __forceinline__ void spmv_rows(const Mat& A, const VT* __restrict__ av, Gather gather, Pre pre,
                                          Epi epi, double* wsm) {
    using acc_t = typename Prec<T>::acc;
    if (A.direct) {   // a direct-form layout gives its kernels no shared memory
        spmv_direct<T, VT>(A, av, gather, pre, epi);
        return;
    }
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
        acc_norm(s);
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
#ifndef SLA_GATHER_U
#define SLA_GATHER_U 8
#endif
constexpr int GATHER_U = SLA_GATHER_U;   // register gathers per lane in flight

template <typename VT, typename T>
__host__ __device__ constexpr size_t async_smem_per_warp(int cap, int bufs) {
    return (size_t)bufs * cap * (sizeof(VT) + sizeof(int)) + (size_t)cap * sizeof(T);
}

// Balanced sum of a staged group of 32 rows (one lane per row; Mat::bal).
// A lane-per-row walk costs the warp as many fp64 steps as the group's
// longest row, because a warp-wide fp64 instruction holds the fp64 pipe for
// the whole warp however many lanes are active.  Here the group's cnt
// staged entries are cut into 32 runs of C = ceil(cnt / 32) entries
// (rounded up to odd, so that the lanes' shared-memory reads fall in
// distinct banks), run l summed by lane l: the warp's fp64 steps are C plus
// the rounds that join the pieces of rows cut by run boundaries.  A piece
// that begins a row is left in the staged vector slot of the row's first
// entry (already consumed by the lane that wrote it); a lane's first piece,
// when it continues a row begun in an earlier run, is its carry, passed to
// the row's lane by shuffles.  A row's sum is its first piece plus the
// carries of the lanes whose runs start inside it, in lane order: a fixed
// order, so the result is reproducible.
// rend: 32 ints of scratch (the group's staged column indices, whose
// gathers have all been issued); lo, hi: this lane's row relative to the
// group's first entry.
template <typename T, typename VT, typename XT>
__device__ __forceinline__ typename Prec<T>::acc balanced_group_sum(const VT* __restrict__ cv, XT* sx, int* rend,
                                                                   int cnt, int lo, int hi) {
    using acc_t = typename Prec<T>::acc;
    const int lane = threadIdx.x & 31;
    rend[lane] = hi;
    __syncwarp();
    const int C = ((cnt + 31) >> 5) | 1;
    int e = lane * C;
    const int e1 = min(e + C, cnt);
    acc_t s = Prec<T>::zero(), carry = Prec<T>::zero();
    if (e < e1) {
        int i = 0;   // row holding entry e: the number of rows that end at or before e
#pragma unroll
        for (int st = 16; st >= 1; st >>= 1)
            if (rend[i + st - 1] <= e) i += st;
        bool cont = e > (i > 0 ? rend[i - 1] : 0);   // the run starts inside row i
        int head = e;                                // first entry of the current piece
        int end = rend[i];
        for (; e < e1; ++e) {
            if (e == end) {
                acc_norm(s);
                if (cont) carry = s;
                else sx[head] = to_w(s);
                s = Prec<T>::zero();
                cont = false;
                head = e;
                do end = rend[++i]; while (end == e);   // past empty rows
            }
            mac(s, cv[e], sx[e]);
        }
        acc_norm(s);
        if (cont) carry = s;
        else sx[head] = to_w(s);
    }
    __syncwarp();
    acc_t tot = hi > lo ? acc_t(ld_w(sx[lo])) : Prec<T>::zero();
    const int first = lo / C + 1;   // first lane whose run starts inside this row
    const int joins = hi > lo ? (hi - 1) / C - lo / C : 0;
    const int rounds = __reduce_max_sync(0xffffffffu, joins);
    for (int k = 0; k < rounds; ++k) {
        const acc_t t = acc_from(carry, min(first + k, 31));
        if (k < joins) acc_add(tot, t);
    }
    return tot;
}

template <typename T, typename VT, typename XT, bool GASYNC, bool COH, class Pre, class Epi>
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
                        if (e < cnt) xv[j] = ld_gather<XT, COH>(v + cc[e]);
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
            // the balanced sum keeps a row's first piece in a staged vector slot
            constexpr bool slot_fits = std::is_same<XT, decltype(to_w(acc_t{}))>::value;
            if (slot_fits && A.bal) {
                if constexpr (slot_fits) s = balanced_group_sum<T>(cv, sx, sc + b * cap, cnt, rlo - k0, rhi - k0);
            } else {
                for (int e = rlo - k0 + sub; e < rhi - k0; e += A.lanes) mac(s, cv[e], sx[e]);
            }
        } else {
            if (bufs == 2 && !early) issue_vc(grp + nwarps, b ^ 1, nk0, nk1);
            s = unstaged_row<T>(A, av, GatherVec<XT, COH>{v}, rlo, rhi);
        }
        acc_norm(s);
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

// Warp pipeline.  As in spmv_rows, a warp takes groups of 32 consecutive
// rows (one row per lane; grid stride over groups), but it moves each
// group's values and column indices into its own ring of A.stages
// shared-memory stages with two bulk asynchronous copies (cp.async.bulk,
// L2 evict-first), whose completion is counted in bytes on the stage's
// mbarrier, issued by lane 0 stages - 1 groups ahead of the group being
// summed.  Once a group's columns have landed the lanes gather the vector
// entries they address into one of two gather buffers with cp.async (L2
// evict-last), one group ahead of the arithmetic.  So while a warp sums
// group t, the gathers of group t+1 and the copies of groups t+2 ..
// t+stages-1 are in flight, and no warp ever waits for another.  Each lane
// then sums its row from shared memory (one fp64 FMA per entry for fp64
// systems).  Copies run from the group's first entry rounded down to a
// multiple of 4 to its end rounded up (bulk copies move 16-byte units
// between 16-byte aligned addresses); entries past the pattern's last
// multiple of 4 are copied with plain loads.  The host uses this form only
// when every group fits a stage (A.ccap entries) and the arrays are 16-byte
// aligned.
// Shared memory per warp (A.wstride doubles): PipeHdr, stages * ccap values,
// stages * ccap columns, 2 * ccap gathered entries.
constexpr int MAX_STAGES = 4;
struct PipeHdr {
    unsigned long long bar[MAX_STAGES];   // one mbarrier per stage
    int k0[MAX_STAGES];                   // first staged entry (multiple of 4)
    int cnt[MAX_STAGES];                  // staged entries
};

template <typename VT, typename XT>
__host__ __device__ constexpr size_t pipe_smem_per_warp(int ccap, int stages) {
    return sizeof(PipeHdr) + (size_t)stages * ccap * (sizeof(VT) + sizeof(int)) + 2 * (size_t)ccap * sizeof(XT);
}

template <typename T, typename VT, typename XT, class Pre, class Epi>
__device__ __forceinline__ void spmv_pipe(const Mat& A, const VT* __restrict__ av, const XT* __restrict__ v,
                                          Pre pre, Epi epi, double* dsm) {
    using acc_t = typename Prec<T>::acc;
    using car_t = decltype(pre(0));
    const int S = A.stages, cap = A.ccap;
    const int lane = threadIdx.x & 31;
    char* base = reinterpret_cast<char*>(dsm + (threadIdx.x >> 5) * A.wstride);
    PipeHdr* hd = reinterpret_cast<PipeHdr*>(base);
    VT* sv = reinterpret_cast<VT*>(base + sizeof(PipeHdr));
    int* sc = reinterpret_cast<int*>(sv + (size_t)S * cap);
    XT* sx = reinterpret_cast<XT*>(sc + (size_t)S * cap);
    const int ngroups = (A.n + 31) >> 5;
    const int g0 = (blockIdx.x * NT + threadIdx.x) >> 5;
    const int gstep = (gridDim.x * NT) >> 5;
    const int m = g0 < ngroups ? (ngroups - 1 - g0) / gstep + 1 : 0;   // groups of this warp
    __syncwarp();   // the warp's slice may still be in use by an earlier pass
    if (m == 0) return;
    const long long nnz4 = A.nnz & ~3LL;

    // Lane 0: copies of the warp's j-th group into stage j % S, given the
    // group's entry range [e0, e1).
    auto issue = [&](int j, int e0, int e1) {
        const int st = j % S;
        const long long k0 = (long long)e0 & ~3LL;
        const long long k1 = ((long long)e1 + 3) & ~3LL;
        long long kb = k1 < nnz4 ? k1 : (nnz4 > k0 ? nnz4 : k0);   // end of the bulk part
        long long ke = k1 < A.nnz ? k1 : A.nnz;                      // end of the staged range
        if (ke - k0 > cap) {   // never expected: the host sized the stages for every group
            atomicOr(A.err, ERR_STAGE);
            kb = ke = k0;
        }
        hd->k0[st] = (int)k0;
        hd->cnt[st] = (int)(ke - k0);
        VT* dv = sv + (size_t)st * cap;
        int* dc = sc + (size_t)st * cap;
        for (long long k = kb; k < ke; ++k) {   // ragged end of the pattern
            dv[k - k0] = av[k];
            dc[k - k0] = A.ci[k];
        }
        const unsigned nb = (unsigned)(kb - k0);
        fence_proxy_async();
        mbar_arrive_expect(&hd->bar[st], nb * (unsigned)(sizeof(VT) + sizeof(int)));
        if (nb) {
            const unsigned long long pol = l2_evict_first();
            bulk_copy(dv, av + k0, nb * (unsigned)sizeof(VT), &hd->bar[st], pol);
            bulk_copy(dc, A.ci + k0, nb * (unsigned)sizeof(int), &hd->bar[st], pol);
        }
    };
    // Entry range of the warp's j-th group (lane 0).
    auto bounds = [&](int j, int& e0, int& e1) {
        const int r0 = (g0 + j * gstep) << 5;
        const int r1 = r0 + 32 < A.n ? r0 + 32 : A.n;
        e0 = ld_nc(A.rp + r0);
        e1 = ld_nc(A.rp + r1);
    };

    int ne0 = 0, ne1 = 0;   // lane 0: range of the next group to issue
    if (lane == 0) {
        for (int st = 0; st < S; ++st) mbar_init(&hd->bar[st], 1);
        fence_barrier_init();
        const int pre_n = S < m ? S : m;
        for (int j = 0; j < pre_n; ++j) {
            int e0, e1;
            bounds(j, e0, e1);
            issue(j, e0, e1);
        }
        if (S < m) bounds(S, ne0, ne1);
    }
    __syncwarp();
    const unsigned long long keep = l2_evict_last();
    auto gather = [&](int st, int gb) {
        const int* cc = sc + (size_t)st * cap;
        XT* dx = sx + (size_t)gb * cap;
        const int cnt = hd->cnt[st];
        for (int e = lane; e < cnt; e += 32) cp_async<sizeof(XT)>(dx + e, v + cc[e], keep);
    };
    // this lane's row of group 0
    int row = (g0 << 5) + lane, rlo = 0, rhi = 0;
    car_t car{};
    if (row < A.n) {
        rlo = ld_nc(A.rp + row);
        rhi = ld_nc(A.rp + row + 1);
        car = pre(row);
    }
    bool ok = mbar_wait(&hd->bar[0], 0);
    if (ok) gather(0, 0);
    cp_commit();
    for (int i = 0; i < m; ++i) {
        const int st = i % S, gb = i & 1;
        int nrow = row + (gstep << 5), nlo = 0, nhi = 0;
        car_t ncar{};
        if (i + 1 < m) {
            if (nrow < A.n) {
                nlo = ld_nc(A.rp + nrow);
                nhi = ld_nc(A.rp + nrow + 1);
                ncar = pre(nrow);
            }
            const int ns = (i + 1) % S;
            const bool w = mbar_wait(&hd->bar[ns], (unsigned)(((i + 1) / S) & 1));
            ok = ok && w;
            if (ok) gather(ns, gb ^ 1);
            cp_commit();
            cp_wait<1>();   // this group's gathers (the next group's may fly)
        } else {
            cp_wait<0>();
        }
        if (__any_sync(0xffffffffu, !ok)) {
            // A copy never landed: record it, let copies still in flight
            // settle (bounded), and leave the stages alone.
            if (lane == 0) {
                atomicOr(A.err, ERR_WAIT);
                note_wait(A.err + 2, -1 - (int)blockIdx.x, i, m, (int)(threadIdx.x >> 5));
                bool settled = true;
                for (int j = i; j < i + S && j < m; ++j)
                    settled = mbar_wait(&hd->bar[j % S], (unsigned)((j / S) & 1)) && settled;
                if (settled)
                    for (int st = 0; st < S; ++st) mbar_inval(&hd->bar[st]);
            }
            cp_wait<0>();
            __syncwarp();
            return;
        }
        __syncwarp();   // every lane's gathers of this group have landed
        acc_t s = Prec<T>::zero();
        if (row < A.n) {
            const int k0 = hd->k0[st];
            const VT* cv = sv + (size_t)st * cap;
            const XT* cx = sx + (size_t)gb * cap;
            const int lo = rlo - k0, hi = rhi - k0;
            if (lo >= 0 && hi <= hd->cnt[st])   // inside the staged range (always, unless ERR_STAGE)
                for (int e = lo; e < hi; ++e) mac(s, cv[e], cx[e]);
            acc_norm(s);
        }
        __syncwarp();   // stage st and gather buffer gb are free
        if (lane == 0 && i + S < m) {
            issue(i + S, ne0, ne1);
            if (i + S + 1 < m) bounds(i + S + 1, ne0, ne1);
        }
        if (row < A.n) epi(row, s, car);
        row = nrow; rlo = nlo; rhi = nhi; car = ncar;
    }
    // every copy has landed: retire the barriers so the slice may be reused
    // (by the register-staged passes, or by the next pass's mbar_init)
    __syncwarp();
    if (lane == 0)
        for (int st = 0; st < S; ++st) mbar_inval(&hd->bar[st]);
    __syncwarp();
}

// Producer/consumer product (FORM 4).  Warps specialise: WS_PROD producer
// warps move data, the other WS_CONS warps only add.  Rows are taken in
// tiles of WS_ROWS consecutive rows (a system's tile c belongs to CTA
// c mod gridDim.x), staged in a ring of A.stages shared-memory stages.  For
// each tile one producer lane bulk-copies the values and column indices
// (cp.async.bulk, L2 evict-first, completion counted in bytes on the
// stage's `full_vc` barrier) up to `stages` tiles ahead; once the columns
// have landed all producer threads gather the vector entries they address
// with cp.async (L2 evict-last) and have the stage's `full_x` barrier
// count their completion (cp.async.mbarrier.arrive).  Each consumer lane
// owns one row of the tile: it waits for both barriers, sums its row from
// shared memory (one fp64 FMA per entry for fp64 systems), runs the
// epilogue and, warp by warp, releases the stage on `empty`.  The fp64 pipe
// is thus fed by warps that never wait on global memory, while the memory
// system is kept busy by warps that never wait on the fp64 pipe.  Copies
// are rounded out to 16-byte units as in spmv_pipe; the host uses this form
// only where every tile fits a stage and the arrays are 16-byte aligned.
// Every wait gives up after WAIT_LIMIT_NS, recording ERR_WAIT.
#ifndef SLA_WS_PROD
#define SLA_WS_PROD 2
#endif
constexpr int WS_PROD = SLA_WS_PROD;
constexpr int WS_CONS = NWARP - WS_PROD;
constexpr int WS_ROWS = 32 * WS_CONS;
struct WsHdr {
    unsigned long long full_vc[MAX_STAGES];
    unsigned long long full_x[MAX_STAGES];
    unsigned long long empty[MAX_STAGES];
    int k0[MAX_STAGES];    // first staged entry (multiple of 4)
    int cnt[MAX_STAGES];   // staged entries
};

template <typename VT, typename XT>
__host__ __device__ constexpr size_t ws_smem_bytes(int tcap, int stages) {
    return sizeof(WsHdr) + (size_t)stages * tcap * (sizeof(VT) + sizeof(int) + sizeof(XT));
}

template <typename T, typename VT, typename XT, class Pre, class Epi>
__device__ __forceinline__ void spmv_ws(const Mat& A, const VT* __restrict__ av, const XT* __restrict__ v, Pre pre,
                                        Epi epi, double* dsm) {
    using acc_t = typename Prec<T>::acc;
    using car_t = decltype(pre(0));
    const int S = A.stages, cap = A.ccap;
    char* base = reinterpret_cast<char*>(dsm);
    WsHdr* hd = reinterpret_cast<WsHdr*>(base);
    VT* sv = reinterpret_cast<VT*>(base + sizeof(WsHdr));
    int* sc = reinterpret_cast<int*>(sv + (size_t)S * cap);
    XT* sx = reinterpret_cast<XT*>(sc + (size_t)S * cap);
    const int ntiles = (A.n + WS_ROWS - 1) / WS_ROWS;
    const int c0 = blockIdx.x, cstep = gridDim.x;
    const int m = c0 < ntiles ? (ntiles - 1 - c0) / cstep + 1 : 0;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    __syncthreads();   // shared memory may still be in use by an earlier pass
    if (m == 0) return;
    if (threadIdx.x == 0) {
        for (int st = 0; st < S; ++st) {
            mbar_init(&hd->full_vc[st], 1);
            mbar_init(&hd->full_x[st], 32 * WS_PROD);
            mbar_init(&hd->empty[st], WS_CONS);
        }
        fence_barrier_init();
    }
    __syncthreads();
    bool ok = true;
    if (warp >= WS_CONS) {
        // ------------------------------------------------ producers
        const int pt = threadIdx.x - 32 * WS_CONS;
        const long long nnz4 = A.nnz & ~3LL;
        const unsigned long long keep = l2_evict_last();
        const unsigned long long strm = l2_evict_first();
        // entry range of the CTA's j-th tile (thread pt == 0)
        auto bounds = [&](int j, int& e0, int& e1) {
            const int r0 = (c0 + j * cstep) * WS_ROWS;
            const int r1 = r0 + WS_ROWS < A.n ? r0 + WS_ROWS : A.n;
            e0 = ld_nc(A.rp + r0);
            e1 = ld_nc(A.rp + r1);
        };
        int ne0 = 0, ne1 = 0;
        if (pt == 0) bounds(0, ne0, ne1);
        int tb = 0, bst = 0, bpar = 1;   // next tile to copy, its stage, the parity of its stage's release
        int gst = 0, gpar = 0;           // stage and parity of the tile being gathered
        for (int t = 0; t < m; ++t) {
            while (tb < m && tb < t + S) {
                if (!mbar_wait(&hd->empty[bst], (unsigned)bpar)) { ok = false; break; }
                if (pt == 0) {
                    const long long k0 = (long long)ne0 & ~3LL;
                    const long long k1 = ((long long)ne1 + 3) & ~3LL;
                    long long kb = k1 < nnz4 ? k1 : (nnz4 > k0 ? nnz4 : k0);
                    long long ke = k1 < A.nnz ? k1 : A.nnz;
                    if (ke - k0 > cap) {   // never expected: the host sized the stages for every tile
                        atomicOr(A.err, ERR_STAGE);
                        kb = ke = k0;
                    }
                    hd->k0[bst] = (int)k0;
                    hd->cnt[bst] = (int)(ke - k0);
                    VT* dv = sv + (size_t)bst * cap;
                    int* dc = sc + (size_t)bst * cap;
                    for (long long k = kb; k < ke; ++k) {   // ragged end of the pattern
                        dv[k - k0] = av[k];
                        dc[k - k0] = A.ci[k];
                    }
                    const unsigned nb = (unsigned)(kb - k0);
                    fence_proxy_async();
                    mbar_arrive_expect(&hd->full_vc[bst], nb * (unsigned)(sizeof(VT) + sizeof(int)));
                    if (nb) {
                        bulk_copy(dv, av + k0, nb * (unsigned)sizeof(VT), &hd->full_vc[bst], strm);
                        bulk_copy(dc, A.ci + k0, nb * (unsigned)sizeof(int), &hd->full_vc[bst], strm);
                    }
                    if (tb + 1 < m) bounds(tb + 1, ne0, ne1);
                }
                ++tb;
                if (++bst == S) { bst = 0; bpar ^= 1; }
            }
            if (!ok) break;
            if (!mbar_wait(&hd->full_vc[gst], (unsigned)gpar)) { ok = false; break; }
            const int* cc = sc + (size_t)gst * cap;
            XT* dx = sx + (size_t)gst * cap;
            const int cnt = hd->cnt[gst];
#pragma unroll 4
            for (int e = pt; e < cnt; e += 32 * WS_PROD) cp_async<sizeof(XT)>(dx + e, v + cc[e], keep);
            cp_async_arrive(&hd->full_x[gst]);
            if (++gst == S) { gst = 0; gpar ^= 1; }
        }
    } else {
        // ------------------------------------------------ consumers
        const int rofs = warp * 32 + lane;
        int row = c0 * WS_ROWS + rofs, rlo = 0, rhi = 0;
        car_t car{};
        if (row < A.n) {
            rlo = ld_nc(A.rp + row);
            rhi = ld_nc(A.rp + row + 1);
            car = pre(row);
        }
        int st = 0, par = 0;
        for (int t = 0; t < m; ++t) {
            const int nrow = row + cstep * WS_ROWS;
            int nlo = 0, nhi = 0;
            car_t ncar{};
            if (t + 1 < m && nrow < A.n) {
                nlo = ld_nc(A.rp + nrow);
                nhi = ld_nc(A.rp + nrow + 1);
                ncar = pre(nrow);
            }
            const bool w = mbar_wait(&hd->full_vc[st], (unsigned)par) && mbar_wait(&hd->full_x[st], (unsigned)par);
            if (__any_sync(0xffffffffu, !w)) { ok = false; break; }
            if (row < A.n) {
                const int k0 = hd->k0[st];
                const VT* cv = sv + (size_t)st * cap;
                const XT* cx = sx + (size_t)st * cap;
                acc_t s = Prec<T>::zero();
                const int lo = rlo - k0, hi = rhi - k0;
                if (lo >= 0 && hi <= hd->cnt[st]) {   // inside the staged range (always, unless ERR_STAGE)
#pragma unroll 4
                    for (int e = lo; e < hi; ++e) mac(s, cv[e], cx[e]);
                }
                acc_norm(s);
                epi(row, s, car);
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&hd->empty[st]);
            if (++st == S) { st = 0; par ^= 1; }
            row = nrow; rlo = nlo; rhi = nhi; car = ncar;
        }
    }
    if (!ok) {
        atomicOr(A.err, ERR_WAIT);
        note_wait(A.err + 2, -1 - (int)blockIdx.x, m, warp, lane);
    }
    cp_wait<0>();
    const int all_ok = __syncthreads_and(ok ? 1 : 0);
    if (threadIdx.x == 0 && all_ok)
        for (int st = 0; st < S; ++st) {
            mbar_inval(&hd->full_vc[st]);
            mbar_inval(&hd->full_x[st]);
            mbar_inval(&hd->empty[st]);
        }
    __syncthreads();
}

// Product with a plain vector gather in one of seven compiled forms (the
// host picks one per matrix, so each kernel instantiation carries a single
// path): FORM 0 register staging (spmv_rows); FORM 1 cp.async value/column
// staging with register gathers; FORM 2 cp.async staging and gathers; FORM 3
// the warp pipeline (spmv_pipe); FORM 4 producer/consumer warps (spmv_ws);
// FORM 5 the direct form (spmv_direct); FORMs 6 and 7 the sliced form
// (spmv_sliced, on the layout's sliced copy of the values; compiled for 4
// and 5 resident CTAs per SM).
template <typename T, int FORM, typename VT, typename XT, bool COH = false, class Pre, class Epi>
__device__ __forceinline__ void spmv_vec(const Mat& A, const VT* __restrict__ av, const XT* v, Pre pre,
                                         Epi epi, double* wsm) {
    if constexpr (FORM == 5) spmv_direct<T, VT>(A, av, GatherVec<XT, COH>{v}, pre, epi);
    else if constexpr (sliced_form(FORM)) {
        constexpr int U = FORM == 7 ? SLA_SLICE_U_SHORT : SLICE_U;
        if (A.swin) spmv_sliced_win<T, VT, U>(A, av, GatherVec<XT, COH>{v}, pre, epi, wsm);
        else spmv_sliced<T, VT, U>(A, av, GatherVec<XT, COH>{v}, pre, epi);
    }
    else if constexpr (FORM == 0) spmv_rows<T, VT>(A, av, GatherVec<XT, COH>{v}, pre, epi, wsm);
    else if constexpr (FORM == 3) spmv_pipe<T, VT, XT>(A, av, v, pre, epi, wsm);
    else if constexpr (FORM == 4) spmv_ws<T, VT, XT>(A, av, v, pre, epi, wsm);
    else spmv_rows_async<T, VT, XT, FORM == 2, COH>(A, av, v, pre, epi, wsm);
}

// ----------------------------------------------------------------- scalar logic
// These run in thread 0 of the last CTA of one system on the system's State
// in device memory, or (c == nullptr) in thread 0 of every CTA of the fused
// kernel on the CTA's shared copy, which CTA 0 publishes afterwards.
__device__ __forceinline__ void count_frozen(Ctrl* c) {
    __threadfence();
    if (atomicAdd(&c->ndone, 1) + 1 == (int)gridDim.y) c->all_done = 1;
}
__device__ __forceinline__ void freeze(State* s, Ctrl* c, int status) {
    s->status = status;
    s->done = 1;
    if (c) count_frozen(c);
}

// After the p.q reduction (and the optional true-residual check).
__device__ __forceinline__ void after_spmv(State* s, Ctrl* c, double delta, bool checked, double tr2) {
    s->xpend = 0;   // the previous iteration's x update has been applied
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
    s->xpend = 1;
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
    s->xpend = 0;
    s->alpha = s->beta = s->rho = s->delta = s->tr2 = s->omega = 0.0;
    if (bb == 0.0) { freeze(s, c, ST_OK); return; }   // x = 0 is exact
    if (!finite(gamma)) { freeze(s, c, ST_BREAKDOWN); return; }
    s->check = (gamma <= s->tol2bb);
    if (!s->check && max_iter <= 0) freeze(s, c, ST_NOT_CONVERGED);
}

// ----------------------------------------------------------------- element-wise arithmetic
// acc += a * b
__device__ __forceinline__ void dot_acc(double& s, double a, double b) { s = fma(a, b, s); }
__device__ __forceinline__ void dot_acc(DF& s, float a, float b) { acc_push(s, two_prod(a, b)); }
__device__ __forceinline__ void dot_acc(DF& s, float2 a, float2 b) { acc_push(s, dprod(ld_w(a), ld_w(b))); }

// b - s for a row sum s
__device__ __forceinline__ double resid(double b, double s) { return b - s; }
__device__ __forceinline__ DF resid(float b, DF s) { return df_add_f(df_neg(s), b); }
__device__ __forceinline__ void sq_acc(double& t, double e) { t = fma(e, e, t); }
__device__ __forceinline__ void sq_acc(DF& t, DF e) {
    DF p = two_prod(e.hi, e.hi);
    p.lo = __fmaf_rn(__fmul_rn(2.0f, e.hi), e.lo, p.lo);
    acc_push(t, p);
}

// -lambda_i x_j, rounded once
__device__ __forceinline__ double neg_prod(double l, double x) { return -l * x; }
__device__ __forceinline__ float neg_prod(float l, float x) { return df_round(two_prod(-l, x)); }

// ----------------------------------------------------------------- SpMV API
// y = A x, and dot[sys] = x.y when dot != nullptr.
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, (FORM == 5 ? SLA_DIRECT_CTAS : SPMV_MIN_CTAS)) k_spmv(Mat A, Sys S, const T* __restrict__ av,
                                                            const T* __restrict__ x, T* __restrict__ y, double* dot) {
    using acc_t = typename Prec<T>::acc;
    SYS_PROLOGUE
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    av += val_offset<FORM>(A, sys, S.nnz); x += vo; y += vo;
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
// ||b - A round(x)||^2 over this CTA's rows (the true-residual check).  For
// the staged forms it is kept out of line: it runs only when the recursive
// residual has met the tolerance, and inlining it would cost the main
// product registers.  The direct form inlines it: there the out-of-line call
// (its stack frame) slowed the product in the running iteration by half
// (measured on B300 at six resident CTAs per SM), while the inlined pass
// fits the same registers.
template <typename T, bool COH>
__device__ __forceinline__ typename Prec<T>::acc residual_direct(const Mat& A, const T* __restrict__ av,
                                                                 const typename Prec<T>::xw* x,
                                                                 const T* __restrict__ b) {
    using acc_t = typename Prec<T>::acc;
    acc_t tr2 = Prec<T>::zero();
    spmv_direct<T, T>(A, av, GatherX<T, COH>{x}, [&](int i) { return b[i]; },
                      [&](int, acc_t s, T bi) { sq_acc(tr2, resid(bi, s)); });
    return tr2;
}
template <typename T, int FORM, bool COH = false>
__device__ __noinline__ typename Prec<T>::acc residual_staged(const Mat& A, const T* __restrict__ av,
                                                              const typename Prec<T>::xw* x,
                                                              const T* __restrict__ b, double* dsm) {
    using acc_t = typename Prec<T>::acc;
    acc_t tr2 = Prec<T>::zero();
    spmv_rows<T, T>(A, av, GatherX<T, COH>{x}, [&](int i) { return b[i]; },
                    [&](int, acc_t s, T bi) { sq_acc(tr2, resid(bi, s)); }, dsm);
    return tr2;
}
template <typename T, bool COH>
__device__ __forceinline__ typename Prec<T>::acc residual_sliced(const Mat& A, const T* __restrict__ sv,
                                                                 const typename Prec<T>::xw* x,
                                                                 const T* __restrict__ b) {
    using acc_t = typename Prec<T>::acc;
    acc_t tr2 = Prec<T>::zero();
    spmv_sliced<T, T>(A, sv, GatherX<T, COH>{x}, [&](int i) { return b[i]; },
                      [&](int, acc_t s, T bi) { sq_acc(tr2, resid(bi, s)); });
    return tr2;
}
template <typename T, int FORM, bool COH = false>
__device__ __forceinline__ typename Prec<T>::acc residual_pass(const Mat& A, const T* __restrict__ av,
                                                               const typename Prec<T>::xw* x,
                                                               const T* __restrict__ b, double* dsm) {
    if constexpr (FORM == 5) return residual_direct<T, COH>(A, av, x, b);
    else if constexpr (sliced_form(FORM)) return residual_sliced<T, COH>(A, av, x, b);
    else return residual_staged<T, FORM, COH>(A, av, x, b, dsm);
}

// q = A p, delta = p.q; with `check` set, ||b - A round(x)||^2 first.
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, (ProductCtas<T, FORM>::value))
    k_spmv_iter(Mat A, Sys S, const T* __restrict__ av, const typename Prec<T>::w* __restrict__ p,
                typename Prec<T>::w* __restrict__ q, const typename Prec<T>::xw* __restrict__ x,
                const T* __restrict__ b) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) {
        // a system frozen in k_update had its last x update applied by k_pupdate
        if (blockIdx.x == 0 && threadIdx.x == 0 && ld_cg(&st->xpend)) st->xpend = 0;
        return;
    }
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    av += val_offset<FORM>(A, sys, S.nnz); p += vo; q += vo; x += vo; b += vo;
    const bool check = ld_cg(&st->check) != 0;
    acc_t tr2 = Prec<T>::zero(), delta = Prec<T>::zero();
    if (check) tr2 = residual_pass<T, FORM>(A, av, x, b, dsm);
    spmv_vec<T, FORM, T, W>(A, av, p, [&](int i) { return ld_vec(p + i); },
                      [&](int i, acc_t s, W pi) {
                          const W qi = to_w(s);
                          st_vec(q + i, qi);
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

// One element of the residual update: r -= alpha q; gamma += r^2; and for
// Jacobi z = r / A_ii (stored for the direction update) with rho' += r z.
template <int PC, typename A, typename W, typename XW>
__device__ __forceinline__ void update_r(A alpha, W& ri, W qi, XW di, W& zi, A& g, A& rz) {
    const A rn = afma(aneg(alpha), ld_w(qi), ld_w(ri));
    ri = to_w(rn);
    acc_fma(g, rn, rn);
    if (PC == 1) {
        const A zz = amul(rn, ld_w(di));
        zi = to_w(zz);
        acc_fma(rz, rn, zz);
    }
}

// Pairs per thread per trip of the streaming kernels (measured on B300
// inside the running iteration: one pair per thread with two resident CTAs
// per SM beats two pairs, or four and eight CTAs per SM, on the 2D, 3D and
// kNN workloads).
#ifndef SLA_VU
#define SLA_VU 1
#endif
constexpr int VU = SLA_VU;

// r -= alpha q; gamma = r.r; rho' = r.z (PC 0: z = r; PC 1: z = r / A_ii,
// stored; PC 2: z comes later from the SPAI kernels).  x is advanced by
// k_pupdate, which reads p anyway, so this kernel touches r, q (and dinv, z).
template <typename T, int PC, bool PAIRS>
__global__ void __launch_bounds__(NT) k_update(Sys S, typename Prec<T>::w* __restrict__ r,
                                               const typename Prec<T>::w* __restrict__ q,
                                               const typename Prec<T>::xw* __restrict__ dinv,
                                               typename Prec<T>::w* __restrict__ z) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    using XW = typename Prec<T>::xw;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    __shared__ double red[RED_DOUBLES];
    r += vo; q += vo;
    if (PC == 1) { dinv += vo; z += vo; }
    const acc_t alpha = Prec<T>::scal(ld_cg(&st->alpha));
    acc_t g = Prec<T>::zero(), rz = Prec<T>::zero();
    if (PAIRS) {
        // VU pairs per thread per trip, all loads issued before any use
        using P2 = typename XPair<W>::type;
        using X2 = typename XPair<XW>::type;
        const int n2 = S.n >> 1;
        const int stride = gridDim.x * NT;
        for (int i0 = blockIdx.x * NT + threadIdx.x; i0 < n2; i0 += VU * stride) {
            P2 q2[VU], r2[VU];
            X2 d2[VU];
#pragma unroll
            for (int u = 0; u < VU; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    q2[u] = ld_vec_last(reinterpret_cast<const P2*>(q) + i);
                    r2[u] = ld_vec(reinterpret_cast<const P2*>(r) + i);
                    if (PC == 1) d2[u] = ld_gather(reinterpret_cast<const X2*>(dinv) + i);
                }
            }
#pragma unroll
            for (int u = 0; u < VU; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    W ra, rb, qa, qb, za{}, zb{};
                    XW da{}, db{};
                    split2(r2[u], ra, rb);
                    split2(q2[u], qa, qb);
                    if (PC == 1) split2(d2[u], da, db);
                    update_r<PC>(alpha, ra, qa, da, za, g, rz);
                    update_r<PC>(alpha, rb, qb, db, zb, g, rz);
                    st_vec(reinterpret_cast<P2*>(r) + i, join2(ra, rb));
                    if (PC == 1) st_vec(reinterpret_cast<P2*>(z) + i, join2(za, zb));
                }
            }
        }
    } else {
        for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
            W ri = ld_vec(r + i), zi{};
            update_r<PC>(alpha, ri, ld_vec_last(q + i), PC == 1 ? ld_gather(dinv + i) : XW{}, zi, g, rz);
            st_vec(r + i, ri);
            if (PC == 1) st_vec(z + i, zi);
        }
    }
    double v[2] = {Prec<T>::total(g), Prec<T>::total(rz)}, tot[2];
    if (grid_sum<2>(v, part, cnt, tot, red) && threadIdx.x == 0)
        after_update(st, S.ctl, tot[0], PC != 2, PC == 0 ? tot[0] : tot[1]);
}

// The iteration's pending x += alpha p (applied even when the system froze
// in k_update), then, while iterating, p = z + beta p, with z = r for
// PC 0.  INIT: p = z only (set-up of SPAI).
template <typename T, bool INIT, bool PAIRS>
__global__ void __launch_bounds__(NT) k_pupdate(Sys S, typename Prec<T>::w* __restrict__ p,
                                                typename Prec<T>::xw* __restrict__ x,
                                                const typename Prec<T>::w* __restrict__ zs) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    using XW = typename Prec<T>::xw;
    SYS_PROLOGUE
    const bool done = ld_cg(&st->done) != 0;
    const bool xp = !INIT && ld_cg(&st->xpend) != 0;
    if (done && !xp) return;
    p += vo; x += vo; zs += vo;
    const acc_t alpha = Prec<T>::scal(xp ? ld_cg(&st->alpha) : 0.0);
    const acc_t beta = Prec<T>::scal(INIT ? 0.0 : ld_cg(&st->beta));
    const bool more = !done;
    if (PAIRS) {
        using P2 = typename XPair<W>::type;
        using X2 = typename XPair<XW>::type;
        const int n2 = S.n >> 1;
        const int stride = gridDim.x * NT;
        for (int i0 = blockIdx.x * NT + threadIdx.x; i0 < n2; i0 += VU * stride) {
            P2 p2[VU], z2[VU];
            X2 x2[VU];
#pragma unroll
            for (int u = 0; u < VU; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    p2[u] = INIT ? P2{} : ld_vec(reinterpret_cast<const P2*>(p) + i);
                    if (xp) x2[u] = ld_vec(reinterpret_cast<const X2*>(x) + i);
                    if (more) z2[u] = ld_vec_last(reinterpret_cast<const P2*>(zs) + i);
                }
            }
#pragma unroll
            for (int u = 0; u < VU; ++u) {
                const int i = i0 + u * stride;
                if (i < n2) {
                    W pa, pb;
                    split2(p2[u], pa, pb);
                    if (xp) {
                        XW xa, xb;
                        split2(x2[u], xa, xb);
                        xa = to_w(afma(alpha, ld_w(pa), ld_w(xa)));
                        xb = to_w(afma(alpha, ld_w(pb), ld_w(xb)));
                        st_vec(reinterpret_cast<X2*>(x) + i, join2(xa, xb));
                    }
                    if (more) {
                        W za, zb;
                        split2(z2[u], za, zb);
                        st_vec(reinterpret_cast<P2*>(p) + i,
                               INIT ? join2(za, zb)
                                    : join2(to_w(afma(beta, ld_w(pa), ld_w(za))), to_w(afma(beta, ld_w(pb), ld_w(zb)))));
                    }
                }
            }
        }
    } else {
        for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += gridDim.x * NT) {
            const W pi = INIT ? W{} : ld_vec(p + i);
            if (xp) st_vec(x + i, to_w(afma(alpha, ld_w(pi), ld_w(ld_vec(x + i)))));
            if (more) st_vec(p + i, INIT ? ld_vec_last(zs + i) : to_w(afma(beta, ld_w(pi), ld_w(ld_vec_last(zs + i)))));
        }
    }
}

// SPAI, first product: t = G^T r (explicit transposed CSR of G; G values
// are per system, [batch][nnz(G)]).
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, (FORM >= 5 ? ProductCtas<T, FORM>::value : SPMV_MIN_CTAS)) k_spai_t(Mat GT, Sys S, long long nnzg,
                                                              const typename Prec<T>::gv* __restrict__ gtv,
                                                              const typename Prec<T>::w* __restrict__ r,
                                                              typename Prec<T>::w* __restrict__ t) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ __align__(16) double dsm[];
    gtv += val_offset<FORM>(GT, sys, nnzg); r += vo; t += vo;
    spmv_vec<T, FORM, typename Prec<T>::gv, W>(GT, gtv, r, [](int) { return W{}; },
                                         [&](int i, acc_t s, W) { st_vec(t + i, to_w(s)); }, dsm);
}

// SPAI, second product: z = G t + eps r, rho' = r.z -> beta (or rho at set-up).
template <typename T, int FORM>
__global__ void __launch_bounds__(NT, (FORM >= 5 ? ProductCtas<T, FORM>::value : SPMV_MIN_CTAS)) k_spai_z(Mat G, Sys S, long long nnzg,
                                                              const typename Prec<T>::gv* __restrict__ gv,
                                                              const typename Prec<T>::w* __restrict__ t,
                                                              const typename Prec<T>::w* __restrict__ r,
                                                              typename Prec<T>::w* __restrict__ z, double eps) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    SYS_PROLOGUE
    if (ld_cg(&st->done)) return;
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    gv += val_offset<FORM>(G, sys, nnzg); t += vo; r += vo; z += vo;
    const acc_t e = Prec<T>::scal(eps);
    acc_t rz = Prec<T>::zero();
    spmv_vec<T, FORM, typename Prec<T>::gv, W>(G, gv, t, [&](int i) { return r[i]; },
                                         [&](int i, acc_t s, W ri) {
                                             const W zi = to_w(afma(e, ld_w(ri), s));
                                             st_vec(z + i, zi);
                                             dot_acc(rz, ri, zi);
                                         },
                                         dsm);
    double v[1] = {Prec<T>::total(rz)}, tot[1];
    if (grid_sum<1>(v, part, cnt, tot, red) && threadIdx.x == 0) new_direction(st, S.ctl, tot[0]);
}

// ----------------------------------------------------------------- fused iteration
// A persistent form of the iteration for CG and Jacobi-PCG: one cooperative
// launch (every CTA resident) runs up to `iters` iterations, the CTAs of a
// system meeting at grid barriers instead of kernel boundaries:
//   A  q = A p, delta = p.q (and ||b - A round(x)||^2 when checking)
//      -> all-reduce -> alpha
//   B  r -= alpha q, z = M^-1 r (stored), gamma = r.r, rho' = r.z
//      -> all-reduce -> beta, convergence test
//   C  x += alpha p, p = z + beta p -> barrier
// x is advanced in C, where p is read anyway, so B reads three vectors and
// C three.  Every CTA sums the partial sums of all CTAs itself, in CTA
// order, so all CTAs hold identical scalars (a shared-memory copy of the
// State, advanced by the same scalar logic as the kernel-per-step path) and
// take identical decisions; CTA 0 publishes the State when the launch ends.
struct GridSync {
    unsigned count;   // arrivals at the current barrier
    unsigned gen;     // completed barriers
};

// Thread 0 of every CTA of a system: arrive and wait for the others.
// Returns false (and records ERR_WAIT) after WAIT_LIMIT_NS.
__device__ __forceinline__ bool grid_arrive_wait(GridSync* g, int* err, unsigned long long limit_ns = WAIT_LIMIT_NS) {
    volatile unsigned* vgen = &g->gen;
    const unsigned gen = *vgen;   // read before arriving: the last arrival advances it
    __threadfence();
    const unsigned arrived = atomicAdd(&g->count, 1u);
    if (arrived == gridDim.x - 1) {
        atomicExch(&g->count, 0u);
        __threadfence();
        atomicAdd(&g->gen, 1u);
        return true;
    }
    const unsigned long long t0 = global_ns();
    for (unsigned k = 0; k < (1u << 31); ++k) {
        if (*vgen != gen) {
            __threadfence();
            return true;
        }
        if (k > 32) __nanosleep(64);
        if ((k & 63u) == 63u && global_ns() - t0 > limit_ns) break;
    }
    atomicOr(err, ERR_GRID);
    note_wait(err + 2, 1 + (int)blockIdx.x, (int)gen, (int)arrived, (int)*((volatile unsigned*)&g->count));
    return false;
}

__device__ __forceinline__ bool grid_barrier(GridSync* g, int* err) {
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) s_ok = grid_arrive_wait(g, err);
    __syncthreads();
    return s_ok != 0;
}

// Sum NV values over the system's CTAs (in CTA order, in every CTA; valid
// in thread 0).  part: [gridDim.x][NV] slots of this reduction.
template <int NV>
__device__ __forceinline__ bool grid_allreduce(double (&v)[NV], double* part, GridSync* g, int* err, double* sm) {
    __shared__ int s_ok;
    block_sum<NV>(v, sm);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) part[blockIdx.x * NV + j] = v[j];
        s_ok = grid_arrive_wait(g, err);
    }
    __syncthreads();
    if (!s_ok) return false;
    double acc[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) acc[j] = 0.0;
    for (int bk = threadIdx.x; bk < (int)gridDim.x; bk += NT) {
#pragma unroll
        for (int j = 0; j < NV; ++j) acc[j] += ld_cg(part + bk * NV + j);
    }
    block_sum<NV>(acc, sm);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) v[j] = acc[j];
    }
    return true;
}

#ifndef SLA_FUSED_MIN_CTAS
#define SLA_FUSED_MIN_CTAS IterMinCtas<T>::value
#endif
template <typename T, int FORM, int PC, bool PAIRS>
__global__ void __launch_bounds__(NT, SLA_FUSED_MIN_CTAS)
    k_cg_fused(Mat A, Sys S, const T* __restrict__ av, typename Prec<T>::w* __restrict__ p,
               typename Prec<T>::w* __restrict__ q, typename Prec<T>::w* __restrict__ r,
               typename Prec<T>::w* __restrict__ z, typename Prec<T>::xw* __restrict__ x,
               const typename Prec<T>::xw* __restrict__ dinv, const T* __restrict__ b, GridSync* gsync,
               int iters) {
    using acc_t = typename Prec<T>::acc;
    using W = typename Prec<T>::w;
    using XW = typename Prec<T>::xw;
    SYS_PROLOGUE
    __shared__ State ls;
    __shared__ int s_was_done;
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    av += ao; p += vo; q += vo; r += vo; z += vo; x += vo; b += vo;
    if (PC == 1) dinv += vo;
    GridSync* gs = gsync + sys;
    double* partA = part;                   // [gridDim.x][2]: delta, ||b - A x||^2
    double* partB = part + 2 * gridDim.x;   // [gridDim.x][2]: gamma, rho'
    int* err = &S.ctl->err;
    if (threadIdx.x == 0) {
        ls = *st;
        s_was_done = ls.done;
    }
    __syncthreads();
    const int stride = gridDim.x * NT;
    for (int it = 0; it < iters && !ls.done; ++it) {
        // A
        const bool check = ls.check != 0;
        acc_t tr2 = Prec<T>::zero(), delta = Prec<T>::zero();
        if (check) tr2 = residual_pass<T, FORM, true>(A, av, x, b, dsm);
        spmv_vec<T, FORM, T, W, true>(A, av, p, [&](int i) { return p[i]; },
                                [&](int i, acc_t s, W pi) {
                                    const W qi = to_w(s);
                                    q[i] = qi;
                                    dot_acc(delta, pi, qi);
                                },
                                dsm);
        double va[2] = {Prec<T>::total(delta), Prec<T>::total(tr2)};
        if (!grid_allreduce<2>(va, partA, gs, err, red)) break;
        if (threadIdx.x == 0) after_spmv(&ls, nullptr, va[0], check, va[1]);
        __syncthreads();
        if (ls.done) break;
        // B
        {
            const acc_t alpha = Prec<T>::scal(ls.alpha);
            acc_t g = Prec<T>::zero(), rz = Prec<T>::zero();
            auto one = [&](W& ri, W qi, XW di, W& zi) { update_r<PC>(alpha, ri, qi, di, zi, g, rz); };
            if (PAIRS) {
                using P2 = typename XPair<W>::type;
                using X2 = typename XPair<XW>::type;
                const int n2 = S.n >> 1;
                for (int i = blockIdx.x * NT + threadIdx.x; i < n2; i += stride) {
                    const P2 q2 = ld_stream(reinterpret_cast<const P2*>(q) + i);
                    P2 r2 = reinterpret_cast<const P2*>(r)[i];
                    X2 d2{};
                    if (PC == 1) d2 = ld_nc(reinterpret_cast<const X2*>(dinv) + i);
                    W ra, rb, qa, qb, za{}, zb{};
                    XW da{}, db{};
                    split2(r2, ra, rb);
                    split2(q2, qa, qb);
                    if (PC == 1) split2(d2, da, db);
                    one(ra, qa, da, za);
                    one(rb, qb, db, zb);
                    reinterpret_cast<P2*>(r)[i] = join2(ra, rb);
                    if (PC == 1) reinterpret_cast<P2*>(z)[i] = join2(za, zb);
                }
            } else {
                for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += stride) {
                    W ri = r[i], zi{};
                    one(ri, ld_stream(q + i), PC == 1 ? dinv[i] : XW{}, zi);
                    r[i] = ri;
                    if (PC == 1) z[i] = zi;
                }
            }
            double vb[2] = {Prec<T>::total(g), Prec<T>::total(rz)};
            if (!grid_allreduce<2>(vb, partB, gs, err, red)) break;
            if (threadIdx.x == 0) after_update(&ls, nullptr, vb[0], true, PC == 0 ? vb[0] : vb[1]);
            __syncthreads();
        }
        // C (x always advances; p only while iterating)
        {
            const acc_t alpha = Prec<T>::scal(ls.alpha);
            const acc_t beta = Prec<T>::scal(ls.beta);
            const bool more = !ls.done;
            const W* zs = PC == 1 ? z : r;
            if (PAIRS) {
                using P2 = typename XPair<W>::type;
                using X2 = typename XPair<XW>::type;
                const int n2 = S.n >> 1;
                for (int i = blockIdx.x * NT + threadIdx.x; i < n2; i += stride) {
                    const P2 p2 = reinterpret_cast<const P2*>(p)[i];
                    const X2 x2 = reinterpret_cast<const X2*>(x)[i];
                    const P2 z2 = reinterpret_cast<const P2*>(zs)[i];
                    W pa, pb, za, zb;
                    XW xa, xb;
                    split2(p2, pa, pb);
                    split2(x2, xa, xb);
                    split2(z2, za, zb);
                    xa = to_w(afma(alpha, ld_w(pa), ld_w(xa)));
                    xb = to_w(afma(alpha, ld_w(pb), ld_w(xb)));
                    reinterpret_cast<X2*>(x)[i] = join2(xa, xb);
                    if (more)
                        reinterpret_cast<P2*>(p)[i] =
                            join2(to_w(afma(beta, ld_w(pa), ld_w(za))), to_w(afma(beta, ld_w(pb), ld_w(zb))));
                }
            } else {
                for (int i = blockIdx.x * NT + threadIdx.x; i < S.n; i += stride) {
                    const W pi = p[i];
                    x[i] = to_w(afma(alpha, ld_w(pi), ld_w(x[i])));
                    if (more) p[i] = to_w(afma(beta, ld_w(pi), ld_w(zs[i])));
                }
            }
        }
        if (threadIdx.x == 0) ls.xpend = 0;   // applied in C
        if (ls.done) break;
        if (!grid_barrier(gs, err)) break;
    }
    __syncthreads();
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        *st = ls;
        if (ls.done && !s_was_done) count_frozen(S.ctl);
    }
}

// ----------------------------------------------------------------- set-up / final
// x = 0, r = b, b copied into the workspace, bb = b.b.
template <typename T>
__global__ void __launch_bounds__(NT) k_init(Sys S, const T* __restrict__ b_user, T* __restrict__ bw,
                                             typename Prec<T>::xw* __restrict__ x, typename Prec<T>::w* __restrict__ r,
                                             double tol, int max_iter) {
    SYS_PROLOGUE
    __shared__ double red[RED_DOUBLES];
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
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
    av += ao; b_user += vo; x0 += vo; bw += vo; x += vo; r += vo;
    acc_t bb = Prec<T>::zero(), g = Prec<T>::zero();
    spmv_rows<T, T>(A, av, GatherVec<T>{x0}, [&](int i) { return b_user[i]; },
                    [&](int i, acc_t s, T bi) {
                        bw[i] = bi;
                        x[i] = x_from(x0[i]);
                        const acc_t ri = resid(bi, s);
                        r[i] = to_w(ri);
                        dot_acc(bb, bi, bi);
                        acc_fma(g, ri, ri);
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
    __shared__ double red[RED_DOUBLES];
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
    extern __shared__ __align__(16) double dsm[];
    __shared__ double red[RED_DOUBLES];
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
    extern __shared__ __align__(16) double dsm[];
    lam += vo; x += vo; dA += ao;
    if (A.direct) {   // thread per row (the layout gives no shared memory)
        for (int row = blockIdx.x * NT + threadIdx.x; row < A.n; row += gridDim.x * NT) {
            const int lo = ld_nc(A.rp + row), hi = ld_nc(A.rp + row + 1);
            const T li = lam[row];
            for (int k = lo; k < hi; ++k) __stcs(dA + k, neg_prod(li, ld_nc(x + ld_stream(A.ci + k))));
        }
        return;
    }
    int* srow = reinterpret_cast<int*>(dsm + (threadIdx.x >> 5) * A.wstride);
    const int lane = threadIdx.x & 31;
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

// ----------------------------------------------------------------- self-test of the bounded waits
// Makes one of the library's device waits run out on purpose, with a short
// limit: which = 0, an mbarrier phase that never completes (nothing
// arrives); which = 1, a grid barrier of two CTAs that only CTA 0 reaches
// (CTA 1 returns at once).  The wait gives up, records its error bit and
// location in `c` as the solver's waits do, and the kernel returns, so the
// context stays usable.
__global__ void k_wait_selftest(int which, unsigned long long limit_ns, Ctrl* c, GridSync* gs) {
    if (which == 0) {
        if (blockIdx.x != 0) return;
        __shared__ unsigned long long bar;
        if (threadIdx.x == 0) {
            mbar_init(&bar, 1);
            fence_barrier_init();
            if (!mbar_wait(&bar, 0, limit_ns)) {
                atomicOr(&c->err, ERR_WAIT);
                note_wait(c->diag, -1 - (int)blockIdx.x, 0, 1, 0);
            }
            mbar_inval(&bar);   // no arrival or copy is pending
        }
        return;
    }
    if (blockIdx.x != 0) return;   // never reaches the barrier
    if (threadIdx.x == 0) grid_arrive_wait(gs, &c->err, limit_ns);
}

}  // namespace sla
