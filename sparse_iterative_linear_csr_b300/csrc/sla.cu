// sla.cu -- C ABI of the sm_103a CSR PCG library (declared in include/sla.h).
//
// Host side of the solver: handle life cycle, device set-up, and the
// iteration driver.  The driver captures `poll_k` CG iterations into one CUDA
// graph per (preconditioner, eps, k) and launches it repeatedly; every kernel
// of an iteration returns at once when its system is frozen, so the host
// only reads the batch-wide "all done" flag (one 4-byte copy to pinned memory
// per graph launch, two launches kept in flight) instead of synchronising
// every iteration.
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>
#include <string>
#include <thread>
#include <type_traits>
#include <vector>

#include "../../include/sla.h"
#include "common.cuh"
#include "kernels.cuh"
#include "bicgstab.cuh"
#include "setup.cuh"
#include "block.cuh"

using namespace sla;

// ===================================================================== errors
static thread_local std::string g_err;
static std::atomic<unsigned long long> g_launches{0};

static sla_status fail(sla_status st, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

// A failed runtime call is reported here and cleared from the runtime's
// last-error slot, so the next launch check does not report it again.
#define CU(call)                                                                              \
    do {                                                                                      \
        cudaError_t e_ = (call);                                                              \
        if (e_ != cudaSuccess) {                                                              \
            (void)cudaGetLastError();                                                         \
            return fail(e_ == cudaErrorMemoryAllocation ? SLA_ERR_NOMEM : SLA_ERR_CUDA,      \
                        "%s failed: %s (%s:%d)", #call, cudaGetErrorString(e_), __FILE__,     \
                        __LINE__);                                                            \
        }                                                                                     \
    } while (0)

#define TRY(expr)                            \
    do {                                     \
        sla_status s_ = (expr);              \
        if (s_ != SLA_OK) return s_;         \
    } while (0)

static sla_status launched() {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SLA_ERR_CUDA, "kernel launch failed: %s", cudaGetErrorString(e));
    return SLA_OK;
}

// ===================================================================== handle
struct DevBuf {
    void* p = nullptr;
    size_t bytes = 0;
    DevBuf() = default;
    DevBuf(const DevBuf&) = delete;
    DevBuf& operator=(const DevBuf&) = delete;
    ~DevBuf() { release(); }
    sla_status alloc(size_t b) {
        release();
        if (b == 0) b = 16;
        cudaError_t e = cudaMalloc(&p, b);
        if (e != cudaSuccess) {
            p = nullptr;
            return fail(SLA_ERR_NOMEM, "cudaMalloc(%zu) failed: %s", b, cudaGetErrorString(e));
        }
        bytes = b;
        return SLA_OK;
    }
    void release() {
        if (p) cudaFree(p);
        p = nullptr;
        bytes = 0;
    }
    template <typename T>
    T* as() const { return static_cast<T*>(p); }
};

// Captured iterations for one (preconditioner, eps, k).  With product
// timing there is one instance per launch slot, each recording its own
// pair of events around its first product kernel (two launches are in
// flight, so one pair of events could be overwritten before it is read).
struct GraphCache {
    cudaGraphExec_t exec[2] = {nullptr, nullptr};
    cudaEvent_t t0[2] = {nullptr, nullptr}, t1[2] = {nullptr, nullptr};
    int k = 0;
    double eps = 0.0;
    int nodes = 0;
    void reset() {
        for (int i = 0; i < 2; ++i) {
            if (exec[i]) cudaGraphExecDestroy(exec[i]);
            if (t0[i]) cudaEventDestroy(t0[i]);
            if (t1[i]) cudaEventDestroy(t1[i]);
            exec[i] = nullptr;
            t0[i] = t1[i] = nullptr;
        }
        k = 0;
        nodes = 0;
    }
};

// Product layout of one matrix: warp staging capacity (entries per group of
// 32 / lanes rows), lanes per row, bulk-copy capacities and stages, the
// compiled form the product kernels use, their dynamic shared memory, and
// CTAs per system.
struct Layout {
    int cap = 32;
    int lanes = 1;
    int gx = 1;
    int gasync = 0;   // gathers by cp.async (scattered columns)
    int ccap = 0;     // warp pipeline: entries per stage (0: a group would not fit)
    int tcap = 0;     // producer/consumer form: entries per tile stage (0: unusable)
    int stages = 0;   // bulk-copy forms: ring stages
    int form = 0;     // compiled form of the product kernels (spmv_vec)
    size_t smem = 0;  // their dynamic shared memory
    int maxrow = 0;   // longest row
    int bal = 0;      // staged groups summed split over the lanes (forms 1 and 2, one lane per row)
    int swin = 0;     // sliced rows sorted within windows of SLICE_WIN rows: a warp per window
    // sliced copy (form 6), owned by the handle's SellBufs
    const int* sptr = nullptr;
    const int* sperm = nullptr;
    const int* scol = nullptr;
    const void* sval = nullptr;
    int nslices = 0;
    long long vstride = 0;
};

// Sliced copy of a matrix (form 6): slice pointers, the row of every slot
// (when rows are reordered within windows), columns, the source CSR entry
// of every sliced entry (-1: padding) and the sliced values [batch][vstride].
struct SellBufs {
    DevBuf sptr, perm, scol, smap, sval;
    long long npad = 0;
    long long vstride = 0;
    int nslices = 0;
    void release() {
        sptr.release(); perm.release(); scol.release(); smap.release(); sval.release();
        npad = vstride = 0;
        nslices = 0;
    }
};

struct sla_csr {
    int n = 0;
    long long nnz = 0;
    int batch = 1;
    sla_dtype dt = SLA_F64;
    size_t es = 8;  // bytes per stored value
    const int* rp = nullptr;
    const int* ci = nullptr;
    const void* vals = nullptr;
    int device = 0;
    int sms = 0;

    Layout LA;         // product layout of A (sla_spmv, the dL/dA pass)
    // The matrix the solve iterates on: A itself, or P A P^T when the handle
    // reorders a scattered pattern (reverse Cuthill-McKee).
    const int* irp = nullptr;
    const int* ici = nullptr;
    const void* ivals = nullptr;
    Layout LI;
    bool reordered = false;
    DevBuf perm, iperm;        // int[n]: new -> old row, old -> new row
    DevBuf prp, pci, psrc;     // permuted pattern; source entry of every permuted entry
    DevBuf pvals;              // permuted values [batch][nnz]
    // Scratch of a values update and the SPAI refresh, kept across calls: a
    // buffer freed per call (cudaFree) would synchronise the whole device,
    // also the caller's copies in flight on other streams.
    DevBuf derr;               // one int: error bits of the diagonal and SPAI value kernels
    DevBuf dorig;              // [batch][n] diagonal in the caller's order (SPAI, reordered handles)
    DevBuf drs;                // [batch][n] 1 / sqrt(A_ii) in the caller's order (SPAI)
    DevBuf gtpos;              // [nnz(G)] entry of A behind each entry of G^T (caller's order)
    DevBuf ptmp;               // 2 x [batch][n] values: permuted right-hand side / initial guess, result
    bool vals_aligned = false;  // values 16-byte aligned for every system (bulk-copy forms)
    bool pipeline = false;      // SLA_WARP_PIPELINE: warp-pipeline product where it applies
    bool ws = false;            // SLA_PRODUCER_CONSUMER: producer/consumer product where it applies
    bool staged = false;        // SLA_STAGED: never the direct form
    bool time_product = false;  // SLA_TIME_PRODUCT: events around one product kernel per graph launch
    double prod_ms = 0.0;       // summed product-kernel durations (sla_product_time)
    long long prod_n = 0;
    bool persistent = false;    // SLA_PERSISTENT: persistent iteration kernel for CG / Jacobi-PCG
    bool coop = false;          // device supports cooperative launches
    DevBuf gsync;               // GridSync per system (fused iteration kernel)
    int diag_err = 0;  // ERR_NO_DIAG | ERR_DIAG_SIGN
    DevBuf diag, dinv;

    // SPAI factor (patterns and layouts built on first use; values again
    // after every sla_csr_update_values)
    bool spai_ready = false;
    bool spai_stale = false;   // values of G, G^T older than the values of A
    // reordered handles: the factors on the caller's ordering and the source
    // entry of every permuted entry
    DevBuf grp0, gci0, gv0, gtrp0, gtci0, gtv0, gsrc, gtsrc;
    long long nnzg = 0;
    long long gstride = 0;  // per-system stride of the G values (nnzg rounded up to even: 16-byte aligned)
    Layout LG, LGT;    // ... of G and G^T
    DevBuf grp, gci, gv, gtrp, gtci, gtv;

    // workspace
    DevBuf x, r, p, q, z, t, bw;
    DevBuf state, ctl, cnt, part, stat;
    int pstride = 0;
    int* h_flag = nullptr;     // pinned [2]
    Stat* h_stat = nullptr;    // pinned [batch]
    cudaEvent_t ev[2] = {nullptr, nullptr};
    cudaStream_t cap = nullptr;  // capture stream
    // graphs: CG per preconditioner (0..2), BiCGStab on A / A^T per
    // preconditioner (3 + 2 * transposed + pc)
    GraphCache graph[7];

    // sliced copies (form 6) of the iteration matrix and of G, G^T
    bool sliced = false;        // SLA_SLICED: sliced product form where it applies
    int split = 0;              // SLA_SPLIT_ROWS: 1, SLA_ROW_WALK: -1, else chosen per matrix
    SellBufs sI, sG, sGT;
    SellBufs sB, sT;            // sliced copies of the BiCGStab matrices (values refilled per solve)

    // BiCGStab (built on first use): the iteration matrix's layout with the
    // register / cp.async forms only (its values may be a handle-owned
    // scaled copy), the shadow residual, the column-scaled values A D^-1;
    // for the adjoint the explicit transpose of the iteration matrix (pattern,
    // source entry of every transposed entry, values per system) and its layout.
    bool bicg_ready = false;
    Layout LB;
    DevBuf rh, bvals;
    bool tr_ready = false;
    Layout LT;
    DevBuf trp, tci, tsrc, tvals;
};

static constexpr size_t WORK_BYTES = 8;  // working vectors: fp64, or a double-float pair
static constexpr int MAX_CAP = 864;  // staging capacity limit (larger groups take the global path)

// Staging form for capacity `cap`: 2 (cp.async, double-buffered values and
// columns) while that fits three CTAs per SM, else 1 (single-buffered) while
// it fits two, else 0 (register staging).
#ifndef SLA_STAGE_CTAS
#define SLA_STAGE_CTAS 3   // resident CTAs per SM double buffering must still allow
#endif
#ifndef SLA_MIN_LANES
#define SLA_MIN_LANES 1    // fewest lanes per row the layout considers
#endif
#ifndef SLA_MIN_LANES_G
#define SLA_MIN_LANES_G SLA_MIN_LANES   // the same for the SPAI factors
#endif
#ifndef SLA_MAX_CAP_G
#define SLA_MAX_CAP_G 864   // staging capacity limit for the SPAI factors (larger groups go unstaged)
#endif
static int staging_form(int cap) {
    const size_t per_sm = 228 * 1024;
    if ((size_t)NWARP * async_smem_per_warp<double, double>(cap, 2) * SLA_STAGE_CTAS <= per_sm) return 2;
    if ((size_t)NWARP * async_smem_per_warp<double, double>(cap, 1) * 2 <= per_sm) return 1;
    return 0;
}
// Dynamic shared memory of the staged-SpMV kernels for capacity `cap`
// (enough for the register form too, which the true-residual pass uses).
static size_t spmv_smem(int cap) {
    const size_t single = (size_t)cap * 2 * sizeof(double);
    const int f = staging_form(cap);
    const size_t piped = f ? async_smem_per_warp<double, double>(cap, f) : 0;
    return (size_t)NWARP * (piped > single ? piped : single);
}
// Resident CTAs per SM of `kern` with `smem` bytes of dynamic shared memory
// (the kernel must already allow that much: allow_smem).
template <typename K>
static sla_status occupancy(K kern, size_t smem, int* out) {
    int nb = 0;
    CU(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, NT, smem));
    *out = nb > 0 ? nb : 1;
    return SLA_OK;
}

// CTAs per system for a kernel walking `units` work units with `per_sm`
// resident CTAs per SM (persistent in x: a multiple of the SM count when
// there is enough work).
static int grid_x(const sla_csr* h, long long units, int per_sm) {
    long long g = (long long)per_sm * h->sms / h->batch;
    if (g > units) g = units;
    if (g < 1) g = 1;
    return (int)g;
}

static long long group_ctas(int n, int lanes) {
    const long long rows = 32 / lanes;
    return (((long long)n + rows - 1) / rows + NWARP - 1) / NWARP;
}
static bool pairs_ok(const sla_csr* h) { return (h->n & 1) == 0; }
static long long vec_units(const sla_csr* h) {
    const long long m = pairs_ok(h) ? h->n / 2 : h->n;
    return (m + NT - 1) / NT;
}

// Allow every staged-SpMV kernel of dtype T (all three staging forms) the
// largest staging slice.
template <typename T, int F>
static sla_status allow_smem_form(int b) {
    CU(cudaFuncSetAttribute(k_spmv<T, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
    CU(cudaFuncSetAttribute(k_spmv_iter<T, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
    CU(cudaFuncSetAttribute(k_spai_t<T, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
    CU(cudaFuncSetAttribute(k_spai_z<T, F>, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
    return SLA_OK;
}

// BiCGStab product kernels (fp64; register and cp.async staging forms).
template <int F>
static sla_status allow_smem_bicg(int b) {
    CU(cudaFuncSetAttribute(k_bicg_v<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
    CU(cudaFuncSetAttribute(k_bicg_t<F>, cudaFuncAttributeMaxDynamicSharedMemorySize, b));
    return SLA_OK;
}

static constexpr int SMEM_CTA_MAX = 222 * 1024;   // dynamic shared memory a CTA may use (227 KB less static)
static constexpr size_t SMEM_SM = 228 * 1024;     // shared memory per SM
static constexpr size_t SMEM_CTA_RESERVE = 6144;  // per-CTA system reserve + static shared memory

template <typename T, int F>
static sla_status allow_smem_fused() {
    CU(cudaFuncSetAttribute(k_cg_fused<T, F, 0, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    CU(cudaFuncSetAttribute(k_cg_fused<T, F, 0, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    CU(cudaFuncSetAttribute(k_cg_fused<T, F, 1, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    CU(cudaFuncSetAttribute(k_cg_fused<T, F, 1, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    return SLA_OK;
}

// cudaFuncSetAttribute acts on the current device's context, so the
// attributes are set once per device ordinal (and per dtype).
static constexpr int SMEM_MAX_DEVICES = 64;
static std::mutex g_smem_mu;

template <typename T>
static sla_status allow_smem() {
    static bool done[SMEM_MAX_DEVICES] = {};
    int dev = 0;
    CU(cudaGetDevice(&dev));
    if (dev < 0 || dev >= SMEM_MAX_DEVICES) return fail(SLA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_smem_mu);
    if (done[dev]) return SLA_OK;
    const int b = (int)spmv_smem(MAX_CAP);
    TRY((allow_smem_form<T, 0>(b)));
    TRY((allow_smem_form<T, 1>(b)));
    TRY((allow_smem_form<T, 2>(b)));
    TRY((allow_smem_form<T, 3>(SMEM_CTA_MAX)));
    TRY((allow_smem_form<T, 4>(SMEM_CTA_MAX)));
    TRY((allow_smem_fused<T, 0>()));
    TRY((allow_smem_fused<T, 1>()));
    TRY((allow_smem_fused<T, 2>()));
    TRY((allow_smem_fused<T, 3>()));
    TRY((allow_smem_fused<T, 4>()));
    CU(cudaFuncSetAttribute(k_init_x0<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    CU(cudaFuncSetAttribute(k_final<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    CU(cudaFuncSetAttribute(k_grad_A<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_CTA_MAX));
    if constexpr (std::is_same<T, double>::value) {
        TRY((allow_smem_bicg<0>(b)));
        TRY((allow_smem_bicg<1>(b)));
        TRY((allow_smem_bicg<2>(b)));
    }
    done[dev] = true;
    return SLA_OK;
}

// Warp pipeline (FORM 3): shared memory per warp for capacity `ccap`, S
// stages and `vb`-byte values (gathered entries sized at 8 bytes, the
// largest).
#ifndef SLA_PIPE_CTAS
#define SLA_PIPE_CTAS 3   // most resident CTAs per SM the warp pipeline aims for
#endif
static size_t pipe_bytes(int ccap, int S, size_t vb) {
    return sizeof(PipeHdr) + (size_t)S * ccap * (vb + sizeof(int)) + 2 * (size_t)ccap * sizeof(double);
}
// Most stages (3 or 4) that fit the most resident CTAs per SM (3 or 2); 0
// when not even two CTAs of three stages fit (the warp-staged forms then
// serve the matrix).
static int pipe_stages(int ccap, size_t vb) {
    for (int ctas = SLA_PIPE_CTAS; ctas >= 2; --ctas)
        for (int S = MAX_STAGES; S >= 3; --S) {
            const size_t b = (size_t)NWARP * pipe_bytes(ccap, S, vb);
            if (b <= (size_t)SMEM_CTA_MAX && (b + SMEM_CTA_RESERVE) * ctas <= SMEM_SM) return S;
        }
    return 0;
}

template <class F>
static void with_form(int form, F&& f) {
    switch (form) {
        case 0: f(std::integral_constant<int, 0>{}); break;
        case 1: f(std::integral_constant<int, 1>{}); break;
        case 2: f(std::integral_constant<int, 2>{}); break;
        case 3: f(std::integral_constant<int, 3>{}); break;
        case 4: f(std::integral_constant<int, 4>{}); break;
        case 6: f(std::integral_constant<int, 6>{}); break;
        case 7: f(std::integral_constant<int, 7>{}); break;
        default: f(std::integral_constant<int, 5>{}); break;
    }
}
// The persistent iteration kernel runs on the CSR arrays: a sliced layout
// (whose rows are also short) takes the direct form there.
static int fused_form(int form) { return sliced_form(form) ? 5 : form; }

// Compiled form, shared memory and CTAs per system of a layout's kernels.
// The warp pipeline needs a group capacity (pattern) and 16-byte aligned
// values (`aligned`); `vb` is the value size in bytes.  Every kernel that
// takes the layout's Mat is launched with L->smem.
// Producer/consumer form (FORM 4): shared memory of a CTA for tile capacity
// `tcap`, S stages, `vb`-byte values (gathered entries sized at 8 bytes).
static size_t ws_bytes(int tcap, int S, size_t vb) {
    return sizeof(WsHdr) + (size_t)S * tcap * (vb + sizeof(int) + sizeof(double));
}
// Most stages (4..2) with two resident CTAs per SM, else three or more stages
// with one; 0 when none fits.
static int ws_stages(int tcap, size_t vb) {
    for (int ctas = 2; ctas >= 1; --ctas)
        for (int S = MAX_STAGES; S >= (ctas == 2 ? 2 : 3); --S) {
            const size_t b = ws_bytes(tcap, S, vb);
            if (b <= (size_t)SMEM_CTA_MAX && (b + SMEM_CTA_RESERVE) * ctas <= SMEM_SM) return S;
        }
    return 0;
}

// Longest row the direct form (FORM 5, thread per row) takes; a matrix with
// longer rows uses the staged forms, whose warps share long rows (measured:
// the kNN Laplacian with 13-28 entries per row runs its product in half the
// time staged).
#ifndef SLA_DIRECT_MAXROW
#define SLA_DIRECT_MAXROW 16
#endif
// The same bound for the SPAI factors G and G^T.
#ifndef SLA_DIRECT_MAXROW_G
#define SLA_DIRECT_MAXROW_G SLA_DIRECT_MAXROW
#endif

template <typename T>
static sla_status set_form(const sla_csr* h, Layout* L, bool aligned, size_t vb,
                           int direct_maxrow = SLA_DIRECT_MAXROW) {
    const int wss = L->tcap > 0 && aligned && h->ws ? ws_stages(L->tcap, vb) : 0;
    L->stages = wss == 0 && L->ccap > 0 && aligned && h->pipeline ? pipe_stages(L->ccap, vb) : 0;
    const bool direct = !h->staged && L->maxrow <= direct_maxrow;
    if (wss == 0 && L->stages == 0 && direct) {
        L->form = 5;
        L->smem = 0;
    } else if (wss > 0) {
        L->form = 4;
        L->stages = wss;
        const size_t rows = (size_t)NWARP * L->cap * 2 * sizeof(double);   // warp staging of the check pass
        const size_t b = ws_bytes(L->tcap, wss, vb);
        L->smem = b > rows ? b : rows;
    } else if (L->stages > 0) {
        L->form = 3;
        L->smem = (size_t)NWARP * pipe_bytes(L->ccap, L->stages, vb);
    } else {
        L->form = staging_form(L->cap) == 0 ? 0 : (L->gasync ? 2 : 1);
        L->smem = spmv_smem(L->cap);
    }
    int per = 1;
    sla_status st = SLA_OK;
    with_form(L->form, [&](auto f) { st = occupancy(k_spmv_iter<T, decltype(f)::value>, L->smem, &per); });
    TRY(st);
    const long long units = L->form == 5   ? ((long long)h->n + NT - 1) / NT
                            : L->form == 4 ? ((long long)h->n + WS_ROWS - 1) / WS_ROWS
                                           : group_ctas(h->n, L->form == 3 ? 1 : L->lanes);
    L->gx = grid_x(h, units, per);
    return SLA_OK;
}

// direct_maxrow: longest row for which the direct form may be chosen (0: never).
static sla_status set_form_any(const sla_csr* h, Layout* L, bool aligned, size_t vb,
                               int direct_maxrow = SLA_DIRECT_MAXROW) {
    return h->dt == SLA_F64 ? set_form<double>(h, L, aligned, vb, direct_maxrow)
                            : set_form<float>(h, L, aligned, vb, direct_maxrow);
}

static bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }
// Values of every system 16-byte aligned (bulk copies of the forms 3 and 4).
static bool vals_aligned(const sla_csr* h, const void* vals) {
    return aligned16(vals) && (h->batch == 1 || ((size_t)h->nnz * h->es) % 16 == 0);
}

// Streaming kernels: two resident CTAs per SM, or SLA_VEC_CTAS_LARGE when
// every thread still makes at least SLA_VEC_TRIPS trips (pairs) at that
// occupancy.  Their per-CTA reduction tail and the fp64 work of each pair
// favour few, long-running threads on small systems; on large ones more
// loads in flight pay.  Measured on B300 inside the running iteration (it/s
// at 2 / 4 / 8 CTAs per SM): 2D 5-point 1M rows 22.1k / 20.3k / 18.0k
// (3.5 trips per thread at 4); 3D 7-point 2M rows 13.4k / 13.1k / 12.0k
// (6.9 trips); kNN SPAI 4M rows 1.78k / 1.82k / 1.80k (13.8 trips).  Two
// pairs per thread per trip (SLA_VU) did not help on any of them.
#ifndef SLA_VEC_CTAS
#define SLA_VEC_CTAS 2
#endif
#ifndef SLA_VEC_CTAS_LARGE
#define SLA_VEC_CTAS_LARGE 4
#endif
#ifndef SLA_VEC_TRIPS
#define SLA_VEC_TRIPS 8
#endif
static int gx_vec(const sla_csr* h) {
    const long long units = vec_units(h);   // CTAs if every thread took one pair
    const int large = grid_x(h, units, SLA_VEC_CTAS_LARGE);
    return units >= (long long)SLA_VEC_TRIPS * large ? large : grid_x(h, units, SLA_VEC_CTAS);
}

static Sys sys_of(sla_csr* h) {
    Sys s;
    s.n = h->n;
    s.nnz = h->nnz;
    s.st = h->state.as<State>();
    s.ctl = h->ctl.as<Ctrl>();
    s.cnt = h->cnt.as<unsigned>();
    s.part = h->part.as<double>();
    s.pstride = h->pstride;
    return s;
}

static Mat mat_of(const int* rp, const int* ci, int n, long long nnz, const Layout& L, int* err) {
    Mat m;
    m.rp = rp;
    m.ci = ci;
    m.n = n;
    m.cap = L.cap;
    m.async = staging_form(L.cap);
    // doubles of shared memory per warp (L.smem / NWARP)
    m.wstride = (int)(L.smem / NWARP / sizeof(double));
    m.lanes = L.form == 3 ? 1 : L.lanes;
    m.bal = L.bal && m.lanes == 1 && (L.form == 1 || L.form == 2) ? 1 : 0;
    m.swin = L.swin && sliced_form(L.form) ? 1 : 0;
    m.lshift = m.lanes == 4 ? 2 : (m.lanes == 2 ? 1 : 0);
    if (L.form == 3) m.cap = L.ccap;   // every group stages in the register-staged passes too
    m.nnz = nnz;
    m.ccap = L.form == 4 ? L.tcap : L.ccap;   // entries per stage of the bulk-copy forms
    m.stages = L.stages;
    m.err = err;
    // kernels on the CSR arrays take the direct form under a sliced layout
    m.direct = (L.form == 5 || sliced_form(L.form)) ? 1 : 0;
    m.sptr = L.sptr;
    m.sperm = L.sperm;
    m.scol = L.scol;
    m.nslices = L.nslices;
    m.vstride = L.vstride;
    return m;
}
static Mat mat_A(const sla_csr* h) { return mat_of(h->rp, h->ci, h->n, h->nnz, h->LA, &h->ctl.as<Ctrl>()->err); }
static Mat mat_I(const sla_csr* h) { return mat_of(h->irp, h->ici, h->n, h->nnz, h->LI, &h->ctl.as<Ctrl>()->err); }
static Mat mat_G(const sla_csr* h) {
    return mat_of(h->grp.as<int>(), h->gci.as<int>(), h->n, h->nnzg, h->LG, &h->ctl.as<Ctrl>()->err);
}
static Mat mat_GT(const sla_csr* h) {
    return mat_of(h->gtrp.as<int>(), h->gtci.as<int>(), h->n, h->nnzg, h->LGT, &h->ctl.as<Ctrl>()->err);
}

// ===================================================================== set-up helpers
static sla_status scan_exclusive(int* d, long long m, cudaStream_t s) {
    const long long nb = (m + SCAN_TILE - 1) / SCAN_TILE;
    if (nb <= 1) {
        k_scan_tile<<<1, SCAN_T, 0, s>>>(d, m, nullptr);
        return launched();
    }
    DevBuf sums;
    TRY(sums.alloc(sizeof(int) * (size_t)nb));
    k_scan_tile<<<(unsigned)nb, SCAN_T, 0, s>>>(d, m, sums.as<int>());
    TRY(launched());
    TRY(scan_exclusive(sums.as<int>(), nb, s));
    k_scan_add<<<(unsigned)nb, SCAN_T, 0, s>>>(d, m, sums.as<int>());
    TRY(launched());
    CU(cudaStreamSynchronize(s));
    return SLA_OK;
}

static sla_status read_int(const int* d, int* out, cudaStream_t s) {
    CU(cudaMemcpyAsync(out, d, sizeof(int), cudaMemcpyDeviceToHost, s));
    CU(cudaStreamSynchronize(s));
    return SLA_OK;
}

static sla_status group_max(const int* rp, int n, int rows, int* out, cudaStream_t s) {
    DevBuf m;
    TRY(m.alloc(sizeof(int)));
    CU(cudaMemsetAsync(m.p, 0, sizeof(int), s));
    const long long ng = ((long long)n + rows - 1) / rows;
    const int g = (ng + 255) / 256 < 2048 ? (int)((ng + 255) / 256) : 2048;
    k_group_max<<<g, 256, 0, s>>>(rp, n, rows, m.as<int>());
    TRY(launched());
    TRY(read_int(m.as<int>(), out, s));
    return SLA_OK;
}

// One lane per row whenever a 32-row group fits a stage (up to MAX_CAP
// entries; the staging form follows from the capacity); otherwise the fewest
// lanes per row whose groups fit.  Measured on B300: for ~15-entry rows
// (kNN graphs) one lane per row with single-stage staging beats two lanes
// per row with pipelined staging.
// Scattered columns: more than 10% of the entries lie farther than 64K
// columns from their row (a 512 KB window of an fp64 vector).
static constexpr int NEAR_WINDOW = 65536;

// Split sums of the staged groups (balanced_group_sum) when the lane-per-row
// walk would take at least SLA_SPLIT_RATIO times the warp-wide fp64 steps
// (k_walk_cost), one lane per row only.  Measured on B300 (product of 4M
// rows, staged form 1): at ratios 1.36 and 1.54 the split product took 2-3%
// longer (its serial chain per group -- row search, unrollable walk, joins
// -- is longer, and the fp64 pipe is not what bounds these products), at
// 2.0 2.5% less, at 2.7, 3.3 and 4.4 22%, 26% and 60% less (groups with a
// few long rows).  The SPAI factors of the reordered kNN Laplacian (about
// 1.3) keep the lane-per-row walk.
#ifndef SLA_SPLIT_RATIO
#define SLA_SPLIT_RATIO 1.8
#endif
static sla_status choose_split(const sla_csr* h, const int* rp, Layout* L, cudaStream_t s) {
    L->bal = 0;
    if (L->lanes != 1 || h->split < 0) return SLA_OK;
    if (h->split > 0) {
        L->bal = 1;
        return SLA_OK;
    }
    DevBuf w;
    TRY(w.alloc(2 * sizeof(unsigned long long)));
    CU(cudaMemsetAsync(w.p, 0, 2 * sizeof(unsigned long long), s));
    const long long ng = ((long long)h->n + 31) / 32;
    const int g = (ng + 255) / 256 < 2048 ? (int)((ng + 255) / 256) : 2048;
    k_walk_cost<<<g, 256, 0, s>>>(rp, h->n, w.as<unsigned long long>());
    TRY(launched());
    unsigned long long c[2] = {0, 0};
    CU(cudaMemcpyAsync(c, w.p, sizeof c, cudaMemcpyDeviceToHost, s));
    CU(cudaStreamSynchronize(s));
    L->bal = c[1] > 0 && (double)c[0] >= SLA_SPLIT_RATIO * (double)c[1] ? 1 : 0;
    return SLA_OK;
}

static sla_status choose_layout(const sla_csr* h, const int* rp, const int* ci, long long nnz, Layout* L,
                                bool aligned, size_t vb, cudaStream_t s, int direct_maxrow = SLA_DIRECT_MAXROW,
                                int min_lanes = SLA_MIN_LANES, int max_cap = MAX_CAP) {
    {
        DevBuf far;
        TRY(far.alloc(sizeof(unsigned long long)));
        CU(cudaMemsetAsync(far.p, 0, sizeof(unsigned long long), s));
        const int g = (h->n + 255) / 256 < 2048 ? (h->n + 255) / 256 : 2048;
        k_far_count<<<g, 256, 0, s>>>(rp, ci, h->n, NEAR_WINDOW, far.as<unsigned long long>());
        TRY(launched());
        unsigned long long f = 0;
        CU(cudaMemcpyAsync(&f, far.p, sizeof f, cudaMemcpyDeviceToHost, s));
        CU(cudaStreamSynchronize(s));
        L->gasync = (double)f > 0.1 * (double)nnz ? 1 : 0;
    }
    TRY(group_max(rp, h->n, 1, &L->maxrow, s));
    for (int lanes = min_lanes; lanes <= 4; lanes *= 2) {
        int m = 0;
        TRY(group_max(rp, h->n, 32 / lanes, &m, s));
        int cap = (m + 31) / 32 * 32;
        if (cap < 32) cap = 32;
        if (cap <= max_cap || lanes == 4) {
            L->cap = cap > max_cap ? max_cap : cap;
            L->lanes = lanes;
            break;
        }
    }
    TRY(choose_split(h, rp, L, s));
    // warp pipeline: largest group of 32 rows, as staged
    L->ccap = 0;
    if (aligned16(rp) && aligned16(ci)) {
        DevBuf m;
        TRY(m.alloc(sizeof(int)));
        CU(cudaMemsetAsync(m.p, 0, sizeof(int), s));
        const long long nc = ((long long)h->n + 31) / 32;
        const int g = (nc + 255) / 256 < 2048 ? (int)((nc + 255) / 256) : 2048;
        k_chunk_max<<<g, 256, 0, s>>>(rp, h->n, 32, m.as<int>());
        TRY(launched());
        int cc = 0;
        TRY(read_int(m.as<int>(), &cc, s));
        L->ccap = cc < 4 ? 4 : cc;
        // producer/consumer form: largest tile of WS_ROWS rows, as staged
        CU(cudaMemsetAsync(m.p, 0, sizeof(int), s));
        const long long nt = ((long long)h->n + WS_ROWS - 1) / WS_ROWS;
        const int gt = (nt + 255) / 256 < 2048 ? (int)((nt + 255) / 256) : 2048;
        k_chunk_max<<<gt, 256, 0, s>>>(rp, h->n, WS_ROWS, m.as<int>());
        TRY(launched());
        int tc = 0;
        TRY(read_int(m.as<int>(), &tc, s));
        L->tcap = tc < 4 ? 4 : tc;
    }
    return set_form_any(h, L, aligned, vb, direct_maxrow);
}

// ===================================================================== reordering
// Reverse Cuthill-McKee order of a pattern read as a graph (row i adjacent
// to the columns of its stored entries): each connected part is walked
// breadth-first from a pseudo-peripheral row (George-Liu search from a row
// of least degree), unvisited neighbours in order of increasing degree,
// and the whole order is reversed.  perm[new] = old.
static void rcm_order(int n, const std::vector<int>& rp, const std::vector<int>& ci, std::vector<int>& perm) {
    std::vector<int> deg(n);
    for (int i = 0; i < n; ++i) deg[i] = rp[i + 1] - rp[i];
    std::vector<int> by_deg(n);
    for (int i = 0; i < n; ++i) by_deg[i] = i;
    std::stable_sort(by_deg.begin(), by_deg.end(), [&](int a, int b) { return deg[a] < deg[b]; });
    std::vector<char> seen(n, 0);
    std::vector<int> stamp(n, -1), queue;
    queue.reserve(n);
    std::vector<int> order;
    order.reserve(n);
    int pass = 0;
    // breadth-first levels from `root` inside its part (without marking
    // `seen`); returns the depth and a least-degree row of the last level
    auto last_level = [&](int root, int& far) {
        ++pass;
        queue.clear();
        queue.push_back(root);
        stamp[root] = pass;
        size_t head = 0;
        int depth = 0;
        while (head < queue.size()) {
            const size_t end = queue.size();
            far = queue[head];
            for (size_t k = head; k < end; ++k)
                if (deg[queue[k]] < deg[far]) far = queue[k];
            for (; head < end; ++head) {
                const int u = queue[head];
                for (int k = rp[u]; k < rp[u + 1]; ++k) {
                    const int v = ci[k];
                    if (stamp[v] != pass && !seen[v]) {
                        stamp[v] = pass;
                        queue.push_back(v);
                    }
                }
            }
            if (queue.size() > end) ++depth;
        }
        return depth;
    };
    std::vector<std::pair<int, int>> nb;
    for (int start : by_deg) {
        if (seen[start]) continue;
        int root = start, far = start;
        int depth = last_level(root, far);
        for (int it = 0; it < 4; ++it) {   // move to a farther row while the depth grows
            int far2 = far;
            const int d2 = last_level(far, far2);
            if (d2 <= depth) break;
            root = far;
            depth = d2;
            far = far2;
        }
        const size_t base = order.size();
        order.push_back(root);
        seen[root] = 1;
        for (size_t head = base; head < order.size(); ++head) {
            const int u = order[head];
            nb.clear();
            for (int k = rp[u]; k < rp[u + 1]; ++k) {
                const int v = ci[k];
                if (!seen[v]) {
                    seen[v] = 1;
                    nb.emplace_back(deg[v], v);
                }
            }
            std::sort(nb.begin(), nb.end());
            for (const auto& e : nb) order.push_back(e.second);
        }
    }
    perm.assign(order.rbegin(), order.rend());
}

// Pattern of P M P^T for perm[new] = old: row i' is old row perm[i'] with
// every column c renamed iperm[c], columns ascending; src[k'] = the entry
// of M that permuted entry k' holds.  Rows are filled by several threads.
static void permute_pattern(int n, const std::vector<int>& rp, const std::vector<int>& ci,
                            const std::vector<int>& perm, const std::vector<int>& iperm, std::vector<int>& rp2,
                            std::vector<int>& ci2, std::vector<int>& src) {
    rp2.assign(n + 1, 0);
    for (int i = 0; i < n; ++i) rp2[i + 1] = rp2[i] + (rp[perm[i] + 1] - rp[perm[i]]);
    ci2.resize(ci.size());
    src.resize(ci.size());
    const int nt = std::max(1, std::min(16, (int)std::thread::hardware_concurrency()));
    std::vector<std::thread> pool;
    for (int t = 0; t < nt; ++t)
        pool.emplace_back([&, t] {
            std::vector<std::pair<int, int>> row;
            for (int i = t; i < n; i += nt) {
                const int o = perm[i];
                row.clear();
                for (int k = rp[o]; k < rp[o + 1]; ++k) row.emplace_back(iperm[ci[k]], k);
                std::sort(row.begin(), row.end());
                for (size_t j = 0; j < row.size(); ++j) {
                    ci2[rp2[i] + j] = row[j].first;
                    src[rp2[i] + j] = row[j].second;
                }
            }
        });
    for (auto& th : pool) th.join();
}

static sla_status to_host(std::vector<int>& out, const int* d, size_t m) {
    out.resize(m);
    if (m) CU(cudaMemcpy(out.data(), d, sizeof(int) * m, cudaMemcpyDeviceToHost));
    return SLA_OK;
}
static sla_status to_device(DevBuf& buf, const std::vector<int>& v) {
    TRY(buf.alloc(sizeof(int) * (v.empty() ? 1 : v.size())));
    if (!v.empty()) CU(cudaMemcpy(buf.p, v.data(), sizeof(int) * v.size(), cudaMemcpyHostToDevice));
    return SLA_OK;
}

// out[s][k] = in[s][map[k]] for k < m, systems strided by `is` / `os`
// elements of `eb` bytes (8: fp64 or a double-float pair; 4: fp32).
static sla_status gather_map(size_t eb, long long m, int batch, const int* map, const void* in, long long is,
                             void* out, long long os, cudaStream_t s) {
    if (m == 0) return SLA_OK;
    const long long tot = m * batch;
    const int g = (int)std::min<long long>((tot + 255) / 256, 8192);
    if (eb == 8)
        k_gather_map<double><<<g, 256, 0, s>>>(m, batch, map, (const double*)in, is, (double*)out, os);
    else
        k_gather_map<float><<<g, 256, 0, s>>>(m, batch, map, (const float*)in, is, (float*)out, os);
    return launched();
}

// ===================================================================== sliced copies
// Rows per window whose slots may be reordered by length: the smallest of
// one, four or sixteen CTAs' slices in one trip of the sliced kernels
// (NWARP slices of 32 rows each) that pads at most SLICE_GOOD_PAD (else the
// least padding), so the rows a window's results go to are written by few
// CTAs at about the same time.  On the kNN Laplacian one CTA's 256 rows pad
// A by 4%, but the SPAI factor (whose row lengths vary most) by 15.5%; 1024
// rows pad it by 4%.
static constexpr int SLICE_WINDOWS[3] = {NWARP * 32, 4 * NWARP * 32, 16 * NWARP * 32};
#ifndef SLA_SLICE_WINDOW_LAST
#define SLA_SLICE_WINDOW_LAST 2   // largest window tried (index into SLICE_WINDOWS)
#endif
#ifndef SLA_SLICE_WIN_EPI
#define SLA_SLICE_WIN_EPI 1       // window-sorted sliced layouts run a warp per window (spmv_sliced_win)
#endif
static_assert(SLICE_WINDOWS[0] == SLICE_WIN, "the smallest sorting window is the kernels' window");
static constexpr double SLICE_GOOD_PAD = 1.06;
// Patterns whose rows hold more than 16 entries take the sliced form by
// default when they hold at least this many on average.
#ifndef SLA_SLICED_MINAVG
#define SLA_SLICED_MINAVG 12.0
#endif
// Sliced rows of at least this many entries on average take the form for 4
// resident CTAs per SM and batches of SLICE_U (6), shorter ones the one for
// 5 and batches of 7 (7).  Measured on B300: 3D 7-point (6.97 entries) form
// 7; kNN Laplacian (14.6) form 6; its SPAI factors (7.8 entries): with form
// 6 in batches of 4, G^T alone sliced, form 6 1.87k CG iterations/s against
// 1.86k; with batches of 6 and both factors sliced, form 7 2.15k against
// 2.12-2.13k.
#ifndef SLA_SLICED_FORM6_MINAVG
#define SLA_SLICED_FORM6_MINAVG 8.0
#endif
// Largest padding (sliced entries / stored entries) for which the sliced
// form is used; for the SPAI factors by default (windows of 256 rows).
#ifndef SLA_SLICED_MAXPAD
#define SLA_SLICED_MAXPAD 1.15
#endif
#ifndef SLA_SLICED_MAXPAD_FACTORS
#define SLA_SLICED_MAXPAD_FACTORS 1.2
#endif

// values: the CSR values the sliced copy mirrors ([batch][is] of eb bytes).
static sla_status sliced_values(const sla_csr* h, SellBufs& B, const void* vals, long long is, size_t eb,
                                cudaStream_t s) {
    if (B.npad == 0) return SLA_OK;
    const long long tot = B.npad * h->batch;
    const int g = (int)std::min<long long>((tot + 255) / 256, 8192);
    if (eb == 8)
        k_gather_map_pad<unsigned long long><<<g, 256, 0, s>>>(B.npad, h->batch, B.smap.as<int>(),
                                                               (const unsigned long long*)vals, is,
                                                               B.sval.as<unsigned long long>(), B.vstride);
    else
        k_gather_map_pad<unsigned><<<g, 256, 0, s>>>(B.npad, h->batch, B.smap.as<int>(), (const unsigned*)vals, is,
                                                     B.sval.as<unsigned>(), B.vstride);
    return launched();
}

// Build the sliced copy of the pattern (rp, ci; nnz entries) and its values
// and switch L to form 6, when the padding stays within SLA_SLICED_MAXPAD;
// otherwise leave L as it is.  Within every window of SLICE_WINDOWS rows the
// rows are ordered by decreasing length when that pads less (the slot ->
// row map is then kept); the kernels write each row's result to its own
// row, so the iteration order is unchanged.
template <typename T>
static sla_status make_sliced(sla_csr* h, const int* d_rp, const int* d_ci, long long nnz, const void* vals,
                              long long is, size_t eb, Layout* L, SellBufs& B, cudaStream_t s,
                              int last_window, double max_pad) {
    const int n = h->n;
    if (nnz == 0 || n < 1) return SLA_OK;
    std::vector<int> rp;
    CU(cudaStreamSynchronize(s));
    TRY(to_host(rp, d_rp, (size_t)n + 1));
    const int nslices = (int)(((long long)n + 31) / 32);
    const long long slots = (long long)nslices * 32;
    auto len = [&](long long r) { return r < n ? rp[r + 1] - rp[r] : 0; };
    // padding of the identity order and of the window-sorted order
    long long pad_id = 0;
    for (int sl = 0; sl < nslices; ++sl) {
        int w = 0;
        for (int l = 0; l < 32; ++l) w = std::max(w, len((long long)sl * 32 + l));
        pad_id += 32LL * w;
    }
    std::vector<int> perm, sptr;
    long long pad_sorted = 0;
    int sort_window = 0;
    for (int wi = 0; wi <= last_window; ++wi) {
        const int window = SLICE_WINDOWS[wi];
        std::vector<int> pw(slots), sw(nslices + 1, 0);
        for (long long t = 0; t < slots; ++t) pw[t] = t < n ? (int)t : n;
        for (long long w0 = 0; w0 < n; w0 += window) {
            const long long w1 = std::min<long long>(w0 + window, n);
            std::stable_sort(pw.begin() + w0, pw.begin() + w1, [&](int a, int b) { return len(a) > len(b); });
        }
        for (int sl = 0; sl < nslices; ++sl) {
            int w = 0;
            for (int l = 0; l < 32; ++l) w = std::max(w, len(pw[(size_t)sl * 32 + l]));
            sw[sl + 1] = (int)std::min<long long>((long long)sw[sl] + 32LL * w, 0x7fffffffLL);
        }
        if (perm.empty() || sw[nslices] < pad_sorted) {
            perm.swap(pw);
            sptr.swap(sw);
            pad_sorted = sptr[nslices];
            sort_window = window;
        }
        if ((double)pad_sorted <= SLICE_GOOD_PAD * (double)nnz) break;
    }
    const bool sorted = pad_sorted < pad_id && (double)pad_id > 1.02 * (double)nnz;
    const long long npad = sorted ? pad_sorted : pad_id;
    if ((double)npad > max_pad * (double)nnz || npad >= 0x7fffffffLL) return SLA_OK;
    if (!sorted) {
        for (int sl = 0; sl < nslices; ++sl) {
            int w = 0;
            for (int l = 0; l < 32; ++l) w = std::max(w, len((long long)sl * 32 + l));
            sptr[sl + 1] = sptr[sl] + 32 * w;
        }
    }
    B.release();
    TRY(to_device(B.sptr, sptr));
    if (sorted) TRY(to_device(B.perm, perm));
    TRY(B.scol.alloc(sizeof(int) * (size_t)npad));
    TRY(B.smap.alloc(sizeof(int) * (size_t)npad));
    B.npad = npad;
    B.vstride = (npad + 1) & ~1LL;   // 16-byte aligned systems
    B.nslices = nslices;
    {
        const int g = (int)std::min<long long>((slots + 255) / 256, 8192);
        k_sell_fill<<<g, 256, 0, s>>>(n, nslices, d_rp, d_ci, B.sptr.as<int>(), sorted ? B.perm.as<int>() : nullptr,
                                      B.scol.as<int>(), B.smap.as<int>());
        TRY(launched());
    }
    TRY(B.sval.alloc(eb * (size_t)B.vstride * h->batch));
    TRY(sliced_values(h, B, vals, is, eb, s));
    // the sliced form for 4 resident CTAs per SM (6) for long rows, for 5 (7)
    // for rows of fewer than SLA_SLICED_FORM6_MINAVG entries on average
    const int form = (double)nnz >= SLA_SLICED_FORM6_MINAVG * (double)n ? 6 : 7;
    // rows sorted within windows of SLICE_WIN rows: a warp per window, the
    // epilogue in row order (spmv_sliced_win), SLICE_WIN sums per warp
    L->swin = SLA_SLICE_WIN_EPI && sorted && sort_window == SLICE_WIN ? 1 : 0;
    L->smem = L->swin ? (size_t)NWARP * SLICE_WIN * sizeof(double) : 0;
    int per = 1;
    if (form == 6) TRY(occupancy(k_spmv_iter<T, 6>, L->smem, &per));
    else TRY(occupancy(k_spmv_iter<T, 7>, L->smem, &per));
    L->form = form;
    L->sptr = B.sptr.as<int>();
    L->sperm = sorted ? B.perm.as<int>() : nullptr;
    L->scol = B.scol.as<int>();
    L->sval = B.sval.p;
    L->nslices = nslices;
    L->vstride = B.vstride;
    L->gx = grid_x(h, (slots + NT - 1) / NT, per);
    return SLA_OK;
}

// Default choice of the sliced form for the iteration matrix (measured on
// B300 inside the running iteration): rows too long for the direct form and
// long enough on average (the kNN Laplacian, 14.6 entries per row: 192
// against 238 us staged), or short rows of at least 4.5 on average (the 3D
// 7-point grid: 51.4 against 55.7 us direct, at 5 CTAs per SM; the 2D
// 5-point grid, once a slot's last entries went as one batch: 25.0 against
// 26.6 us, and 53.9 against 68.5 us for 64 fp32 systems on one 256^2 grid);
// the direct form stays for shorter rows.  (The 64^2 5-point grid, launch
// bound, measured 57.2k against 58.2k CG iterations/s sliced.)  The SPAI
// factors take their own rule (build_spai).
#ifndef SLA_SLICED_MINAVG_SHORT
#define SLA_SLICED_MINAVG_SHORT 4.5
#endif
static bool sliced_by_default(const sla_csr* h, const Layout& L, long long nnz) {
    const double avg = (double)nnz / (double)h->n;
    if (L.maxrow > SLA_DIRECT_MAXROW) return avg >= SLA_SLICED_MINAVG;
    return avg >= SLA_SLICED_MINAVG_SHORT;
}

static sla_status make_sliced_any(sla_csr* h, const int* d_rp, const int* d_ci, long long nnz, const void* vals,
                                  long long is, size_t eb, Layout* L, SellBufs& B, cudaStream_t s,
                                  int last_window = SLA_SLICE_WINDOW_LAST, double max_pad = SLA_SLICED_MAXPAD) {
    return h->dt == SLA_F64 ? make_sliced<double>(h, d_rp, d_ci, nnz, vals, is, eb, L, B, s, last_window, max_pad)
                            : make_sliced<float>(h, d_rp, d_ci, nnz, vals, is, eb, L, B, s, last_window, max_pad);
}

// Iterate on P A P^T (reverse Cuthill-McKee): permuted pattern and values
// owned by the handle, with the permutation both ways.
static sla_status make_reordered(sla_csr* h, cudaStream_t s) {
    const int n = h->n;
    std::vector<int> rp, ci, perm, iperm, rp2, ci2, src;
    CU(cudaStreamSynchronize(s));
    TRY(to_host(rp, h->rp, (size_t)n + 1));
    TRY(to_host(ci, h->ci, (size_t)h->nnz));
    rcm_order(n, rp, ci, perm);
    iperm.resize(n);
    for (int i = 0; i < n; ++i) iperm[perm[i]] = i;
    permute_pattern(n, rp, ci, perm, iperm, rp2, ci2, src);
    TRY(to_device(h->perm, perm));
    TRY(to_device(h->iperm, iperm));
    TRY(to_device(h->prp, rp2));
    TRY(to_device(h->pci, ci2));
    TRY(to_device(h->psrc, src));
    TRY(h->pvals.alloc(h->es * (size_t)h->nnz * h->batch));
    TRY(gather_map(h->es, h->nnz, h->batch, h->psrc.as<int>(), h->vals, h->nnz, h->pvals.p, h->nnz, s));
    TRY(h->ptmp.alloc(2 * h->es * (size_t)n * h->batch));
    h->irp = h->prp.as<int>();
    h->ici = h->pci.as<int>();
    h->ivals = h->pvals.p;
    h->reordered = true;
    return SLA_OK;
}

static sla_status compute_diag(sla_csr* h, cudaStream_t s) {
    if (!h->derr.p) TRY(h->derr.alloc(sizeof(int)));
    DevBuf& err = h->derr;
    CU(cudaMemsetAsync(err.p, 0, sizeof(int), s));
    const int g = (h->n + 255) / 256 < 4096 ? (h->n + 255) / 256 : 4096;
    if (h->dt == SLA_F64)
        k_diag<double><<<g, 256, 0, s>>>(h->n, h->nnz, h->batch, h->irp, h->ici, (const double*)h->ivals,
                                         h->diag.as<double>(), err.as<int>());
    else
        k_diag<float><<<g, 256, 0, s>>>(h->n, h->nnz, h->batch, h->irp, h->ici, (const float*)h->ivals,
                                        h->diag.as<double>(), err.as<int>());
    TRY(launched());
    const size_t m = (size_t)h->batch * h->n;
    if (h->dt == SLA_F64) k_recip<double><<<4096, 256, 0, s>>>(m, h->diag.as<double>(), h->dinv.as<double>());
    else k_recip<float2><<<4096, 256, 0, s>>>(m, h->diag.as<double>(), h->dinv.as<float2>());
    TRY(launched());
    TRY(read_int(err.as<int>(), &h->diag_err, s));
    return SLA_OK;
}


static sla_status ensure_pstride(sla_csr* h);

// Values of G and G^T from the current values of A (on the caller's
// ordering, where G is defined), then -- unless fill_only -- for a reordered
// handle gathered into the permuted factors, and into their sliced copies.
// The patterns, permutation maps and layouts were built once by build_spai
// (which calls this with fill_only before the maps exist).
static sla_status spai_values(sla_csr* h, cudaStream_t s, bool fill_only = false) {
    if (h->diag_err & ERR_NO_DIAG) return fail(SLA_ERR_INVALID, "SPAI needs every diagonal entry stored");
    if (h->diag_err & ERR_DIAG_SIGN) return fail(SLA_ERR_INVALID, "SPAI needs a positive diagonal");
    const int n = h->n;
    const int g = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    if (!h->derr.p) TRY(h->derr.alloc(sizeof(int)));
    DevBuf& err = h->derr;
    CU(cudaMemsetAsync(err.p, 0, sizeof(int), s));
    DevBuf& dorig = h->dorig;
    const double* dbase = h->diag.as<double>();
    if (h->reordered) {
        if (dorig.bytes < sizeof(double) * (size_t)n * h->batch) TRY(dorig.alloc(sizeof(double) * (size_t)n * h->batch));
        TRY(gather_map(8, n, h->batch, h->iperm.as<int>(), h->diag.p, n, dorig.p, n, s));
        dbase = dorig.as<double>();
    }
    // caller-ordered factors: the final ones, or the sources of the permuted ones
    DevBuf& grp = h->reordered ? h->grp0 : h->grp;
    DevBuf& gci = h->reordered ? h->gci0 : h->gci;
    DevBuf& gvb = h->reordered ? h->gv0 : h->gv;
    DevBuf& gtrp = h->reordered ? h->gtrp0 : h->gtrp;
    DevBuf& gtci = h->reordered ? h->gtci0 : h->gtci;
    DevBuf& gtvb = h->reordered ? h->gtv0 : h->gtv;
    if (h->drs.bytes < sizeof(double) * (size_t)n * h->batch) TRY(h->drs.alloc(sizeof(double) * (size_t)n * h->batch));
    {
        const long long m = (long long)n * h->batch;
        const int gr = (int)std::min<long long>((m + 255) / 256, 4096);
        k_rsqrt_diag<<<gr, 256, 0, s>>>((int)m, dbase, h->drs.as<double>());
        TRY(launched());
    }
    // positions of G^T's values in A, found by the first fill (system 0)
    const bool have_pos = h->gtpos.p != nullptr && h->gtpos.bytes >= sizeof(int) * (size_t)h->nnzg;
    if (!have_pos) TRY(h->gtpos.alloc(sizeof(int) * (size_t)(h->nnzg > 0 ? h->nnzg : 1)));
    for (int sy = 0; sy < h->batch; ++sy) {
        const double* dg = h->drs.as<double>() + (size_t)sy * n;
        double* gv = gvb.as<double>() + (size_t)sy * h->gstride;     // 8-byte slots: fp64, or a
        double* gtv = gtvb.as<double>() + (size_t)sy * h->gstride;   // double-float pair for fp32
        if (h->dt == SLA_F64) {
            const double* av = (const double*)h->vals + (size_t)sy * h->nnz;
            k_fill_G<double, double><<<g, 256, 0, s>>>(n, h->rp, h->ci, av, dg, grp.as<int>(), gci.as<int>(), gv);
            TRY(launched());
            k_fill_GT<double, double><<<g, 256, 0, s>>>(n, h->rp, h->ci, av, dg, gtrp.as<int>(), gtci.as<int>(), gtv,
                                                        h->gtpos.as<int>(), have_pos, err.as<int>());
        } else {
            const float* av = (const float*)h->vals + (size_t)sy * h->nnz;
            k_fill_G<float, float2><<<g, 256, 0, s>>>(n, h->rp, h->ci, av, dg, grp.as<int>(), gci.as<int>(),
                                                      reinterpret_cast<float2*>(gv));
            TRY(launched());
            k_fill_GT<float, float2><<<g, 256, 0, s>>>(n, h->rp, h->ci, av, dg, gtrp.as<int>(), gtci.as<int>(),
                                                       reinterpret_cast<float2*>(gtv), h->gtpos.as<int>(), have_pos, err.as<int>());
        }
        TRY(launched());
    }
    int e = 0;
    TRY(read_int(err.as<int>(), &e, s));
    if (e & ERR_ASYM) return fail(SLA_ERR_INVALID, "SPAI needs a structurally symmetric matrix");
    if (fill_only) return SLA_OK;
    if (h->reordered) {
        TRY(gather_map(8, h->nnzg, h->batch, h->gsrc.as<int>(), h->gv0.p, h->gstride, h->gv.p, h->gstride, s));
        TRY(gather_map(8, h->nnzg, h->batch, h->gtsrc.as<int>(), h->gtv0.p, h->gstride, h->gtv.p, h->gstride, s));
    }
    if (sliced_form(h->LG.form)) TRY(sliced_values(h, h->sG, h->gv.p, h->gstride, 8, s));
    if (sliced_form(h->LGT.form)) TRY(sliced_values(h, h->sGT, h->gtv.p, h->gstride, 8, s));
    h->spai_stale = false;
    return SLA_OK;
}

// The SPAI factor's patterns (G on tril(A) and its explicit transpose, on
// the caller's ordering; for a reordered handle also permuted like A, with
// the source entry of every permuted entry) and layouts, once per handle;
// then its values.
// Work units (warps' groups, tiles, thread rows or slices, in CTAs of NT
// threads) of a layout's product kernels.
static long long layout_units(const sla_csr* h, const Layout& L) {
    if (sliced_form(L.form)) return ((long long)L.nslices * 32 + NT - 1) / NT;
    if (L.form == 5) return ((long long)h->n + NT - 1) / NT;
    if (L.form == 4) return ((long long)h->n + WS_ROWS - 1) / WS_ROWS;
    return group_ctas(h->n, L.form == 3 ? 1 : L.lanes);
}

// The SPAI products take their grids from their own kernels' occupancy,
// in the staged forms at most SLA_SPAI_CTAS resident CTAs per SM (their
// staging shared memory competes with L1).  Measured on B300 (SPAI
// factors of the reordered kNN Laplacian, 4M rows, staged form 1): 3 CTAs
// per SM 1.78k CG iterations/s; 4 (k_spai_t fits 4 by its own occupancy)
// 1.73k -- the staging shared memory then leaves too little L1 for the
// gathered vector; 2 1.66k.
#ifndef SLA_SPAI_CTAS
#define SLA_SPAI_CTAS 3
#endif
static int spai_ctas(const Layout& L, int per) {
    return L.form <= 4 && per > SLA_SPAI_CTAS ? SLA_SPAI_CTAS : per;
}
template <typename T>
static sla_status spai_grids(sla_csr* h) {
    int per = 1;
    sla_status st = SLA_OK;
    with_form(h->LGT.form, [&](auto f) { st = occupancy(k_spai_t<T, decltype(f)::value>, h->LGT.smem, &per); });
    TRY(st);
    h->LGT.gx = grid_x(h, layout_units(h, h->LGT), spai_ctas(h->LGT, per));
    with_form(h->LG.form, [&](auto f) { st = occupancy(k_spai_z<T, decltype(f)::value>, h->LG.smem, &per); });
    TRY(st);
    h->LG.gx = grid_x(h, layout_units(h, h->LG), spai_ctas(h->LG, per));
    return SLA_OK;
}

static sla_status build_spai(sla_csr* h, cudaStream_t s) {
    if (h->diag_err & ERR_NO_DIAG) return fail(SLA_ERR_INVALID, "SPAI needs every diagonal entry stored");
    if (h->diag_err & ERR_DIAG_SIGN) return fail(SLA_ERR_INVALID, "SPAI needs a positive diagonal");
    const int n = h->n;
    DevBuf& grp = h->reordered ? h->grp0 : h->grp;
    DevBuf& gtrp = h->reordered ? h->gtrp0 : h->gtrp;
    TRY(grp.alloc(sizeof(int) * (size_t)(n + 1)));
    TRY(gtrp.alloc(sizeof(int) * (size_t)(n + 1)));
    const int g = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
    k_tri_count<<<g, 256, 0, s>>>(n, h->rp, h->ci, grp.as<int>(), gtrp.as<int>());
    TRY(launched());
    CU(cudaMemsetAsync(grp.as<int>() + n, 0, sizeof(int), s));
    CU(cudaMemsetAsync(gtrp.as<int>() + n, 0, sizeof(int), s));
    TRY(scan_exclusive(grp.as<int>(), n + 1, s));
    TRY(scan_exclusive(gtrp.as<int>(), n + 1, s));
    int ng = 0, ngt = 0;
    TRY(read_int(grp.as<int>() + n, &ng, s));
    TRY(read_int(gtrp.as<int>() + n, &ngt, s));
    if (ng != ngt) return fail(SLA_ERR_INVALID, "SPAI needs a structurally symmetric matrix");
    h->nnzg = ng;
    h->gstride = ((long long)ng + 1) & ~1LL;
    DevBuf& gci = h->reordered ? h->gci0 : h->gci;
    DevBuf& gtci = h->reordered ? h->gtci0 : h->gtci;
    TRY(gci.alloc(sizeof(int) * (size_t)ng));
    TRY(gtci.alloc(sizeof(int) * (size_t)ng));
    TRY(h->gv.alloc(sizeof(double) * (size_t)h->gstride * h->batch));
    TRY(h->gtv.alloc(sizeof(double) * (size_t)h->gstride * h->batch));
    if (h->reordered) {
        TRY(h->gv0.alloc(sizeof(double) * (size_t)h->gstride * h->batch));
        TRY(h->gtv0.alloc(sizeof(double) * (size_t)h->gstride * h->batch));
    }
    TRY(spai_values(h, s, true));   // fills the caller-ordered patterns too
    if (h->reordered) {
        std::vector<int> perm, iperm;
        TRY(to_host(perm, h->perm.as<int>(), (size_t)n));
        iperm.resize(n);
        for (int i = 0; i < n; ++i) iperm[perm[i]] = i;
        DevBuf* pats[2][4] = {{&h->grp0, &h->gci0, &h->grp, &h->gci}, {&h->gtrp0, &h->gtci0, &h->gtrp, &h->gtci}};
        DevBuf* srcs[2] = {&h->gsrc, &h->gtsrc};
        for (int f = 0; f < 2; ++f) {
            std::vector<int> rp, ci, rp2, ci2, src;
            TRY(to_host(rp, pats[f][0]->as<int>(), (size_t)n + 1));
            TRY(to_host(ci, pats[f][1]->as<int>(), (size_t)ng));
            permute_pattern(n, rp, ci, perm, iperm, rp2, ci2, src);
            TRY(to_device(*pats[f][2], rp2));
            TRY(to_device(*pats[f][3], ci2));
            TRY(to_device(*srcs[f], src));
        }
        TRY(gather_map(8, ng, h->batch, h->gsrc.as<int>(), h->gv0.p, h->gstride, h->gv.p, h->gstride, s));
        TRY(gather_map(8, ng, h->batch, h->gtsrc.as<int>(), h->gtv0.p, h->gstride, h->gtv.p, h->gstride, s));
    }
    TRY(choose_layout(h, h->grp.as<int>(), h->gci.as<int>(), ng, &h->LG, true, sizeof(double), s,
                      SLA_DIRECT_MAXROW_G, SLA_MIN_LANES_G, SLA_MAX_CAP_G));
    TRY(choose_layout(h, h->gtrp.as<int>(), h->gtci.as<int>(), ng, &h->LGT, true, sizeof(double), s,
                      SLA_DIRECT_MAXROW_G, SLA_MIN_LANES_G, SLA_MAX_CAP_G));
    // Sliced factors.  By default G and G^T take the sliced form with rows
    // sorted by length within windows of 256 rows (a warp per window, the
    // epilogue in row order; the gathers stay near the row) when that pads
    // at most SLA_SLICED_MAXPAD_FACTORS; with SLA_SLICED in the iteration
    // matrix's windows (up to 4096 rows, least padding).  Measured on B300
    // (SPAI factors of the reordered kNN Laplacian, 4M rows, CG
    // iterations/s): both staged 1.80k.  With the epilogue in slot order:
    // G^T sliced 1.86k, G sliced 1.72k (G's kernel also reads r and reduces
    // r.z at every row, which the slot order scatters), both 1.75k, both in
    // windows of up to 1024 rows 1.56k.  With the window epilogue (and the
    // iteration matrix's product on it too): G^T sliced 1.96k, both 2.04k.
    if (h->sliced) {
        TRY(make_sliced_any(h, h->grp.as<int>(), h->gci.as<int>(), ng, h->gv.p, h->gstride, 8, &h->LG, h->sG, s));
        TRY(make_sliced_any(h, h->gtrp.as<int>(), h->gtci.as<int>(), ng, h->gtv.p, h->gstride, 8, &h->LGT, h->sGT,
                            s));
    } else if (!h->pipeline && !h->ws && !h->staged) {
        TRY(make_sliced_any(h, h->grp.as<int>(), h->gci.as<int>(), ng, h->gv.p, h->gstride, 8, &h->LG, h->sG, s, 0,
                            SLA_SLICED_MAXPAD_FACTORS));
        TRY(make_sliced_any(h, h->gtrp.as<int>(), h->gtci.as<int>(), ng, h->gtv.p, h->gstride, 8, &h->LGT, h->sGT,
                            s, 0, SLA_SLICED_MAXPAD_FACTORS));
    }
    TRY(h->dt == SLA_F64 ? spai_grids<double>(h) : spai_grids<float>(h));
    TRY(h->t.alloc(WORK_BYTES * (size_t)n * h->batch));
    h->spai_ready = true;
    h->spai_stale = false;
    return ensure_pstride(h);
}

static sla_status ensure_pstride(sla_csr* h) {
    int m = gx_vec(h);
    m = m > h->LA.gx ? m : h->LA.gx;
    m = m > h->LI.gx ? m : h->LI.gx;
    // the fused iteration kernel: two reductions of two values per CTA, at
    // most as many CTAs as fit resident (2048 threads per SM)
    const int fused = (int)((long long)(2048 / NT) * h->sms / h->batch) + 1;
    m = m > fused ? m : fused;
    if (h->spai_ready) {
        m = m > h->LG.gx ? m : h->LG.gx;
        m = m > h->LGT.gx ? m : h->LGT.gx;
    }
    if (h->bicg_ready) m = m > h->LB.gx ? m : h->LB.gx;
    if (h->tr_ready) m = m > h->LT.gx ? m : h->LT.gx;
    const int need = 4 * m;
    if (need <= h->pstride) return SLA_OK;
    TRY(h->part.alloc(sizeof(double) * (size_t)need * h->batch));
    h->pstride = need;
    for (auto& g : h->graph) g.reset();
    return SLA_OK;
}

// ===================================================================== kernels per iteration
template <typename T, bool PAIRS>
static sla_status enqueue_iteration(sla_csr* h, int pc, double eps, cudaStream_t s, int* nodes, cudaEvent_t ev0,
                                    cudaEvent_t ev1) {
    const Sys S = sys_of(h);
    const Mat A = mat_I(h);
    const T* av = (const T*)h->ivals;
    using W = typename Prec<T>::w;
    W* r = h->r.as<W>();
    W* p = h->p.as<W>();
    W* q = h->q.as<W>();
    using XW = typename Prec<T>::xw;
    using GV = typename Prec<T>::gv;
    XW* x = h->x.as<XW>();
    const XW* dinv = h->dinv.as<XW>();
    const dim3 gs(h->LI.gx, h->batch), gv(gx_vec(h), h->batch);
    // external event-record nodes (a plain record inside a capture only
    // orders streams within the graph)
    if (ev0) CU(cudaEventRecordWithFlags(ev0, s, cudaEventRecordExternal));
    const T* avi = sliced_form(h->LI.form) ? (const T*)h->LI.sval : av;
    with_form(h->LI.form, [&](auto f) {
        k_spmv_iter<T, decltype(f)::value><<<gs, NT, h->LI.smem, s>>>(A, S, avi, p, q, x, h->bw.as<T>());
    });
    TRY(launched());
    if (ev1) CU(cudaEventRecordWithFlags(ev1, s, cudaEventRecordExternal));
    if (pc == SLA_PC_SPAI) {
        k_update<T, 2, PAIRS><<<gv, NT, 0, s>>>(S, r, q, dinv, h->z.as<W>());
        TRY(launched());
        const Mat GT = mat_GT(h);
        const Mat G = mat_G(h);
        const GV* gtv = sliced_form(h->LGT.form) ? (const GV*)h->LGT.sval : h->gtv.as<GV>();
        const GV* gvv = sliced_form(h->LG.form) ? (const GV*)h->LG.sval : h->gv.as<GV>();
        with_form(h->LGT.form, [&](auto f) {
        k_spai_t<T, decltype(f)::value><<<dim3(h->LGT.gx, h->batch), NT, h->LGT.smem, s>>>(GT, S, h->gstride,
                                                                                        gtv, r, h->t.as<W>());
        });
        TRY(launched());
        with_form(h->LG.form, [&](auto f) {
        k_spai_z<T, decltype(f)::value><<<dim3(h->LG.gx, h->batch), NT, h->LG.smem, s>>>(
            G, S, h->gstride, gvv, h->t.as<W>(), r, h->z.as<W>(), eps);
        });
        TRY(launched());
        k_pupdate<T, false, PAIRS><<<gv, NT, 0, s>>>(S, p, x, h->z.as<W>());
        TRY(launched());
        *nodes += 5;
    } else if (pc == SLA_PC_JACOBI) {
        k_update<T, 1, PAIRS><<<gv, NT, 0, s>>>(S, r, q, dinv, h->z.as<W>());
        TRY(launched());
        k_pupdate<T, false, PAIRS><<<gv, NT, 0, s>>>(S, p, x, h->z.as<W>());
        TRY(launched());
        *nodes += 3;
    } else {
        k_update<T, 0, PAIRS><<<gv, NT, 0, s>>>(S, r, q, dinv, h->z.as<W>());
        TRY(launched());
        k_pupdate<T, false, PAIRS><<<gv, NT, 0, s>>>(S, p, x, r);
        TRY(launched());
        *nodes += 3;
    }
    return SLA_OK;
}

template <typename T>
static sla_status enqueue_iteration_any(sla_csr* h, int pc, double eps, cudaStream_t s, int* nodes,
                                        cudaEvent_t ev0 = nullptr, cudaEvent_t ev1 = nullptr) {
    return pairs_ok(h) ? enqueue_iteration<T, true>(h, pc, eps, s, nodes, ev0, ev1)
                       : enqueue_iteration<T, false>(h, pc, eps, s, nodes, ev0, ev1);
}

// Capture k iterations into gc (enq(stream, &nodes, ev0, ev1) enqueues one,
// recording ev0 / ev1 around its product kernel when they are given): one
// instance per launch slot when `timed`, with events around the middle
// iteration's product (clear of the graph launch's own start-up), else one.
template <class Enq>
static sla_status capture_graph(sla_csr* h, GraphCache& gc, int k, double eps, bool timed, Enq enq) {
    if (gc.exec[0] && gc.k == k && gc.eps == eps) return SLA_OK;
    gc.reset();
    const int inst = timed ? 2 : 1;
    int nodes = 0;
    for (int slot = 0; slot < inst; ++slot) {
        if (timed) {
            CU(cudaEventCreate(&gc.t0[slot]));
            CU(cudaEventCreate(&gc.t1[slot]));
        }
        CU(cudaStreamBeginCapture(h->cap, cudaStreamCaptureModeThreadLocal));
        nodes = 0;
        sla_status st = SLA_OK;
        for (int i = 0; i < k && st == SLA_OK; ++i)
            st = enq(h->cap, &nodes, i == k / 2 ? gc.t0[slot] : nullptr, i == k / 2 ? gc.t1[slot] : nullptr);
        cudaGraph_t graph = nullptr;
        cudaError_t e = cudaStreamEndCapture(h->cap, &graph);
        // launches made during capture were counted; they only run when the graph does
        g_launches.fetch_sub((unsigned long long)nodes, std::memory_order_relaxed);
        if (st != SLA_OK) {
            if (graph) cudaGraphDestroy(graph);
            gc.reset();
            return st;
        }
        if (e != cudaSuccess) {
            gc.reset();
            return fail(SLA_ERR_CUDA, "graph capture failed: %s", cudaGetErrorString(e));
        }
        e = cudaGraphInstantiate(&gc.exec[slot], graph, 0);
        cudaGraphDestroy(graph);
        if (e != cudaSuccess) {
            gc.exec[slot] = nullptr;
            gc.reset();
            return fail(SLA_ERR_CUDA, "graph instantiate failed: %s", cudaGetErrorString(e));
        }
    }
    gc.k = k;
    gc.eps = eps;
    gc.nodes = nodes;
    return SLA_OK;
}

template <typename T>
static sla_status get_graph(sla_csr* h, int pc, double eps, int k, GraphCache** out) {
    GraphCache& gc = h->graph[pc];
    TRY(capture_graph(h, gc, k, eps, h->time_product,
                      [&](cudaStream_t s, int* nodes, cudaEvent_t e0, cudaEvent_t e1) {
                          return enqueue_iteration_any<T>(h, pc, eps, s, nodes, e0, e1);
                      }));
    *out = &gc;
    return SLA_OK;
}

// ===================================================================== fused iteration
// Grid of the persistent iteration kernel: every CTA must be resident (a
// cooperative launch), so at most the occupancy times the SM count, spread
// over the batch; 0 when not even one CTA per system fits.
template <typename T, int PC, bool PAIRS>
static sla_status fused_grid(const sla_csr* h, int* gx) {
    int per = 0;
    cudaError_t e = cudaSuccess;
    with_form(fused_form(h->LI.form), [&](auto f) {
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_cg_fused<T, decltype(f)::value, PC, PAIRS>, NT,
                                                          h->LI.smem);
    });
    if (e != cudaSuccess) return fail(SLA_ERR_CUDA, "occupancy query failed: %s", cudaGetErrorString(e));
    long long g = (long long)per * h->sms / h->batch;
    const long long rows_work = fused_form(h->LI.form) == 5 ? ((long long)h->n + NT - 1) / NT
                                                : group_ctas(h->n, h->LI.form == 3 ? 1 : h->LI.lanes);
    const long long work = std::max(rows_work, vec_units(h));
    if (g > work) g = work;
    *gx = (int)g;
    return SLA_OK;
}

template <typename T, int PC, bool PAIRS>
static sla_status launch_fused(sla_csr* h, int gx, int iters, cudaStream_t s) {
    using W = typename Prec<T>::w;
    using XW = typename Prec<T>::xw;
    Mat A = mat_I(h);
    Sys S = sys_of(h);
    const T* av = (const T*)h->ivals;
    W* p = h->p.as<W>();
    W* q = h->q.as<W>();
    W* r = h->r.as<W>();
    W* z = h->z.as<W>();
    XW* x = h->x.as<XW>();
    const XW* dinv = h->dinv.as<XW>();
    const T* b = h->bw.as<T>();
    GridSync* gsy = h->gsync.as<GridSync>();
    void* args[] = {&A, &S, &av, &p, &q, &r, &z, &x, &dinv, &b, &gsy, &iters};
    cudaError_t e = cudaSuccess;
    with_form(fused_form(h->LI.form), [&](auto f) {
        e = cudaLaunchCooperativeKernel((const void*)k_cg_fused<T, decltype(f)::value, PC, PAIRS>,
                                        dim3((unsigned)gx, (unsigned)h->batch), dim3(NT), args, h->LI.smem, s);
    });
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (e != cudaSuccess) return fail(SLA_ERR_CUDA, "cooperative launch failed: %s", cudaGetErrorString(e));
    return SLA_OK;
}

template <typename T>
static sla_status fused_grid_any(const sla_csr* h, int pc, int* gx) {
    const bool pr = pairs_ok(h);
    if (pc == SLA_PC_JACOBI) return pr ? fused_grid<T, 1, true>(h, gx) : fused_grid<T, 1, false>(h, gx);
    return pr ? fused_grid<T, 0, true>(h, gx) : fused_grid<T, 0, false>(h, gx);
}
template <typename T>
static sla_status launch_fused_any(sla_csr* h, int pc, int gx, int iters, cudaStream_t s) {
    const bool pr = pairs_ok(h);
    if (pc == SLA_PC_JACOBI)
        return pr ? launch_fused<T, 1, true>(h, gx, iters, s) : launch_fused<T, 1, false>(h, gx, iters, s);
    return pr ? launch_fused<T, 0, true>(h, gx, iters, s) : launch_fused<T, 0, false>(h, gx, iters, s);
}

// ===================================================================== solve driver
static sla_status from_code(int c) {
    switch (c) {
        case ST_OK: return SLA_OK;
        case ST_NOT_CONVERGED: return SLA_ERR_NOT_CONVERGED;
        default: return SLA_ERR_BREAKDOWN;
    }
}

// Run the iteration in batches -- launch(slot) issues one: a graph of k
// iterations or one persistent kernel -- two in flight, reading the
// device's all-frozen flag after each, until it is set, cap_launches
// batches have run or the host timeout has passed; then drain the stream.
// With gc set, the product-kernel time of every launch during which some
// system stayed live throughout is summed into the handle.
template <class Launch>
static sla_status poll_loop(sla_csr* h, const sla_pcg_opts* o, long long cap_launches, GraphCache* gc,
                            cudaStream_t s, bool* finished_out, bool* timed_out_out, Launch launch) {
    const auto t0 = std::chrono::steady_clock::now();
    int head = 0, inflight = 0;
    long long issued = 0;
    bool finished = false, timed_out = false;
    bool prev_done = false;   // the launch before the oldest in flight left every system frozen
    while (!finished) {
        if (issued < cap_launches && !timed_out) {
            const int slot = (head + inflight) & 1;
            TRY(launch(slot));
            CU(cudaMemcpyAsync(&h->h_flag[slot], &h->ctl.as<Ctrl>()->all_done, sizeof(int),
                               cudaMemcpyDeviceToHost, s));
            CU(cudaEventRecord(h->ev[slot], s));
            ++inflight;
            ++issued;
            if (inflight < 2) continue;
        }
        if (inflight == 0) break;
        // wait for the oldest launch
        const int slot = head;
        if (o->timeout_s > 0) {
            for (;;) {
                cudaError_t q = cudaEventQuery(h->ev[slot]);
                if (q == cudaSuccess) break;
                if (q != cudaErrorNotReady) return fail(SLA_ERR_CUDA, "event query: %s", cudaGetErrorString(q));
                const double el = std::chrono::duration<double>(std::chrono::steady_clock::now() - t0).count();
                if (el > o->timeout_s) timed_out = true;
                std::this_thread::sleep_for(std::chrono::microseconds(50));
            }
        } else {
            CU(cudaEventSynchronize(h->ev[slot]));
        }
        if (gc && !prev_done && !h->h_flag[slot]) {   // live systems from start to end
            float ms = 0.0f;
            CU(cudaEventElapsedTime(&ms, gc->t0[slot], gc->t1[slot]));
            h->prod_ms += ms;
            h->prod_n += 1;
        }
        prev_done = h->h_flag[slot] != 0;
        head ^= 1;
        --inflight;
        if (h->h_flag[slot]) finished = true;
        if ((issued >= cap_launches || timed_out) && inflight == 0) break;
    }
    // drain (kernels of a finished batch return at once)
    CU(cudaStreamSynchronize(s));
    *finished_out = finished;
    *timed_out_out = timed_out;
    return SLA_OK;
}

// After the final pass (k_final) is enqueued: device error bits, then the
// per-system statistics into info[] and the call's status.
static sla_status collect(sla_csr* h, bool finished, bool timed_out, const sla_pcg_opts* o, sla_solve_info* info,
                          cudaStream_t s, const char* breakdown_msg) {
    CU(cudaMemcpyAsync(h->h_stat, h->stat.p, sizeof(Stat) * h->batch, cudaMemcpyDeviceToHost, s));
    Ctrl dc;
    CU(cudaMemcpyAsync(&dc, h->ctl.p, sizeof(Ctrl), cudaMemcpyDeviceToHost, s));
    CU(cudaStreamSynchronize(s));
    if (dc.err & ERR_STAGE) return fail(SLA_ERR_CUDA, "a staged range exceeded its stage; results invalid");
    if (dc.err & (ERR_WAIT | ERR_GRID))
        return fail(SLA_ERR_CUDA, "a device wait gave up (%s; at %d: %d %d %d); results invalid",
                    (dc.err & ERR_GRID) ? "grid barrier" : "bulk copy", dc.diag[0], dc.diag[1], dc.diag[2],
                    dc.diag[3]);

    sla_status ret = SLA_OK;
    for (int i = 0; i < h->batch; ++i) {
        const Stat& st = h->h_stat[i];
        sla_status si = from_code(st.status);
        if (!st.done) si = timed_out ? SLA_ERR_TIMEOUT : SLA_ERR_NOT_CONVERGED;  // host stopped first
        if (info) {
            info[i].iters = st.iters;
            info[i].rel_res_recursive = st.rel_rec;
            info[i].rel_res_true = st.rel_true;
            info[i].status = si;
        }
        if (ret == SLA_OK && si != SLA_OK) ret = si;
    }
    if (!finished && !timed_out)
        return fail(SLA_ERR_NOT_CONVERGED, "iteration launches exhausted before the device froze");
    if (ret == SLA_ERR_TIMEOUT) return fail(ret, "timeout after %.3f s", o->timeout_s);
    if (ret != SLA_OK) fail(ret, ret == SLA_ERR_BREAKDOWN ? breakdown_msg : "not converged within max_iter");
    return ret;
}

template <typename T>
static sla_status solve_impl(sla_csr* h, const T* b, T* x_user, const sla_pcg_opts* o, sla_solve_info* info,
                             cudaStream_t s) {
    const int pc = (int)o->pc;
    if (pc == SLA_PC_JACOBI && (h->diag_err & ERR_NO_DIAG))
        return fail(SLA_ERR_INVALID, "Jacobi needs every diagonal entry stored");
    if (pc == SLA_PC_SPAI && !h->spai_ready) TRY(build_spai(h, s));
    if (pc == SLA_PC_SPAI && h->spai_stale) TRY(spai_values(h, s));
    TRY(ensure_pstride(h));
    const int k = o->poll_k > 0 ? o->poll_k : 32;
    const double eps = pc == SLA_PC_SPAI ? o->eps : 0.0;
    // A CUDA graph of k iterations of one kernel per step; with
    // SLA_PERSISTENT, CG and Jacobi-PCG instead run as the persistent
    // iteration kernel wherever every CTA can be resident.
    int gxf = 0;
    if (pc != SLA_PC_SPAI && h->coop && h->persistent) TRY(fused_grid_any<T>(h, pc, &gxf));
    const bool fused = gxf >= 1;
    GraphCache* gc = nullptr;
    if (!fused) TRY(get_graph<T>(h, pc, eps, k, &gc));

    const Sys S = sys_of(h);
    const Mat A = mat_I(h);
    const T* av = (const T*)h->ivals;
    const dim3 gs(h->LI.gx, h->batch), gv(gx_vec(h), h->batch);
    using W = typename Prec<T>::w;
    W* r = h->r.as<W>();
    W* p = h->p.as<W>();
    using XW = typename Prec<T>::xw;
    using GV = typename Prec<T>::gv;
    XW* x = h->x.as<XW>();
    const XW* dinv = h->dinv.as<XW>();

    CU(cudaMemsetAsync(h->ctl.p, 0, sizeof(Ctrl), s));
    CU(cudaMemsetAsync(h->gsync.p, 0, sizeof(GridSync) * h->batch, s));
    // a reordered handle iterates on P b (and P x0) and returns P^T x
    const T* b_it = b;
    const T* x0_it = x_user;
    T* x_it = x_user;
    if (h->reordered) {
        T* tb = h->ptmp.as<T>();
        T* tx = tb + (size_t)h->batch * h->n;
        TRY(gather_map(sizeof(T), h->n, h->batch, h->perm.as<int>(), b, h->n, tb, h->n, s));
        if (o->use_x0) TRY(gather_map(sizeof(T), h->n, h->batch, h->perm.as<int>(), x_user, h->n, tx, h->n, s));
        b_it = tb;
        x0_it = tx;
        x_it = tx;
    }
    if (o->use_x0) {
        k_init_x0<T><<<gs, NT, h->LI.smem, s>>>(A, S, av, b_it, x0_it, h->bw.as<T>(), x, r, o->tol, o->max_iter);
    } else {
        k_init<T><<<gv, NT, 0, s>>>(S, b_it, h->bw.as<T>(), x, r, o->tol, o->max_iter);
    }
    TRY(launched());
    if (pc == SLA_PC_SPAI) {
        const Mat GT = mat_GT(h);
        const Mat G = mat_G(h);
        const GV* gtv = sliced_form(h->LGT.form) ? (const GV*)h->LGT.sval : h->gtv.as<GV>();
        const GV* gvv = sliced_form(h->LG.form) ? (const GV*)h->LG.sval : h->gv.as<GV>();
        with_form(h->LGT.form, [&](auto f) {
        k_spai_t<T, decltype(f)::value><<<dim3(h->LGT.gx, h->batch), NT, h->LGT.smem, s>>>(GT, S, h->gstride,
                                                                                       gtv, r, h->t.as<W>());
        });
        TRY(launched());
        with_form(h->LG.form, [&](auto f) {
        k_spai_z<T, decltype(f)::value><<<dim3(h->LG.gx, h->batch), NT, h->LG.smem, s>>>(
            G, S, h->gstride, gvv, h->t.as<W>(), r, h->z.as<W>(), eps);
        });
        TRY(launched());
        k_pupdate<T, true, false><<<gv, NT, 0, s>>>(S, p, x, h->z.as<W>());
    } else if (pc == SLA_PC_JACOBI) {
        k_init_dir<T, 1><<<gv, NT, 0, s>>>(S, p, r, dinv);
    } else {
        k_init_dir<T, 0><<<gv, NT, 0, s>>>(S, p, r, dinv);
    }
    TRY(launched());

    const long long cap_launches = ((long long)o->max_iter + 2LL * k + 2) / k + 2;
    const bool timing = !fused && h->time_product;
    bool finished = false, timed_out = false;
    TRY(poll_loop(h, o, cap_launches, timing ? gc : nullptr, s, &finished, &timed_out, [&](int slot) {
        if (fused) return launch_fused_any<T>(h, pc, gxf, k, s);
        CU(cudaGraphLaunch(gc->exec[timing ? slot : 0], s));
        g_launches.fetch_add((unsigned long long)gc->nodes, std::memory_order_relaxed);
        return SLA_OK;
    }));

    k_final<T><<<gs, NT, h->LI.smem, s>>>(A, S, av, x, h->bw.as<T>(), x_it, h->stat.as<Stat>());
    TRY(launched());
    if (h->reordered) TRY(gather_map(sizeof(T), h->n, h->batch, h->iperm.as<int>(), x_it, h->n, x_user, h->n, s));
    return collect(h, finished, timed_out, o, info, s, "breakdown (p.Ap <= 0, r.z <= 0 or non-finite value)");
}

// ===================================================================== BiCGStab
// Dispatch over the register / cp.async staging forms, the direct form and
// the sliced forms (the BiCGStab product kernels are built for these only).
template <class F>
static void with_form_rc(int form, F&& f) {
    switch (form) {
        case 0: f(std::integral_constant<int, 0>{}); break;
        case 1: f(std::integral_constant<int, 1>{}); break;
        case 5: f(std::integral_constant<int, 5>{}); break;
        case 6: f(std::integral_constant<int, 6>{}); break;
        case 7: f(std::integral_constant<int, 7>{}); break;
        default: f(std::integral_constant<int, 2>{}); break;
    }
}

// Pattern of M^T: row j lists the rows i of the entries (i, j) of M in
// ascending order; src[k'] = the entry of M that transposed entry k' holds.
static void transpose_pattern(int n, const std::vector<int>& rp, const std::vector<int>& ci, std::vector<int>& trp,
                              std::vector<int>& tci, std::vector<int>& src) {
    trp.assign(n + 1, 0);
    for (size_t k = 0; k < ci.size(); ++k) trp[ci[k] + 1] += 1;
    for (int j = 0; j < n; ++j) trp[j + 1] += trp[j];
    std::vector<int> next(trp.begin(), trp.end() - 1);
    tci.resize(ci.size());
    src.resize(ci.size());
    for (int i = 0; i < n; ++i)
        for (int k = rp[i]; k < rp[i + 1]; ++k) {
            const int d = next[ci[k]]++;
            tci[d] = i;
            src[d] = k;
        }
}

// Workspace of BiCGStab (and, for `transposed`, the explicit transpose of
// the iteration matrix); built once per handle.  Its products take the
// staged forms, or the sliced form where the CG products' default would
// (a handle-owned sliced copy whose values bicg_impl refills from the
// iterated values every solve).  Measured on B300, 3D convection-diffusion
// system: the direct form's product was slower than the staged one inside
// the BiCGStab iteration (71.9 against 65.1 us), unlike in the CG iteration.
#ifndef SLA_BICG_SLICED
#define SLA_BICG_SLICED 1
#endif
static bool bicg_sliced(const sla_csr* h, const Layout& L) {
    return h->dt == SLA_F64 && SLA_BICG_SLICED && !h->pipeline && !h->ws && !h->staged &&
           (h->sliced || sliced_by_default(h, L, h->nnz));
}
static sla_status ensure_bicg(sla_csr* h, bool transposed, cudaStream_t s) {
    if (!h->bicg_ready) {
        TRY(h->rh.alloc(sizeof(double) * (size_t)h->n * h->batch));
        h->LB = h->LI;   // the CG layout's pattern analysis; its own form (and sliced copy) below
        TRY(set_form_any(h, &h->LB, false, sizeof(double), 0));
        if (bicg_sliced(h, h->LB))
            TRY(make_sliced_any(h, h->irp, h->ici, h->nnz, h->ivals, h->nnz, 8, &h->LB, h->sB, s));
        h->bicg_ready = true;
    }
    if (transposed && !h->tr_ready) {
        std::vector<int> rp, ci, trp, tci, src;
        CU(cudaStreamSynchronize(s));
        TRY(to_host(rp, h->irp, (size_t)h->n + 1));
        TRY(to_host(ci, h->ici, (size_t)h->nnz));
        transpose_pattern(h->n, rp, ci, trp, tci, src);
        TRY(to_device(h->trp, trp));
        TRY(to_device(h->tci, tci));
        TRY(to_device(h->tsrc, src));
        TRY(h->tvals.alloc(sizeof(double) * (size_t)h->nnz * h->batch));
        TRY(choose_layout(h, h->trp.as<int>(), h->tci.as<int>(), h->nnz, &h->LT, false, sizeof(double), s, 0));
        if (bicg_sliced(h, h->LT))
            TRY(make_sliced_any(h, h->trp.as<int>(), h->tci.as<int>(), h->nnz, h->ivals, h->nnz, 8, &h->LT, h->sT,
                                s));
        h->tr_ready = true;
    }
    return ensure_pstride(h);
}

// One BiCGStab iteration on the matrix (M, av): five kernels.
// a0, dsc: the unscaled values and the diagonal when the iteration runs on
// the column-scaled values (right Jacobi), else null.
template <int W>
static sla_status enqueue_bicg(sla_csr* h, const Mat& M, const Layout& L, const double* av, const double* a0,
                               const double* dsc, cudaStream_t s, int* nodes, cudaEvent_t ev0, cudaEvent_t ev1) {
    const Sys S = sys_of(h);
    double* y = h->x.as<double>();
    double* r = h->r.as<double>();   // r, and s over it
    double* p = h->p.as<double>();
    double* v = h->q.as<double>();
    double* t = h->z.as<double>();
    const double* rh = h->rh.as<double>();
    const dim3 gs(L.gx, h->batch), gv(gx_vec(h), h->batch);
    if (ev0) CU(cudaEventRecordWithFlags(ev0, s, cudaEventRecordExternal));
    with_form_rc(L.form, [&](auto f) {
        k_bicg_v<decltype(f)::value><<<gs, NT, L.smem, s>>>(M, S, av, p, v, rh, y, h->bw.as<double>(), a0, dsc);
    });
    TRY(launched());
    if (ev1) CU(cudaEventRecordWithFlags(ev1, s, cudaEventRecordExternal));
    k_bicg_s<W><<<gv, NT, 0, s>>>(S, r, v);
    TRY(launched());
    with_form_rc(L.form, [&](auto f) { k_bicg_t<decltype(f)::value><<<gs, NT, L.smem, s>>>(M, S, av, r, t); });
    TRY(launched());
    k_bicg_xr<W><<<gv, NT, 0, s>>>(S, y, p, r, t, rh);
    TRY(launched());
    k_bicg_p<W><<<gv, NT, 0, s>>>(S, p, r, v);
    TRY(launched());
    *nodes += 5;
    return SLA_OK;
}

// Solve A x = b (transposed: A^T x = b) by BiCGStab on the iteration matrix
// (P A P^T when the handle reorders; b and x are permuted in and out).
static sla_status bicg_impl(sla_csr* h, bool transposed, const double* b, double* x_user, const sla_pcg_opts* o,
                            sla_solve_info* info, cudaStream_t s) {
    const int pc = (int)o->pc;
    if (pc == SLA_PC_JACOBI && (h->diag_err & ERR_NO_DIAG))
        return fail(SLA_ERR_INVALID, "Jacobi needs every diagonal entry stored");
    TRY(ensure_bicg(h, transposed, s));
    const int k = o->poll_k > 0 ? o->poll_k : 32;
    const Sys S = sys_of(h);
    int* err = &h->ctl.as<Ctrl>()->err;
    // the matrix as stored (initial residual, final check) and as iterated
    const int* mrp = transposed ? h->trp.as<int>() : h->irp;
    const int* mci = transposed ? h->tci.as<int>() : h->ici;
    const Layout& L = transposed ? h->LT : h->LB;
    const Mat M = mat_of(mrp, mci, h->n, h->nnz, L, err);
    const double* uv = (const double*)h->ivals;
    if (transposed) {
        TRY(gather_map(8, h->nnz, h->batch, h->tsrc.as<int>(), h->ivals, h->nnz, h->tvals.p, h->nnz, s));
        uv = h->tvals.as<double>();
    }
    const double* itv = uv;
    if (pc == SLA_PC_JACOBI) {
        if (!h->bvals.p) {
            TRY(h->bvals.alloc(sizeof(double) * (size_t)h->nnz * h->batch));
            for (int g = 3; g < 7; ++g) h->graph[g].reset();
        }
        if (h->nnz > 0) {
            const long long blocks = (h->nnz + NT - 1) / NT;
            const dim3 gsc((unsigned)std::min<long long>(blocks, 4096), h->batch);
            k_bicg_colscale<<<gsc, NT, 0, s>>>(h->nnz, h->n, mci, uv, h->diag.as<double>(), h->bvals.as<double>());
            TRY(launched());
        }
        itv = h->bvals.as<double>();
    }
    if (sliced_form(L.form)) {   // the sliced copy holds this solve's iterated values
        TRY(sliced_values(h, transposed ? h->sT : h->sB, itv, h->nnz, 8, s));
        itv = (const double*)L.sval;
    }
    GraphCache& gc = h->graph[3 + 2 * (transposed ? 1 : 0) + (pc == SLA_PC_JACOBI ? 1 : 0)];
    TRY(capture_graph(h, gc, k, 0.0, h->time_product, [&](cudaStream_t cs, int* nodes, cudaEvent_t e0,
                                                            cudaEvent_t e1) {
        const double* a0 = pc == SLA_PC_JACOBI ? uv : nullptr;
        const double* dsc = pc == SLA_PC_JACOBI ? h->diag.as<double>() : nullptr;
        return pairs_ok(h) ? enqueue_bicg<2>(h, M, L, itv, a0, dsc, cs, nodes, e0, e1)
                           : enqueue_bicg<1>(h, M, L, itv, a0, dsc, cs, nodes, e0, e1);
    }));

    const dim3 gs(L.gx, h->batch), gv(gx_vec(h), h->batch);
    double* x = h->x.as<double>();
    double* r = h->r.as<double>();
    CU(cudaMemsetAsync(h->ctl.p, 0, sizeof(Ctrl), s));
    const double* b_it = b;
    const double* x0_it = x_user;
    double* x_it = x_user;
    if (h->reordered) {
        double* tb = h->ptmp.as<double>();
        double* tx = tb + (size_t)h->batch * h->n;
        TRY(gather_map(8, h->n, h->batch, h->perm.as<int>(), b, h->n, tb, h->n, s));
        if (o->use_x0) TRY(gather_map(8, h->n, h->batch, h->perm.as<int>(), x_user, h->n, tx, h->n, s));
        b_it = tb;
        x0_it = tx;
        x_it = tx;
    }
    if (o->use_x0) {
        k_init_x0<double><<<gs, NT, L.smem, s>>>(M, S, uv, b_it, x0_it, h->bw.as<double>(), x, r, o->tol,
                                                 o->max_iter);
    } else {
        k_init<double><<<gv, NT, 0, s>>>(S, b_it, h->bw.as<double>(), x, r, o->tol, o->max_iter);
    }
    TRY(launched());
    if (pc == SLA_PC_JACOBI && o->use_x0) {   // y = D x0
        k_bicg_scale<true><<<gv, NT, 0, s>>>(S, x, h->diag.as<double>());
        TRY(launched());
    }
    if (pairs_ok(h)) k_bicg_dir<2><<<gv, NT, 0, s>>>(S, r, h->rh.as<double>(), h->p.as<double>());
    else k_bicg_dir<1><<<gv, NT, 0, s>>>(S, r, h->rh.as<double>(), h->p.as<double>());
    TRY(launched());

    const long long cap_launches = ((long long)o->max_iter + 2LL * k + 2) / k + 2;
    bool finished = false, timed_out = false;
    TRY(poll_loop(h, o, cap_launches, h->time_product ? &gc : nullptr, s, &finished, &timed_out, [&](int slot) {
        CU(cudaGraphLaunch(gc.exec[h->time_product ? slot : 0], s));
        g_launches.fetch_add((unsigned long long)gc.nodes, std::memory_order_relaxed);
        return SLA_OK;
    }));

    if (pc == SLA_PC_JACOBI) {   // x = D^-1 y
        k_bicg_scale<false><<<gv, NT, 0, s>>>(S, x, h->diag.as<double>());
        TRY(launched());
    }
    k_final<double><<<gs, NT, L.smem, s>>>(M, S, uv, x, h->bw.as<double>(), x_it, h->stat.as<Stat>());
    TRY(launched());
    if (h->reordered) TRY(gather_map(8, h->n, h->batch, h->iperm.as<int>(), x_it, h->n, x_user, h->n, s));
    return collect(h, finished, timed_out, o, info, s, "breakdown (r^.r or r^.v zero, omega zero or non-finite value)");
}

// ===================================================================== C ABI
extern "C" {

void sla_pcg_opts_default(sla_pcg_opts* o) {
    if (!o) return;
    o->tol = 1e-8;
    o->max_iter = 10000;
    o->pc = SLA_PC_NONE;
    o->eps = 1e-3;
    o->poll_k = 32;
    o->use_x0 = 0;
    o->timeout_s = 0.0;
}

const char* sla_last_error(void) { return g_err.c_str(); }

unsigned long long sla_launch_count(void) { return g_launches.load(); }

static void destroy_handle(sla_csr* h) {
    if (!h) return;
    for (auto& g : h->graph) g.reset();
    if (h->cap) cudaStreamDestroy(h->cap);
    for (auto& e : h->ev) if (e) cudaEventDestroy(e);
    if (h->h_flag) cudaFreeHost(h->h_flag);
    if (h->h_stat) cudaFreeHost(h->h_stat);
    delete h;  // DevBuf members free themselves below via release()
}

sla_status sla_csr_destroy(sla_handle h) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    DevBuf* bufs[] = {&h->diag, &h->dinv, &h->grp, &h->gci, &h->gv, &h->gtrp, &h->gtci, &h->gtv,
                      &h->x, &h->r, &h->p, &h->q, &h->z, &h->t, &h->bw, &h->state,
                      &h->ctl, &h->cnt, &h->part, &h->stat, &h->gsync, &h->perm, &h->iperm,
                      &h->prp, &h->pci, &h->psrc, &h->pvals, &h->ptmp};
    for (DevBuf* b : bufs) b->release();
    destroy_handle(h);
    return SLA_OK;
}

sla_status sla_csr_create(int n, long long nnz, int batch, sla_dtype dt, const int* d_row_ptr,
                          const int* d_col_idx, const void* d_vals, unsigned flags, void* stream,
                          sla_handle* out) {
    if (!out) return fail(SLA_ERR_INVALID, "out is null");
    *out = nullptr;
    if (n < 1) return fail(SLA_ERR_INVALID, "n must be >= 1 (got %d)", n);
    if (nnz < 0 || nnz > 2147483647LL) return fail(SLA_ERR_INVALID, "nnz must be in [0, 2^31) (got %lld)", nnz);
    if (batch < 1) return fail(SLA_ERR_INVALID, "batch must be >= 1 (got %d)", batch);
    if (dt != SLA_F64 && dt != SLA_F32) return fail(SLA_ERR_INVALID, "unknown dtype %d", (int)dt);
    if (!d_row_ptr || (nnz > 0 && (!d_col_idx || !d_vals))) return fail(SLA_ERR_INVALID, "null CSR pointer");
    cudaStream_t s = (cudaStream_t)stream;

    sla_csr* h = new sla_csr();
    h->n = n;
    h->nnz = nnz;
    h->batch = batch;
    h->dt = dt;
    h->es = dt == SLA_F64 ? 8 : 4;
    h->rp = d_row_ptr;
    h->ci = d_col_idx;
    h->vals = d_vals;
    auto bail = [&](sla_status st) {
        std::string msg = g_err;
        sla_csr_destroy(h);
        g_err = msg;
        return st;
    };
#define HTRY(expr)                                 \
    do {                                           \
        sla_status s_ = (expr);                    \
        if (s_ != SLA_OK) return bail(s_);         \
    } while (0)
#define HCU(call)                                                                                   \
    do {                                                                                            \
        cudaError_t e_ = (call);                                                                    \
        if (e_ != cudaSuccess)                                                                      \
            return bail(fail(SLA_ERR_CUDA, "%s failed: %s", #call, cudaGetErrorString(e_)));       \
    } while (0)

    HCU(cudaGetDevice(&h->device));
    HCU(cudaDeviceGetAttribute(&h->sms, cudaDevAttrMultiProcessorCount, h->device));
    HCU(cudaStreamCreateWithFlags(&h->cap, cudaStreamNonBlocking));
    HCU(cudaEventCreateWithFlags(&h->ev[0], cudaEventDisableTiming));
    HCU(cudaEventCreateWithFlags(&h->ev[1], cudaEventDisableTiming));
    HCU(cudaHostAlloc((void**)&h->h_flag, 2 * sizeof(int), cudaHostAllocDefault));
    HCU(cudaHostAlloc((void**)&h->h_stat, sizeof(Stat) * batch, cudaHostAllocDefault));
    h->h_flag[0] = h->h_flag[1] = 0;

    if (flags & SLA_VALIDATE) {
        DevBuf err;
        HTRY(err.alloc(sizeof(int)));
        HCU(cudaMemsetAsync(err.p, 0, sizeof(int), s));
        const int g = (n + 255) / 256 < 4096 ? (n + 255) / 256 : 4096;
        k_validate<<<g, 256, 0, s>>>(n, nnz, d_row_ptr, d_col_idx, err.as<int>());
        HTRY(launched());
        int e = 0;
        HTRY(read_int(err.as<int>(), &e, s));
        if (e)
            return bail(fail(SLA_ERR_INVALID, "malformed CSR:%s%s%s", (e & ERR_ROWPTR) ? " row_ptr" : "",
                             (e & ERR_COL_RANGE) ? " column out of range" : "",
                             (e & ERR_COL_ORDER) ? " columns not strictly ascending" : ""));
    }
    HTRY(dt == SLA_F64 ? allow_smem<double>() : allow_smem<float>());
    h->vals_aligned = vals_aligned(h, d_vals);
    h->pipeline = (flags & SLA_WARP_PIPELINE) != 0;
    h->ws = (flags & SLA_PRODUCER_CONSUMER) != 0;
    h->staged = (flags & SLA_STAGED) != 0;
    h->time_product = (flags & SLA_TIME_PRODUCT) != 0;
    h->persistent = (flags & SLA_PERSISTENT) != 0;
    h->sliced = (flags & SLA_SLICED) != 0;
    h->split = (flags & SLA_ROW_WALK) ? -1 : (flags & SLA_SPLIT_ROWS) ? 1 : 0;
    {
        int coop = 0;
        HCU(cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, h->device));
        h->coop = coop != 0;
    }
    HTRY(choose_layout(h, d_row_ptr, d_col_idx, nnz, &h->LA, h->vals_aligned, h->es, s));
    // the matrix the solve iterates on: A, or P A P^T for a scattered
    // pattern (its gathers then stay near the row)
    h->irp = d_row_ptr;
    h->ici = d_col_idx;
    h->ivals = d_vals;
    h->LI = h->LA;
    const bool reorder = nnz > 0 && !(flags & SLA_NO_REORDER) && ((flags & SLA_REORDER) || h->LA.gasync);
    if (reorder) {
        HTRY(make_reordered(h, s));
        const bool al = h->batch == 1 || ((size_t)nnz * h->es) % 16 == 0;
        HTRY(choose_layout(h, h->irp, h->ici, nnz, &h->LI, al, h->es, s));
    }
    if (!h->pipeline && !h->ws && !h->staged && (h->sliced || sliced_by_default(h, h->LI, nnz)))
        HTRY(make_sliced_any(h, h->irp, h->ici, nnz, h->ivals, nnz, h->es, &h->LI, h->sI, s));
    const size_t vn = (size_t)n * batch;
    HTRY(h->diag.alloc(sizeof(double) * vn));
    HTRY(h->dinv.alloc(sizeof(double) * vn));
    HTRY(compute_diag(h, s));
    HTRY(h->x.alloc(sizeof(double) * vn));
    HTRY(h->r.alloc(WORK_BYTES * vn));
    HTRY(h->p.alloc(WORK_BYTES * vn));
    HTRY(h->q.alloc(WORK_BYTES * vn));
    HTRY(h->z.alloc(WORK_BYTES * vn));
    HTRY(h->gsync.alloc(sizeof(GridSync) * batch));
    HCU(cudaMemsetAsync(h->gsync.p, 0, sizeof(GridSync) * batch, s));
    HTRY(h->bw.alloc(h->es * vn));
    HTRY(h->state.alloc(sizeof(State) * batch));
    HTRY(h->ctl.alloc(sizeof(Ctrl)));
    HTRY(h->cnt.alloc(sizeof(unsigned) * batch));
    HTRY(h->stat.alloc(sizeof(Stat) * batch));
    HCU(cudaMemsetAsync(h->cnt.p, 0, sizeof(unsigned) * batch, s));
    HCU(cudaMemsetAsync(h->ctl.p, 0, sizeof(Ctrl), s));
    HCU(cudaMemsetAsync(h->state.p, 0, sizeof(State) * batch, s));
    HTRY(ensure_pstride(h));
    HCU(cudaStreamSynchronize(s));
#undef HTRY
#undef HCU
    *out = h;
    return SLA_OK;
}

sla_status sla_product_time(sla_handle h, double* total_ms, long long* samples, int reset) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (total_ms) *total_ms = h->prod_ms;
    if (samples) *samples = h->prod_n;
    if (reset) {
        h->prod_ms = 0.0;
        h->prod_n = 0;
    }
    return SLA_OK;
}

sla_status sla_csr_layout(sla_handle h, int* form, int* ctas, int* reordered) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (form) *form = h->LI.form;
    if (ctas) *ctas = h->LI.gx;
    if (reordered) *reordered = h->reordered ? 1 : 0;
    return SLA_OK;
}

sla_status sla_csr_layout_of(sla_handle h, int which, int* form, int* ctas, int* split) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (which < 0 || which > 4) return fail(SLA_ERR_INVALID, "which = %d: 0 to 4", which);
    if ((which == 1 || which == 2) && !h->spai_ready) return fail(SLA_ERR_INVALID, "no SPAI factor yet");
    if (which == 3 && !h->bicg_ready) return fail(SLA_ERR_INVALID, "no BiCGStab solve yet");
    if (which == 4 && !h->tr_ready) return fail(SLA_ERR_INVALID, "no BiCGStab adjoint yet");
    const Layout& L = which == 0 ? h->LI : which == 1 ? h->LG : which == 2 ? h->LGT : which == 3 ? h->LB : h->LT;
    if (form) *form = L.form;
    if (ctas) *ctas = L.gx;
    if (split) *split = L.bal && L.lanes == 1 && (L.form == 1 || L.form == 2) ? 1 : 0;
    return SLA_OK;
}

sla_status sla_csr_update_values(sla_handle h, const void* d_vals, void* stream) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (!d_vals && h->nnz > 0) return fail(SLA_ERR_INVALID, "null values");
    cudaStream_t s = (cudaStream_t)stream;
    const bool moved = d_vals != h->vals;
    h->vals = d_vals;
    h->spai_stale = true;   // G, G^T values recomputed by the next SPAI solve
    // The CUDA graphs hold the pointers their kernels read.  Rebuilt: all of
    // them when the layout changes (below); when the caller's values moved,
    // those that read them -- CG on neither a permuted nor a sliced copy,
    // BiCGStab on A (its unsliced product and its Jacobi residual check)
    // unless the handle reorders.  The handle's own copies (permuted,
    // sliced, G, G^T, the transpose) keep their buffers and are refreshed
    // in place.
    if (moved && !h->reordered) {
        if (!sliced_form(h->LI.form))
            for (int g = 0; g < 3; ++g) h->graph[g].reset();
        h->graph[3].reset();
        h->graph[4].reset();
    }
    if (vals_aligned(h, d_vals) != h->vals_aligned) {
        for (auto& g : h->graph) g.reset();
        h->vals_aligned = !h->vals_aligned;
        TRY(set_form_any(h, &h->LA, h->vals_aligned, h->es));
        if (!h->reordered) {
            const bool was_sliced = sliced_form(h->LI.form);
            h->LI = h->LA;
            if (was_sliced) TRY(make_sliced_any(h, h->irp, h->ici, h->nnz, d_vals, h->nnz, h->es, &h->LI, h->sI, s));
        }
        TRY(ensure_pstride(h));
    }
    if (h->reordered) TRY(gather_map(h->es, h->nnz, h->batch, h->psrc.as<int>(), d_vals, h->nnz, h->pvals.p, h->nnz, s));
    else h->ivals = d_vals;
    if (sliced_form(h->LI.form)) TRY(sliced_values(h, h->sI, h->ivals, h->nnz, h->es, s));
    TRY(compute_diag(h, s));
    CU(cudaStreamSynchronize(s));
    return SLA_OK;
}

static sla_status spmv_common(sla_handle h, const void* d_x, void* d_y, double* d_dot, void* stream) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (!d_x || !d_y) return fail(SLA_ERR_INVALID, "null vector");
    cudaStream_t s = (cudaStream_t)stream;
    const Sys S = sys_of(h);
    // the sliced copy of the iteration matrix serves A itself when the
    // handle does not reorder
    const bool sl = !h->reordered && sliced_form(h->LI.form);
    const Layout& L = sl ? h->LI : h->LA;
    const Mat A = sl ? mat_I(h) : mat_A(h);
    const void* vals = sl ? L.sval : h->vals;
    const dim3 g(L.gx, h->batch);
    const size_t sm = L.smem;
    with_form(L.form, [&](auto f) {
        constexpr int F = decltype(f)::value;
        if (h->dt == SLA_F64)
            k_spmv<double, F><<<g, NT, sm, s>>>(A, S, (const double*)vals, (const double*)d_x, (double*)d_y, d_dot);
        else
            k_spmv<float, F><<<g, NT, sm, s>>>(A, S, (const float*)vals, (const float*)d_x, (float*)d_y, d_dot);
    });
    return launched();
}

sla_status sla_spmm(sla_handle h, const void* d_X, void* d_Y, int k, void* stream) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (h->batch != 1) return fail(SLA_ERR_INVALID, "sla_spmm needs a single-system handle (batch = 1)");
    if (k < 0) return fail(SLA_ERR_INVALID, "k must be >= 0 (got %d)", k);
    if (k == 0) return SLA_OK;
    if (!d_X || !d_Y) return fail(SLA_ERR_INVALID, "null block");
    if (k > 65535) return fail(SLA_ERR_INVALID, "k must be <= 65535 (got %d)", k);
    cudaStream_t s = (cudaStream_t)stream;
    Sys S = sys_of(h);
    S.nnz = 0;   // every column of the block is multiplied by the same values
    // the sliced copy of the iteration matrix serves A itself when the
    // handle does not reorder (as in sla_spmv)
    const bool sl = !h->reordered && sliced_form(h->LI.form);
    const Layout& L = sl ? h->LI : h->LA;
    Mat A = sl ? mat_I(h) : mat_A(h);
    A.vstride = 0;   // likewise for the sliced values
    const void* vals = sl ? L.sval : h->vals;
    const dim3 g(L.gx, k);
    const size_t sm = L.smem;
    with_form(L.form, [&](auto f) {
        constexpr int F = decltype(f)::value;
        if (h->dt == SLA_F64)
            k_spmv<double, F><<<g, NT, sm, s>>>(A, S, (const double*)vals, (const double*)d_X, (double*)d_Y,
                                                nullptr);
        else
            k_spmv<float, F><<<g, NT, sm, s>>>(A, S, (const float*)vals, (const float*)d_X, (float*)d_Y,
                                               nullptr);
    });
    return launched();
}

sla_status sla_spmv(sla_handle h, const void* d_x, void* d_y, void* stream) {
    return spmv_common(h, d_x, d_y, nullptr, stream);
}

sla_status sla_spmv_dot(sla_handle h, const void* d_x, void* d_y, double* d_dot, void* stream) {
    if (!d_dot) return fail(SLA_ERR_INVALID, "null dot");
    return spmv_common(h, d_x, d_y, d_dot, stream);
}

static sla_status check_opts(const sla_pcg_opts* o) {
    if (!o) return fail(SLA_ERR_INVALID, "null options");
    if (!(o->tol > 0.0)) return fail(SLA_ERR_INVALID, "tol must be > 0");
    if (o->max_iter < 0) return fail(SLA_ERR_INVALID, "max_iter must be >= 0");
    if (o->pc != SLA_PC_NONE && o->pc != SLA_PC_JACOBI && o->pc != SLA_PC_SPAI)
        return fail(SLA_ERR_INVALID, "unknown preconditioner %d", (int)o->pc);
    if (o->pc == SLA_PC_SPAI && !(o->eps >= 0.0)) return fail(SLA_ERR_INVALID, "eps must be >= 0");
    if (o->poll_k < 0) return fail(SLA_ERR_INVALID, "poll_k must be >= 0");
    return SLA_OK;
}

sla_status sla_pcg_solve(sla_handle h, const void* d_b, void* d_x, const sla_pcg_opts* opts,
                         sla_solve_info* info, void* stream) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (!d_b || !d_x) return fail(SLA_ERR_INVALID, "null vector");
    TRY(check_opts(opts));
    cudaStream_t s = (cudaStream_t)stream;
    if (h->dt == SLA_F64) return solve_impl<double>(h, (const double*)d_b, (double*)d_x, opts, info, s);
    return solve_impl<float>(h, (const float*)d_b, (float*)d_x, opts, info, s);
}

// dL/dA_k = -lambda_row(k) x_col(k) on A's own pattern and ordering.
static sla_status grad_A(sla_csr* h, const void* d_x, const void* d_lam, void* d_dLdA, cudaStream_t s) {
    if (!d_dLdA || h->nnz == 0) return SLA_OK;
    const Sys S = sys_of(h);
    const Mat A = mat_A(h);
    const dim3 g(h->LA.gx, h->batch);
    if (h->dt == SLA_F64)
        k_grad_A<double><<<g, NT, h->LA.smem, s>>>(A, S, (const double*)d_lam, (const double*)d_x, (double*)d_dLdA);
    else
        k_grad_A<float><<<g, NT, h->LA.smem, s>>>(A, S, (const float*)d_lam, (const float*)d_x, (float*)d_dLdA);
    TRY(launched());
    CU(cudaStreamSynchronize(s));
    return SLA_OK;
}

// A solve status after which the gradient is still formed (x holds the last iterate).
static bool solved_or_stopped(sla_status st) {
    return st == SLA_OK || st == SLA_ERR_NOT_CONVERGED || st == SLA_ERR_BREAKDOWN || st == SLA_ERR_TIMEOUT;
}

sla_status sla_adjoint(sla_handle h, const void* d_x, const void* d_g, const sla_pcg_opts* opts, void* d_dLdb,
                       void* d_dLdA, sla_solve_info* info, void* stream) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (!d_x || !d_g || !d_dLdb) return fail(SLA_ERR_INVALID, "null vector");
    TRY(check_opts(opts));
    cudaStream_t s = (cudaStream_t)stream;
    sla_pcg_opts o = *opts;
    o.use_x0 = 0;
    sla_status st = h->dt == SLA_F64
                        ? solve_impl<double>(h, (const double*)d_g, (double*)d_dLdb, &o, info, s)
                        : solve_impl<float>(h, (const float*)d_g, (float*)d_dLdb, &o, info, s);
    if (!solved_or_stopped(st)) return st;
    TRY(grad_A(h, d_x, d_dLdb, d_dLdA, s));
    return st;
}

static sla_status check_bicg(sla_handle h, const sla_pcg_opts* o) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    TRY(check_opts(o));
    if (o->pc == SLA_PC_SPAI) return fail(SLA_ERR_INVALID, "BiCGStab takes SLA_PC_NONE or SLA_PC_JACOBI");
    if (h->dt != SLA_F64) return fail(SLA_ERR_UNSUPPORTED, "BiCGStab is built for fp64 systems only");
    return SLA_OK;
}

sla_status sla_bicgstab_solve(sla_handle h, const void* d_b, void* d_x, const sla_pcg_opts* opts,
                              sla_solve_info* info, void* stream) {
    TRY(check_bicg(h, opts));
    if (!d_b || !d_x) return fail(SLA_ERR_INVALID, "null vector");
    return bicg_impl(h, false, (const double*)d_b, (double*)d_x, opts, info, (cudaStream_t)stream);
}

sla_status sla_bicgstab_adjoint(sla_handle h, const void* d_x, const void* d_g, const sla_pcg_opts* opts,
                                void* d_dLdb, void* d_dLdA, sla_solve_info* info, void* stream) {
    TRY(check_bicg(h, opts));
    if (!d_x || !d_g || !d_dLdb) return fail(SLA_ERR_INVALID, "null vector");
    cudaStream_t s = (cudaStream_t)stream;
    sla_pcg_opts o = *opts;
    o.use_x0 = 0;
    sla_status st = bicg_impl(h, true, (const double*)d_g, (double*)d_dLdb, &o, info, s);
    if (!solved_or_stopped(st)) return st;
    TRY(grad_A(h, d_x, d_dLdb, d_dLdA, s));
    return st;
}

// Thread-FMA rate of the fp64 pipe: every thread runs PROBE_CHAINS
// independent chains of dependent fp64 FMAs (enough in flight to keep the
// pipe issuing), on a grid of every SM at full occupancy.  The result is
// stored so the chains are not optimised away.
static constexpr int PROBE_CHAINS = 8;
__global__ void __launch_bounds__(NT) k_fp64_probe(double* out, int iters, double m, double c) {
    double a[PROBE_CHAINS];
#pragma unroll
    for (int j = 0; j < PROBE_CHAINS; ++j) a[j] = 1e-3 * (threadIdx.x + j);
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < PROBE_CHAINS; ++j) a[j] = fma(a[j], m, c);
    }
    double t = 0.0;
#pragma unroll
    for (int j = 0; j < PROBE_CHAINS; ++j) t += a[j];
    out[blockIdx.x * NT + threadIdx.x] = t;
}

sla_status sla_fp64_fma_rate(double* fma_per_s, void* stream) {
    if (!fma_per_s) return fail(SLA_ERR_INVALID, "null output");
    cudaStream_t s = (cudaStream_t)stream;
    int dev = 0, sms = 0, per = 0;
    CU(cudaGetDevice(&dev));
    CU(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    CU(cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, k_fp64_probe, NT, 0));
    if (per < 1) per = 1;
    const int grid = per * sms;
    DevBuf out;
    TRY(out.alloc(sizeof(double) * (size_t)grid * NT));
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    CU(cudaEventCreate(&e0));
    CU(cudaEventCreate(&e1));
    const int iters = 4096;
    float best = 0.0f;
    sla_status st = SLA_OK;
    for (int rep = 0; rep < 4 && st == SLA_OK; ++rep) {   // the first launch warms up
        cudaEventRecord(e0, s);
        k_fp64_probe<<<grid, NT, 0, s>>>(out.as<double>(), iters, 0.999999, 1e-7);
        st = launched();
        cudaEventRecord(e1, s);
        if (st == SLA_OK && cudaEventSynchronize(e1) == cudaSuccess) {
            float ms = 0.0f;
            cudaEventElapsedTime(&ms, e0, e1);
            if (rep > 0 && (best == 0.0f || ms < best)) best = ms;
        }
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    TRY(st);
    if (!(best > 0.0f)) return fail(SLA_ERR_CUDA, "fp64 probe could not be timed");
    *fma_per_s = (double)grid * NT * iters * PROBE_CHAINS / (best * 1e-3);
    return SLA_OK;
}

// ===================================================================== block arithmetic
// CTAs per SM of the Gram kernel's grid.  Measured on B300 (LOBPCG on the
// 128^3 Laplacian, k = 8, block kept full, ms per iteration): 2 / 3 / 4 CTAs
// per SM 24.9 / 22.8 / 22.3 (the Gram matrices of LOBPCG need at most 4
// result entries per thread: 64 registers, 4 CTAs resident).
#ifndef SLA_GRAM_CTAS
#define SLA_GRAM_CTAS 4
#endif
static int gram_grid(long long n) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const long long chunks = (n + GRAM_COLS - 1) / GRAM_COLS;
    long long g = (long long)SLA_GRAM_CTAS * sms;
    if (g > chunks) g = chunks;
    return (int)(g < 1 ? 1 : g);
}

sla_status sla_block_gram_work(int ka, int kb, int mode, long long n, long long* doubles) {
    if (!doubles) return fail(SLA_ERR_INVALID, "null output");
    if (ka < 1 || kb < 1 || ka > GRAM_MAXK || kb > GRAM_MAXK)
        return fail(SLA_ERR_INVALID, "block sizes must be in [1, %d] (got %d, %d)", GRAM_MAXK, ka, kb);
    if (mode != GRAM_FULL && mode != GRAM_SYM && mode != GRAM_DIAG && mode != GRAM_UPPER)
        return fail(SLA_ERR_INVALID, "unknown mode %d", mode);
    if (mode != GRAM_FULL && ka != kb) return fail(SLA_ERR_INVALID, "this mode needs ka == kb");
    if (n < 0) return fail(SLA_ERR_INVALID, "n must be >= 0");
    *doubles = (long long)gram_grid(n > 0 ? n : 1) * gram_pairs(ka, kb, mode);
    return SLA_OK;
}

sla_status sla_block_gram(int ka, int kb, long long n, const double* d_A, const double* d_B, int mode, double* d_G,
                          double* d_work, long long work_doubles, void* stream) {
    long long need = 0;
    TRY(sla_block_gram_work(ka, kb, mode, n, &need));
    if (!d_A || !d_G || (!gram_one_block(mode) && !d_B) || !d_work) return fail(SLA_ERR_INVALID, "null pointer");
    if (work_doubles < need) return fail(SLA_ERR_INVALID, "workspace too small (%lld < %lld doubles)", work_doubles, need);
    cudaStream_t s = (cudaStream_t)stream;
    if (n == 0) {
        CU(cudaMemsetAsync(d_G, 0, sizeof(double) * (size_t)(mode == GRAM_DIAG ? ka : ka * kb), s));
        return SLA_OK;
    }
    const int grid = gram_grid(n);
    const double* B = gram_one_block(mode) ? d_A : d_B;
    const int ppt = (gram_pairs(ka, kb, mode) + NT - 1) / NT;   // result entries per thread
    if (ppt <= 2) k_gram_partial<2><<<grid, NT, 0, s>>>(ka, kb, n, d_A, B, mode, d_work);
    else if (ppt <= 4) k_gram_partial<4><<<grid, NT, 0, s>>>(ka, kb, n, d_A, B, mode, d_work);
    else if (ppt <= 8) k_gram_partial<8><<<grid, NT, 0, s>>>(ka, kb, n, d_A, B, mode, d_work);
    else k_gram_partial<GRAM_PER_THREAD><<<grid, NT, 0, s>>>(ka, kb, n, d_A, B, mode, d_work);
    TRY(launched());
    const int npairs = gram_pairs(ka, kb, mode);
    k_gram_reduce<<<(npairs + NT - 1) / NT, NT, 0, s>>>(ka, kb, mode, grid, d_work, d_G);
    return launched();
}

sla_status sla_block_update(int ks, int kc, long long n, const double* d_C, const double* d_S, const double* d_Yin,
                            double* d_Y, void* stream) {
    if (ks < 1 || kc < 1 || ks > GRAM_MAXK || kc > GRAM_MAXK)
        return fail(SLA_ERR_INVALID, "block sizes must be in [1, %d] (got %d, %d)", GRAM_MAXK, ks, kc);
    if (n < 0) return fail(SLA_ERR_INVALID, "n must be >= 0");
    if (!d_C || !d_S || !d_Y) return fail(SLA_ERR_INVALID, "null pointer");
    if (n == 0) return SLA_OK;
    cudaStream_t s = (cudaStream_t)stream;
    int dev = 0, sms = 148;
    CU(cudaGetDevice(&dev));
    CU(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    long long g = (n + NT - 1) / NT;
    if (g > 8LL * sms) g = 8LL * sms;
    k_block_update<<<(unsigned)g, NT, 0, s>>>(ks, kc, n, d_C, d_S, d_Yin, d_Y);
    return launched();
}

// ===================================================================== partitioned CG steps
static int local_grid(long long n) {
    int dev = 0, sms = 148;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    long long g = (n + NT - 1) / NT;
    if (g > 2LL * sms) g = 2LL * sms;
    return (int)(g < 1 ? 1 : g);
}

sla_status sla_cg_local_work(int n, long long* doubles) {
    if (!doubles) return fail(SLA_ERR_INVALID, "null output");
    if (n < 0) return fail(SLA_ERR_INVALID, "n must be >= 0");
    *doubles = 2LL * local_grid(n);
    return SLA_OK;
}

sla_status sla_cg_local_update(int n, double alpha, const double* d_p, const double* d_q, const double* d_dinv,
                               double* d_x, double* d_r, double* d_z, double* d_dots, double* d_work,
                               long long work_doubles, void* stream) {
    long long need = 0;
    TRY(sla_cg_local_work(n, &need));
    if ((n > 0 && (!d_p || !d_q || !d_x || !d_r || !d_z)) || !d_dots || !d_work)
        return fail(SLA_ERR_INVALID, "null pointer");
    if (work_doubles < need) return fail(SLA_ERR_INVALID, "workspace too small (%lld < %lld doubles)", work_doubles, need);
    cudaStream_t s = (cudaStream_t)stream;
    const int g = local_grid(n);
    k_cg_local_update<<<g, NT, 0, s>>>(n, alpha, d_p, d_q, d_dinv, d_x, d_r, d_z, d_work);
    TRY(launched());
    k_pair_reduce<<<1, 32, 0, s>>>(g, d_work, d_dots);
    return launched();
}

sla_status sla_cg_local_direction(int n, double beta, const double* d_z, double* d_p, void* stream) {
    if (n < 0) return fail(SLA_ERR_INVALID, "n must be >= 0");
    if (n > 0 && (!d_z || !d_p)) return fail(SLA_ERR_INVALID, "null pointer");
    if (n == 0) return SLA_OK;
    k_cg_local_direction<<<local_grid(n), NT, 0, (cudaStream_t)stream>>>(n, beta, d_z, d_p);
    return launched();
}

sla_status sla_grad_A(sla_handle h, const void* d_lam, const void* d_x, void* d_dLdA, void* stream) {
    if (!h) return fail(SLA_ERR_INVALID, "null handle");
    if (!d_lam || !d_x || (!d_dLdA && h->nnz > 0)) return fail(SLA_ERR_INVALID, "null vector");
    return grad_A(h, d_x, d_lam, d_dLdA, (cudaStream_t)stream);
}

sla_status sla_wait_selftest(int which, double limit_s, void* stream) {
    if (which != 0 && which != 1) return fail(SLA_ERR_INVALID, "which must be 0 (mbarrier) or 1 (grid barrier)");
    if (!(limit_s > 0.0) || limit_s > 1.0) return fail(SLA_ERR_INVALID, "limit_s must be in (0, 1]");
    cudaStream_t s = (cudaStream_t)stream;
    DevBuf ctl, gs;
    TRY(ctl.alloc(sizeof(Ctrl)));
    TRY(gs.alloc(sizeof(GridSync)));
    CU(cudaMemsetAsync(ctl.p, 0, sizeof(Ctrl), s));
    CU(cudaMemsetAsync(gs.p, 0, sizeof(GridSync), s));
    k_wait_selftest<<<2, 32, 0, s>>>(which, (unsigned long long)(limit_s * 1e9), ctl.as<Ctrl>(), gs.as<GridSync>());
    TRY(launched());
    Ctrl dc;
    CU(cudaMemcpyAsync(&dc, ctl.p, sizeof(Ctrl), cudaMemcpyDeviceToHost, s));
    CU(cudaStreamSynchronize(s));
    if (dc.err & (ERR_WAIT | ERR_GRID))
        return fail(SLA_ERR_CUDA, "a device wait gave up (%s; at %d: %d %d %d)",
                    (dc.err & ERR_GRID) ? "grid barrier" : "bulk copy", dc.diag[0], dc.diag[1], dc.diag[2],
                    dc.diag[3]);
    return SLA_OK;
}

}  // extern "C"

// ===================================================================== allocation-free SpMV + dot
// Scratch of sla_spmv_dot_static, in file-scope device memory instead of a
// handle: one arrival counter per system (first STATIC_COUNTER_BYTES) and the
// per-CTA partial sums of x.y (the rest).  Every GPU that loads this library
// holds these bytes until the process exits.  Host code must not pass the
// symbol itself to a kernel (on the host it names a host-side stand-in):
// static_scratch() looks up its device address once per device.
static constexpr int STATIC_MAX_BATCH = 64;
static constexpr int STATIC_COUNTER_BYTES = 256;                 // 64 counters, one per system
static constexpr int STATIC_PARTIALS = 4096;                     // partial sums shared by all systems
static constexpr size_t STATIC_SCRATCH_BYTES = STATIC_COUNTER_BYTES + STATIC_PARTIALS * sizeof(double);
static constexpr int STATIC_CAP = 256;                           // staged entries per 32-row group
static __device__ __align__(256) unsigned char g_static_scratch[STATIC_SCRATCH_BYTES];

static constexpr int STATIC_MAX_DEVICES = 64;
static std::mutex g_static_mu;
static void* g_static_ptr[STATIC_MAX_DEVICES] = {};

// Device address of g_static_scratch on the current device (looked up on the
// first call made with that device current, then cached).
static sla_status static_scratch(void** out) {
    int dev = 0;
    CU(cudaGetDevice(&dev));
    if (dev < 0 || dev >= STATIC_MAX_DEVICES) return fail(SLA_ERR_UNSUPPORTED, "device ordinal %d out of range", dev);
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
        void* ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess || !ptr)
            return fail(SLA_ERR_CUDA, "cudaGetSymbolAddress(scratch) failed: %s", cudaGetErrorString(e));
        g_static_ptr[dev] = ptr;
    }
    *out = g_static_ptr[dev];
    return SLA_OK;
}

template <typename T>
static sla_status spmv_dot_static_impl(int n, long long nnz, int batch, const int* rp, const int* ci,
                                       const T* vals, const T* x, T* y, double* dot, cudaStream_t s) {
    void* scratch = nullptr;
    TRY(static_scratch(&scratch));
    TRY(allow_smem<T>());
    int dev = 0, sms = 0, per = 0;
    CU(cudaGetDevice(&dev));
    CU(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    const size_t smem = spmv_smem(STATIC_CAP);
    TRY(occupancy(k_spmv<T, 1>, smem, &per));   // STATIC_CAP fits the pipelined form
    long long gx = (long long)per * sms / batch;
    if (gx > group_ctas(n, 1)) gx = group_ctas(n, 1);
    if (gx > STATIC_PARTIALS / batch) gx = STATIC_PARTIALS / batch;
    if (gx < 1) gx = 1;
    unsigned* counters = static_cast<unsigned*>(scratch);
    double* partials = reinterpret_cast<double*>(static_cast<unsigned char*>(scratch) + STATIC_COUNTER_BYTES);
    // The counters must start at zero; the partial sums are always written before they are read.
    CU(cudaMemsetAsync(counters, 0, sizeof(unsigned) * batch, s));
    Sys S;
    S.n = n;
    S.nnz = nnz;
    S.st = nullptr;    // k_spmv keeps no solver state
    S.ctl = nullptr;
    S.cnt = counters;
    S.part = partials;
    S.pstride = (int)gx;
    Layout L;
    L.cap = STATIC_CAP;
    L.lanes = 1;
    L.gasync = 0;
    L.form = 1;
    L.smem = smem;
    const Mat A = mat_of(rp, ci, n, nnz, L, nullptr);
    k_spmv<T, 1><<<dim3((unsigned)gx, batch), NT, smem, s>>>(A, S, vals, x, y, dot);
    return launched();
}

extern "C" sla_status sla_spmv_dot_static(int n, long long nnz, int batch, sla_dtype dt, const int* d_row_ptr,
                                          const int* d_col_idx, const void* d_vals, const void* d_x, void* d_y,
                                          double* d_dot, void* stream) {
    if (n < 1) return fail(SLA_ERR_INVALID, "n must be >= 1 (got %d)", n);
    if (nnz < 0 || nnz > 2147483647LL) return fail(SLA_ERR_INVALID, "nnz must be in [0, 2^31) (got %lld)", nnz);
    if (batch < 1 || batch > STATIC_MAX_BATCH)
        return fail(SLA_ERR_INVALID, "batch must be in [1, %d] for the allocation-free entry point (got %d)",
                    STATIC_MAX_BATCH, batch);
    if (dt != SLA_F64 && dt != SLA_F32) return fail(SLA_ERR_INVALID, "unknown dtype %d", (int)dt);
    if (!d_row_ptr || (nnz > 0 && (!d_col_idx || !d_vals)) || !d_x || !d_y || !d_dot)
        return fail(SLA_ERR_INVALID, "null pointer");
    cudaStream_t s = (cudaStream_t)stream;
    if (dt == SLA_F64)
        return spmv_dot_static_impl<double>(n, nnz, batch, d_row_ptr, d_col_idx, (const double*)d_vals,
                                            (const double*)d_x, (double*)d_y, d_dot, s);
    return spmv_dot_static_impl<float>(n, nnz, batch, d_row_ptr, d_col_idx, (const float*)d_vals,
                                       (const float*)d_x, (float*)d_y, d_dot, s);
}

