// common.cuh -- shared device definitions of the sm_103a CSR PCG library:
// per-system solver state, deterministic block/grid reductions, storage
// precision helpers and cache-hinted loads.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

namespace sla {

constexpr int NT = 256;          // threads per CTA for every kernel here
constexpr int NWARP = NT / 32;
constexpr int SPMV_MIN_CTAS = 4; // resident CTAs per SM the staged-SpMV kernels are compiled for
// Resident CTAs per SM the CG product kernel (which also carries the residual
// check) is compiled for: fp64 measured faster unspilled at 3 than spilled
// at 4; fp32 fits 4 unspilled.
#ifndef SLA_ITER_CTAS_F64
#define SLA_ITER_CTAS_F64 3
#endif
template <typename T> struct IterMinCtas { static constexpr int value = SLA_ITER_CTAS_F64; };
template <> struct IterMinCtas<float> { static constexpr int value = 4; };
// Resident CTAs per SM the product kernels are compiled for in the direct
// form (thread per row, no staging): occupancy is what hides its latency.
// Measured on B300 inside the running iteration (c4, c2): 4 beats 6 and 8,
// which thrash the caches the iteration's other kernels leave filled.
#ifndef SLA_DIRECT_CTAS
#define SLA_DIRECT_CTAS 4
#endif
// The sliced form (no staging either) is compiled twice: FORM 6 for
// SLA_SLICED_CTAS resident CTAs per SM (long rows, whose scattered gathers
// want the caches to themselves: on the kNN Laplacian 5 and 6 CTAs per SM
// took 270 and 303 us against 191 us at 4) and FORM 7 for SLA_SLICED_CTAS_SHORT
// (short rows: the 3D 7-point product 51.4 us at 5 against 55.6 us at 4).
#ifndef SLA_SLICED_CTAS
#define SLA_SLICED_CTAS 4
#endif
#ifndef SLA_SLICED_CTAS_SHORT
#define SLA_SLICED_CTAS_SHORT 5
#endif
__host__ __device__ constexpr bool sliced_form(int form) { return form == 6 || form == 7; }
// fp32 systems (fp32 values, double-float vectors) in the short-row form
// take 8 (32 registers, a few spilled): measured on 64 fp32 systems on one
// 256^2 5-point grid, 5 / 6 / 8 CTAs per SM 570k / 578k / 595k
// system-iterations/s (product 53.7 / 52.5 / 49.5 us; 7 compiles to the
// same 32 registers as 8).  fp64 keeps 5 (6 slowed the 2D and 3D grids by
// 6% and 3%).
#ifndef SLA_SLICED_CTAS_SHORT_F32
#define SLA_SLICED_CTAS_SHORT_F32 8
#endif
template <typename T, int FORM> struct ProductCtas {
    static constexpr int value = FORM == 5   ? SLA_DIRECT_CTAS
                                 : FORM == 6 ? SLA_SLICED_CTAS
                                 : FORM == 7 ? (sizeof(T) == 4 ? SLA_SLICED_CTAS_SHORT_F32 : SLA_SLICED_CTAS_SHORT)
                                             : IterMinCtas<T>::value;
};

// Outcome codes mirrored from sla_status (kept numerically equal).
enum : int { ST_OK = 0, ST_NOT_CONVERGED = 4, ST_BREAKDOWN = 5 };
// Device error bit in Ctrl::err.
enum : int { ERR_WAIT = 1 << 8, ERR_GRID = 1 << 9, ERR_STAGE = 1 << 10 };
// Record where the first wait gave up (diagnostics for the host's message).
__device__ __forceinline__ void note_wait(int* diag, int who, int a, int b, int c) {
    if (atomicCAS(diag, 0, who) == 0) {
        diag[1] = a;
        diag[2] = b;
        diag[3] = c;
    }
}

// Solver state of one system, in device memory.  Written only by the last
// CTA of a kernel (thread 0), read by every CTA of the following kernels.
struct State {
    double rho;       // r.z of the current direction
    double alpha;     // rho / p.q of the current iteration
    double beta;      // r.z(new) / r.z(old)
    double gamma;     // r.r after the last update
    double bb;        // b.b
    double tol2bb;    // tol^2 * b.b
    double tr2;       // ||b - A x||^2 of the last true-residual check
    double delta;     // p.q of the last iteration (BiCGStab: r^.v)
    double omega;     // BiCGStab: the stabilising step (t.s) / (t.t)
    int iter;         // products A p done in the loop
    int max_iter;
    int done;         // 1: frozen (converged, not converged at cap, or breakdown)
    int status;       // ST_*
    int check;        // 1: the recursive residual met tol; next SpMV pass checks the true residual
    int rho_bad;      // r.z <= 0 seen while a check was pending
    int phase;        // 0 = set-up (p = z), 1 = iterating
    int xpend;        // x += alpha p of the current iteration not yet applied
};

// Batch-wide control block (per-system CTA arrival counters live in a
// separate array, one per system, each reset by the last CTA to arrive).
struct Ctrl {
    int all_done;     // every system frozen
    int ndone;        // systems frozen so far
    int err;          // error bits (ERR_WAIT: a bulk-copy wait gave up; ERR_GRID: a grid barrier did)
    int pad;
    int diag[4];      // where the first wait gave up: CTA + 1 (negative for a copy wait), then details
};

// ----------------------------------------------------------------- loads
template <typename T>
__device__ __forceinline__ T ld_stream(const T* p) { return __ldcs(p); }   // evict-first
template <typename T>
__device__ __forceinline__ T ld_nc(const T* p) { return __ldg(p); }        // read-only path
template <typename T>
__device__ __forceinline__ T ld_cg(const T* p) { return __ldcg(p); }       // L2 only (coherent)
// Plain (weak, L1-cached) loads the compiler cannot turn into read-only-path
// loads: for vectors a persistent kernel rewrites between grid barriers
// (the read-only path may only serve data no thread writes during the kernel).
__device__ __forceinline__ double ld_coh(const double* p) {
    double v;
    asm volatile("ld.global.f64 %0, [%1];\n" : "=d"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float ld_coh(const float* p) {
    float v;
    asm volatile("ld.global.f32 %0, [%1];\n" : "=f"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ float2 ld_coh(const float2* p) {
    float2 v;
    asm volatile("ld.global.v2.f32 {%0, %1}, [%2];\n" : "=f"(v.x), "=f"(v.y) : "l"(p));
    return v;
}

// Asynchronous global -> shared copies (cp.async, 4 or 8 bytes per thread),
// cached at L1 with an L2 evict-first policy: the streamed matrix arrays are
// read once per product and must not push the gathered vector out of L2.
__device__ __forceinline__ unsigned long long l2_evict_first() {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
// For gathered vector entries, which every product re-reads: keep them in L2.
__device__ __forceinline__ unsigned long long l2_evict_last() {
    unsigned long long pol;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
// SLA_L2_KEEP = 1 marks every working-vector access L2 evict-last and the
// matrix stream evict-first, so that the vectors (read and rewritten every
// iteration) would stay resident in L2.  Measured on B300 (c2, c4, the 3D
// convection-diffusion BiCGStab): no change in iterations per second, since
// the iteration is bound by fp64 throughput and load latency rather than by
// the vectors' HBM traffic; off by default.  Policies come from a pure asm,
// so the compiler hoists them out of loops.
#ifndef SLA_L2_KEEP
#define SLA_L2_KEEP 0
#endif
__device__ __forceinline__ unsigned long long pol_keep() {
    unsigned long long pol;
    asm("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
__device__ __forceinline__ unsigned long long pol_stream() {
    unsigned long long pol;
    asm("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;\n" : "=l"(pol));
    return pol;
}
// 4-, 8- and 16-byte loads and stores with an L2 policy (any trivially
// copyable type of that size).  NC: read-only path (data not written during
// the kernel).
template <bool NC, typename T>
__device__ __forceinline__ T ld_pol(const T* p, unsigned long long pol) {
    static_assert(sizeof(T) == 4 || sizeof(T) == 8 || sizeof(T) == 16, "size");
    T out;
    if constexpr (sizeof(T) == 4) {
        unsigned v;
        if (NC) asm("ld.global.nc.L2::cache_hint.b32 %0, [%1], %2;\n" : "=r"(v) : "l"(p), "l"(pol));
        else asm("ld.global.L2::cache_hint.b32 %0, [%1], %2;\n" : "=r"(v) : "l"(p), "l"(pol));
        memcpy(&out, &v, 4);
    } else if constexpr (sizeof(T) == 8) {
        unsigned long long v;
        if (NC) asm("ld.global.nc.L2::cache_hint.b64 %0, [%1], %2;\n" : "=l"(v) : "l"(p), "l"(pol));
        else asm("ld.global.L2::cache_hint.b64 %0, [%1], %2;\n" : "=l"(v) : "l"(p), "l"(pol));
        memcpy(&out, &v, 8);
    } else {
        unsigned long long a, b;
        if (NC) asm("ld.global.nc.L2::cache_hint.v2.b64 {%0, %1}, [%2], %3;\n" : "=l"(a), "=l"(b) : "l"(p), "l"(pol));
        else asm("ld.global.L2::cache_hint.v2.b64 {%0, %1}, [%2], %3;\n" : "=l"(a), "=l"(b) : "l"(p), "l"(pol));
        unsigned long long v[2] = {a, b};
        memcpy(&out, v, 16);
    }
    return out;
}
template <typename T>
__device__ __forceinline__ void st_pol(T* p, const T& val, unsigned long long pol) {
    static_assert(sizeof(T) == 4 || sizeof(T) == 8 || sizeof(T) == 16, "size");
    if constexpr (sizeof(T) == 4) {
        unsigned v;
        memcpy(&v, &val, 4);
        asm volatile("st.global.L2::cache_hint.b32 [%0], %1, %2;\n" :: "l"(p), "r"(v), "l"(pol) : "memory");
    } else if constexpr (sizeof(T) == 8) {
        unsigned long long v;
        memcpy(&v, &val, 8);
        asm volatile("st.global.L2::cache_hint.b64 [%0], %1, %2;\n" :: "l"(p), "l"(v), "l"(pol) : "memory");
    } else {
        unsigned long long v[2];
        memcpy(v, &val, 16);
        asm volatile("st.global.L2::cache_hint.v2.b64 [%0], {%1, %2}, %3;\n" :: "l"(p), "l"(v[0]), "l"(v[1]), "l"(pol)
                     : "memory");
    }
}
// A working-vector load / store (kept in L2 when SLA_L2_KEEP) and a matrix
// stream load (evict-first).
template <typename T>
__device__ __forceinline__ T ld_vec(const T* p) {
    if constexpr (SLA_L2_KEEP) return ld_pol<false>(p, pol_keep());
    else return *p;
}
template <typename T>
__device__ __forceinline__ T ld_vec_last(const T* p) {   // last read of the vector in this kernel
    if constexpr (SLA_L2_KEEP) return ld_pol<false>(p, pol_keep());
    else return __ldcs(p);
}
template <typename T>
__device__ __forceinline__ void st_vec(T* p, const T& v) {
    if constexpr (SLA_L2_KEEP) st_pol(p, v, pol_keep());
    else *p = v;
}
template <typename T>
__device__ __forceinline__ T ld_mat(const T* p) {
    if constexpr (SLA_L2_KEEP) return ld_pol<true>(p, pol_stream());
    else return __ldcs(p);
}

template <int BYTES>
__device__ __forceinline__ void cp_async(void* smem, const void* gmem, unsigned long long pol) {
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.ca.shared.global.L2::cache_hint [%0], [%1], %2, %3;\n" ::"r"(s), "l"(gmem), "n"(BYTES),
                 "l"(pol)
                 : "memory");
}
__device__ __forceinline__ void cp_commit() { asm volatile("cp.async.commit_group;\n" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N) : "memory"); }

// ----------------------------------------------------------------- bulk copies
// One-shot mbarriers (one arrival per phase, completion counted in bytes)
// and bulk asynchronous global -> shared copies (cp.async.bulk): the copy
// engine moves a contiguous range of 16-byte units and signals the
// barrier when its bytes have landed.
__device__ __forceinline__ unsigned smem_u32(const void* p) { return (unsigned)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// Ends a barrier's life: required before its memory is used for anything
// else (including another mbar_init), once no arrival or copy is pending.
__device__ __forceinline__ void mbar_inval(unsigned long long* bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// Makes initialised barriers visible to the asynchronous (copy) proxy.
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}
// Orders this thread's earlier shared-memory accesses before later
// asynchronous-proxy accesses (a stage is refilled after it was read).
#ifndef SLA_PROXY_FENCE
#define SLA_PROXY_FENCE 1
#endif
__device__ __forceinline__ void fence_proxy_async() {
#if SLA_PROXY_FENCE
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
#endif
}

__device__ __forceinline__ void mbar_arrive_expect(unsigned long long* bar, unsigned bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
// One arrival (count 1).
__device__ __forceinline__ void mbar_arrive(unsigned long long* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
// An arrival on `bar` once every cp.async this thread issued so far has
// landed (the barrier's expected count includes these arrivals).
__device__ __forceinline__ void cp_async_arrive(unsigned long long* bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];\n" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_test(unsigned long long* bar, unsigned parity) {
    unsigned ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
__device__ __forceinline__ unsigned long long global_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}
// Wait for phase `parity` of `bar` to complete; gives up (returns false)
// after about WAIT_LIMIT_NS, so a copy that never lands cannot hang the GPU.
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;   // 1 s
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity,
                                          unsigned long long limit_ns = WAIT_LIMIT_NS) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (unsigned k = 1; k < (1u << 30); ++k) {
        if (mbar_test(bar, parity)) return true;
        if ((k & 255u) == 0 && global_ns() - t0 > limit_ns) return false;
    }
    return false;
}
// `bytes` (a multiple of 16) from global `src` to shared `dst`, both 16-byte
// aligned; completion is counted on `bar`.
__device__ __forceinline__ void bulk_copy(void* dst, const void* src, unsigned bytes, unsigned long long* bar,
                                          unsigned long long pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;\n" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Value stored at the system's precision, returned as the fp64 value it holds.
template <typename T>
__device__ __forceinline__ double rnd(double v) { return (double)(T)v; }

// ----------------------------------------------------------------- reductions
__device__ __forceinline__ double warp_sum(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_down_sync(0xffffffffu, v, o);
    return v;
}

// Sum NV values over the CTA in a fixed order; the result is valid in thread 0.
// Every thread parks its values in shared memory and warp 0 alone adds
// them up (NT / 32 per lane, then a shuffle tree): on B300 every fp64 add
// of every lane costs issue slots of the narrow fp64 pipe, so a shuffle
// tree in all warps (5 adds per value per thread) was measurably slower.
constexpr int RED_DOUBLES = 2 * NT;   // shared memory of block_sum<2>
template <int NV>
__device__ __forceinline__ void block_sum(double (&v)[NV], double* sm /* [NV][NT] */) {
    static_assert(NV * NT <= RED_DOUBLES, "reduction buffer too small");
    __syncthreads();   // the buffer may still be read by an earlier reduction
#pragma unroll
    for (int j = 0; j < NV; ++j) sm[j * NT + threadIdx.x] = v[j];
    __syncthreads();
    if (threadIdx.x < 32) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            double s = 0.0;
#pragma unroll
            for (int k = 0; k < NT / 32; ++k) s += sm[j * NT + k * 32 + threadIdx.x];
            v[j] = warp_sum(s);
        }
    }
    __syncthreads();
}

// Every CTA publishes NV partial sums at part[blockIdx.x * NV + j] and
// arrives on the counter; returns true in the last CTA to arrive, where
// `tot` then holds the grid totals (summed in CTA order: deterministic for a
// fixed grid).  The last CTA resets the counter.  Must be called by all
// threads of every CTA of the grid.
template <int NV>
__device__ __forceinline__ bool grid_sum(double (&v)[NV], double* part, unsigned* counter,
                                         double (&tot)[NV], double* sm) {
    __shared__ int s_last;
    block_sum<NV>(v, sm);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) part[blockIdx.x * NV + j] = v[j];
        __threadfence();
        unsigned prev = atomicAdd(counter, 1u);
        s_last = (prev == gridDim.x - 1);
    }
    __syncthreads();
    if (!s_last) return false;
    __threadfence();
    double acc[NV];
#pragma unroll
    for (int j = 0; j < NV; ++j) acc[j] = 0.0;
    for (int b = threadIdx.x; b < (int)gridDim.x; b += NT) {
#pragma unroll
        for (int j = 0; j < NV; ++j) acc[j] += ld_cg(part + b * NV + j);
    }
    block_sum<NV>(acc, sm);
    if (threadIdx.x == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) tot[j] = acc[j];
        *counter = 0u;
    }
    return true;
}

__device__ __forceinline__ bool finite(double v) { return isfinite(v); }

}  // namespace sla
