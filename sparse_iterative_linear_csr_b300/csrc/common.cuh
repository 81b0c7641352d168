// common.cuh -- shared device definitions of the sm_103a CSR PCG library:
// per-system solver state, deterministic block/grid reductions, storage
// precision helpers and cache-hinted loads.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sla {

constexpr int NT = 256;          // threads per CTA for every kernel here
constexpr int NWARP = NT / 32;
constexpr int SPMV_MIN_CTAS = 4; // resident CTAs per SM the staged-SpMV kernels are compiled for
// Resident CTAs per SM the CG product kernel (which also carries the residual
// check) is compiled for: fp64 measured faster unspilled at 3 than spilled
// at 4; fp32 fits 4 unspilled.
template <typename T> struct IterMinCtas { static constexpr int value = 3; };
template <> struct IterMinCtas<float> { static constexpr int value = 4; };
constexpr int MAXR = NT;         // rows per row block (one row per thread)

// Outcome codes mirrored from sla_status (kept numerically equal).
enum : int { ST_OK = 0, ST_NOT_CONVERGED = 4, ST_BREAKDOWN = 5 };

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
    double delta;     // p.q of the last iteration
    int iter;         // products A p done in the loop
    int max_iter;
    int done;         // 1: frozen (converged, not converged at cap, or breakdown)
    int status;       // ST_*
    int check;        // 1: the recursive residual met tol; next SpMV pass checks the true residual
    int rho_bad;      // r.z <= 0 seen while a check was pending
    int phase;        // 0 = set-up (p = z), 1 = iterating
    int pad;
};

// Batch-wide control block (per-system CTA arrival counters live in a
// separate array, one per system, each reset by the last CTA to arrive).
struct Ctrl {
    int all_done;     // every system frozen
    int ndone;        // systems frozen so far
    int err;          // set-up / validation error bits
    int pad;
};

// ----------------------------------------------------------------- loads
template <typename T>
__device__ __forceinline__ T ld_stream(const T* p) { return __ldcs(p); }   // evict-first
template <typename T>
__device__ __forceinline__ T ld_nc(const T* p) { return __ldg(p); }        // read-only path
template <typename T>
__device__ __forceinline__ T ld_cg(const T* p) { return __ldcg(p); }       // L2 only (coherent)

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
template <int NV>
__device__ __forceinline__ void block_sum(double (&v)[NV], double* sm /* [NV][NWARP] */) {
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
#pragma unroll
    for (int j = 0; j < NV; ++j) v[j] = warp_sum(v[j]);
    __syncthreads();
    if (lane == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) sm[j * NWARP + w] = v[j];
    }
    __syncthreads();
    if (threadIdx.x == 0) {
#pragma unroll
        for (int j = 0; j < NV; ++j) {
            double s = 0.0;
#pragma unroll
            for (int k = 0; k < NWARP; ++k) s += sm[j * NWARP + k];
            v[j] = s;
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
