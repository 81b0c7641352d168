// block.cuh -- dense arithmetic on tall blocks of vectors (fp64), for the
// block eigensolver (torch-sla §3, .eigsh, here LOBPCG): the Gram matrix of
// two blocks and the product of a block with a small matrix.  A block of k
// vectors of length n is stored vector after vector ([k][n], row-major).
//
// Both are fp64-throughput bound (B300 issues 2 fp64 FMAs per clock per SM):
// the Gram matrix of blocks of ka and kb vectors is ka kb n FMAs, read from
// 8 (ka + kb) n bytes.  The kernels keep the fp64 pipe fed: the Gram kernel
// stages 32 columns of both blocks in shared memory per step and gives every
// thread a few entries of the small result; the update kernel keeps the
// small matrix in shared memory and each thread a column of the block.
#pragma once

#include "common.cuh"

namespace sla {

constexpr int GRAM_COLS = 32;    // columns of both blocks staged per step
constexpr int GRAM_MAXK = 64;    // largest block of either operand
constexpr int GRAM_PER_THREAD = (GRAM_MAXK * GRAM_MAXK + NT - 1) / NT;

// Modes of the Gram kernels: every entry, the upper triangle (A = B,
// mirrored), the diagonal only (A = B: the squared norms of A's vectors), or
// the upper triangle of A B^T for two blocks whose product is symmetric
// (such as S^T (A S) for a symmetric A), mirrored.
enum : int { GRAM_FULL = 0, GRAM_SYM = 1, GRAM_DIAG = 2, GRAM_UPPER = 3 };
__host__ __device__ constexpr bool gram_triangle(int mode) { return mode == GRAM_SYM || mode == GRAM_UPPER; }
__host__ __device__ constexpr bool gram_one_block(int mode) { return mode == GRAM_SYM || mode == GRAM_DIAG; }
__host__ __device__ constexpr int gram_pairs(int ka, int kb, int mode) {
    return mode == GRAM_FULL ? ka * kb : gram_triangle(mode) ? ka * (ka + 1) / 2 : ka;
}

// Entry p of the result: (i, j) = (p / kb, p % kb); in GRAM_SYM and
// GRAM_UPPER modes only i <= j, enumerated row by row; in GRAM_DIAG mode
// (p, p).
__device__ __forceinline__ void gram_pair(int p, int ka, int kb, int mode, int& i, int& j) {
    if (mode == GRAM_FULL) {
        i = p / kb;
        j = p - i * kb;
        return;
    }
    if (mode == GRAM_DIAG) {
        i = j = p;
        return;
    }
    // row i holds kb - i entries: find the row by walking (ka <= 64)
    i = 0;
    int start = 0;
    while (p >= start + (kb - i)) {
        start += kb - i;
        ++i;
    }
    j = i + (p - start);
}

// Partial Gram matrices: CTA c sums the column chunks c, c + gridDim.x, ...
// and writes its ka x kb (or upper-triangle) partial sums to part[c][...].
// PT: result entries per thread; the launch takes the fewest that cover the
// pairs, so small Gram matrices hold fewer registers and more CTAs fit.
template <int PT>
__global__ void __launch_bounds__(NT) k_gram_partial(int ka, int kb, long long n, const double* __restrict__ A,
                                                      const double* __restrict__ B, int mode,
                                                      double* __restrict__ part) {
    __shared__ double sA[GRAM_MAXK][GRAM_COLS + 1];
    __shared__ double sB[GRAM_MAXK][GRAM_COLS + 1];
    const bool sym = gram_one_block(mode);   // one operand: B = A
    const int npairs = gram_pairs(ka, kb, mode);
    double acc[PT];
    int pi[PT], pj[PT];
#pragma unroll
    for (int q = 0; q < PT; ++q) {
        acc[q] = 0.0;
        const int p = threadIdx.x + q * NT;
        if (p < npairs) gram_pair(p, ka, kb, mode, pi[q], pj[q]);
        else pi[q] = pj[q] = 0;
    }
    const long long nchunks = (n + GRAM_COLS - 1) / GRAM_COLS;
    for (long long ch = blockIdx.x; ch < nchunks; ch += gridDim.x) {
        const long long l0 = ch * GRAM_COLS;
        __syncthreads();   // the previous chunk's reads are done
        for (int t = threadIdx.x; t < ka * GRAM_COLS; t += NT) {
            const int r = t / GRAM_COLS, c = t - r * GRAM_COLS;
            const long long l = l0 + c;
            sA[r][c] = l < n ? ld_stream(A + (size_t)r * n + l) : 0.0;
        }
        if (!sym)
            for (int t = threadIdx.x; t < kb * GRAM_COLS; t += NT) {
                const int r = t / GRAM_COLS, c = t - r * GRAM_COLS;
                const long long l = l0 + c;
                sB[r][c] = l < n ? ld_stream(B + (size_t)r * n + l) : 0.0;
            }
        __syncthreads();
        const double(*tb)[GRAM_COLS + 1] = sym ? sA : sB;
#pragma unroll
        for (int q = 0; q < PT; ++q) {
            if (threadIdx.x + q * NT >= npairs) break;
            const double* ra = sA[pi[q]];
            const double* rb = tb[pj[q]];
            double s = acc[q];
#pragma unroll 8
            for (int c = 0; c < GRAM_COLS; ++c) s = fma(ra[c], rb[c], s);
            acc[q] = s;
        }
    }
#pragma unroll
    for (int q = 0; q < PT; ++q) {
        const int p = threadIdx.x + q * NT;
        if (p < npairs) part[(size_t)blockIdx.x * npairs + p] = acc[q];
    }
}

// G = the sum of the partials over the CTAs, in CTA order (deterministic);
// GRAM_SYM and GRAM_UPPER mirror the upper triangle; GRAM_DIAG writes G[i]
// (a vector).
__global__ void __launch_bounds__(NT) k_gram_reduce(int ka, int kb, int mode, int nparts,
                                                     const double* __restrict__ part, double* __restrict__ G) {
    const int npairs = gram_pairs(ka, kb, mode);
    for (int p = blockIdx.x * NT + threadIdx.x; p < npairs; p += gridDim.x * NT) {
        double s = 0.0;
        for (int c = 0; c < nparts; ++c) s += part[(size_t)c * npairs + p];
        if (mode == GRAM_DIAG) {
            G[p] = s;
            continue;
        }
        int i, j;
        gram_pair(p, ka, kb, mode, i, j);
        G[i * kb + j] = s;
        if (gram_triangle(mode)) G[j * kb + i] = s;
    }
}

// Y[r] = sum_i C[i][r] S[i] (+ Yin[r]) for r < kc: the block S ([ks][n])
// times the small matrix C ([ks][kc]), each thread a column of the block.
// Outputs go in groups of UPD_R (registers), inputs in groups of UPD_S.
// Yin may be Y (each entry is read once, then written by the same thread).
constexpr int UPD_R = 16;
constexpr int UPD_S = 8;
__global__ void __launch_bounds__(NT) k_block_update(int ks, int kc, long long n, const double* __restrict__ C,
                                                      const double* __restrict__ S, const double* Yin, double* Y) {
    __shared__ double sC[GRAM_MAXK * GRAM_MAXK];
    for (int t = threadIdx.x; t < ks * kc; t += NT) sC[t] = C[t];
    __syncthreads();
    for (long long l = blockIdx.x * (long long)NT + threadIdx.x; l < n; l += (long long)gridDim.x * NT) {
        for (int r0 = 0; r0 < kc; r0 += UPD_R) {
            double y[UPD_R];
#pragma unroll
            for (int u = 0; u < UPD_R; ++u)
                y[u] = (Yin && r0 + u < kc) ? Yin[(size_t)(r0 + u) * n + l] : 0.0;
            for (int i0 = 0; i0 < ks; i0 += UPD_S) {
                double sv[UPD_S];
#pragma unroll
                for (int v = 0; v < UPD_S; ++v) sv[v] = i0 + v < ks ? S[(size_t)(i0 + v) * n + l] : 0.0;
#pragma unroll
                for (int v = 0; v < UPD_S; ++v) {
                    if (i0 + v >= ks) break;
                    const double* crow = sC + (i0 + v) * kc + r0;
#pragma unroll
                    for (int u = 0; u < UPD_R; ++u)
                        if (r0 + u < kc) y[u] = fma(crow[u], sv[v], y[u]);
                }
            }
#pragma unroll
            for (int u = 0; u < UPD_R; ++u)
                if (r0 + u < kc) Y[(size_t)(r0 + u) * n + l] = y[u];
        }
    }
}

// ----------------------------------------------------------------- local CG steps of a partitioned solve
// One rank's part of a CG step on its owned entries (n of them): x += alpha p,
// r -= alpha q, z = dinv * r (z = r without dinv), and its partial sums of
// r.r and r.z (per CTA, summed in CTA order by k_pair_reduce).
__global__ void __launch_bounds__(NT) k_cg_local_update(int n, double alpha, const double* __restrict__ p,
                                                         const double* __restrict__ q,
                                                         const double* __restrict__ dinv, double* __restrict__ x,
                                                         double* __restrict__ r, double* __restrict__ z,
                                                         double* __restrict__ part) {
    __shared__ double red[RED_DOUBLES];
    double v[2] = {0.0, 0.0};
    for (int i = blockIdx.x * NT + threadIdx.x; i < n; i += gridDim.x * NT) {
        x[i] = fma(alpha, p[i], x[i]);
        const double ri = fma(-alpha, q[i], r[i]);
        r[i] = ri;
        const double zi = dinv ? ri * dinv[i] : ri;
        z[i] = zi;
        v[0] = fma(ri, ri, v[0]);
        v[1] = fma(ri, zi, v[1]);
    }
    block_sum<2>(v, red);
    if (threadIdx.x == 0) {
        part[2 * blockIdx.x] = v[0];
        part[2 * blockIdx.x + 1] = v[1];
    }
}

__global__ void __launch_bounds__(32) k_pair_reduce(int nparts, const double* __restrict__ part,
                                                     double* __restrict__ out) {
    if (threadIdx.x < 2) {
        double s = 0.0;
        for (int c = 0; c < nparts; ++c) s += part[2 * c + threadIdx.x];
        out[threadIdx.x] = s;
    }
}

// p = z + beta p on the owned entries.
__global__ void __launch_bounds__(NT) k_cg_local_direction(int n, double beta, const double* __restrict__ z,
                                                            double* __restrict__ p) {
    for (int i = blockIdx.x * NT + threadIdx.x; i < n; i += gridDim.x * NT) p[i] = fma(beta, p[i], z[i]);
}

}  // namespace sla
