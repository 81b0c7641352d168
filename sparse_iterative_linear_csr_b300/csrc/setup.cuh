// setup.cuh -- once-per-pattern (and once-per-values) device set-up:
// CSR validation, diagonal extraction, the per-warp staging capacity of the
// SpMV, an exclusive scan, and the closed-form SPAI factor G on tril(A) with
// its explicit transpose.
#pragma once

#include "common.cuh"
#include "df.cuh"

namespace sla {

enum : int {
    ERR_ROWPTR = 1,       // row_ptr[0] != 0, row_ptr[n] != nnz, or decreasing
    ERR_COL_RANGE = 2,    // a column outside [0, n)
    ERR_COL_ORDER = 4,    // columns not strictly ascending within a row
    ERR_NO_DIAG = 8,      // some A_ii not stored
    ERR_DIAG_SIGN = 16,   // some A_ii <= 0 (or not finite)
    ERR_ASYM = 32,        // pattern not symmetric (G^T construction)
};

// Structure check, one thread per row.  Column reads stay inside
// [row_ptr[i], row_ptr[i+1]) only after that range was found valid.
__global__ void k_validate(int n, long long nnz, const int* __restrict__ rp, const int* __restrict__ ci,
                           int* err) {
    int bits = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int a = rp[i], b = rp[i + 1];
        if (i == 0 && a != 0) bits |= ERR_ROWPTR;
        if (i == n - 1 && (long long)b != nnz) bits |= ERR_ROWPTR;
        if (a < 0 || b < a || (long long)b > nnz) { bits |= ERR_ROWPTR; continue; }
        int prev = -1;
        for (int k = a; k < b; ++k) {
            const int c = ci[k];
            if (c < 0 || c >= n) bits |= ERR_COL_RANGE;
            if (c <= prev) bits |= ERR_COL_ORDER;
            prev = c;
        }
    }
    if (bits) atomicOr(err, bits);
}

// Position of column c in row i (columns ascending), or -1.
__device__ __forceinline__ int find_col(const int* __restrict__ ci, int a, int b, int c) {
    int lo = a, hi = b;
    while (lo < hi) {
        const int m = (lo + hi) >> 1;
        if (ci[m] < c) lo = m + 1; else hi = m;
    }
    return (lo < b && ci[lo] == c) ? lo : -1;
}

// diag[s*n + i] = A_ii of system s (fp64); error bits for a missing or a
// non-positive diagonal entry.
template <typename T>
__global__ void k_diag(int n, long long nnz, int batch, const int* __restrict__ rp, const int* __restrict__ ci,
                       const T* __restrict__ av, double* diag, int* err) {
    int bits = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int k = find_col(ci, rp[i], rp[i + 1], i);
        for (int s = 0; s < batch; ++s) {
            if (k < 0) { diag[(size_t)s * n + i] = 0.0; bits |= ERR_NO_DIAG; continue; }
            const double d = (double)av[(size_t)s * nnz + k];
            diag[(size_t)s * n + i] = d;
            if (!(d > 0.0) || !isfinite(d)) bits |= ERR_DIAG_SIGN;
        }
    }
    if (bits) atomicOr(err, bits);
}

// Stored form of an fp64 set-up value: fp64 itself, or a double-float pair
// for fp32 systems.
__device__ __forceinline__ void put(double* dst, double v) { *dst = v; }
__device__ __forceinline__ void put(float2* dst, double v) {
    const DF d = df_from_double(v);
    *dst = make_float2(d.hi, d.lo);
}

template <typename W>
__global__ void k_recip(size_t m, const double* __restrict__ d, W* __restrict__ dinv) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < m; i += (size_t)gridDim.x * blockDim.x)
        put(dinv + i, 1.0 / d[i]);
}

// ----------------------------------------------------------------- row groups
// Largest number of stored entries in any group of R consecutive rows (the
// shared-memory staging capacity a warp needs for the SpMV).
__global__ void k_group_max(const int* __restrict__ rp, int n, int R, int* out) {
    const long long ng = ((long long)n + R - 1) / R;
    int m = 0;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < ng; g += (long long)gridDim.x * blockDim.x) {
        const long long r0 = g * R;
        const long long r1 = r0 + R < n ? r0 + R : n;
        m = max(m, rp[r1] - rp[r0]);
    }
    if (m) atomicMax(out, m);
}

// Warp-wide fp64 steps of the two ways a staged warp can sum a group of 32
// rows (one lane per row), summed over the groups:
//   out[0]: a lane per row -- the group's longest row;
//   out[1]: the entries split evenly, C = ceil(cnt / 32) rounded up to odd
//           per lane, plus the shuffle-add rounds that join the pieces of
//           split rows (the most pieces any row of the group has past its
//           first).
// (balanced_group_sum in kernels.cuh is the second way.)
__global__ void k_walk_cost(const int* __restrict__ rp, int n, unsigned long long* out) {
    const long long ng = ((long long)n + 31) / 32;
    unsigned long long row_walk = 0, split_walk = 0;
    for (long long g = blockIdx.x * (long long)blockDim.x + threadIdx.x; g < ng; g += (long long)gridDim.x * blockDim.x) {
        const long long r0 = g * 32;
        const long long r1 = r0 + 32 < n ? r0 + 32 : n;
        const int k0 = rp[r0];
        const int cnt = rp[r1] - k0;
        if (cnt == 0) continue;
        const int C = ((cnt + 31) >> 5) | 1;
        int longest = 0, joins = 0;
        for (long long r = r0; r < r1; ++r) {
            const int lo = rp[r] - k0, hi = rp[r + 1] - k0;
            longest = max(longest, hi - lo);
            if (hi > lo) joins = max(joins, (hi - 1) / C - lo / C);
        }
        row_walk += longest;
        split_walk += C + joins;
    }
    if (row_walk) atomicAdd(out, row_walk);
    if (split_walk) atomicAdd(out + 1, split_walk);
}

// Largest staged range of a run of R consecutive rows (a warp-pipeline group
// or a producer/consumer tile), the range's ends rounded out to multiples of
// 4 entries as the bulk copies move it.
__global__ void k_chunk_max(const int* __restrict__ rp, int n, int R, int* out) {
    const long long nc = ((long long)n + R - 1) / R;
    int m = 0;
    for (long long c = blockIdx.x * (long long)blockDim.x + threadIdx.x; c < nc; c += (long long)gridDim.x * blockDim.x) {
        const long long r0 = c * R;
        const long long r1 = r0 + R < n ? r0 + R : n;
        const long long k0 = (long long)rp[r0] & ~3LL;
        const long long k1 = ((long long)rp[r1] + 3) & ~3LL;
        m = max(m, (int)(k1 - k0));
    }
    if (m) atomicMax(out, m);
}

// out[s * os + i] = in[s * is + map[i]] for i < m and every system s:
// permuted vectors (map = permutation) and permuted values (map = source
// entry of each permuted entry).
template <typename T>
__global__ void k_gather_map(long long m, int batch, const int* __restrict__ map, const T* __restrict__ in,
                             long long is, T* __restrict__ out, long long os) {
    const long long total = m * batch;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const long long s = t / m, i = t - s * m;
        out[s * os + i] = in[s * is + map[i]];
    }
}

// out[s * os + i] = in[s * is + map[i]], or 0 where map[i] < 0: the sliced
// copy of the values (map = source CSR entry of every sliced entry, -1 for
// padding).  T is an unsigned type of the value's size (bits are copied).
template <typename T>
__global__ void k_gather_map_pad(long long m, int batch, const int* __restrict__ map, const T* __restrict__ in,
                                 long long is, T* __restrict__ out, long long os) {
    const long long total = m * batch;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < total;
         t += (long long)gridDim.x * blockDim.x) {
        const long long s = t / m, i = t - s * m;
        const int k = map[i];
        out[s * os + i] = k >= 0 ? in[s * is + k] : T(0);
    }
}

// Sliced pattern: slot t = 32 * slice + lane holds row perm[t] (t itself
// when perm is null; >= n: an empty slot); its entry j (j < the slice's
// width) goes to sptr[slice] + 32 j + lane.  Entries past the row's length
// are padding: column = the row itself (0 for an empty slot), source -1.
__global__ void k_sell_fill(int n, int nslices, const int* __restrict__ rp, const int* __restrict__ ci,
                            const int* __restrict__ sptr, const int* __restrict__ perm, int* __restrict__ scol,
                            int* __restrict__ smap) {
    const long long slots = (long long)nslices * 32;
    for (long long t = blockIdx.x * (long long)blockDim.x + threadIdx.x; t < slots;
         t += (long long)gridDim.x * blockDim.x) {
        const int sl = (int)(t >> 5), lane = (int)(t & 31);
        const int base = sptr[sl];
        const int w = (sptr[sl + 1] - base) >> 5;
        const int row = perm ? perm[t] : (int)t;
        const int lo = row < n ? rp[row] : 0;
        const int len = row < n ? rp[row + 1] - lo : 0;
        const int fill = row < n ? row : 0;
        for (int j = 0; j < w; ++j) {
            const int idx = base + 32 * j + lane;
            scol[idx] = j < len ? ci[lo + j] : fill;
            smap[idx] = j < len ? lo + j : -1;
        }
    }
}

// Number of stored entries whose column is more than `w` away from the row.
__global__ void k_far_count(const int* __restrict__ rp, const int* __restrict__ ci, int n, int w,
                            unsigned long long* out) {
    unsigned long long c = 0;
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        for (int k = rp[i]; k < rp[i + 1]; ++k) c += (abs(ci[k] - i) > w);
    if (c) atomicAdd(out, c);
}

// ----------------------------------------------------------------- scan
// Exclusive prefix sum, SCAN_T threads x SCAN_V items per CTA; CTA totals go
// to `sums` and are scanned recursively by the host driver.
constexpr int SCAN_T = 1024, SCAN_V = 8, SCAN_TILE = SCAN_T * SCAN_V;

__global__ void __launch_bounds__(SCAN_T) k_scan_tile(int* d, long long m, int* sums) {
    __shared__ int wsum[SCAN_T / 32];
    const long long base = (long long)blockIdx.x * SCAN_TILE + (long long)threadIdx.x * SCAN_V;
    int v[SCAN_V], tsum = 0;
#pragma unroll
    for (int j = 0; j < SCAN_V; ++j) {
        v[j] = (base + j < m) ? d[base + j] : 0;
        const int t = v[j];
        v[j] = tsum;
        tsum += t;
    }
    const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
    int incl = tsum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {
        int s = wsum[lane];
        int si = s;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, si, o);
            if (lane >= o) si += y;
        }
        wsum[lane] = si - s;  // exclusive over warps
        if (lane == 31 && sums) sums[blockIdx.x] = si;
    }
    __syncthreads();
    const int off = wsum[w] + incl - tsum;
#pragma unroll
    for (int j = 0; j < SCAN_V; ++j)
        if (base + j < m) d[base + j] = v[j] + off;
}

__global__ void k_scan_add(int* d, long long m, const int* __restrict__ sums) {
    const long long base = (long long)blockIdx.x * SCAN_TILE;
    const int add = sums[blockIdx.x];
    for (int j = threadIdx.x; j < SCAN_TILE; j += blockDim.x)
        if (base + j < m) d[base + j] += add;
}

// ----------------------------------------------------------------- SPAI factor
// Closed-form factor on the pattern of tril(A) ("Learning Sparse Approximate
// Inverse Preconditioners ...": M^-1 = G G^T + eps I with G sparse lower
// triangular): G_ii = A_ii^-1/2, G_ij = -A_ij / (2 sqrt(A_ii A_jj)), j < i.
// Row i of G is the prefix of row i of A with columns <= i; row j of G^T
// holds G_ij for the columns i >= j of row j of A (the pattern is symmetric),
// each value read from row i of A, so G^T is a true transpose of G.

// cntG[i] = #{cols <= i in row i}, cntGT[i] = #{cols >= i in row i}
__global__ void k_tri_count(int n, const int* __restrict__ rp, const int* __restrict__ ci, int* cntG,
                            int* cntGT) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        const int a = rp[i], b = rp[i + 1];
        int lo = a, hi = b;  // first column > i
        while (lo < hi) {
            const int m = (lo + hi) >> 1;
            if (ci[m] <= i) lo = m + 1; else hi = m;
        }
        const int le = lo - a;
        const int has_diag = (lo > a && ci[lo - 1] == i);
        cntG[i] = le;
        cntGT[i] = (b - a) - le + has_diag;
    }
}

// rs[i] = 1 / sqrt(A_ii): the factor's entries are G_ii = rs_i and
// G_ij = -A_ij rs_i rs_j / 2, so each entry costs two products instead of a
// square root and a division (both long sequences on the fp64 pipe).
__global__ void k_rsqrt_diag(int n, const double* __restrict__ diag, double* __restrict__ rs) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        rs[i] = 1.0 / sqrt(diag[i]);
}

template <typename T, typename GV>
__global__ void k_fill_G(int n, const int* __restrict__ rp, const int* __restrict__ ci, const T* __restrict__ av,
                         const double* __restrict__ rs, const int* __restrict__ grp, int* gci, GV* gv) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
        int m = grp[i];
        const int end = grp[i + 1];
        const double ri = rs[i];
        for (int k = rp[i]; m < end; ++k, ++m) {
            const int j = ci[k];
            gci[m] = j;
            put(gv + m, (j == i) ? ri : -0.5 * (double)av[k] * ri * rs[j]);
        }
    }
}

// gtpos[m]: the entry of A whose value G^T's entry m takes (row i, column
// j of A for G^T's row j, column i; -1 for the diagonal).  The first fill
// (have_pos false) finds it by a search of row i and records it; later
// fills, after a values update, read it.
template <typename T, typename GV>
__global__ void k_fill_GT(int n, const int* __restrict__ rp, const int* __restrict__ ci, const T* __restrict__ av,
                          const double* __restrict__ rs, const int* __restrict__ gtrp, int* gtci, GV* gtv,
                          int* gtpos, bool have_pos, int* err) {
    int bits = 0;
    for (int j = blockIdx.x * blockDim.x + threadIdx.x; j < n; j += gridDim.x * blockDim.x) {
        int m = gtrp[j];
        const int end = gtrp[j + 1];
        const double rj = rs[j];
        const int b = rp[j + 1];
        for (int k = b - (end - m); k < b; ++k, ++m) {
            const int i = ci[k];   // i >= j
            gtci[m] = i;
            if (i == j) {
                if (!have_pos) gtpos[m] = -1;
                put(gtv + m, rj);
                continue;
            }
            int pos;
            if (have_pos) {
                pos = gtpos[m];
            } else {
                pos = find_col(ci, rp[i], rp[i + 1], j);
                gtpos[m] = pos;
            }
            if (pos < 0) { bits |= ERR_ASYM; put(gtv + m, 0.0); continue; }
            put(gtv + m, -0.5 * (double)av[pos] * rs[i] * rj);
        }
    }
    if (bits) atomicOr(err, bits);
}

}  // namespace sla
