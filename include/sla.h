/*
 * sla.h -- C ABI of the B300 (sm_103a) sparse iterative linear solver:
 * preconditioned conjugate gradient on a CSR matrix and its adjoint, and
 * BiCGStab with its transpose adjoint for nonsymmetric systems.
 *
 * Sources of the operations (page title, then section):
 *  - "torch-sla: Differentiable Sparse Linear Algebra with Adjoint Solvers and
 *    Sparse Tensor Parallelism for PyTorch" (arXiv 2601.13994):
 *      §3 sparse tensor types: one matrix, or a batch of matrices sharing one
 *         sparsity pattern whose set-up is reused across the batch; the
 *         .matvec and .solve methods;
 *      §3 autograd wrapper: forward stashes (A, x), backward runs one adjoint
 *         solve;
 *      §3.3 distributed CG: the CG recurrence with the inner products <r,r>
 *         and <p,Ap>; the adjoint A^T lambda = dL/dx and the matrix gradient
 *         -lambda_i x_j on the stored non-zeros;
 *      §4 Table 3: CG with Jacobi preconditioning; §4 Figure 2: an absolute /
 *         relative stopping tolerance on the residual;
 *      §3 backends paragraph: BiCGStab beside CG among the iterative methods.
 *  - BiCGStab itself: van der Vorst, SIAM J. Sci. Stat. Comput. 13(2), 1992,
 *    as laid out in Barrett et al., "Templates for the Solution of Linear
 *    Systems" (SIAM, 1994), §2.3.8.
 *  - "Learning Sparse Approximate Inverse Preconditioners for Conjugate
 *    Gradient Solvers on GPUs" (author responses): the factored
 *    preconditioner M^-1 = G G^T + eps I applied with two SpMVs (Reviewer umir
 *    Concern 1; Reviewer GmV6 Concern 3 for eps).  G is the closed-form factor
 *    on the pattern of tril(A): G_ii = A_ii^-1/2,
 *    G_ij = -A_ij / (2 sqrt(A_ii A_jj)) for j < i.
 *
 * Conventions for every call
 *  - Pointers named d_* are device pointers owned by the caller.  The matrix
 *    arrays passed to sla_csr_create must stay alive and unchanged for the
 *    life of the handle (sla_csr_update_values swaps in new values).
 *  - CSR: row_ptr int32[n+1] with row_ptr[0] = 0 and row_ptr[n] = nnz;
 *    col_idx int32[nnz], strictly ascending within each row, 0 <= col < n;
 *    values [batch][nnz] in the handle's dtype (fp64 or fp32), system s at
 *    offset s*nnz.
 *  - Vectors of a batch are [batch][n], system s at offset s*n.
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  All device
 *    work of a call is ordered on it.  The solve and adjoint calls return
 *    after the solve has finished on the device (they synchronise `stream`);
 *    sla_spmv and sla_spmv_dot return without synchronising.
 *  - One call at a time per handle: the handle owns the solver workspace.
 *  - Every function returns SLA_OK or an error code; sla_last_error() gives
 *    a message for the calling thread's last error.
 */
#ifndef SLA_H
#define SLA_H

#ifdef __cplusplus
extern "C" {
#endif

typedef struct sla_csr* sla_handle;

typedef enum {
    SLA_OK = 0,
    SLA_ERR_INVALID = 1,        /* bad argument or malformed CSR */
    SLA_ERR_CUDA = 2,           /* a CUDA runtime call failed */
    SLA_ERR_NOMEM = 3,          /* device or pinned allocation failed */
    SLA_ERR_NOT_CONVERGED = 4,  /* max_iter reached; x holds the last iterate */
    SLA_ERR_BREAKDOWN = 5,      /* CG: p.Ap <= 0, r.z <= 0; BiCGStab: r^.r or r^.v = 0, omega = 0;
                                   or a non-finite value */
    SLA_ERR_TIMEOUT = 6,        /* host wall-clock limit; x holds the last iterate */
    SLA_ERR_UNSUPPORTED = 7     /* valid request this build does not serve */
} sla_status;

typedef enum { SLA_F64 = 0, SLA_F32 = 1 } sla_dtype;

typedef enum {
    SLA_PC_NONE = 0,    /* z = r */
    SLA_PC_JACOBI = 1,  /* z_i = r_i / A_ii */
    SLA_PC_SPAI = 2     /* z = G (G^T r) + eps r */
} sla_pc;

/* sla_csr_create flags */
#define SLA_VALIDATE 1u     /* check the CSR structure on the device; SLA_ERR_INVALID on failure */
#define SLA_WARP_PIPELINE 2u /* use the warp-pipeline product where it applies (see sla_csr_layout) */
#define SLA_PERSISTENT 4u    /* CG / Jacobi-PCG: one persistent iteration kernel per poll interval
                                instead of a CUDA graph of one kernel per step (see sla_pcg_solve) */
#define SLA_TIME_PRODUCT 8u  /* time one product kernel per graph launch (sla_product_time) */
#define SLA_PRODUCER_CONSUMER 16u /* use the producer/consumer product where it applies (see sla_csr_layout) */
#define SLA_REORDER 32u      /* always iterate on the reordered matrix (see sla_pcg_solve) */
#define SLA_NO_REORDER 64u   /* never reorder */
#define SLA_STAGED 128u      /* never use the direct or sliced product forms, for any matrix of the
                                solves (see sla_csr_layout) */
#define SLA_SLICED 256u      /* use the sliced product form wherever it pads little, also for the
                                SPAI factors (see sla_csr_layout) */
#define SLA_SPLIT_ROWS 512u  /* staged forms 1 and 2 with one lane per row: always sum a group with
                                its entries split evenly over the lanes (see sla_csr_layout) */
#define SLA_ROW_WALK 1024u   /* never split a group's entries: every lane sums its own row
                                (takes precedence over SLA_SPLIT_ROWS) */

typedef struct {
    double tol;        /* stop when ||r||_2 <= tol ||b||_2 and the true residual of
                          the returned x meets the same bound; tol > 0 */
    int max_iter;      /* cap on iterations per system (CG: products A p; BiCGStab:
                          iterations of two products); >= 0 */
    sla_pc pc;         /* preconditioner */
    double eps;        /* SPAI shift (ignored otherwise), >= 0 */
    int poll_k;        /* iterations between host checks of the device flag; 0 = default (32) */
    int use_x0;        /* nonzero: d_x holds the initial guess on entry */
    double timeout_s;  /* host wall-clock limit per call; <= 0 = none */
} sla_pcg_opts;

typedef struct {
    int iters;                 /* iterations performed in the loop (CG: products A p;
                                  BiCGStab: iterations of two products) */
    double rel_res_recursive;  /* ||r||_2 / ||b||_2 of the recursively updated r */
    double rel_res_true;       /* ||b - A x||_2 / ||b||_2 for the returned x */
    sla_status status;         /* per-system outcome */
} sla_solve_info;

/* Fill *o with defaults: tol 1e-8, max_iter 10000, SLA_PC_NONE, eps 1e-3,
 * poll_k 32, use_x0 0, timeout_s 0.  The keyword defaults of torch-sla §3
 * (.solve with per-call overrides); eps = 1e-3 is the learned-SPAI shift
 * (Reviewer GmV6 Concern 3). */
void sla_pcg_opts_default(sla_pcg_opts* o);

/*
 * Create a handle for an n x n CSR matrix (or a batch of `batch` matrices on
 * one pattern).  Defined by torch-sla §3, sparse tensor types: one sparse
 * matrix, or a batch of matrices that share one sparsity pattern so that the
 * set-up done once (here the analysis below; there the symbolic
 * factorisation or communication buffers) is reused across the batch and
 * across solves.  Analyses the pattern on the device: the product layout
 * (sla_csr_layout), the diagonal, and on first SPAI use the factor G and its
 * explicit transpose.
 * n >= 1, 0 <= nnz < 2^31, batch >= 1.  The handle keeps the three pointers
 * (it copies nothing but derived data).  With SLA_VALIDATE the structure is
 * checked first (monotone row_ptr, row_ptr[0] = 0, row_ptr[n] = nnz, columns
 * in range and strictly ascending).  A missing or non-positive diagonal entry
 * is reported when a solve asks for a preconditioner that needs it.
 * Synchronises `stream`.
 */
sla_status sla_csr_create(int n, long long nnz, int batch, sla_dtype dt,
                          const int* d_row_ptr, const int* d_col_idx, const void* d_vals,
                          unsigned flags, void* stream, sla_handle* out);

/*
 * Product layout of the matrix the solves iterate on -- A, or P A P^T when
 * the handle reorders (see sla_pcg_solve) -- for diagnostics.  The pages have
 * no counterpart (it reports this implementation's choices):
 *  *form: 0 register-staged warp groups, 1 warp groups with asynchronous
 *         value/column staging, 2 the same with asynchronous gathers,
 *         3 the warp pipeline (each warp bulk-copies its 32-row groups into
 *         a ring of shared-memory stages; needs 16-byte aligned row_ptr,
 *         col_idx and values of every system, and groups that fit shared
 *         memory; only with SLA_WARP_PIPELINE);
 *         4 producer/consumer warps (2 warps bulk-copy and gather tiles of
 *         192 rows into a ring of shared-memory stages, 6 warps add; same
 *         alignment conditions; only with SLA_PRODUCER_CONSUMER, which
 *         takes precedence over SLA_WARP_PIPELINE);
 *         5 direct: one thread per row, no shared-memory staging, kernels
 *         built for high occupancy -- the default whenever no row has more
 *         than 16 entries and the sliced form (below) does not apply, unless
 *         SLA_STAGED, SLA_WARP_PIPELINE or SLA_PRODUCER_CONSUMER asks
 *         otherwise; otherwise 0, 1 or 2;
 *         6 and 7 sliced (not with SLA_STAGED, SLA_WARP_PIPELINE or
 *         SLA_PRODUCER_CONSUMER): a handle-owned copy of the iteration
 *         matrix in slices of 32 rows stored column by column (rows
 *         reordered by length within windows of 256, 1024 or 4096 rows when
 *         that pads less), used when padding adds at most 15% entries; one
 *         thread per row, coalesced value and column loads; 6 for rows of
 *         at least 8 entries on average, 7 (more resident CTAs) for
 *         shorter ones.  The default for the iteration matrix when some row
 *         has more than 16 entries and rows hold at least 12 on average, or
 *         when no row has more than 16 and rows hold at least 4.5 on average;
 *         with SLA_SLICED wherever it applies, the SPAI factors included.
 *         Costs (8 + value size) bytes per sliced entry of device memory,
 *         and the values are copied again by sla_csr_update_values.
 *         The SPAI factors G and G^T take the sliced form whenever rows
 *         sorted within windows of 256 rows pad them by at most 20% (unless
 *         SLA_STAGED, SLA_WARP_PIPELINE or SLA_PRODUCER_CONSUMER), else
 *         their forms by the rule above; a sliced matrix whose rows are
 *         sorted within windows of 256 rows runs a warp per window, with the
 *         per-row work after the sums (the vector updates) in row order;
 *         the BiCGStab products always take a staged form (0, 1 or 2).
 *         In forms 1 and 2 with one lane per row a warp sums its group of
 *         32 rows either lane by lane (each lane its own row: as many
 *         warp-wide fp64 steps as the group's longest row) or split (the
 *         group's entries cut into 32 even runs, one per lane, the pieces of
 *         cut rows joined by shuffles in lane order).  The split is taken
 *         when the lane-per-row walk would cost at least 1.8 times as many
 *         warp-wide fp64 steps over the whole matrix (groups holding a few
 *         rows far longer than the rest), always with SLA_SPLIT_ROWS, never
 *         with SLA_ROW_WALK;
 *  *ctas: CTAs per system of the product kernels;
 *  *reordered: 1 when the solves iterate on P A P^T.
 * Any pointer may be NULL.  SLA_ERR_INVALID for a null handle.
 */
sla_status sla_csr_layout(sla_handle h, int* form, int* ctas, int* reordered);

/*
 * The same report for one matrix of the solves (no counterpart in the
 * pages): which = 0 the iteration matrix, 1 the SPAI factor G, 2 its
 * transpose G^T (built by the handle's first SPAI solve), 3 the matrix the
 * BiCGStab products iterate on (built by the first BiCGStab solve), 4 its
 * explicit transpose (built by the first BiCGStab adjoint); SLA_ERR_INVALID
 * before those are built.  *split: 1 when its staged groups are summed
 * split (see sla_csr_layout).  Any output pointer may be NULL.
 * SLA_ERR_INVALID for a null handle or another `which`.
 */
sla_status sla_csr_layout_of(sla_handle h, int which, int* form, int* ctas, int* split);

/*
 * Measurement hook; the pages have no counterpart.
 * Live duration of the first product kernel of an iteration (CG: q = A p
 * fused with p.q; BiCGStab: v = A p fused with r^.v; either with the
 * pending true-residual check), for handles created with SLA_TIME_PRODUCT:
 * every graph launch of sla_pcg_solve / sla_adjoint / sla_bicgstab_solve /
 * sla_bicgstab_adjoint records CUDA events on
 * the solve's stream around the product kernel of its middle iteration,
 * and the solve adds that duration once the launch has finished, for
 * launches that neither start nor end with every system frozen (a system
 * that freezes within a launch makes its later kernels return at once).  Returns the summed duration in
 * milliseconds and the number of launches timed since creation or the last
 * reset; nonzero `reset` clears both after reading.  The persistent
 * iteration kernel (SLA_PERSISTENT) is not timed.  Either output pointer
 * may be NULL.  SLA_ERR_INVALID for a null handle.
 */
sla_status sla_product_time(sla_handle h, double* total_ms, long long* samples, int reset);

/* Replace the values (same pattern, same dtype, [batch][nnz]); recomputes the
 * value-dependent set-up (diagonal, G, G^T).  torch-sla §3, sparse tensor
 * types: the pattern-dependent set-up is kept and reused when only the
 * values change (the shared-pattern case).  Synchronises `stream`.  The
 * handle keeps d_vals as it kept the values passed to sla_csr_create. */
sla_status sla_csr_update_values(sla_handle h, const void* d_vals, void* stream);

/* y = A x for every system (torch-sla §3, .matvec).  d_x, d_y: [batch][n]. */
sla_status sla_spmv(sla_handle h, const void* d_x, void* d_y, void* stream);

/* y = A x and d_dot[s] = x_s . y_s (fp64, one per system) in one fused pass:
 * the q = A p, delta = <p,Ap> step of CG (torch-sla §3.3, distributed CG).
 * d_dot: device double[batch].  Does not synchronise. */
sla_status sla_spmv_dot(sla_handle h, const void* d_x, void* d_y, double* d_dot, void* stream);

/*
 * Block product (the A-times-a-block step of torch-sla §3's .eigsh, here
 * LOBPCG): Y[:, j] = A X[:, j] for the k columns of a block stored
 * column after column (d_X, d_Y: [k][n], column j at offset j*n), in the
 * handle's dtype.  Needs a single-system handle (batch = 1); 0 <= k <= 65535.
 * Same product kernels as sla_spmv, with every column reading the same
 * values (the block eigensolver's A times a block).  Does not synchronise.
 */
sla_status sla_spmm(sla_handle h, const void* d_X, void* d_Y, int k, void* stream);

/*
 * Solve A x = b by preconditioned CG (torch-sla §3.3, distributed CG: the CG
 * recurrence with the inner products <r,r> and <p,Ap>; torch-sla §4 Table 3:
 * CG with Jacobi preconditioning, opts->pc = SLA_PC_JACOBI; the learned-SPAI
 * author responses, Reviewer umir Concern 1 and Reviewer GmV6 Concern 3:
 * M^-1 = G G^T + eps I applied by two SpMVs, opts->pc = SLA_PC_SPAI; torch-sla
 * §4 Figure 2: the stopping tolerance on the residual), every system of a
 * batch independently
 * (converged systems are frozen while the others continue).  d_b, d_x:
 * [batch][n].  x0 = 0 unless opts->use_x0.  info: host array of `batch`
 * entries, filled on return.  Returns SLA_OK when every system converged,
 * else the first non-OK per-system status (x still holds each system's last
 * iterate).  ||b|| = 0 gives x = 0 after 0 iterations.  Reordering: when
 * the pattern is scattered (more than 10% of its entries lie farther than
 * 65536 columns from their row) or SLA_REORDER is given, and SLA_NO_REORDER
 * is not, the handle iterates on P A P^T with P a reverse Cuthill-McKee
 * permutation of the pattern (computed on the host at creation), P b and
 * P x0, and returns P^T x: the same method (the SPAI factor is still built
 * on the caller's ordering and then permuted), rounded in a different
 * order.  sla_spmv and the dL/dA pass always use the caller's arrays.
 * fp32 handles run
 * the recurrence at fp64-equivalent precision (working vectors as
 * double-float pairs) and round x to fp32 on return.  The host issues
 * opts->poll_k iterations per launch -- a CUDA graph of one kernel per CG
 * step, or with SLA_PERSISTENT (CG and Jacobi only) one persistent
 * cooperative kernel -- keeps two launches in flight and reads one device
 * flag per launch; a device wait that gives up (never expected) returns
 * SLA_ERR_CUDA with its location in sla_last_error().
 */
sla_status sla_pcg_solve(sla_handle h, const void* d_b, void* d_x, const sla_pcg_opts* opts,
                         sla_solve_info* info, void* stream);

/*
 * Adjoint of x = A^-1 b for an upstream gradient g = dL/dx: solves
 * A^T lambda = g with the same options (A^T = A: CG needs a symmetric
 * matrix), then writes dL/db = lambda into d_dLdb [batch][n] and
 * dL/dA_k = -lambda_row(k) * x_col(k) for every stored entry k into d_dLdA
 * [batch][nnz] (torch-sla §3.3, adjoint paragraph).  d_x is the forward
 * solution.  d_dLdA may be NULL to skip the matrix gradient.
 */
sla_status sla_adjoint(sla_handle h, const void* d_x, const void* d_g, const sla_pcg_opts* opts,
                       void* d_dLdb, void* d_dLdA, sla_solve_info* info, void* stream);

/*
 * Solve a general (nonsymmetric) A x = b by BiCGStab (van der Vorst 1992;
 * the right-preconditioned form of Barrett et al., "Templates for the
 * Solution of Linear Systems", §2.3.8, shadow residual r^ = r0) -- the
 * nonsymmetric Krylov solver of torch-sla's iterative backends (§3, backends
 * paragraph).
 *  - fp64 handles only (SLA_ERR_UNSUPPORTED for fp32).  opts->pc is
 *    SLA_PC_NONE or SLA_PC_JACOBI (right preconditioning by diag(A), which
 *    must be stored; applied as the column scaling A diag(A)^-1 of a
 *    handle-owned copy of the values); SLA_PC_SPAI is SLA_ERR_INVALID.
 *    opts->eps is ignored.
 *  - Layout, batching, x0, polling, reordering and timeout as for
 *    sla_pcg_solve; info[s].iters counts BiCGStab iterations (two products
 *    each).  Stopping: ||r|| <= tol ||b|| on the recursive residual,
 *    confirmed on the true residual of x before returning SLA_OK.
 *  - SLA_ERR_BREAKDOWN when r^.r or r^.v is zero or not finite, or when
 *    omega = (t.s)/(t.t) is zero while the residual test fails.
 *  - The first call allocates the shadow residual (and, for Jacobi, a copy
 *    of the values: batch x nnz doubles); later calls allocate nothing.
 */
sla_status sla_bicgstab_solve(sla_handle h, const void* d_b, void* d_x, const sla_pcg_opts* opts,
                              sla_solve_info* info, void* stream);

/*
 * Adjoint of x = A^-1 b for a general A (torch-sla §3.3, adjoint
 * paragraph): solves A^T lambda = g by BiCGStab on an explicit transpose of
 * A -- its pattern built on the host at the first call and kept by the
 * handle, its values gathered from the current values on every call -- then
 * writes dL/db = lambda into d_dLdb and dL/dA_k = -lambda_row(k) x_col(k)
 * into d_dLdA (NULL skips it), as sla_adjoint.  Options and errors as for
 * sla_bicgstab_solve (use_x0 is ignored).  The transpose costs
 * nnz ints x 3 plus batch x nnz doubles of device memory.
 */
sla_status sla_bicgstab_adjoint(sla_handle h, const void* d_x, const void* d_g, const sla_pcg_opts* opts,
                                void* d_dLdb, void* d_dLdA, sla_solve_info* info, void* stream);

/*
 * Allocation-free y = A x and d_dot[s] = x_s . y_s (the same fused kernel as
 * sla_spmv_dot), without a handle.  The pages have no counterpart: this entry
 * point exists for callers that cannot let a library allocate device
 * memory -- programs that own all device memory through their own allocator
 * or memory budget, and latency-critical loops where cudaMalloc / cudaFree
 * would synchronise the device.  It calls no cudaMalloc, cudaFree or other
 * allocating routine; the caller passes every input and output.
 *  - Arguments as for sla_csr_create plus the vectors of sla_spmv_dot:
 *    CSR arrays (structure not checked here), d_x and d_y [batch][n] in the
 *    dtype, d_dot double[batch].  1 <= batch <= 64; a larger batch returns
 *    SLA_ERR_INVALID.
 *  - Its scratch (64 arrival counters and 4096 partial sums, about 33 KB) is
 *    a fixed array in device memory that every GPU loading this library
 *    holds until the process exits.  Every call shares it: each call first
 *    clears the counters on `stream`, so calls that overlap on the GPU (on
 *    different streams, or from several threads) race and must not be used.
 *  - The first call with a given device current looks up the scratch's
 *    device address (cudaGetSymbolAddress) and caches it; make that first
 *    call before any stream capture.
 *  - Returns without synchronising `stream`.
 */
sla_status sla_spmv_dot_static(int n, long long nnz, int batch, sla_dtype dt, const int* d_row_ptr,
                               const int* d_col_idx, const void* d_vals, const void* d_x, void* d_y,
                               double* d_dot, void* stream);

/*
 * Measurement hook; the pages have no counterpart.  Measures the device's
 * fp64 fused multiply-add rate (thread FMAs per second): a kernel of
 * independent fp64 FMA chains on every SM at full occupancy, timed with CUDA
 * events on `stream` (best of three launches after one warm-up).  This is
 * the fp64 roof beside the HBM roof: an fp64 SpMV spends one FMA per stored
 * entry.  Allocates a small output buffer; synchronises `stream`.
 */
sla_status sla_fp64_fma_rate(double* fma_per_s, void* stream);

/*
 * Dense steps of the block eigensolver (torch-sla §3, .eigsh; here LOBPCG,
 * Knyazev, SIAM J. Sci. Comput. 23(2), 2001: Rayleigh-Ritz over a basis of
 * blocks, kept orthonormal).  A block of k vectors of length n is stored
 * vector after vector (device double [k][n]); small matrices are row-major.
 *
 * sla_block_gram: G = A B^T, G[i][j] = A_i . B_j, for blocks A [ka][n] and
 * B [kb][n] (1 <= ka, kb <= 64), into d_G (device double [ka][kb]).
 * mode 0: every entry; mode 1 (B = A, ka = kb; d_B may be NULL): only
 * i <= j, mirrored; mode 2 (B = A): only the diagonal, the squared norms of
 * A's vectors, into d_G[0..ka); mode 3 (ka = kb, for blocks whose product
 * is symmetric, such as S and A S for a symmetric A): only i <= j of A B^T,
 * mirrored.  Sums are fp64, split over CTAs and added in
 * a fixed order (deterministic).  d_work: caller-owned device scratch of at
 * least the number of doubles sla_block_gram_work returns for the same
 * (ka, kb, mode, n).  Two kernels; does not synchronise.  SLA_ERR_INVALID
 * for sizes out of range, an unknown mode, null pointers or too small a
 * workspace.
 */
sla_status sla_block_gram_work(int ka, int kb, int mode, long long n, long long* doubles);
sla_status sla_block_gram(int ka, int kb, long long n, const double* d_A, const double* d_B, int mode, double* d_G,
                          double* d_work, long long work_doubles, void* stream);

/*
 * sla_block_update: Y[r] = sum_i C[i][r] S[i] (+ Yin[r]) for r < kc, i.e.
 * Y = C^T S (+ Yin): the block S [ks][n] times the small matrix C (device
 * double [ks][kc]), 1 <= ks, kc <= 64; d_Yin may be NULL or equal d_Y (an
 * in-place update); d_Y must not overlap d_S.  fp64, one kernel; does not
 * synchronise.
 */
sla_status sla_block_update(int ks, int kc, long long n, const double* d_C, const double* d_S, const double* d_Yin,
                            double* d_Y, void* stream);

/*
 * dL/dA_k = -lambda_row(k) x_col(k) for every stored entry k of the handle's
 * matrix (the matrix-gradient step of sla_adjoint, torch-sla §3.3 adjoint
 * paragraph, on its own): d_lam, d_x [batch][n], d_dLdA [batch][nnz], the
 * handle's dtype.  Used by the row-partitioned solve, where lambda and x come
 * from a partitioned solve and x carries the halo.  Synchronises `stream`.
 */
sla_status sla_grad_A(sla_handle h, const void* d_lam, const void* d_x, void* d_dLdA, void* stream);

/*
 * Local steps of the row-partitioned CG (torch-sla §3.3, distributed CG:
 * each rank updates its owned entries, and the inner products are all-reduced
 * over the ranks by the caller).  fp64, device pointers, n owned entries.
 * sla_cg_local_update: x += alpha p, r -= alpha q, z = dinv * r (z = r when
 * d_dinv is NULL), and d_dots (device double[2]) = this rank's r.r and r.z
 * (summed in a fixed order: deterministic); d_work: caller-owned scratch of
 * at least sla_cg_local_work(n) doubles.  sla_cg_local_direction:
 * p = z + beta p.  Neither synchronises.
 */
sla_status sla_cg_local_work(int n, long long* doubles);
sla_status sla_cg_local_update(int n, double alpha, const double* d_p, const double* d_q, const double* d_dinv,
                               double* d_x, double* d_r, double* d_z, double* d_dots, double* d_work,
                               long long work_doubles, void* stream);
sla_status sla_cg_local_direction(int n, double beta, const double* d_z, double* d_p, void* stream);

/*
 * Self-test of the bounded device waits; the pages have no counterpart.
 * Every wait of this library's kernels (on an mbarrier phase, or on the
 * other CTAs at a grid barrier) gives up after a time limit, records where,
 * and lets its kernel return, so a wait that never ends cannot hang the GPU;
 * the call that launched it then returns SLA_ERR_CUDA with the location in
 * sla_last_error().  This call makes one such wait run out on purpose with
 * a short limit: which = 0 waits on an mbarrier nothing arrives at, which =
 * 1 on a two-CTA grid barrier that one CTA never reaches.  0 < limit_s <= 1.
 * Returns SLA_ERR_CUDA with the wait's message (the expected outcome), or
 * SLA_OK if the wait ended (never expected); the device stays usable.
 * Allocates a few bytes of device memory; synchronises `stream`.
 */
sla_status sla_wait_selftest(int which, double limit_s, void* stream);

/* Free the handle and everything it owns (not the caller's arrays).  The
 * pages have no counterpart (a resource-release call of this C interface).
 * A NULL handle returns SLA_ERR_INVALID.  Must not run while a call on the
 * handle is in flight on another thread. */
sla_status sla_csr_destroy(sla_handle h);

/* Message for the calling thread's last error ("" if none).  The pages have
 * no counterpart (error reporting of this C interface).  The string belongs
 * to the library and stays valid until the thread's next failing call. */
const char* sla_last_error(void);

/* Number of kernels this library has launched in the process (graph nodes
 * count once per graph launch).  Diagnostics for benchmarks; the pages have
 * no counterpart. */
unsigned long long sla_launch_count(void);

#ifdef __cplusplus
}
#endif
#endif /* SLA_H */
