/*
 * oracle.c -- plain, slow, single-threaded fp64 reference for the CSR PCG
 * solve and its adjoint.  TEST INFRASTRUCTURE ONLY: the library never calls
 * it.  Only the tests, the smoke check and the benchmark's CPU-baseline leg
 * load it.  It shares no code, header or constant with the CUDA library.
 *
 * What it follows
 *   - CSR SpMV y = A x: the matvec of torch-sla (arXiv 2601.13994), §3 "sparse
 *     tensor types" (.matvec) and §4 Figure 2 (scatter-based SpMV), written as
 *     the plain definition y_i = sum_k A_ik x_k in stored order.
 *   - Conjugate gradient with a preconditioner (torch-sla §3.3 "Distributed
 *     CG": the Krylov recurrence with the inner products <r,r> and <p,Ap>;
 *     §4 Table 3: CG with Jacobi preconditioning), in the Hestenes-Stiefel
 *     order: q = A p, alpha = rho / p.q, x += alpha p, r -= alpha q,
 *     z = M^-1 r, beta = r.z / rho, p = z + beta p.
 *   - Factored sparse approximate inverse M^-1 = G G^T + eps I ("Learning
 *     Sparse Approximate Inverse Preconditioners for Conjugate Gradient
 *     Solvers on GPUs", author responses: Reviewer GmV6 Concern 3 for the
 *     eps I term, Reviewer umir Concern 1 for M^-1 r = G G^T r applied by
 *     SpMV, Reviewer Rbu2 Concern 3 for A^-1 ~ G G^T with G sparse).  The
 *     pages learn G with a graph network; here G is the closed-form stand-in
 *     on the pattern of tril(A): G_ii = A_ii^-1/2,
 *     G_ij = -A_ij / (2 sqrt(A_ii A_jj)) for j < i.
 *   - Adjoint (torch-sla §3.3, last paragraph, and §3.2 as summarised in §3):
 *     solve A^T lambda = dL/dx, then dL/db = lambda and
 *     dL/dA_ij = -lambda_i x_j on the stored non-zeros.
 *
 * Readings where the pages are silent
 *   - Stopping: ||r||_2 <= tol ||b||_2 on the recursive residual, tested right
 *     after the r update; when it holds, the true residual of the returned x
 *     is computed and the solve stops only if that is <= tol ||b|| as well;
 *     otherwise the iteration continues.  x0 = 0 unless given.  ||b|| = 0
 *     returns x = 0 after 0 iterations.
 *   - Iterations = number of products A p inside the loop.
 *   - Breakdown: p.q <= 0 or not finite, r.z <= 0 or not finite, or a
 *     non-finite ||r||^2.
 *   - fp32 systems (f32 != 0): "fp32 values" are the matrix values, b and
 *     the returned x (A, b passed here as the exact doubles).  The recurrence
 *     itself runs at fp64 precision: all arithmetic is fp64 and the working
 *     vectors (q, r, z, p, t) are not rounded; x is rounded to fp32 when it
 *     is returned, and the true-residual test uses that rounded x (as do the
 *     returned lambda and dL/dA of the adjoint).
 *
 * Build: gcc -O2 -ffp-contract=off -shared -fPIC (no fused multiply-add, so
 * every product is rounded before it is added).
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

#define OR_PC_NONE 0
#define OR_PC_JACOBI 1
#define OR_PC_SPAI 2

#define OR_OK 0
#define OR_NOT_CONVERGED 1
#define OR_BREAKDOWN 2
#define OR_INVALID 3

/* Value as returned to the caller: rounded to fp32 for fp32 systems. */
static double stor(double v, int f32) { return f32 ? (double)(float)v : v; }

static double dot(int n, const double* u, const double* v) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += u[i] * v[i];
    return s;
}

/* y = A x, each row summed in stored order starting from 0. */
void oracle_spmv(int n, const int* rp, const int* ci, const double* a,
                 const double* x, double* y) {
    for (int i = 0; i < n; ++i) {
        double s = 0.0;
        for (int k = rp[i]; k < rp[i + 1]; ++k) s += a[k] * x[ci[k]];
        y[i] = s;
    }
}

/* Diagonal of A; returns 0 if some A_ii is missing. */
static int diagonal(int n, const int* rp, const int* ci, const double* a, double* d) {
    for (int i = 0; i < n; ++i) {
        int found = 0;
        for (int k = rp[i]; k < rp[i + 1]; ++k)
            if (ci[k] == i) { d[i] = a[k]; found = 1; }
        if (!found) return 0;
    }
    return 1;
}

/* Number of stored entries of tril(A) (columns <= row). */
long long oracle_spai_nnz(int n, const int* rp, const int* ci) {
    long long c = 0;
    for (int i = 0; i < n; ++i)
        for (int k = rp[i]; k < rp[i + 1]; ++k)
            if (ci[k] <= i) ++c;
    return c;
}

/* G on the pattern of tril(A).  grp[n+1], gci[nnzG], gv[nnzG] are outputs.
 * Returns OR_INVALID if a diagonal entry is missing or not positive. */
int oracle_spai_factor(int n, const int* rp, const int* ci, const double* a,
                       int* grp, int* gci, double* gv) {
    double* d = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!diagonal(n, rp, ci, a, d)) { free(d); return OR_INVALID; }
    for (int i = 0; i < n; ++i)
        if (!(d[i] > 0.0)) { free(d); return OR_INVALID; }
    int m = 0;
    grp[0] = 0;
    for (int i = 0; i < n; ++i) {
        for (int k = rp[i]; k < rp[i + 1]; ++k) {
            int j = ci[k];
            if (j > i) continue;
            gci[m] = j;
            if (j == i) gv[m] = 1.0 / sqrt(d[i]);
            else gv[m] = -a[k] / (2.0 * sqrt(d[i] * d[j]));
            ++m;
        }
        grp[i + 1] = m;
    }
    free(d);
    return OR_OK;
}

/* z = G (G^T r) + eps r.  t = G^T r is formed by scattering the rows of G
 * (t_j += G_ij r_i, rows in ascending order), so no transposed copy of G is
 * built.  (f32 is accepted for symmetry with the solver; working vectors are
 * fp64 in both modes.) */
void oracle_spai_apply(int n, const int* grp, const int* gci, const double* gv,
                       double eps, int f32, const double* r, double* t, double* z) {
    for (int j = 0; j < n; ++j) t[j] = 0.0;
    for (int i = 0; i < n; ++i)
        for (int k = grp[i]; k < grp[i + 1]; ++k) t[gci[k]] += gv[k] * r[i];
    for (int i = 0; i < n; ++i) {
        double s = 0.0;
        for (int k = grp[i]; k < grp[i + 1]; ++k) s += gv[k] * t[gci[k]];
        z[i] = s + eps * r[i];
    }
}

/* ||b - A xo||^2 with every row sum in fp64. */
static double true_res2(int n, const int* rp, const int* ci, const double* a,
                        const double* b, const double* xo) {
    double s = 0.0;
    for (int i = 0; i < n; ++i) {
        double y = 0.0;
        for (int k = rp[i]; k < rp[i + 1]; ++k) y += a[k] * xo[ci[k]];
        double e = b[i] - y;
        s += e * e;
    }
    return s;
}

typedef struct {
    int pc;
    double eps;
    int f32;
    double* dinv_src;      /* Jacobi: A_ii */
    int* grp; int* gci; double* gv; double* t;   /* SPAI */
} precond;

static void apply_precond(const precond* M, int n, const double* r, double* z) {
    if (M->pc == OR_PC_JACOBI) {
        for (int i = 0; i < n; ++i) z[i] = r[i] / M->dinv_src[i];
    } else if (M->pc == OR_PC_SPAI) {
        oracle_spai_apply(n, M->grp, M->gci, M->gv, M->eps, M->f32, r, M->t, z);
    } else {
        for (int i = 0; i < n; ++i) z[i] = r[i];
    }
}

/*
 * Solve A x = b.  x: on entry the initial guess if use_x0, on exit the
 * solution (rounded to fp32 values when f32).  Returns a status code; iters,
 * rel_rec (||r||/||b||, recursive) and rel_true (||b - A x||/||b|| for the
 * returned x) are written when non-null.
 */
int oracle_pcg(int n, const int* rp, const int* ci, const double* a,
               const double* b, double* x, double tol, int max_iter, int pc,
               double eps, int f32, int use_x0, int* iters, double* rel_rec,
               double* rel_true) {
    if (n < 0 || tol <= 0.0 || max_iter < 0) return OR_INVALID;
    size_t sz = sizeof(double) * (size_t)(n > 0 ? n : 1);
    double* xi = (double*)malloc(sz);
    double* xo = (double*)malloc(sz);
    double* r = (double*)malloc(sz);
    double* z = (double*)malloc(sz);
    double* p = (double*)malloc(sz);
    double* q = (double*)malloc(sz);
    precond M;
    memset(&M, 0, sizeof M);
    M.pc = pc; M.eps = eps; M.f32 = f32;
    int status = OR_OK, k = 0;
    double gamma = 0.0, tr2 = 0.0;

    double bb = dot(n, b, b);
    if (pc == OR_PC_JACOBI) {
        M.dinv_src = (double*)malloc(sz);
        if (!diagonal(n, rp, ci, a, M.dinv_src)) { status = OR_INVALID; goto done; }
    } else if (pc == OR_PC_SPAI) {
        long long ng = oracle_spai_nnz(n, rp, ci);
        M.grp = (int*)malloc(sizeof(int) * (size_t)(n + 1));
        M.gci = (int*)malloc(sizeof(int) * (size_t)(ng > 0 ? ng : 1));
        M.gv = (double*)malloc(sizeof(double) * (size_t)(ng > 0 ? ng : 1));
        M.t = (double*)malloc(sz);
        if (oracle_spai_factor(n, rp, ci, a, M.grp, M.gci, M.gv) != OR_OK) {
            status = OR_INVALID; goto done;
        }
    }

    if (bb == 0.0) {
        for (int i = 0; i < n; ++i) x[i] = 0.0;
        if (iters) *iters = 0;
        if (rel_rec) *rel_rec = 0.0;
        if (rel_true) *rel_true = 0.0;
        goto done;
    }

    /* r = b - A x0 (or b), z = M^-1 r, p = z, rho = r.z */
    if (use_x0) {
        for (int i = 0; i < n; ++i) xi[i] = x[i];
        oracle_spmv(n, rp, ci, a, xi, q);
        for (int i = 0; i < n; ++i) r[i] = b[i] - q[i];
    } else {
        for (int i = 0; i < n; ++i) { xi[i] = 0.0; r[i] = b[i]; }
    }
    apply_precond(&M, n, r, z);
    for (int i = 0; i < n; ++i) p[i] = z[i];
    double rho = dot(n, r, z);
    gamma = dot(n, r, r);
    double tol2bb = tol * tol * bb;

    for (;;) {
        if (!isfinite(gamma)) { status = OR_BREAKDOWN; break; }
        if (gamma <= tol2bb) {
            for (int i = 0; i < n; ++i) xo[i] = stor(xi[i], f32);
            tr2 = true_res2(n, rp, ci, a, b, xo);
            if (tr2 <= tol2bb) { status = OR_OK; break; }
        }
        if (k >= max_iter) { status = OR_NOT_CONVERGED; break; }
        if (k > 0) {
            apply_precond(&M, n, r, z);
            double rho_new = dot(n, r, z);
            if (!(rho_new > 0.0) || !isfinite(rho_new)) { status = OR_BREAKDOWN; break; }
            double beta = rho_new / rho;
            rho = rho_new;
            for (int i = 0; i < n; ++i) p[i] = z[i] + beta * p[i];
        }
        oracle_spmv(n, rp, ci, a, p, q);
        double delta = dot(n, p, q);
        if (!(delta > 0.0) || !isfinite(delta)) { status = OR_BREAKDOWN; break; }
        double alpha = rho / delta;
        for (int i = 0; i < n; ++i) {
            xi[i] = xi[i] + alpha * p[i];
            r[i] = r[i] - alpha * q[i];
        }
        ++k;
        gamma = dot(n, r, r);
    }

    for (int i = 0; i < n; ++i) x[i] = stor(xi[i], f32);
    if (iters) *iters = k;
    if (rel_rec) *rel_rec = sqrt(gamma / bb);
    if (rel_true) *rel_true = sqrt(true_res2(n, rp, ci, a, b, x) / bb);

done:
    free(xi); free(xo); free(r); free(z); free(p); free(q);
    free(M.dinv_src); free(M.grp); free(M.gci); free(M.gv); free(M.t);
    return status;
}

/* A^T in CSR (columns ascending within each row): a counting pass over the
 * columns, then rows of A visited in ascending order. */
static void transpose(int n, const int* rp, const int* ci, const double* a,
                      int* trp, int* tci, double* ta) {
    int nnz = rp[n];
    for (int j = 0; j <= n; ++j) trp[j] = 0;
    for (int k = 0; k < nnz; ++k) trp[ci[k] + 1]++;
    for (int j = 0; j < n; ++j) trp[j + 1] += trp[j];
    int* fill = (int*)malloc(sizeof(int) * (size_t)(n > 0 ? n : 1));
    for (int j = 0; j < n; ++j) fill[j] = trp[j];
    for (int i = 0; i < n; ++i)
        for (int k = rp[i]; k < rp[i + 1]; ++k) {
            int pos = fill[ci[k]]++;
            tci[pos] = i;
            ta[pos] = a[k];
        }
    free(fill);
}

/*
 * Matrix gradient on the stored pattern (torch-sla §3.3, adjoint paragraph):
 * dL/dA_k = -lambda_row(k) * x_col(k) for every stored entry k, rounded to
 * fp32 in fp32 mode.
 */
void oracle_grad_A(int n, const int* rp, const int* ci, const double* lam,
                   const double* x, int f32, double* dlda) {
    for (int i = 0; i < n; ++i)
        for (int k = rp[i]; k < rp[i + 1]; ++k)
            dlda[k] = stor(-lam[i] * x[ci[k]], f32);
}

/*
 * Adjoint of x = A^-1 b for the upstream gradient g = dL/dx:
 * solve A^T lambda = g (same preconditioner kind, tolerance and iteration
 * cap), then dL/db = lambda and dL/dA_k = -lambda_row(k) * x_col(k) for every
 * stored entry k.  In fp32 mode lambda is rounded to fp32 as it is returned
 * and dL/dA is formed from that rounded lambda, then rounded.  dlda = NULL
 * skips the matrix gradient (x is then not read).
 */
int oracle_adjoint(int n, const int* rp, const int* ci, const double* a,
                   const double* x, const double* g, double tol, int max_iter,
                   int pc, double eps, int f32, double* dldb, double* dlda,
                   int* iters, double* rel_rec, double* rel_true) {
    int nnz = rp[n];
    int* trp = (int*)malloc(sizeof(int) * (size_t)(n + 1));
    int* tci = (int*)malloc(sizeof(int) * (size_t)(nnz > 0 ? nnz : 1));
    double* ta = (double*)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
    transpose(n, rp, ci, a, trp, tci, ta);
    int st = oracle_pcg(n, trp, tci, ta, g, dldb, tol, max_iter, pc, eps, f32, 0,
                        iters, rel_rec, rel_true);
    if (st != OR_INVALID && dlda) oracle_grad_A(n, rp, ci, dldb, x, f32, dlda);
    free(trp); free(tci); free(ta);
    return st;
}

/* ||b - A x||_2 / ||b||_2 (0 when b = 0). */
double oracle_rel_residual(int n, const int* rp, const int* ci, const double* a,
                           const double* b, const double* x) {
    double bb = dot(n, b, b);
    if (bb == 0.0) return 0.0;
    return sqrt(true_res2(n, rp, ci, a, b, x) / bb);
}

/*
 * BiCGStab for a general (nonsymmetric) A x = b, right-preconditioned
 * (M = diag(A) for pc = OR_PC_JACOBI, M = I for OR_PC_NONE): the algorithm
 * of van der Vorst (SIAM J. Sci. Stat. Comput. 13(2), 1992) as laid out in
 * Barrett et al., "Templates for the Solution of Linear Systems" (SIAM,
 * 1994), section 2.3.8, with the shadow residual r^ = r0.  One iteration is
 * the pair of products A p^ and A s^.  Stopping as in oracle_pcg: the
 * recursive residual ||r|| <= tol ||b|| (tested after the x / r update, and
 * before the first iteration), confirmed on the true residual of the
 * returned x, otherwise the iteration continues.  omega = (t.s)/(t.t), or 0
 * when t = 0.  Breakdown: rho = r^.r or sigma = r^.v zero or not finite, a
 * non-finite ||r||^2, or omega = 0 while the residual test fails.
 */
int oracle_bicgstab(int n, const int* rp, const int* ci, const double* a,
                    const double* b, double* x, double tol, int max_iter, int pc,
                    int use_x0, int* iters, double* rel_rec, double* rel_true) {
    if (n < 0 || tol <= 0.0 || max_iter < 0 || (pc != OR_PC_NONE && pc != OR_PC_JACOBI)) return OR_INVALID;
    size_t sz = sizeof(double) * (size_t)(n > 0 ? n : 1);
    double *xi = (double*)malloc(sz), *r = (double*)malloc(sz), *rh = (double*)malloc(sz);
    double *p = (double*)malloc(sz), *ph = (double*)malloc(sz), *v = (double*)malloc(sz);
    double *s = (double*)malloc(sz), *sh = (double*)malloc(sz), *t = (double*)malloc(sz);
    double *d = (double*)malloc(sz), *xo = (double*)malloc(sz);
    int status = OR_OK, k = 0;
    double gamma = 0.0;
    double bb = dot(n, b, b);
    if (pc == OR_PC_JACOBI && !diagonal(n, rp, ci, a, d)) { status = OR_INVALID; goto done; }
    if (bb == 0.0) {
        for (int i = 0; i < n; ++i) x[i] = 0.0;
        if (iters) *iters = 0;
        if (rel_rec) *rel_rec = 0.0;
        if (rel_true) *rel_true = 0.0;
        goto done;
    }
    if (use_x0) {
        for (int i = 0; i < n; ++i) xi[i] = x[i];
        oracle_spmv(n, rp, ci, a, xi, v);
        for (int i = 0; i < n; ++i) r[i] = b[i] - v[i];
    } else {
        for (int i = 0; i < n; ++i) { xi[i] = 0.0; r[i] = b[i]; }
    }
    for (int i = 0; i < n; ++i) { rh[i] = r[i]; p[i] = 0.0; v[i] = 0.0; }
    gamma = dot(n, r, r);
    double tol2bb = tol * tol * bb, rho_prev = 1.0, alpha = 1.0, omega = 1.0;
    for (;;) {
        if (!isfinite(gamma)) { status = OR_BREAKDOWN; break; }
        if (gamma <= tol2bb) {
            for (int i = 0; i < n; ++i) xo[i] = xi[i];
            if (true_res2(n, rp, ci, a, b, xo) <= tol2bb) { status = OR_OK; break; }
        } else if (k > 0 && omega == 0.0) {
            status = OR_BREAKDOWN;
            break;
        }
        if (k >= max_iter) { status = OR_NOT_CONVERGED; break; }
        double rho = dot(n, rh, r);
        if (rho == 0.0 || !isfinite(rho)) { status = OR_BREAKDOWN; break; }
        if (k == 0) {
            for (int i = 0; i < n; ++i) p[i] = r[i];
        } else {
            double beta = (rho / rho_prev) * (alpha / omega);
            for (int i = 0; i < n; ++i) p[i] = r[i] + beta * (p[i] - omega * v[i]);
        }
        for (int i = 0; i < n; ++i) ph[i] = pc == OR_PC_JACOBI ? p[i] / d[i] : p[i];
        oracle_spmv(n, rp, ci, a, ph, v);
        double sigma = dot(n, rh, v);
        if (sigma == 0.0 || !isfinite(sigma)) { status = OR_BREAKDOWN; break; }
        alpha = rho / sigma;
        for (int i = 0; i < n; ++i) {
            s[i] = r[i] - alpha * v[i];
            sh[i] = pc == OR_PC_JACOBI ? s[i] / d[i] : s[i];
        }
        oracle_spmv(n, rp, ci, a, sh, t);
        double tt = dot(n, t, t), ts = dot(n, t, s);
        omega = tt > 0.0 ? ts / tt : 0.0;
        if (!isfinite(omega)) { status = OR_BREAKDOWN; break; }
        for (int i = 0; i < n; ++i) {
            xi[i] = xi[i] + alpha * ph[i] + omega * sh[i];
            r[i] = s[i] - omega * t[i];
        }
        gamma = dot(n, r, r);
        rho_prev = rho;
        ++k;
    }
    for (int i = 0; i < n; ++i) x[i] = xi[i];
    if (iters) *iters = k;
    if (rel_rec) *rel_rec = sqrt(gamma / bb);
    if (rel_true) *rel_true = sqrt(true_res2(n, rp, ci, a, b, x) / bb);
done:
    free(xi); free(r); free(rh); free(p); free(ph); free(v); free(s); free(sh); free(t); free(d); free(xo);
    return status;
}

/* Adjoint of x = A^-1 b for a general A: solve A^T lambda = g by BiCGStab on
 * the explicit transpose, then dL/db = lambda and dL/dA_k = -lambda_row(k)
 * x_col(k) on the stored entries (torch-sla §3.3, adjoint paragraph). */
int oracle_bicgstab_adjoint(int n, const int* rp, const int* ci, const double* a,
                            const double* x, const double* g, double tol, int max_iter,
                            int pc, double* dldb, double* dlda, int* iters,
                            double* rel_rec, double* rel_true) {
    int nnz = rp[n];
    int* trp = (int*)malloc(sizeof(int) * (size_t)(n + 1));
    int* tci = (int*)malloc(sizeof(int) * (size_t)(nnz > 0 ? nnz : 1));
    double* ta = (double*)malloc(sizeof(double) * (size_t)(nnz > 0 ? nnz : 1));
    transpose(n, rp, ci, a, trp, tci, ta);
    int st = oracle_bicgstab(n, trp, tci, ta, g, dldb, tol, max_iter, pc, 0, iters, rel_rec, rel_true);
    if (st != OR_INVALID)
        for (int i = 0; i < n; ++i)
            for (int k = rp[i]; k < rp[i + 1]; ++k) dlda[k] = -dldb[i] * x[ci[k]];
    free(trp); free(tci); free(ta);
    return st;
}
