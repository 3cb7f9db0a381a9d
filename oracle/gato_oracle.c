/*
 * gato_oracle.c -- plain fp64 CPU oracle for the batched KKT path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the package's smoke check and the bench's
 * CPU-baseline leg do.  It shares no code with the CUDA library.
 *
 * Everything here follows "GATO: GPU-Accelerated and Batched Trajectory
 * Optimization for Scalable Edge Model Predictive Control" (the GATO paper):
 *   Sec. II, eq. (1)   the LQ subproblem (Q, R, q, r, A, B, e, x_s)
 *   Sec. II, eq. (2)   the KKT system in dz = [dx_k; du_k], multipliers lambda
 *   Sec. II, eqs. (4)-(6)  Schur complement S = C G^-1 C^T, gamma, theta/phi/
 *                      zeta, and the symmetric stair preconditioner Phi^-1
 *   Sec. II            PCG on Phi^-1 S lambda = Phi^-1 gamma to tolerance eps
 *   Sec. III-A         parallel line search, alpha = beta^-i, L1 merit
 * The pages' display equations were lost in extraction; the forms used here
 * are the readings written beside each function.
 *
 * Conventions (one solve): N knots x_0..x_{N-1}, controls u_0..u_{N-2}.
 *   Q [N][n][n]  R [N-1][m][m]  q [N][n]  r [N-1][m]
 *   A [N-1][n][n]  B [N-1][n][m]  e [N-1][n]  s0 [n]
 *   dX [N][n]  dU [N-1][m]  lambda [N][n]
 * Block-tridiagonal matrices: diagonal blocks Dg [N][n][n]; the sub-diagonal
 * block (j, j-1) is stored at Off[j-1] ([N-1][n][n]); (j-1, j) is its transpose.
 * All matrices row-major, all arithmetic double.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* small dense helpers                                                       */
/* ------------------------------------------------------------------------ */

/* In-place Cholesky a = L L^T (lower triangle of a holds L, upper zeroed).
 * Returns 0, or -1 on a non-positive pivot. */
static int chol(int n, double *a)
{
    for (int j = 0; j < n; ++j) {
        double d = a[j * n + j];
        for (int k = 0; k < j; ++k) d -= a[j * n + k] * a[j * n + k];
        if (!(d > 0.0)) return -1;
        d = sqrt(d);
        a[j * n + j] = d;
        for (int i = j + 1; i < n; ++i) {
            double s = a[i * n + j];
            for (int k = 0; k < j; ++k) s -= a[i * n + k] * a[j * n + k];
            a[i * n + j] = s / d;
        }
        for (int k = j + 1; k < n; ++k) a[j * n + k] = 0.0;
    }
    return 0;
}

/* Solve L y = b (forward) in place. */
static void lower_solve(int n, const double *L, double *b)
{
    for (int i = 0; i < n; ++i) {
        double s = b[i];
        for (int k = 0; k < i; ++k) s -= L[i * n + k] * b[k];
        b[i] = s / L[i * n + i];
    }
}

/* Solve L^T x = b (backward) in place. */
static void upper_t_solve(int n, const double *L, double *b)
{
    for (int i = n - 1; i >= 0; --i) {
        double s = b[i];
        for (int k = i + 1; k < n; ++k) s -= L[k * n + i] * b[k];
        b[i] = s / L[i * n + i];
    }
}

/* inv = a^-1 for SPD a, column by column through its Cholesky factor. */
static int spd_inverse(int n, const double *a, double *inv)
{
    double *L = malloc(sizeof(double) * n * n);
    double *col = malloc(sizeof(double) * n);
    memcpy(L, a, sizeof(double) * n * n);
    int rc = chol(n, L);
    if (rc == 0) {
        for (int c = 0; c < n; ++c) {
            for (int i = 0; i < n; ++i) col[i] = (i == c) ? 1.0 : 0.0;
            lower_solve(n, L, col);
            upper_t_solve(n, L, col);
            for (int i = 0; i < n; ++i) inv[i * n + c] = col[i];
        }
    }
    free(L);
    free(col);
    return rc;
}

/* C = op(A) * op(B) with A (r x k or k x r), B (k x c or c x k). */
static void gemm(int r, int c, int k, const double *A, int ta, const double *B,
                 int tb, double *C)
{
    for (int i = 0; i < r; ++i)
        for (int j = 0; j < c; ++j) {
            double s = 0.0;
            for (int l = 0; l < k; ++l) {
                double a = ta ? A[l * r + i] : A[i * k + l];
                double b = tb ? B[j * k + l] : B[l * c + j];
                s += a * b;
            }
            C[i * c + j] = s;
        }
}

/* y = op(A) x, A is r x c (op = transpose when t). */
static void gemv(int r, int c, const double *A, int t, const double *x, double *y)
{
    int rows = t ? c : r;
    int cols = t ? r : c;
    for (int i = 0; i < rows; ++i) {
        double s = 0.0;
        for (int l = 0; l < cols; ++l) s += (t ? A[l * c + i] : A[i * c + l]) * x[l];
        y[i] = s;
    }
}

static double dot(int n, const double *a, const double *b)
{
    double s = 0.0;
    for (int i = 0; i < n; ++i) s += a[i] * b[i];
    return s;
}

/* ------------------------------------------------------------------------ */
/* Dense KKT system (eq. (2)): the definition the Schur path must reproduce. */
/* ------------------------------------------------------------------------ */
/*
 * Reading of eq. (1)-(2):  minimise sum_k 1/2 dz_k^T G_k dz_k + g_k^T dz_k with
 * G_k = diag(Q_k, R_k), g_k = [q_k; r_k] (G_{N-1} = Q_{N-1}, g_{N-1} = q_{N-1}),
 * subject to   -dx_0 = -s0          (initial condition, s0 = x_s - xbar_0)
 *              A_k dx_k + B_k du_k - dx_{k+1} = -e_k,   k = 0..N-2.
 * KKT:  [G C^T; C 0] [dz; lambda] = [-g; c],   c_0 = -s0, c_{k+1} = -e_k.
 * Primal ordering z = [dx_0, du_0, dx_1, du_1, ..., dx_{N-1}], then lambda_0..N-1.
 */
static int zx(int k, int n, int m) { return k * (n + m); }
static int zu(int k, int n, int m) { return k * (n + m) + n; }

static void kkt_assemble(int N, int n, int m, const double *Q, const double *R,
                         const double *q, const double *r, const double *A,
                         const double *B, const double *e, const double *s0,
                         double *K, double *rhs)
{
    const int nz = (N - 1) * (n + m) + n;
    const int dim = nz + N * n;
    memset(K, 0, sizeof(double) * dim * dim);
    for (int k = 0; k < N; ++k) {
        for (int i = 0; i < n; ++i) {
            for (int j = 0; j < n; ++j)
                K[(zx(k, n, m) + i) * dim + zx(k, n, m) + j] = Q[k * n * n + i * n + j];
            rhs[zx(k, n, m) + i] = -q[k * n + i];
        }
        if (k < N - 1)
            for (int i = 0; i < m; ++i) {
                for (int j = 0; j < m; ++j)
                    K[(zu(k, n, m) + i) * dim + zu(k, n, m) + j] = R[k * m * m + i * m + j];
                rhs[zu(k, n, m) + i] = -r[k * m + i];
            }
    }
    /* constraint rows: row block j of C sits at K rows nz + j*n */
    for (int i = 0; i < n; ++i) {
        int row = nz + i;
        K[row * dim + zx(0, n, m) + i] = -1.0;
        K[(zx(0, n, m) + i) * dim + row] = -1.0;
        rhs[row] = -s0[i];
    }
    for (int k = 0; k < N - 1; ++k)
        for (int i = 0; i < n; ++i) {
            int row = nz + (k + 1) * n + i;
            for (int j = 0; j < n; ++j) {
                double a = A[k * n * n + i * n + j];
                K[row * dim + zx(k, n, m) + j] = a;
                K[(zx(k, n, m) + j) * dim + row] = a;
            }
            for (int j = 0; j < m; ++j) {
                double b = B[k * n * m + i * m + j];
                K[row * dim + zu(k, n, m) + j] = b;
                K[(zu(k, n, m) + j) * dim + row] = b;
            }
            K[row * dim + zx(k + 1, n, m) + i] = -1.0;
            K[(zx(k + 1, n, m) + i) * dim + row] = -1.0;
            rhs[row] = -e[k * n + i];
        }
}

/* Symmetric LDL^T without pivoting, natural order; solves K x = b in place. */
static int ldlt_solve(int dim, double *K, double *b)
{
    for (int j = 0; j < dim; ++j) {
        double d = K[j * dim + j];
        for (int k = 0; k < j; ++k) d -= K[j * dim + k] * K[j * dim + k] * K[k * dim + k];
        if (d == 0.0 || !isfinite(d)) return -1;
        K[j * dim + j] = d;
        for (int i = j + 1; i < dim; ++i) {
            double s = K[i * dim + j];
            for (int k = 0; k < j; ++k) s -= K[i * dim + k] * K[j * dim + k] * K[k * dim + k];
            K[i * dim + j] = s / d;
        }
    }
    for (int i = 0; i < dim; ++i)
        for (int k = 0; k < i; ++k) b[i] -= K[i * dim + k] * b[k];
    for (int i = 0; i < dim; ++i) b[i] /= K[i * dim + i];
    for (int i = dim - 1; i >= 0; --i)
        for (int k = i + 1; k < dim; ++k) b[i] -= K[k * dim + i] * b[k];
    return 0;
}

/* Gaussian elimination with partial pivoting; solves K x = b in place. */
static int lu_solve(int dim, double *K, double *b)
{
    for (int j = 0; j < dim; ++j) {
        int p = j;
        double best = fabs(K[j * dim + j]);
        for (int i = j + 1; i < dim; ++i)
            if (fabs(K[i * dim + j]) > best) { best = fabs(K[i * dim + j]); p = i; }
        if (best == 0.0) return -1;
        if (p != j) {
            for (int c = 0; c < dim; ++c) {
                double t = K[j * dim + c]; K[j * dim + c] = K[p * dim + c]; K[p * dim + c] = t;
            }
            double t = b[j]; b[j] = b[p]; b[p] = t;
        }
        for (int i = j + 1; i < dim; ++i) {
            double f = K[i * dim + j] / K[j * dim + j];
            if (f == 0.0) continue;
            for (int c = j; c < dim; ++c) K[i * dim + c] -= f * K[j * dim + c];
            b[i] -= f * b[j];
        }
    }
    for (int i = dim - 1; i >= 0; --i) {
        double s = b[i];
        for (int c = i + 1; c < dim; ++c) s -= K[i * dim + c] * b[c];
        b[i] = s / K[i * dim + i];
    }
    return 0;
}

/* Dense KKT solve.  method 0 = LDL^T (no pivoting), 1 = partial-pivot LU.
 * Returns 0, or -1 if the factorisation broke down. */
int oracle_kkt_dense(int N, int n, int m, const double *Q, const double *R,
                     const double *q, const double *r, const double *A,
                     const double *B, const double *e, const double *s0,
                     int method, double *dX, double *dU, double *lambda)
{
    const int nz = (N - 1) * (n + m) + n;
    const int dim = nz + N * n;
    double *K = malloc(sizeof(double) * dim * dim);
    double *x = malloc(sizeof(double) * dim);
    if (!K || !x) { free(K); free(x); return -2; }
    kkt_assemble(N, n, m, Q, R, q, r, A, B, e, s0, K, x);
    int rc = method == 0 ? ldlt_solve(dim, K, x) : lu_solve(dim, K, x);
    if (rc == 0) {
        for (int k = 0; k < N; ++k) {
            for (int i = 0; i < n; ++i) dX[k * n + i] = x[zx(k, n, m) + i];
            if (k < N - 1)
                for (int i = 0; i < m; ++i) dU[k * m + i] = x[zu(k, n, m) + i];
        }
        for (int i = 0; i < N * n; ++i) lambda[i] = x[nz + i];
    }
    free(K);
    free(x);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Schur complement, eqs. (4)-(6)                                            */
/* ------------------------------------------------------------------------ */
/*
 * S = C G^-1 C^T, gamma = -c - C G^-1 g (block rows j = 0..N-1):
 *   S_00 = Q_0^-1                         gamma_0 = s0 + Q_0^-1 q_0
 *   S_jj = theta_{j-1} = A_{j-1} Q_{j-1}^-1 A_{j-1}^T + B_{j-1} R_{j-1}^-1 B_{j-1}^T + Q_j^-1
 *   S_{j,j-1} = phi_{j-1} = -A_{j-1} Q_{j-1}^-1
 *   gamma_j = e_{j-1} + zeta_{j-1},
 *   zeta_{j-1} = -A_{j-1} Q_{j-1}^-1 q_{j-1} - B_{j-1} R_{j-1}^-1 r_{j-1} + Q_j^-1 q_j
 * Returns 0, or -1 if some Q_k or R_k is not positive definite.
 */
int oracle_schur(int N, int n, int m, const double *Q, const double *R,
                 const double *q, const double *r, const double *A,
                 const double *B, const double *e, const double *s0,
                 double *Dg, double *Off, double *gamma)
{
    int rc = 0;
    double *Qi = malloc(sizeof(double) * N * n * n);
    double *Ri = malloc(sizeof(double) * (N > 1 ? (N - 1) : 1) * m * m);
    double *T1 = malloc(sizeof(double) * n * n);
    double *T2 = malloc(sizeof(double) * n * (n > m ? n : m));
    double *w = malloc(sizeof(double) * n);
    for (int k = 0; k < N; ++k)
        if (spd_inverse(n, Q + k * n * n, Qi + k * n * n)) rc = -1;
    for (int k = 0; k < N - 1; ++k)
        if (spd_inverse(m, R + k * m * m, Ri + k * m * m)) rc = -1;

    /* block row 0 */
    memcpy(Dg, Qi, sizeof(double) * n * n);
    gemv(n, n, Qi, 0, q, w);
    for (int i = 0; i < n; ++i) gamma[i] = s0[i] + w[i];

    for (int j = 1; j < N; ++j) {
        const int k = j - 1;
        const double *Ak = A + k * n * n, *Bk = B + k * n * m;
        const double *Qk = Qi + k * n * n, *Rk = Ri + k * m * m, *Qj = Qi + j * n * n;
        double *D = Dg + j * n * n, *O = Off + k * n * n, *g = gamma + j * n;
        gemm(n, n, n, Ak, 0, Qk, 0, T1);               /* T1 = A Q^-1          */
        gemm(n, n, n, T1, 0, Ak, 1, D);                /* D  = A Q^-1 A^T      */
        gemm(n, m, m, Bk, 0, Rk, 0, T2);               /* T2 = B R^-1          */
        for (int i = 0; i < n; ++i)
            for (int c = 0; c < n; ++c) {
                double s = 0.0;
                for (int l = 0; l < m; ++l) s += T2[i * m + l] * Bk[c * m + l];
                D[i * n + c] += s + Qj[i * n + c];     /* + B R^-1 B^T + Q_j^-1 */
            }
        for (int i = 0; i < n * n; ++i) O[i] = -T1[i]; /* phi = -A Q^-1        */
        /* zeta = -A Q_k^-1 q_k - B R_k^-1 r_k + Q_j^-1 q_j ; gamma_j = e_k + zeta */
        gemv(n, n, T1, 0, q + k * n, w);
        for (int i = 0; i < n; ++i) g[i] = e[k * n + i] - w[i];
        gemv(n, m, T2, 0, r + k * m, w);
        for (int i = 0; i < n; ++i) g[i] -= w[i];
        gemv(n, n, Qj, 0, q + j * n, w);
        for (int i = 0; i < n; ++i) g[i] += w[i];
    }
    free(Qi); free(Ri); free(T1); free(T2); free(w);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Symmetric stair preconditioner, eq. (6)                                   */
/* ------------------------------------------------------------------------ */
/*
 * Reading: Phi^-1 = D^-1 - D^-1 (L + L^T) D^-1, with D the block diagonal of S
 * and L its strictly-lower block part: block-tridiagonal with diagonal blocks
 * D_j^-1 and sub-diagonal blocks -D_j^-1 S_{j,j-1} D_{j-1}^-1.
 * Returns 0, or -1 if some diagonal block of S is not positive definite.
 */
int oracle_stair(int N, int n, const double *Dg, const double *Off, double *Pd,
                 double *Po)
{
    int rc = 0;
    double *T = malloc(sizeof(double) * n * n);
    for (int j = 0; j < N; ++j)
        if (spd_inverse(n, Dg + j * n * n, Pd + j * n * n)) rc = -1;
    for (int j = 1; j < N; ++j) {
        gemm(n, n, n, Pd + j * n * n, 0, Off + (j - 1) * n * n, 0, T);
        gemm(n, n, n, T, 0, Pd + (j - 1) * n * n, 0, Po + (j - 1) * n * n);
        for (int i = 0; i < n * n; ++i) Po[(j - 1) * n * n + i] = -Po[(j - 1) * n * n + i];
    }
    free(T);
    return rc;
}

/* y = M x for block-tridiagonal symmetric M (Dg, Off). */
static void bt_matvec(int N, int n, const double *Dg, const double *Off,
                      const double *x, double *y)
{
    double *t = malloc(sizeof(double) * n);
    for (int j = 0; j < N; ++j) {
        double *yj = y + j * n;
        gemv(n, n, Dg + j * n * n, 0, x + j * n, yj);
        if (j > 0) {
            gemv(n, n, Off + (j - 1) * n * n, 0, x + (j - 1) * n, t);
            for (int i = 0; i < n; ++i) yj[i] += t[i];
        }
        if (j < N - 1) {
            gemv(n, n, Off + j * n * n, 1, x + (j + 1) * n, t);
            for (int i = 0; i < n; ++i) yj[i] += t[i];
        }
    }
    free(t);
}

/* Dense S or Phi^-1 from its blocks (for checks on small cases). */
void oracle_bt_dense(int N, int n, const double *Dg, const double *Off, double *M)
{
    const int d = N * n;
    memset(M, 0, sizeof(double) * d * d);
    for (int j = 0; j < N; ++j)
        for (int a = 0; a < n; ++a)
            for (int b = 0; b < n; ++b) {
                M[(j * n + a) * d + j * n + b] = Dg[j * n * n + a * n + b];
                if (j > 0) {
                    double o = Off[(j - 1) * n * n + a * n + b];
                    M[(j * n + a) * d + (j - 1) * n + b] = o;
                    M[((j - 1) * n + b) * d + j * n + a] = o;
                }
            }
}

/* ------------------------------------------------------------------------ */
/* Preconditioned conjugate gradient on S lambda = gamma                     */
/* ------------------------------------------------------------------------ */
/*
 * Standard PCG with preconditioner Phi^-1, from lambda0 (zero when NULL):
 *   r = gamma - S lambda, z = Phi^-1 r, p = z, eta = r^T z, eta0 = eta
 *   repeat: v = S p; alpha = eta / p^T v; lambda += alpha p; r -= alpha v;
 *           z = Phi^-1 r; eta' = r^T z; stop when converged;
 *           p = z + (eta'/eta) p; eta = eta'
 * Convergence (tested on the recursively updated r, also before the first
 * iteration):
 *   stop_rule 0: relative residual  ||r||_2 <= eps ||gamma||_2
 *   stop_rule 1: preconditioned     r^T Phi^-1 r <= eps^2 eta0
 *   stop_rule 2: block-Jacobi-scaled residual r^T D^-1 r <= eps^2 gamma^T D^-1 gamma,
 *                D^-1 = Pd, the diagonal blocks of Phi^-1
 * Returns 0 if converged, 1 if max_iters was reached; *iters = iterations run.
 * With eps = 0 and max_iters = k the result is exactly the k-th iterate.
 */
/* x^T blockdiag(Pd) x */
static double dinv_norm2(int N, int n, const double *Pd, const double *x)
{
    double s = 0.0;
    double *t = malloc(sizeof(double) * n);
    for (int j = 0; j < N; ++j) {
        gemv(n, n, Pd + j * n * n, 0, x + j * n, t);
        s += dot(n, x + j * n, t);
    }
    free(t);
    return s;
}

static int pcg_converged(int rule, int N, int n, const double *Pd, const double *rv,
                         double eta, double eta0, double ref, double eps)
{
    if (rule == 0) return dot(N * n, rv, rv) <= eps * eps * ref;
    if (rule == 2) return dinv_norm2(N, n, Pd, rv) <= eps * eps * ref;
    return eta <= eps * eps * eta0;
}

int oracle_pcg(int N, int n, const double *Dg, const double *Off, const double *Pd,
               const double *Po, const double *gamma, const double *lambda0,
               double eps, int max_iters, int stop_rule, double *lambda, int *iters)
{
    const int d = N * n;
    double *rv = malloc(sizeof(double) * d), *z = malloc(sizeof(double) * d);
    double *p = malloc(sizeof(double) * d), *v = malloc(sizeof(double) * d);
    int it = 0;
    for (int i = 0; i < d; ++i) lambda[i] = lambda0 ? lambda0[i] : 0.0;
    bt_matvec(N, n, Dg, Off, lambda, v);
    for (int i = 0; i < d; ++i) rv[i] = gamma[i] - v[i];
    bt_matvec(N, n, Pd, Po, rv, z);
    memcpy(p, z, sizeof(double) * d);
    double eta = dot(d, rv, z);
    const double eta0 = eta;
    const double ref = stop_rule == 2 ? dinv_norm2(N, n, Pd, gamma) : dot(d, gamma, gamma);
    int done = pcg_converged(stop_rule, N, n, Pd, rv, eta, eta0, ref, eps);
    while (!done && it < max_iters) {
        ++it;
        bt_matvec(N, n, Dg, Off, p, v);
        double alpha = eta / dot(d, p, v);
        for (int i = 0; i < d; ++i) { lambda[i] += alpha * p[i]; rv[i] -= alpha * v[i]; }
        bt_matvec(N, n, Pd, Po, rv, z);
        double eta_new = dot(d, rv, z);
        done = pcg_converged(stop_rule, N, n, Pd, rv, eta_new, eta0, ref, eps);
        if (done) break;
        double beta = eta_new / eta;
        for (int i = 0; i < d; ++i) p[i] = z[i] + beta * p[i];
        eta = eta_new;
    }
    *iters = it;
    free(rv); free(z); free(p); free(v);
    return done ? 0 : 1;
}

/* ------------------------------------------------------------------------ */
/* Direct block-tridiagonal Cholesky solve of S lambda = gamma (reference)   */
/* ------------------------------------------------------------------------ */
/*
 * S = L L^T with L block lower bidiagonal: L_0 = chol(S_00),
 * W_j = S_{j,j-1} L_{j-1}^-T, L_j = chol(S_jj - W_j W_j^T); then a forward
 * and a backward block substitution.  Returns 0 or -1 (not positive definite).
 */
int oracle_block_cholesky(int N, int n, const double *Dg, const double *Off,
                          const double *gamma, double *lambda)
{
    int rc = 0;
    double *L = malloc(sizeof(double) * N * n * n);
    double *W = malloc(sizeof(double) * (N > 1 ? N - 1 : 1) * n * n);
    double *y = malloc(sizeof(double) * N * n);
    double *t = malloc(sizeof(double) * n);
    memcpy(L, Dg, sizeof(double) * n * n);
    if (chol(n, L)) rc = -1;
    for (int j = 1; j < N && rc == 0; ++j) {
        double *Wj = W + (j - 1) * n * n, *Lj = L + j * n * n;
        const double *Lp = L + (j - 1) * n * n;
        /* W_j = O_j L_{j-1}^-T: each row w of W_j solves L_{j-1} w^T = o^T */
        for (int a = 0; a < n; ++a) {
            for (int b = 0; b < n; ++b) t[b] = Off[(j - 1) * n * n + a * n + b];
            lower_solve(n, Lp, t);
            for (int b = 0; b < n; ++b) Wj[a * n + b] = t[b];
        }
        gemm(n, n, n, Wj, 0, Wj, 1, Lj);
        for (int i = 0; i < n * n; ++i) Lj[i] = Dg[j * n * n + i] - Lj[i];
        if (chol(n, Lj)) rc = -1;
    }
    if (rc == 0) {
        for (int j = 0; j < N; ++j) {
            for (int i = 0; i < n; ++i) y[j * n + i] = gamma[j * n + i];
            if (j > 0) {
                gemv(n, n, W + (j - 1) * n * n, 0, y + (j - 1) * n, t);
                for (int i = 0; i < n; ++i) y[j * n + i] -= t[i];
            }
            lower_solve(n, L + j * n * n, y + j * n);
        }
        for (int j = N - 1; j >= 0; --j) {
            for (int i = 0; i < n; ++i) lambda[j * n + i] = y[j * n + i];
            if (j < N - 1) {
                gemv(n, n, W + j * n * n, 1, lambda + (j + 1) * n, t);
                for (int i = 0; i < n; ++i) lambda[j * n + i] -= t[i];
            }
            upper_t_solve(n, L + j * n * n, lambda + j * n);
        }
    }
    free(L); free(W); free(y); free(t);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Recovery of dz from lambda, eq. (4): dz = -G^-1 (g + C^T lambda)          */
/* ------------------------------------------------------------------------ */
/*
 *   dx_k = -Q_k^-1 (q_k - lambda_k + A_k^T lambda_{k+1})   (no A term at N-1)
 *   du_k = -R_k^-1 (r_k + B_k^T lambda_{k+1})
 * Returns 0, or -1 if some Q_k or R_k is not positive definite.
 */
int oracle_recover(int N, int n, int m, const double *Q, const double *R,
                   const double *q, const double *r, const double *A,
                   const double *B, const double *lambda, double *dX, double *dU)
{
    int rc = 0;
    const int w = n > m ? n : m;
    double *L = malloc(sizeof(double) * w * w);
    double *t = malloc(sizeof(double) * w);
    for (int k = 0; k < N; ++k) {
        double *x = dX + k * n;
        for (int i = 0; i < n; ++i) x[i] = q[k * n + i] - lambda[k * n + i];
        if (k < N - 1) {
            gemv(n, n, A + k * n * n, 1, lambda + (k + 1) * n, t);
            for (int i = 0; i < n; ++i) x[i] += t[i];
        }
        memcpy(L, Q + k * n * n, sizeof(double) * n * n);
        if (chol(n, L)) { rc = -1; continue; }
        lower_solve(n, L, x);
        upper_t_solve(n, L, x);
        for (int i = 0; i < n; ++i) x[i] = -x[i];
    }
    for (int k = 0; k < N - 1; ++k) {
        double *u = dU + k * m;
        gemv(n, m, B + k * n * m, 1, lambda + (k + 1) * n, t);
        for (int i = 0; i < m; ++i) u[i] = r[k * m + i] + t[i];
        memcpy(L, R + k * m * m, sizeof(double) * m * m);
        if (chol(m, L)) { rc = -1; continue; }
        lower_solve(m, L, u);
        upper_t_solve(m, L, u);
        for (int i = 0; i < m; ++i) u[i] = -u[i];
    }
    free(L); free(t);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* L1 merit and the parallel line search (Sec. III-A)                        */
/* ------------------------------------------------------------------------ */
/*
 * Reading: M(alpha) = J(zbar + alpha dz) + mu * ||c(zbar + alpha dz)||_1 with
 * zbar = 0, evaluated by its full formula at x = alpha dx, u = alpha du:
 *   J = sum_k 1/2 x_k^T Q_k x_k + q_k^T x_k + sum_{k<N-1} 1/2 u_k^T R_k u_k + r_k^T u_k
 *   ||c||_1 = ||x_0 - s0||_1 + sum_{k<N-1} ||A_k x_k + B_k u_k + e_k - x_{k+1}||_1
 * Returns the merit; *J_out and *viol_out receive the two parts.
 */
double oracle_merit(int N, int n, int m, const double *Q, const double *R,
                    const double *q, const double *r, const double *A,
                    const double *B, const double *e, const double *s0,
                    const double *dX, const double *dU, double alpha, double mu,
                    double *J_out, double *viol_out)
{
    const int w = n > m ? n : m;
    double *x = malloc(sizeof(double) * n), *xn = malloc(sizeof(double) * n);
    double *u = malloc(sizeof(double) * (m > 0 ? m : 1)), *t = malloc(sizeof(double) * w);
    double J = 0.0, viol = 0.0;
    for (int k = 0; k < N; ++k) {
        for (int i = 0; i < n; ++i) x[i] = alpha * dX[k * n + i];
        gemv(n, n, Q + k * n * n, 0, x, t);
        J += 0.5 * dot(n, x, t) + dot(n, q + k * n, x);
        if (k == 0)
            for (int i = 0; i < n; ++i) viol += fabs(x[i] - s0[i]);
        if (k < N - 1) {
            for (int i = 0; i < m; ++i) u[i] = alpha * dU[k * m + i];
            gemv(m, m, R + k * m * m, 0, u, t);
            J += 0.5 * dot(m, u, t) + dot(m, r + k * m, u);
            for (int i = 0; i < n; ++i) xn[i] = alpha * dX[(k + 1) * n + i];
            for (int i = 0; i < n; ++i) {
                double s = e[k * n + i] - xn[i];
                for (int j = 0; j < n; ++j) s += A[k * n * n + i * n + j] * x[j];
                for (int j = 0; j < m; ++j) s += B[k * n * m + i * m + j] * u[j];
                viol += fabs(s);
            }
        }
    }
    free(x); free(xn); free(u); free(t);
    if (J_out) *J_out = J;
    if (viol_out) *viol_out = viol;
    return J + mu * viol;
}

/*
 * Candidates: merit[0] at alpha = 0, merit[1 + i] at alpha = beta^-i,
 * i = 0..n_alpha-1.  best = argmin_i merit[1 + i] (lowest i on ties); the step
 * is accepted iff merit[1 + best] < merit[0], otherwise best = -1.
 * Returns best.
 */
int oracle_linesearch(int N, int n, int m, const double *Q, const double *R,
                      const double *q, const double *r, const double *A,
                      const double *B, const double *e, const double *s0,
                      const double *dX, const double *dU, int n_alpha,
                      double beta, double mu, double *merit)
{
    merit[0] = oracle_merit(N, n, m, Q, R, q, r, A, B, e, s0, dX, dU, 0.0, mu, 0, 0);
    int best = 0;
    double alpha = 1.0;
    for (int i = 0; i < n_alpha; ++i) {
        merit[1 + i] = oracle_merit(N, n, m, Q, R, q, r, A, B, e, s0, dX, dU, alpha, mu, 0, 0);
        if (merit[1 + i] < merit[1 + best]) best = i;
        alpha /= beta;
    }
    return merit[1 + best] < merit[0] ? best : -1;
}

/* ------------------------------------------------------------------------ */
/* Whole path for one solve: Schur, stair, PCG, recovery, line search        */
/* ------------------------------------------------------------------------ */
/* Returns a status bitmask: 1 PCG reached max_iters, 2 non-positive pivot,
 * 4 line search found no decrease. */
int oracle_solve_kkt(int N, int n, int m, const double *Q, const double *R,
                     const double *q, const double *r, const double *A,
                     const double *B, const double *e, const double *s0,
                     double eps, int max_iters, int stop_rule, int n_alpha,
                     double beta, double mu, double *dX, double *dU, double *lambda, int *iters,
                     double *merit, int *best)
{
    int status = 0;
    double *Dg = malloc(sizeof(double) * N * n * n);
    double *Off = malloc(sizeof(double) * (N > 1 ? N - 1 : 1) * n * n);
    double *Pd = malloc(sizeof(double) * N * n * n);
    double *Po = malloc(sizeof(double) * (N > 1 ? N - 1 : 1) * n * n);
    double *gamma = malloc(sizeof(double) * N * n);
    if (oracle_schur(N, n, m, Q, R, q, r, A, B, e, s0, Dg, Off, gamma)) status |= 2;
    if (oracle_stair(N, n, Dg, Off, Pd, Po)) status |= 2;
    if (oracle_pcg(N, n, Dg, Off, Pd, Po, gamma, 0, eps, max_iters, stop_rule, lambda, iters))
        status |= 1;
    if (oracle_recover(N, n, m, Q, R, q, r, A, B, lambda, dX, dU)) status |= 2;
    *best = oracle_linesearch(N, n, m, Q, R, q, r, A, B, e, s0, dX, dU, n_alpha, beta, mu, merit);
    if (*best < 0) status |= 4;
    free(Dg); free(Off); free(Pd); free(Po); free(gamma);
    return status;
}

/* ------------------------------------------------------------------------ */
/* SQP on a linear model with rho damping (Sec. II steps 1-3; Sec. IV-C)     */
/* ------------------------------------------------------------------------ */
/*
 * The problem (a linear model in place of the robot dynamics):
 *   minimize  J(X, U) = sum_k 1/2 x_k^T Q_k x_k + q_k^T x_k
 *                     + sum_{k<N-1} 1/2 u_k^T R_k u_k + r_k^T u_k
 *   s.t.      x_0 = xs,   x_{k+1} = A_k x_k + B_k u_k + c_k.
 * One SQP iteration at the nominal (X, U), in the paper's three steps:
 *   1. the quadratic program of the expansion along (X, U) -- exact for this
 *      model: gradients q_k + Q_k x_k and r_k + R_k u_k, defects
 *      e_k = A_k x_k + B_k u_k + c_k - x_{k+1} and s0 = xs - x_0, with the
 *      damping rho added to the diagonal of every Q_k (Sec. IV-C);
 *   2. its KKT solution dz (computed exactly here: Schur complement, block
 *      Cholesky, recovery);
 *   3. the line search on the L1 merit of the problem itself (undamped Q):
 *      oracle_linesearch on the expansion's data gives M(X + a dX, U + a dU)
 *      - J(X, U), and (X, U) += a* dz when a candidate beats a = 0.
 * The damping follows the line search (reading of "adjusted after each SQP
 * iteration based on the status of the line search"): rho <- max(rho / f,
 * rho_min) after an accepted step, min(rho f, rho_max) after a failed one.
 * Outputs: X, U updated in place; merit_hist[0] the merit at the start and
 * merit_hist[t + 1] after iteration t; best_hist[t] the line-search index
 * (-1 on failure); rho_hist[t] the rho of iteration t and rho_hist[iters] the
 * final one; lambda the multipliers of the last subproblem.  Returns a
 * status mask: 2 a non-positive pivot, 4 some line search failed.
 */
int oracle_sqp_linear(int N, int n, int m, const double *Q, const double *R,
                      const double *q, const double *r, const double *A,
                      const double *B, const double *c, const double *xs, int iters,
                      double rho, double rho_factor, double rho_min, double rho_max,
                      int n_alpha, double beta, double mu, double *X, double *U,
                      double *lambda, double *merit_hist, int *best_hist, double *rho_hist)
{
    const int K = N > 1 ? N - 1 : 1;
    int status = 0;
    double *Qd = malloc(sizeof(double) * N * n * n);
    double *qt = malloc(sizeof(double) * N * n), *rt = malloc(sizeof(double) * K * m);
    double *et = malloc(sizeof(double) * K * n), *s0t = malloc(sizeof(double) * n);
    double *Dg = malloc(sizeof(double) * N * n * n), *Off = malloc(sizeof(double) * K * n * n);
    double *gamma = malloc(sizeof(double) * N * n);
    double *dX = malloc(sizeof(double) * N * n), *dU = malloc(sizeof(double) * K * m);
    double *merit = malloc(sizeof(double) * (n_alpha + 1));
    double *t = malloc(sizeof(double) * (n > m ? n : m));
    for (int it = 0; it < iters; ++it) {
        /* step 1: expansion along (X, U) and J(X, U) */
        double J = 0.0;
        for (int k = 0; k < N; ++k) {
            const double *x = X + k * n;
            gemv(n, n, Q + k * n * n, 0, x, t);
            for (int i = 0; i < n; ++i) qt[k * n + i] = t[i] + q[k * n + i];
            J += 0.5 * dot(n, x, t) + dot(n, q + k * n, x);
            for (int i = 0; i < n * n; ++i) Qd[k * n * n + i] = Q[k * n * n + i];
            for (int i = 0; i < n; ++i) Qd[k * n * n + i * n + i] += rho;
            if (k < N - 1) {
                const double *u = U + k * m;
                gemv(m, m, R + k * m * m, 0, u, t);
                for (int i = 0; i < m; ++i) rt[k * m + i] = t[i] + r[k * m + i];
                J += 0.5 * dot(m, u, t) + dot(m, r + k * m, u);
                for (int i = 0; i < n; ++i) {
                    double s = c[k * n + i] - X[(k + 1) * n + i];
                    for (int j = 0; j < n; ++j) s += A[k * n * n + i * n + j] * x[j];
                    for (int j = 0; j < m; ++j) s += B[k * n * m + i * m + j] * u[j];
                    et[k * n + i] = s;
                }
            }
        }
        for (int i = 0; i < n; ++i) s0t[i] = xs[i] - X[i];
        rho_hist[it] = rho;
        /* step 2: the damped subproblem's KKT solution */
        if (oracle_schur(N, n, m, Qd, R, qt, rt, A, B, et, s0t, Dg, Off, gamma) ||
            oracle_block_cholesky(N, n, Dg, Off, gamma, lambda) ||
            oracle_recover(N, n, m, Qd, R, qt, rt, A, B, lambda, dX, dU))
            status |= 2;
        /* step 3: line search on the problem's own merit */
        const int best = oracle_linesearch(N, n, m, Q, R, qt, rt, A, B, et, s0t, dX, dU,
                                           n_alpha, beta, mu, merit);
        if (it == 0) merit_hist[0] = J + merit[0];
        best_hist[it] = best;
        if (best >= 0) {
            double alpha = 1.0;
            for (int i = 0; i < best; ++i) alpha /= beta;
            for (int i = 0; i < N * n; ++i) X[i] += alpha * dX[i];
            for (int i = 0; i < (N - 1) * m; ++i) U[i] += alpha * dU[i];
            merit_hist[it + 1] = J + merit[1 + best];
            rho = rho / rho_factor;
            if (rho < rho_min) rho = rho_min;
        } else {
            status |= 4;
            merit_hist[it + 1] = J + merit[0];
            rho = rho * rho_factor;
            if (rho > rho_max) rho = rho_max;
        }
    }
    rho_hist[iters] = rho;
    free(Qd); free(qt); free(rt); free(et); free(s0t); free(Dg); free(Off); free(gamma);
    free(dX); free(dU); free(merit); free(t);
    return status;
}
