/*
 * gato.h -- C ABI of the GB300 (sm_103a) batched KKT solver.
 *
 * The solver takes a batch of M independent linear-quadratic trajectory
 * subproblems (GATO paper, "GATO: GPU-Accelerated and Batched Trajectory
 * Optimization for Scalable Edge Model Predictive Control", Sec. II eq. (1))
 * and runs the data-parallel half of one SQP iteration on the GPU:
 *
 *   gato_form_schur   Schur complement S = C G^-1 C^T, gamma and the symmetric
 *                     stair preconditioner Phi^-1 (Sec. II eqs. (4)-(6)),
 *   gato_pcg_solve    batched preconditioned CG on S lambda = gamma (Sec. II)
 *                     and recovery of dz = -G^-1 (g + C^T lambda) (eq. (4)),
 *   gato_linesearch   the parallel line search over alpha = beta^-i with the
 *                     L1 merit J + mu ||c||_1 (Sec. III-A),
 *   gato_solve_kkt    all of the above, in order, on one stream,
 *   gato_apply_step   the update Z <- Z + alpha* dZ (Sec. III-A).
 *
 * Problem layout (all pointers are fp32 DEVICE memory, dense row-major,
 * solve-major then knot-major, no padding; the caller owns every buffer):
 *   Q  [M][N][n][n]    state cost Hessians (symmetric positive definite)
 *   R  [M][N-1][m][m]  control cost Hessians (symmetric positive definite)
 *   q  [M][N][n]       state cost gradients
 *   r  [M][N-1][m]     control cost gradients
 *   A  [M][N-1][n][n]  dynamics Jacobians wrt x
 *   B  [M][N-1][n][m]  dynamics Jacobians wrt u
 *   e  [M][N-1][n]     defects f(x_k, u_k) - x_{k+1}
 *   s0 [M][n]          initial-state error x_s - x_0
 * N counts state knots x_0..x_{N-1}; there are N-1 controls.  When N == 1
 * the [N-1] arrays are empty and their pointers may be NULL.
 *
 * Constraints of the QP:  dx_0 = s0,  A_k dx_k + B_k du_k + e_k = dx_{k+1}.
 * Multipliers follow  G dz + C^T lambda = -g  with C's row for dx_0 equal to
 * -I, so lambda_0 = Q_0 dx_0 + q_0 + A_0^T lambda_1 and so on.
 *
 * Streams and errors: every call is asynchronous on `stream` (a cudaStream_t
 * passed as void*, NULL = legacy default stream) and never synchronises the
 * device.  Return values: GATO_OK, or a negative call-level error (nothing
 * was launched unless the error is GATO_ERR_CUDA).  Per-solve outcomes are
 * OR-ed into the caller's device array `status[M]` (uint32, not cleared by
 * the library: zero it before the first call); see GATO_STATUS_*.
 * Device code never traps and every loop is bounded.
 */
#ifndef GATO_H
#define GATO_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* call-level return codes */
#define GATO_OK 0
#define GATO_ERR_INVALID_ARG (-1)  /* NULL pointer, M/N/n/m out of range      */
#define GATO_ERR_UNSUPPORTED (-2)  /* sizes beyond the kernels' limits         */
#define GATO_ERR_CUDA (-3)         /* a CUDA call or kernel launch failed     */
#define GATO_ERR_NO_MEMORY (-4)    /* workspace allocation failed             */

/* per-solve status bits (device array status[M]) */
#define GATO_STATUS_PCG_MAX_ITERS 1u      /* PCG stopped at pcg_max_iters          */
#define GATO_STATUS_NONPOSITIVE_PIVOT 2u  /* a Cholesky pivot of Q_k, R_k or S_jj
                                             was <= 0 or not finite: flagged, not
                                             repaired (the pivot is replaced by 1
                                             so that the arithmetic stays finite) */
#define GATO_STATUS_LINESEARCH_FAILED 4u  /* no candidate beat M(0); best = -1     */
#define GATO_STATUS_NONFINITE 8u          /* a NaN/Inf reached a PCG reduction or
                                             a merit value                          */
#define GATO_STATUS_BOUNDS 16u            /* library built with GATO_DEBUG_BOUNDS
                                             only: a device index check failed and
                                             the access was skipped (never set by
                                             the normal build)                      */

/* PCG stopping rules (GATO paper Sec. II: "up to tolerance eps") */
#define GATO_STOP_RESIDUAL 0       /* ||gamma - S lambda||_2 <= eps ||gamma||_2   */
#define GATO_STOP_PRECOND 1        /* r^T Phi^-1 r <= eps^2 (r0^T Phi^-1 r0)      */
#define GATO_STOP_SCALED 2         /* ||r||_{D^-1} <= eps ||gamma||_{D^-1}, D the
                                      block diagonal of S                         */

/* PCG kernel selection (gato_set_pcg_kernel) */
#define GATO_PCG_AUTO 0            /* for 7 <= n <= 16 the wide-tile kernel when
                                      N <= 128 and the cluster kernel (2 or 4
                                      CTAs per solve) when 128 < N <= 512; for
                                      16 < n <= 64 the register-row kernel, with
                                      a solve over a cluster of 2, 4 or 8 CTAs
                                      where one CTA cannot hold it (N ceil(n/R)
                                      threads beyond the register budget: N > 18
                                      at n = 36); else the generic kernel         */
#define GATO_PCG_GENERIC 1         /* always the generic kernel                   */
#define GATO_PCG_WIDE 2            /* the wide-tile kernel (two threads per
                                      coupling block, rows over all 2H columns)
                                      where it applies, else as GATO_PCG_AUTO     */
#define GATO_PCG_TILE 3            /* the four-thread tile kernel (H x H tiles)
                                      where it applies, else as GATO_PCG_AUTO     */
#define GATO_PCG_ROWS 4            /* the register-row kernel (whole rows of the
                                      two coupling blocks around a knot per
                                      thread) for any n <= 64, one CTA per solve
                                      or its cluster form (up to 8 CTAs), else
                                      as GATO_PCG_AUTO                            */
#define GATO_PCG_QUAD 5            /* the four-thread kernel with row quarters
                                      over all n columns (7 <= n <= 16,
                                      N <= 128; column sums reduced by warp
                                      shuffles within the quad) where it
                                      applies, else as GATO_PCG_AUTO.  AUTO
                                      takes it at n = 12, and elsewhere where
                                      the wide-tile kernel would leave each SM
                                      with at most four working warps (2N
                                      threads per solve, as many solves per SM
                                      as the batch and the occupancy give)        */
/* reported in gato_stats.pcg_kernel only (not choices of gato_set_pcg_kernel) */
#define GATO_PCG_CLUSTER 6         /* the wide-tile iteration over a cluster of
                                      2 or 4 CTAs per solve (128 < N <= 512)      */
#define GATO_PCG_DOUBLE_FLOAT 7    /* the double-float kernel (pcg_precision FF),
                                      one CTA or a cluster of two per solve       */

/* Arithmetic of the main PCG solve (gato_params.pcg_precision).  The
 * iteration count of CG in finite precision grows with the rounding unit:
 * on long, poorly conditioned horizons fp32 PCG needs 3-25 % more iterations
 * than fp64 PCG to reach the same relative residual, and a stated
 * iteration cap can stop it first.  The double-float kernel carries the
 * vectors, products, inner products and CG scalars as pairs of floats
 * (about 48 significand bits), at fp32 instruction speed, on the operator
 * formed in fp32; it follows the fp64 iteration count closely and costs
 * several times the fp32 kernels' time per iteration. */
#define GATO_PCG_PRECISION_FP32 0  /* fp32 vectors and sums (default)           */
#define GATO_PCG_PRECISION_FF 1    /* double-float: one block per solve, one
                                      thread per row of S (two when N n > 1024),
                                      any n <= 64 with N n <= 2048 (N n <= 1024
                                      when n > 16) and the blocks in shared
                                      memory; larger sizes are rejected with
                                      GATO_ERR_UNSUPPORTED                       */

/* How refinement corrections are solved (gato_params.refine_solver). */
#define GATO_REFINE_SOLVER_SAME 0    /* with the main solve's solver: PCG to
                                        refine_eps, or the direct solve's factors
                                        (default)                                 */
#define GATO_REFINE_SOLVER_DIRECT 1  /* with the cyclic-reduction factorisation of
                                        the same S (bdsv), factored once per call
                                        when the main solve is PCG: each correction
                                        is then a substitution, exact for the
                                        fp32-formed S                             */

/* Linear solver of S lambda = gamma (gato_params.linsys).  The direct solver
 * (bdsv) factors the block-tridiagonal S exactly instead of iterating; the
 * GATO documentation measures it about linear in the horizon N and faster
 * than PCG from N = 256 (its BDSV_HORIZON policy), which GATO_LINSYS_AUTO
 * follows with the threshold gato_params.bdsv_horizon. */
#define GATO_LINSYS_AUTO 0         /* PCG when N < bdsv_horizon, else the cyclic-
                                      reduction direct solve (default)            */
#define GATO_LINSYS_PCG 1          /* always PCG                                  */
#define GATO_LINSYS_BDSV 2         /* direct solve, cyclic reduction (odd knots
                                      first, ceil(log2 N) levels)                 */
#define GATO_LINSYS_BDSV_CHRONO 3  /* direct solve, block Cholesky in
                                      chronological order (block Thomas)          */

/* direct-solve kernel selection (gato_set_bdsv_kernel) */
#define GATO_BDSV_KERNEL_AUTO 0    /* register kernel for cyclic reduction when
                                      n <= 16, else the shared-memory kernel      */
#define GATO_BDSV_KERNEL_SHARED 1  /* always the shared-memory kernel             */

/* formation kernel selection (gato_set_form_kernel) */
#define GATO_FORM_AUTO 0           /* register kernels when n, m <= 16, else the
                                      shared-memory kernels                        */
#define GATO_FORM_SHARED 1         /* always the shared-memory kernels           */

/* merit kernels (gato_params.merit_kernel) */
#define GATO_MERIT_FUSED 0         /* knots read once, candidates in factored
                                      form (default): a half-warp per knot and the
                                      blocks of a solve summed in block order when
                                      n, m <= 16, else one block per solve        */
#define GATO_MERIT_PER_CANDIDATE 1 /* one block of merit_threads per (knot,
                                      candidate), full formula per candidate      */

/* Limits of the library. */
#define GATO_MAX_STATE 64          /* n <= 64 */
#define GATO_MAX_CONTROL 64        /* m <= 64 */
#define GATO_MAX_ALPHA 31          /* n_alpha <= 31 */
#define GATO_NOALLOC_MAX_BYTES (32u * 1024u * 1024u) /* scratch of gato_solve_kkt_noalloc */

typedef struct gato_params {
    float pcg_eps;       /* PCG tolerance eps (default 1e-6)                     */
    int pcg_max_iters;   /* PCG iteration cap (default 200)                       */
    int stop_rule;       /* GATO_STOP_* (default GATO_STOP_RESIDUAL)              */
    int refine_steps;    /* gato_solve_kkt only: rounds of iterative refinement of
                            the KKT solution, residual in compensated fp32
                            (default 0)                                            */
    int n_alpha;         /* line-search candidates A (default 8)                  */
    float beta;          /* alpha_i = beta^-i, beta > 1 (default 2)               */
    float mu;            /* L1 penalty weight (default 10)                        */
    int merit_threads;   /* threads per merit block, 32..256, multiple of 32
                            (default 64); results are bit-identical at any size   */
    float refine_eps;    /* PCG tolerance of each refinement correction, on the
                            preconditioned residual sqrt(r^T Phi^-1 r / r0^T Phi^-1
                            r0); 0 means pcg_eps (default 0.1: a correction only
                            needs a digit)                                         */
    int merit_kernel;    /* GATO_MERIT_FUSED (default) or GATO_MERIT_PER_CANDIDATE */
    int linsys;          /* GATO_LINSYS_* (default GATO_LINSYS_AUTO)              */
    int bdsv_horizon;    /* GATO_LINSYS_AUTO: direct solve when N >= bdsv_horizon
                            (default 256); >= 1                                    */
    int pcg_precision;   /* GATO_PCG_PRECISION_* of the main PCG solve (default
                            GATO_PCG_PRECISION_FP32); refinement corrections are
                            always solved in fp32                                  */
    int refine_solver;   /* GATO_REFINE_SOLVER_* (default GATO_REFINE_SOLVER_SAME) */
} gato_params;

/* SQP loop on a linear model (gato_sqp_linear). */
typedef struct gato_sqp_params {
    int iters;           /* SQP iterations of one call, >= 1 (default 10)          */
    float rho_factor;    /* > 1: after each line search rho <- max(rho / factor,
                            rho_min) when a step was accepted, min(rho * factor,
                            rho_max) when none was (default 10)                    */
    float rho_min;       /* 0 <= rho_min <= rho_max (default 1e-8)                  */
    float rho_max;       /* (default 10)                                            */
    int warm_start;      /* 1: each PCG solve starts from the current lambda (the
                            caller's on entry, then the previous iteration's);
                            0: from zero (default 1)                               */
    int use_graph;       /* 1: one iteration is recorded as a CUDA graph once and
                            replayed (default); 0: launched kernel by kernel      */
} gato_sqp_params;

typedef struct gato_stats {
    float form_us;       /* device time of the last call's stages (microseconds), */
    float pcg_us;        /* filled only when timing was enabled with              */
    float refine_us;     /* gato_set_timing; -1 for a stage that did not run.     */
    float merit_us;      /* pcg_us: the linear solve (PCG, or the direct solve's  */
    float total_us;      /* factorisation and substitution); refine_us: every
                            refinement round (residual, right-hand side, solve).  */
    int pcg_kernel;      /* the kernel the last call's main PCG solve ran: a
                            GATO_PCG_* value other than AUTO (WIDE, TILE, QUAD,
                            ROWS, GENERIC, CLUSTER or DOUBLE_FLOAT); 0 when the
                            call ran no PCG solve.  Filled with or without
                            timing.                                              */
    int refine_kernel;   /* the same for the refinement corrections' PCG solves
                            (0 when they were direct or did not run)             */
} gato_stats;

typedef struct gato_handle gato_handle;

/* Default parameters (values above). */
void gato_default_params(gato_params* p);
void gato_default_sqp_params(gato_sqp_params* sp);

/* Creates a solver for M solves of N knots, n states and m controls on the
 * current CUDA device and allocates its device workspace (one cudaMalloc of
 * the bytes given at gato_solve_kkt_noalloc below, plus 512 bytes for each of
 * GATO_MAX_PARTS possible parts).  *h receives the handle, which the caller
 * releases with gato_destroy.  Errors: INVALID_ARG (h NULL, M, N, n or
 * m < 1), UNSUPPORTED (n or m above the limits), NO_MEMORY, CUDA. */
int gato_create(gato_handle** h, int M, int N, int n, int m);

/* Frees the workspace and the handle (waits for nothing: the caller must make
 * sure no call using the handle is still running). NULL is ignored. */
void gato_destroy(gato_handle* h);

/* Turns per-stage CUDA-event timing on (1) or off (0).  When on, calls record
 * events on their stream; gato_get_stats synchronises on the last one. */
int gato_set_timing(gato_handle* h, int on);

/* Stage times of the last call (see gato_stats). */
int gato_get_stats(gato_handle* h, gato_stats* out);

/* Chooses the PCG kernel (GATO_PCG_AUTO, GATO_PCG_GENERIC, GATO_PCG_WIDE,
 * GATO_PCG_TILE, GATO_PCG_ROWS or GATO_PCG_QUAD) for later calls.
 * Both give the same PCG iterates up to rounding; the generic kernel covers
 * every supported size.  Errors: INVALID_ARG. */
int gato_set_pcg_kernel(gato_handle* h, int kind);

/* Chooses the direct-solve kernels (GATO_BDSV_KERNEL_AUTO or
 * GATO_BDSV_KERNEL_SHARED) for later calls; both compute the same
 * factorisation up to rounding.  Errors: INVALID_ARG. */
int gato_set_bdsv_kernel(gato_handle* h, int kind);

/* Chooses the formation kernels (GATO_FORM_AUTO or GATO_FORM_SHARED) for later
 * calls; both compute the same blocks up to rounding.  Errors: INVALID_ARG. */
int gato_set_form_kernel(gato_handle* h, int kind);

/* a1 + a2.  Forms, per solve and knot (GATO paper Sec. II, eqs. (4)-(6)):
 *   S_00 = Q_0^-1, S_jj = A_{j-1} Q_{j-1}^-1 A_{j-1}^T + B_{j-1} R_{j-1}^-1 B_{j-1}^T + Q_j^-1,
 *   S_{j,j-1} = -A_{j-1} Q_{j-1}^-1,
 *   gamma_0 = s0 + Q_0^-1 q_0,
 *   gamma_j = e_{j-1} - A_{j-1} Q_{j-1}^-1 q_{j-1} - B_{j-1} R_{j-1}^-1 r_{j-1} + Q_j^-1 q_j,
 * and the symmetric stair preconditioner
 *   Phi^-1 = D^-1 - D^-1 (L + L^T) D^-1   (D = blockdiag(S), L = S's lower blocks)
 * in the factored form the PCG kernel uses (Cholesky factors of S_jj and the
 * scaled coupling blocks L_j^-1 S_{j,j-1} L_{j-1}^-T).  Everything goes to
 * the handle's workspace; inputs are read only during this call.
 * Inputs as in the layout above; status[M] as above. */
int gato_form_schur(gato_handle* h, const float* Q, const float* R, const float* q,
                    const float* r, const float* A, const float* B, const float* e,
                    const float* s0, uint32_t* status, void* stream);

/* Copies the explicit blocks formed by the last gato_form_schur into caller
 * buffers (any may be NULL): S_diag [M][N][n][n], S_off [M][N-1][n][n] (block
 * (j, j-1) at index j-1), gamma [M][N][n], Phi_diag [M][N][n][n], Phi_off
 * [M][N-1][n][n].  Device-to-device copies on `stream`.  The solve applies
 * Phi^-1 in factored form, so the explicit Phi^-1 blocks are formed from
 * those factors on the first request after a formation (two kernels on
 * `stream`, before the copies). */
int gato_get_schur(gato_handle* h, float* S_diag, float* S_off, float* gamma,
                   float* Phi_diag, float* Phi_off, void* stream);

/* a3 + a4.  Batched PCG on S lambda = gamma with Phi^-1 (GATO paper Sec. II),
 * one thread block per solve, from lambda0 [M][N][n] (NULL = zero), stopping
 * by p->stop_rule at p->pcg_eps or after p->pcg_max_iters iterations; then
 *   dx_k = -Q_k^-1 (q_k - lambda_k + A_k^T lambda_{k+1}),
 *   du_k = -R_k^-1 (r_k + B_k^T lambda_{k+1})            (eq. (4)).
 * Outputs: lambda [M][N][n], dX [M][N][n], dU [M][N-1][m], iters [M] (int32).
 * Requires a preceding gato_form_schur on the same handle (stream-ordered).
 * p->refine_steps is ignored here (see gato_solve_kkt). */
int gato_pcg_solve(gato_handle* h, const gato_params* p, const float* lambda0,
                   float* lambda, float* dX, float* dU, int32_t* iters,
                   uint32_t* status, void* stream);

/* Direct solve of S lambda = gamma (f1 of the GATO documentation's linear
 * solvers, "bdsv"): the block-tridiagonal S is factored exactly, in the
 * block-Jacobi-scaled form S_hat = L^-1 S L^-T (identity diagonal blocks,
 * coupling blocks L_j^-1 S_{j,j-1} L_{j-1}^-T), by cyclic reduction
 * (p->linsys = GATO_LINSYS_BDSV or AUTO: odd knots eliminated first, then the
 * odd ones of the reduced chain, ceil(log2 N) levels, one thread block per
 * solve) or by block Cholesky in chronological order (GATO_LINSYS_BDSV_CHRONO,
 * the block Thomas algorithm); then lambda, and dz by eq. (4) as in
 * gato_pcg_solve.  Outputs as gato_pcg_solve; iters [M] gets 0.  A pivot of a
 * reduced block that is <= 0 sets GATO_STATUS_NONPOSITIVE_PIVOT, a non-finite
 * lambda GATO_STATUS_NONFINITE.  Requires a preceding gato_form_schur on the
 * same handle.  Errors: INVALID_ARG (also p->linsys = GATO_LINSYS_PCG). */
int gato_bdsv_solve(gato_handle* h, const gato_params* p, float* lambda, float* dX,
                    float* dU, int32_t* iters, uint32_t* status, void* stream);

/* a5 + a6.  Parallel line search (GATO paper Sec. III-A): for alpha = 0 and
 * alpha_i = beta^-i (i = 0..n_alpha-1), with x = alpha dx, u = alpha du,
 *   M(alpha) = sum_k 1/2 x_k^T Q_k x_k + q_k^T x_k + 1/2 u_k^T R_k u_k + r_k^T u_k
 *            + mu (||x_0 - s0||_1 + sum_k ||A_k x_k + B_k u_k + e_k - x_{k+1}||_1),
 * with the fused kernel (default) or one thread block per (knot, candidate)
 * (p->merit_kernel); knot sums in a fixed order, so results are reproducible
 * and, for the per-candidate kernel, identical at any p->merit_threads.
 * merit [M][n_alpha+1]: merit[.][0] is alpha = 0, merit[.][1+i] is beta^-i.
 * best [M]: argmin_i merit[1+i] (lowest i on ties) if it is below merit[0],
 * else -1 with GATO_STATUS_LINESEARCH_FAILED. */
int gato_linesearch(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                    const float* q, const float* r, const float* A, const float* B,
                    const float* e, const float* s0, const float* dX, const float* dU,
                    float* merit, int32_t* best, uint32_t* status, void* stream);

/* gato_form_schur + the linear solve (gato_pcg_solve, or gato_bdsv_solve as
 * p->linsys selects) + gato_linesearch on one stream.  With p->refine_steps =
 * k > 0 the KKT solution is refined k times: the residual of the full KKT
 * system is formed from the inputs in compensated fp32 (error-free products
 * and sums, about as accurate as fp64 accumulation), the correction is solved
 * with the same S (PCG to p->refine_eps on the correction system's relative
 * preconditioned residual, or the direct solve's factors: those of a direct
 * main solve, or with p->refine_solver = GATO_REFINE_SOLVER_DIRECT the
 * cyclic-reduction factorisation of the same S, formed once beside the PCG
 * main solve on an internal stream of the lowest priority and joined before
 * the first correction), and added to dz and lambda; iters then counts the
 * PCG iterations of every solve of the call (a direct correction adds none).
 * The batch runs as gato_set_parts parts of consecutive solves,
 * concurrently on internal streams ordered after the work already on `stream`
 * (which waits for them); the outputs do not depend on the part count.  The
 * parts' workspaces are views into the handle's own allocation (nothing is
 * allocated by the call, which can be captured into a CUDA graph), so a call
 * in parts overwrites the handle's formation: call gato_form_schur again
 * before gato_get_schur, gato_pcg_solve or gato_bdsv_solve. */
int gato_solve_kkt(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                   const float* q, const float* r, const float* A, const float* B,
                   const float* e, const float* s0, float* dX, float* dU, float* lambda,
                   int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                   void* stream);

/* The update Z <- Z + alpha* dZ (GATO paper Sec. III-A): X [M][N][n] and
 * U [M][N-1][m] are updated in place with alpha* = beta^-best per solve;
 * solves with best < 0 are left unchanged. */
int gato_apply_step(gato_handle* h, const gato_params* p, const int32_t* best,
                    const float* dX, const float* dU, float* X, float* U, void* stream);

/* SQP on a linear model (GATO paper Sec. II, the three steps repeated; the
 * rho damping and its line-search-driven adjustment of Sec. IV-C).  Each of
 * the M problems is
 *   minimise  sum_k 1/2 x_k^T Q_k x_k + q_k^T x_k + sum_{k<N-1} 1/2 u_k^T R_k u_k + r_k^T u_k
 *   s.t.      x_0 = xs,  x_{k+1} = A_k x_k + B_k u_k + c_k,
 * with c [M][N-1][n] and xs [M][n] in place of e and s0 and the other inputs
 * laid out as for gato_solve_kkt.  Starting from the trajectories X
 * [M][N][n], U [M][N-1][m] (updated in place), each iteration
 *   1. expands the problem along (X, U) (exact for this model): gradients
 *      Q_k x_k + q_k, R_k u_k + r_k, defects A_k x_k + B_k u_k + c_k - x_{k+1},
 *      xs - x_0, and adds rho[j] to the diagonal of every Q_k of problem j;
 *   2. solves that KKT system as gato_solve_kkt does (p->linsys, refinement;
 *      PCG warm-started from lambda when sp->warm_start);
 *   3. runs the line search on the problem's own L1 merit (undamped Q) and
 *      steps (X, U) += alpha* dz when a candidate beats alpha = 0;
 *   4. divides rho[j] by sp->rho_factor after an accepted step and multiplies
 *      it after a failed line search, clamped to [rho_min, rho_max].
 * rho [M] (in/out) is the per-problem damping: for a sweep over rho, give the
 * M slots the same problem and different initial rho.  lambda [M][N][n]
 * (in/out) holds the multipliers of the last subproblem.  merit_hist
 * [M][iters+1] receives the merit J + mu ||c||_1 at the start (column 0) and
 * after each iteration; iters_hist [M][iters] (may be NULL) the PCG
 * iterations of each (0 for a direct solve).  status [M] accumulates the
 * bits of every iteration (4: some line search failed).  Stage timing is not
 * recorded.  With sp->use_graph, the first call records one iteration as a
 * CUDA graph on a private stream and later calls with the same arguments
 * and parameters replay it; any change of a pointer or a parameter records
 * it again.  Errors: INVALID_ARG (a NULL input, iters < 1, rho bounds). */
int gato_sqp_linear(gato_handle* h, const gato_params* p, const gato_sqp_params* sp,
                    const float* Q, const float* R, const float* q, const float* r,
                    const float* A, const float* B, const float* c, const float* xs,
                    float* X, float* U, float* lambda, float* rho, float* merit_hist,
                    int32_t* iters_hist, uint32_t* status, void* stream);

/* gato_solve_kkt without a handle and without allocating anything.  The
 * paper has no counterpart: this entry point exists for callers that cannot
 * allocate device memory while they run, such as a real-time MPC loop whose
 * memory is fixed at start-up, or a host framework that owns every device
 * allocation.  Arguments are those of gato_solve_kkt plus the sizes (M, N,
 * n, m); the caller still provides every input and output.  The solver's
 * scratch is one static device array of GATO_NOALLOC_MAX_BYTES that every GPU
 * loading this library holds until the process exits; a problem needs
 *   4 (M (9 r(N n^2) + 3 r((N-1) n^2) + r((N-1) m^2) + r((N-1) n m) + 17 r(N n)
 *        + 6 r((N-1) m) + 2 r(N) + 64 N + 36) + M + 64) bytes of it,
 *   r(x) = max(64, x rounded up to a multiple of 64)
 * (exactly; for instance 46 solves of N = 64, n = 14, m = 7 fit and 47 do
 * not), and larger problems are rejected with GATO_ERR_UNSUPPORTED before
 * anything is launched (use gato_create for those).  The first call on each
 * device looks up the array's device address; make that first call before
 * any stream capture.  The address is cached with the identifier of the
 * device's CUDA context and looked up again when that changes (after a
 * cudaDeviceReset).  All calls share the array and it keeps the previous
 * call's contents (every entry is written before it is read, so nothing needs
 * clearing); calls that overlap on the GPU race on it, so the caller must
 * serialise them.  Never calls cudaMalloc, cudaFree or any allocating
 * routine. */
int gato_solve_kkt_noalloc(const gato_params* p, int M, int N, int n, int m, const float* Q,
                           const float* R, const float* q, const float* r, const float* A,
                           const float* B, const float* e, const float* s0, float* dX,
                           float* dU, float* lambda, int32_t* iters, float* merit,
                           int32_t* best, uint32_t* status, void* stream);

/* fp32 FMA throughput probe (a measurement helper; the paper has no
 * counterpart).  The PCG kernels keep their operator on chip, so the bound
 * of their roofline is the SM's fp32 FMA rate, which this probe measures
 * rather than assuming the nominal unit count.  Launches `blocks` blocks of
 * `threads` threads (a multiple of 32, at most 1024) on `stream`; every
 * thread runs eight independent FMA chains for 16 `trips` FMAs each, as
 * scalar fma.rn.f32 (packed = 0) or as half as many packed two-lane
 * fma.rn.f32x2 instructions (packed = 1).  sink [blocks] floats of device
 * memory is never written in practice (only under a condition that cannot
 * hold).  Returns the floating-point operations of the launch (2 per FMA),
 * or a negative GATO_ERR_* (INVALID_ARG, CUDA).  The caller times it. */
long long gato_probe_fp32(int packed, int blocks, int threads, int trips, float* sink,
                          void* stream);

/* Largest number of parts gato_solve_kkt and gato_solve_kkt_host split a
 * batch into (gato_set_parts). */
#define GATO_MAX_PARTS 8

/* gato_solve_kkt on HOST buffers: every input and output pointer (same
 * shapes and layouts as gato_solve_kkt) is host memory.  The paper has no
 * counterpart; it serves callers whose batch lives in host memory.  The call
 * splits the batch into parts of consecutive solves (gato_set_parts) and
 * runs each part on an internal stream: copy its inputs to the device, solve
 * it as gato_solve_kkt does, copy its outputs back.  The copies of one part
 * overlap the solves of the others; nothing overlaps the first part's input
 * copy, so with three parts or more that part is about half the size of the
 * others.  Each part's arithmetic is that of
 * gato_solve_kkt on the same solves, so the outputs are identical.
 * status[M] is in/out here too: it is copied in with the inputs, the bits
 * are OR-ed into it, and it is copied back.  Host buffers should be pinned
 * (cudaHostAlloc or cudaHostRegister); with pageable memory the copies are
 * staged by the driver and do not overlap.  The work is ordered after the
 * work already on `stream`, and `stream` waits for all of it: synchronise
 * `stream` before reading the outputs or reusing the inputs.  The first call
 * allocates device staging buffers for the inputs and outputs of all M
 * solves; later calls reuse them.  Stage timing is recorded only for a
 * single part.  Errors: INVALID_ARG, NO_MEMORY,
 * CUDA. */
int gato_solve_kkt_host(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                        const float* q, const float* r, const float* A, const float* B,
                        const float* e, const float* s0, float* dX, float* dU, float* lambda,
                        int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                        void* stream);

/* Number of parts gato_solve_kkt and gato_solve_kkt_host split a batch into:
 * 1 .. GATO_MAX_PARTS (capped at M), or 0 for the automatic choice (the
 * default): one part below 64 solves, two below 128, four from 128; but for
 * gato_solve_kkt with direct corrections after a PCG main solve
 * (refine_solver = GATO_REFINE_SOLVER_DIRECT, refine_steps > 0), whose
 * factorisation already runs beside the PCG on a low-priority stream, one
 * part while the PCG kernel holds the whole batch at once (its resident
 * blocks over the device: one solve per SM at N = 128, n = 14, more at
 * shorter horizons) and two beyond.  The
 * parts of a call run concurrently on internal streams of the highest
 * priority, each on its own sub-batch workspace, so the kernels of one part
 * fill the SMs that another part's leave idle (the last wave of its PCG, its
 * shorter stages).
 * Errors: INVALID_ARG. */
int gato_set_parts(gato_handle* h, int parts);

/* The number of parts the last gato_solve_kkt or gato_solve_kkt_host call on
 * this handle ran into *parts; before any such call, the number a
 * gato_solve_kkt call with the default parameters would run.
 * Errors: INVALID_ARG. */
int gato_get_parts(const gato_handle* h, int* parts);

#ifdef __cplusplus
}
#endif

#endif /* GATO_H */
