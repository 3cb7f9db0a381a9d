// gato_internal.cuh -- shared declarations of the CUDA library (not part of
// the C ABI): the handle, the workspace layout, and warp-level dense helpers
// for the small per-knot matrices (n, m <= 64) kept in shared memory.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "gato.h"

namespace gato {

// ---------------------------------------------------------------------------
// workspace: every array is [M][per-solve stride] floats; strides are rounded
// up to 64 floats (256 bytes) so that each solve's slice is 16-byte aligned
// for bulk copies.
// ---------------------------------------------------------------------------
// right-hand side data of one linear system S lambda = gamma (the problem's
// own, or the correction system of iterative refinement)
struct Rhs {
    float* gamma;  // [N][n]
    float* ghat;   // [N][n] L_j^-1 gamma_j
    float* avec;   // [N][n] -Q_k^-1 q_k
    float* bvec;   // [N-1][m] -R_k^-1 r_k
};

struct Work {
    int M, N, n, m;
    size_t sNnn;   // N n n
    size_t sKnn;   // (N-1) n n
    size_t sKmm;   // (N-1) m m
    size_t sKnm;   // (N-1) n m
    size_t sNn;    // N n
    size_t sN;     // N
    size_t sKm;    // (N-1) m
    size_t sK2;    // N (GATO_MAX_ALPHA + 1): float2 merit partials per solve
    // matrix part of the Schur formation
    float* Qinv;   // [N] Q_k^-1
    float* Rinv;   // [N-1] R_k^-1
    float* O;      // [N-1] S_{j,j-1} = -A_{j-1} Q_{j-1}^-1, at index j-1
    float* V;      // [N-1] B_k R_k^-1  (n x m)
    float* D;      // [N] S_jj
    float* L;      // [N] chol(S_jj), lower, full n x n
    float* Linv;   // [N] L_j^-1, lower
    float* Pd;     // [N] S_jj^-1 (diagonal blocks of Phi^-1)
    float* Po;     // [N-1] -S_jj^-1 S_{j,j-1} S_{j-1,j-1}^-1 (off-diagonal blocks of Phi^-1)
    float* Nh;     // [N-1] L_j^-1 S_{j,j-1} L_{j-1}^-T (scaled coupling blocks)
    float* dlow;   // [N] 1 / ||L_j^-1||_F^2, a lower bound on the smallest
                   //     eigenvalue of S_jj (1 / trace(S_jj^-1))
    // vector part: rhs[0] for the problem, rhs[1] for refinement corrections
    Rhs rhs[2];
    // iterative refinement: right-hand side of the correction system, and
    // the correction itself; these are stored densely ([M][N][n], [M][N-1][m],
    // [M][n]) inside their (larger) strided slots
    float* q2;     // [N][n]
    float* r2;     // [N-1][m]
    float* e2;     // [N-1][n]
    float* s02;    // [n]
    float* dlam;   // [N][n]
    float* ddX;    // [N][n]
    float* ddU;    // [N-1][m]
    // direct block-tridiagonal solve of S_hat lambda_hat = ghat (S_hat =
    // L^-1 S L^-T: identity diagonal blocks, coupling blocks Nhat_j).
    // Cyclic reduction: for a knot eliminated at stride s >= 2, Bd holds
    // F = C^-1 (C C^T its reduced diagonal block), Be X = F E (E its coupling
    // to the active knot s to the left) and By Y = F E_right^T; knot 0 ends
    // with F_0 of the last reduced block in Bd.  Chronological order: Bd holds
    // F_j = C_j^-1 and Be W_j = Nhat_j F_{j-1}^T of S_hat = L L^T, L block
    // lower bidiagonal with diagonal C_j and sub-diagonal W_j.
    float* Bd;     // [N] n x n
    float* Be;     // [N] n x n
    float* By;     // [N] n x n
    float* Bv;     // [N][n] vector scratch of the substitution when it does not
    float* Bg;     // [N][n] fit in shared memory
    // SQP loop on the linear model: the expansion along the current
    // trajectory (dense [M][...] like the caller's arrays), per-knot cost
    // partials, and the iteration's step, merits and counters
    float* Qd;     // [N][n][n] Q_k + rho I
    float* qt;     // [N][n]    Q_k x_k + q_k
    float* rt;     // [N-1][m]  R_k u_k + r_k
    float* et;     // [N-1][n]  A_k x_k + B_k u_k + c_k - x_{k+1}
    float* s0t;    // [n]       xs - x_0
    float* Jk;     // [N]       cost of knot k at the current trajectory (stride sN)
    float* sdX;    // [N][n]    the step
    float* sdU;    // [N-1][m]
    float* smerit; // [n_alpha + 1] (dense [M][n_alpha + 1])
    int* sbest;    // [M]
    int* siters;   // [M]
    int* sqpt;     // [M] iterations done in the current call
    // line search partial sums
    float2* mpart; // [(A+1)][N] (cost, violation) per knot and candidate
    int* queue;    // work counters of the persistent kernels (not per solve)
    int* mcount;   // [M] merit blocks arrived per solve (zeroed before each launch)
    // the current call's status[M] (may be NULL): where the index checks of
    // the debug build record GATO_STATUS_BOUNDS; set by every entry point
    // before it launches
    uint32_t* status;
};

}  // namespace gato

struct gato_handle {
    gato::Work w;
    int device;
    int smem_optin;     // bytes of dynamic shared memory a block may opt into
    int num_sms;
    void* base;         // the single workspace allocation
    size_t bytes;
    int timing;
    int pcg_kernel;         // GATO_PCG_* selected by gato_set_pcg_kernel
    int pcg_ran;            // GATO_PCG_* kernel of the last main PCG launch (0: none)
    int refine_ran;         // ... and of the last correction PCG launch
    int batch_M;            // solves running at the same time as this handle's: the
                            // whole batch when the handle is one part of it (0: w.M)
    // a low-priority stream, and the events that fork work onto it and join
    // it back, for work that may run beside the main solve (the corrections'
    // factorisation); side is NULL where there is none (the allocation-free
    // entry), and that work then runs in stream order
    cudaStream_t side;
    cudaEvent_t ev_fork, ev_join;
    int bdsv_kernel;        // GATO_BDSV_KERNEL_* selected by gato_set_bdsv_kernel
    int force_smem_form;    // GATO_FORM_SHARED selected by gato_set_form_kernel
    int phi_pending;        // the last formation left the explicit Phi^-1 blocks unformed
    int phi_smem;           // ... and it ran the shared-memory kernels (form them there)
    cudaEvent_t ev[5];  // start, after form, after PCG, after refinement, after merit
    int ev_used[5];
    gato_stats last;
    // one SQP iteration recorded as a CUDA graph, with the arguments it was
    // recorded for (replayed while they stay the same)
    cudaStream_t capture_stream;
    cudaGraphExec_t sqp_exec;
    unsigned char sqp_key[512];
    // gato_set_parts: requested part count (0 = automatic), and the streams,
    // sub-batch handles and (host entry only) staging buffers of the current
    // one
    int parts;
    int parts_last;  // parts the last gato_solve_kkt / _host call ran (0: none yet)
    struct gato_parts* pipe;
};

namespace gato {
// gato_parts.cu
size_t parts_extra_bytes();       // allocation beyond the handle's own workspace
int parts_init(gato_handle* h);   // streams and events of the parts (gato_create)
void parts_free(gato_handle* h);  // releases h->pipe
int parts_for(const gato_handle* h, const gato_params* p, bool host);
// a stream of the device's lowest priority (work that fills idle SMs) or
// highest (the solve's own stages), and the two fork/join events
cudaError_t side_stream_create(cudaStream_t* st, cudaEvent_t* fork, cudaEvent_t* join);
cudaError_t priority_stream_create(cudaStream_t* st, bool highest);
// gato_solve_kkt on parts of the batch, concurrently on internal streams;
// with `host`, every pointer is host memory and is staged through device
// buffers.  Returns a GATO_* code.
int run_parts(gato_handle* h, const gato_params* p, const float* Q, const float* R,
              const float* q, const float* r, const float* A, const float* B, const float* e,
              const float* s0, float* dX, float* dU, float* lambda, int32_t* iters, float* merit,
              int32_t* best, uint32_t* status, cudaStream_t user, bool host);
}

namespace gato {

// ---------------------------------------------------------------------------
// launchers (defined in form_schur.cu, pcg.cu, merit.cu); return cudaError_t
// ---------------------------------------------------------------------------
cudaError_t launch_form_matrices(gato_handle* h, const float* Q, const float* R,
                                 const float* A, const float* B, uint32_t* status,
                                 cudaStream_t st);
// register formation for n, m <= 16 (form_rows.cu)
bool rows_formation_supported(const Work& w);
cudaError_t launch_form_rows(gato_handle* h, const float* Q, const float* R, const float* A,
                             const float* B, uint32_t* status, cudaStream_t st);
// the explicit Phi^-1 blocks after a register formation (form_rows.cu)
cudaError_t launch_form_phi(gato_handle* h, cudaStream_t st);
cudaError_t launch_form_phi_smem(gato_handle* h, cudaStream_t st);
cudaError_t launch_form_rhs(gato_handle* h, int set, const float* q, const float* r,
                            const float* e, const float* s0, size_t s0_stride, cudaStream_t st);
cudaError_t launch_pcg(gato_handle* h, const gato_params* p, const float* lambda0,
                       float* lambda, float* dX, float* dU, int32_t* iters,
                       uint32_t* status, cudaStream_t st);
// rhs set `set`; acc_iters != 0: iterations are added to iters[] instead of stored
cudaError_t launch_pcg_ex(gato_handle* h, const gato_params* p, int set, const float* lambda0,
                          float* lambda, float* dX, float* dU, int32_t* iters, int acc_iters,
                          uint32_t* status, cudaStream_t st);
cudaError_t launch_kkt_residual(gato_handle* h, const float* Q, const float* R,
                                const float* q, const float* r, const float* A,
                                const float* B, const float* e, const float* s0,
                                const float* dX, const float* dU, const float* lambda,
                                cudaStream_t st);
cudaError_t launch_accumulate(gato_handle* h, float* lambda, float* dX, float* dU,
                              int32_t* iters, cudaStream_t st);
cudaError_t launch_merit(gato_handle* h, const gato_params* p, const float* Q,
                         const float* R, const float* q, const float* r, const float* A,
                         const float* B, const float* e, const float* s0, const float* dX,
                         const float* dU, float* merit, int32_t* best, uint32_t* status,
                         cudaStream_t st);
cudaError_t launch_apply_step(gato_handle* h, const gato_params* p, const int32_t* best,
                              const float* dX, const float* dU, float* X, float* U,
                              cudaStream_t st);
// direct solve (bdsv.cu): factorisation of S_hat in the order `order`
// (GATO_LINSYS_BDSV or GATO_LINSYS_BDSV_CHRONO), then substitution for the
// right-hand side set `set` and recovery of dz; iters[] gets 0 (or nothing
// added when acc_iters)
cudaError_t launch_bdsv_factor(gato_handle* h, int order, uint32_t* status, cudaStream_t st);
cudaError_t launch_bdsv_solve(gato_handle* h, int order, int set, float* lambda, float* dX,
                              float* dU, int32_t* iters, int acc_iters, uint32_t* status,
                              cudaStream_t st);

// workspace layout shared by gato_create and the allocation-free entry point:
// sets every pointer of w from base (when base != NULL) and returns the bytes
size_t carve_workspace(Work& w, int M, int N, int n, int m, float* base);
bool params_valid(const gato_params* p);
// the double-float PCG kernel takes N knots of n states within smem_limit
// bytes of shared memory per block (pcg_ff.cu)
bool pcg_ff_fits(int N, int n, size_t smem_limit);
// the kernels p asks for take the sizes of w: false when p asks for the
// double-float PCG and the linear solver is PCG but the kernel cannot take
// them (checked before anything is launched)
bool sizes_supported(const Work& w, const gato_params* p, int smem_limit);
// the linear solver a call with parameters p uses: GATO_LINSYS_PCG,
// GATO_LINSYS_BDSV or GATO_LINSYS_BDSV_CHRONO
int linsys_for(const gato_params* p, int N);
// solves one PCG launch over the handle's whole batch holds at once (pcg.cu)
int pcg_solves_per_wave(const gato_handle* h, const gato_params* p);
// formation with Q_form, right-hand side, linear solve (from lambda0 when not
// NULL), refinement rounds and line search with Q_merit, on stream st; the
// handle's timing events are recorded when `timed`
cudaError_t run_kkt_core(gato_handle* h, const gato_params* p, const float* Q_form,
                         const float* Q_merit, const float* R, const float* q, const float* r,
                         const float* A, const float* B, const float* e, const float* s0,
                         const float* lambda0, float* dX, float* dU, float* lambda,
                         int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                         cudaStream_t st, bool timed);
// SQP loop kernels (sqp.cu)
cudaError_t launch_sqp_linearize(gato_handle* h, const float* Q, const float* R, const float* q,
                                 const float* r, const float* A, const float* B, const float* c,
                                 const float* xs, const float* X, const float* U,
                                 const float* rho, cudaStream_t st);
cudaError_t launch_sqp_step(gato_handle* h, const gato_params* p, const gato_sqp_params* sp,
                            float* X, float* U, float* rho, float* merit_hist,
                            int32_t* iters_hist, cudaStream_t st);
// the whole gato_solve_kkt sequence on stream st (events recorded when the
// handle times)
cudaError_t run_solve_kkt(gato_handle* h, const gato_params* p, const float* Q, const float* R,
                          const float* q, const float* r, const float* A, const float* B,
                          const float* e, const float* s0, float* dX, float* dU, float* lambda,
                          int32_t* iters, float* merit, int32_t* best, uint32_t* status,
                          cudaStream_t st);

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

// ---------------------------------------------------------------------------
// index checks of the debug build (compiled with -DGATO_DEBUG_BOUNDS=1, the
// stand-in for a memory checker): an index outside its array, or a layout
// that does not fit the block's dynamic shared memory, is recorded as
// GATO_STATUS_BOUNDS in the call's status[sol] and the check returns false,
// so that the caller skips the access.  Nothing traps.  In the normal build
// both checks are the constant true and vanish.
// ---------------------------------------------------------------------------
#ifndef GATO_DEBUG_BOUNDS
#define GATO_DEBUG_BOUNDS 0
#endif

__device__ __forceinline__ bool gb_ok(long long idx, long long limit, uint32_t* status, int sol)
{
#if GATO_DEBUG_BOUNDS
    if (idx >= 0 && idx < limit) return true;
    if (status) atomicOr(status + sol, GATO_STATUS_BOUNDS);
    return false;
#else
    (void)idx;
    (void)limit;
    (void)status;
    (void)sol;
    return true;
#endif
}

// the block's layout needs `bytes` of dynamic shared memory
__device__ __forceinline__ bool gb_smem(size_t bytes, uint32_t* status, int sol)
{
#if GATO_DEBUG_BOUNDS
    unsigned dyn;
    asm volatile("mov.u32 %0, %%dynamic_smem_size;" : "=r"(dyn));
    if (bytes <= dyn) return true;
    if (status) atomicOr(status + sol, GATO_STATUS_BOUNDS);
    return false;
#else
    (void)bytes;
    (void)status;
    (void)sol;
    return true;
#endif
}

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ float warp_sum(float v)
{
    // xor butterfly: every lane ends with the same, order-fixed sum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// dst[0..count) = s * src[0..count), lanes over elements.  The loads are
// issued in batches (eight per lane, 128-bit when both ends are 16-byte
// aligned and count is a multiple of 4) before their stores, so that a
// matrix copied from global memory costs a few memory latencies rather than
// one per 32 elements.
__device__ __forceinline__ void warp_copy(float* dst, const float* src, int count,
                                          float s = 1.f)
{
    const int lane = lane_id();
    if ((((uintptr_t)dst | (uintptr_t)src) & 15) == 0 && (count & 3) == 0) {
        const float4* s4 = reinterpret_cast<const float4*>(src);
        float4* d4 = reinterpret_cast<float4*>(dst);
        const int c4 = count >> 2;
        int i = lane;
        for (; i + 7 * 32 < c4; i += 8 * 32) {
            float4 v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = s4[i + 32 * k];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                d4[i + 32 * k] = make_float4(s * v[k].x, s * v[k].y, s * v[k].z, s * v[k].w);
        }
        for (; i < c4; i += 32) {
            const float4 v = s4[i];
            d4[i] = make_float4(s * v.x, s * v.y, s * v.z, s * v.w);
        }
        return;
    }
    int i = lane;
    for (; i + 7 * 32 < count; i += 8 * 32) {
        float v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) v[k] = src[i + 32 * k];
#pragma unroll
        for (int k = 0; k < 8; ++k) dst[i + 32 * k] = s * v[k];
    }
    for (; i < count; i += 32) dst[i] = s * src[i];
}

// In-place lower Cholesky a = L L^T of the n x n row-major matrix in shared
// memory (only the lower triangle is read; the strict upper triangle is
// zeroed).  Right-looking, one row per lane.  A pivot that is <= 0 or not
// finite is flagged (return false) and replaced by 1 so that the rest of the
// factorisation stays finite.
__device__ inline bool warp_cholesky(float* a, int n)
{
    const int lane = lane_id();
    bool ok = true;
    for (int k = 0; k < n; ++k) {
        __syncwarp();
        const float d = a[k * n + k];
        const bool bad = !(d > 0.f) || !isfinite(d);
        ok = ok && !bad;
        const float s = bad ? 1.f : sqrtf(d);
        const float inv = 1.f / s;
        __syncwarp();
        if (lane == 0) a[k * n + k] = s;
        for (int i = k + 1 + lane; i < n; i += 32) a[i * n + k] *= inv;
        __syncwarp();
        for (int i = k + 1 + lane; i < n; i += 32) {
            const float lik = a[i * n + k];
            for (int j = k + 1; j <= i; ++j) a[i * n + j] -= lik * a[j * n + k];
        }
    }
    __syncwarp();
    for (int t = lane; t < n * n; t += 32)
        if (t % n > t / n) a[t] = 0.f;
    __syncwarp();
    return ok;
}

// Linv = L^-1 for lower-triangular L (forward substitution, one column per lane).
__device__ inline void warp_lower_inverse(const float* L, float* Linv, int n)
{
    for (int c = lane_id(); c < n; c += 32) {
        for (int i = 0; i < c; ++i) Linv[i * n + c] = 0.f;
        for (int i = c; i < n; ++i) {
            float x = (i == c) ? 1.f : 0.f;
            for (int k = c; k < i; ++k) x -= L[i * n + k] * Linv[k * n + c];
            Linv[i * n + c] = x / L[i * n + i];
        }
    }
    __syncwarp();
}

// out = Linv^T Linv (the inverse of L L^T); bitwise symmetric.
__device__ inline void warp_gram_lower(const float* Linv, float* out, int n)
{
    for (int t = lane_id(); t < n * n; t += 32) {
        const int i = t / n, j = t - (t / n) * n;
        float s = 0.f;
        for (int k = i > j ? i : j; k < n; ++k) s += Linv[k * n + i] * Linv[k * n + j];
        out[t] = s;
    }
    __syncwarp();
}

// dst (cols x rows, row-major) = src^T for a row-major rows x cols src: the
// reads are contiguous, the writes strided (once per element)
__device__ inline void warp_transpose(const float* src, int rows, int cols, float* dst)
{
    for (int t = lane_id(); t < rows * cols; t += 32) {
        const int i = t / cols, j = t - i * cols;
        dst[j * rows + i] = src[t];
    }
    __syncwarp();
}

// C (r x c) = s * op(A) op(B) (+ C when acc).  op(A) is r x kk: A row-major
// r x kk, or kk x r when TA.  op(B) is kk x c: B row-major kk x c, or c x kk
// when TB.  Any of the pointers may be global or shared.
template <bool TA, bool TB>
__device__ inline void warp_gemm(int r, int c, int kk, const float* A, const float* B,
                                 float* C, float s, bool acc)
{
    if (!TB && (c & 3) == 0 &&
        ((reinterpret_cast<uintptr_t>(B) | reinterpret_cast<uintptr_t>(C)) & 15) == 0) {
        // four adjacent columns per lane: one load of A and one 128-bit load of
        // B per four FMAs; every element accumulates in the same order as the
        // one-element loop below, so the results are the same
        const int c4 = c >> 2;
        const float4* B4 = reinterpret_cast<const float4*>(B);
        float4* C4 = reinterpret_cast<float4*>(C);
        for (int t = lane_id(); t < r * c4; t += 32) {
            const int i = t / c4, j4 = t - (t / c4) * c4;
            float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
            for (int l = 0; l < kk; ++l) {
                const float a = TA ? A[l * r + i] : A[i * kk + l];
                const float4 b = B4[l * c4 + j4];
                v.x += a * b.x;
                v.y += a * b.y;
                v.z += a * b.z;
                v.w += a * b.w;
            }
            if (acc) {
                float4 o = C4[t];
                o.x += s * v.x;
                o.y += s * v.y;
                o.z += s * v.z;
                o.w += s * v.w;
                C4[t] = o;
            } else {
                C4[t] = make_float4(s * v.x, s * v.y, s * v.z, s * v.w);
            }
        }
        __syncwarp();
        return;
    }
    for (int t = lane_id(); t < r * c; t += 32) {
        const int i = t / c, j = t - (t / c) * c;
        float v = 0.f;
        for (int l = 0; l < kk; ++l) {
            const float a = TA ? A[l * r + i] : A[i * kk + l];
            const float b = TB ? B[j * kk + l] : B[l * c + j];
            v += a * b;
        }
        C[t] = acc ? C[t] + s * v : s * v;
    }
    __syncwarp();
}

// y (rows) = s * op(M) x (+ y when acc); M row-major rows x cols (cols x rows when T).
template <bool T>
__device__ inline void warp_gemv(int rows, int cols, const float* M, const float* x,
                                 float* y, float s, bool acc)
{
    for (int i = lane_id(); i < rows; i += 32) {
        float v = 0.f;
        for (int l = 0; l < cols; ++l) v += (T ? M[l * rows + i] : M[i * cols + l]) * x[l];
        y[i] = acc ? y[i] + s * v : s * v;
    }
    __syncwarp();
}

// sum_{c in [lo, hi)} M[c * stride] x(c): with NPX > 0 (hi <= NPX) unrolled
// and predicated so that all loads are in flight at once
template <int NPX, typename XFn>
__device__ __forceinline__ float strided_dot(const float* M, int stride, XFn x, int lo, int hi)
{
    float s = 0.f;
    if constexpr (NPX > 0) {
        float mv[NPX], xv[NPX];
#pragma unroll
        for (int c = 0; c < NPX; ++c) {
            const bool in = c >= lo && c < hi;
            mv[c] = in ? M[c * stride] : 0.f;
            xv[c] = in ? x(c) : 0.f;
        }
#pragma unroll
        for (int c = 0; c < NPX; ++c) s = fmaf(mv[c], xv[c], s);
    } else {
        for (int c = lo; c < hi; ++c) s += M[c * stride] * x(c);
    }
    return s;
}

// Recovery after a solve of S_hat lambda_hat = ghat (GATO paper, eq. (4)):
// lambda = L^-T lambda_hat, then dx_k = -Q_k^-1 q_k + Q_k^-1 lambda_k
// + S_{k+1,k}^T lambda_{k+1} and du_k = -R_k^-1 r_k - (B_k R_k^-1)^T
// lambda_{k+1}, with the -Q^-1 q and -R^-1 r parts taken from the rhs set.
// Block-wide (all threads of the block, one solve); lhat(j, a) reads
// lambda_hat; lsm is an N n scratch in shared memory.  NPX > 0 (n <= NPX)
// unrolls the dot products.
template <int NPX = 0, typename LhatFn>
__device__ inline void recover_dz(const Work& w, const Rhs& rhs, float* lambda, float* dX,
                                  float* dU, int sol, LhatFn lhat, float* lsm)
{
    const int N = w.N, n = w.n, m = w.m, Nn = N * n, T = blockDim.x, tid = threadIdx.x;
    const float* gLi = w.Linv + sol * w.sNnn;
    for (int i = tid; i < Nn; i += T) {
        const int j = i / n, a = i - j * n;
        const float* Li = gLi + (size_t)j * n * n;
        const float x = strided_dot<NPX>(Li + a, n, [&](int b) { return lhat(j, b); }, a, n);
        lambda[(size_t)sol * Nn + i] = x;
        lsm[i] = x;
    }
    __syncthreads();
    const float* Qi = w.Qinv + sol * w.sNnn;
    const float* Ob = w.O + sol * w.sKnn;
    const float* av = rhs.avec + sol * w.sNn;
    for (int i = tid; i < Nn; i += T) {
        const int k = i / n, a = i - k * n;
        const float* lk = lsm + k * n;
        float x = av[i];
        x += strided_dot<NPX>(Qi + (size_t)k * n * n + a * n, 1, [&](int b) { return lk[b]; },
                              0, n);
        if (k < N - 1) {
            const float* lk1 = lsm + (k + 1) * n;
            // S_{k+1,k}, column a
            x += strided_dot<NPX>(Ob + (size_t)k * n * n + a, n, [&](int b) { return lk1[b]; },
                                  0, n);
        }
        dX[(size_t)sol * Nn + i] = x;
    }
    const int Km = (N - 1) * m;
    const float* Vb = w.V + sol * w.sKnm;
    const float* bv = rhs.bvec + sol * w.sKm;
    for (int t = tid; t < Km; t += T) {
        const int k = t / m, c = t - k * m;
        const float* lk1 = lsm + (k + 1) * n;
        // column c of B_k R_k^-1
        const float u = strided_dot<NPX>(Vb + (size_t)k * n * m + c, m,
                                         [&](int b) { return lk1[b]; }, 0, n);
        dU[(size_t)sol * Km + t] = bv[t] - u;
    }
}

#endif  // __CUDACC__

}  // namespace gato
