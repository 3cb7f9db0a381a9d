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
    // line search partial sums
    float2* mpart; // [(A+1)][N] (cost, violation) per knot and candidate
    int* queue;    // work counters of the persistent kernels (not per solve)
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
    int force_smem_form;    // GATO_FORM_SHARED selected by gato_set_form_kernel
    cudaEvent_t ev[5];  // start, after form, after PCG, after refinement, after merit
    int ev_used[5];
    gato_stats last;
};

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

// ---------------------------------------------------------------------------
// device helpers
// ---------------------------------------------------------------------------
#ifdef __CUDACC__

__device__ __forceinline__ int lane_id() { return threadIdx.x & 31; }

__device__ __forceinline__ float warp_sum(float v)
{
    // xor butterfly: every lane ends with the same, order-fixed sum
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// dst[0..count) = s * src[0..count), lanes over elements
__device__ __forceinline__ void warp_copy(float* dst, const float* src, int count,
                                          float s = 1.f)
{
    for (int i = lane_id(); i < count; i += 32) dst[i] = s * src[i];
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

// C (r x c) = s * op(A) op(B) (+ C when acc).  op(A) is r x kk: A row-major
// r x kk, or kk x r when TA.  op(B) is kk x c: B row-major kk x c, or c x kk
// when TB.  Any of the pointers may be global or shared.
template <bool TA, bool TB>
__device__ inline void warp_gemm(int r, int c, int kk, const float* A, const float* B,
                                 float* C, float s, bool acc)
{
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

#endif  // __CUDACC__

}  // namespace gato
