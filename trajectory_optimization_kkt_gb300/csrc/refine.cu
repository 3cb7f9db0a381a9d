// refine.cu -- mixed-precision iterative refinement of the KKT solution.
//
// Not on the GATO pages: fp32 cannot hold S to the accuracy some workloads
// need (with Q_k's diagonal scaled over four decades, rounding S alone moves
// dz by a few 1e-4).  Refinement forms the residual of the full KKT system
// (GATO paper, Sec. II eq. (2)) in extended precision from the caller's data
// and solves the correction with the same S and Phi^-1 (classical iterative
// refinement; the mixed-precision form as analysed by Carson & Higham, SIAM
// J. Sci. Comput. 40(2), 2018).  The residual's sums of products use the
// compensated dot product of Ogita, Rump & Oishi ("Accurate sum and dot
// product", SIAM J. Sci. Comput. 26(6), 2005, Algorithm Dot2): error-free
// products by FMA and error-free sums (Knuth's TwoSum) accumulate the
// rounding errors separately, so the result is as accurate as if computed
// in twice the working precision and then rounded -- at fp32 speed, which on
// this GPU is far above its fp64 rate.  The correction system is the KKT
// system with
//   q'_k = Q_k dx_k + q_k - lambda_k + A_k^T lambda_{k+1}
//   r'_k = R_k du_k + r_k + B_k^T lambda_{k+1}
//   s0'  = s0 - dx_0
//   e'_k = e_k + A_k dx_k + B_k du_k - dx_{k+1}
// in place of (q, r, s0, e); its solution is added to (dz, lambda).
#include "gato_internal.cuh"

namespace gato {
namespace {

// Compensated accumulator: s + c carries the sum to about u^2 relative error.
// The intrinsics keep the compiler from contracting or reassociating the
// error-free transformations.
struct Acc2 {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float v)
    {
        const float t = __fadd_rn(s, v);
        const float z = __fsub_rn(t, s);
        c = __fadd_rn(c, __fadd_rn(__fsub_rn(s, __fsub_rn(t, z)), __fsub_rn(v, z)));
        s = t;
    }
    __device__ __forceinline__ void add_prod(float x, float y)
    {
        const float p = __fmul_rn(x, y);
        const float pe = __fmaf_rn(x, y, -p);  // x*y = p + pe exactly
        add(p);
        c = __fadd_rn(c, pe);
    }
    __device__ __forceinline__ float value() const { return __fadd_rn(s, c); }
};

// one warp per knot, lanes over rows, compensated sums; the correction's data
// (q2, r2, e2, s02) is written densely, like the caller's q, r, e, s0
__global__ void k_kkt_residual(Work w, const float* __restrict__ Q, const float* __restrict__ R,
                               const float* __restrict__ q, const float* __restrict__ r,
                               const float* __restrict__ A, const float* __restrict__ B,
                               const float* __restrict__ e, const float* __restrict__ s0,
                               const float* __restrict__ dX, const float* __restrict__ dU,
                               const float* __restrict__ lam)
{
    const int n = w.n, m = w.m, N = w.N;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5, lane = lane_id();
    const long g = (long)blockIdx.x * wpb + warp;
    if (g >= (long)w.M * N) return;
    const int sol = (int)(g / N), k = (int)(g % N);
    const size_t K = (size_t)(N - 1);
    const float* x = dX + ((size_t)sol * N + k) * n;
    const float* l = lam + ((size_t)sol * N + k) * n;
    const float* Qk = Q + ((size_t)sol * N + k) * n * n;
    for (int a = lane; a < n; a += 32) {
        Acc2 acc;
        acc.add(q[((size_t)sol * N + k) * n + a]);
        acc.add(-l[a]);
        for (int b = 0; b < n; ++b) acc.add_prod(Qk[a * n + b], x[b]);
        if (k < N - 1) {
            const float* Ak = A + ((size_t)sol * K + k) * n * n;
            for (int b = 0; b < n; ++b) acc.add_prod(Ak[b * n + a], l[n + b]);
        }
        w.q2[((size_t)sol * N + k) * n + a] = acc.value();
    }
    if (k == 0)
        for (int a = lane; a < n; a += 32) {
            Acc2 acc;
            acc.add(s0[(size_t)sol * n + a]);
            acc.add(-x[a]);
            w.s02[(size_t)sol * n + a] = acc.value();
        }
    if (k < N - 1) {
        const float* u = dU + ((size_t)sol * K + k) * m;
        const float* Rk = R + ((size_t)sol * K + k) * m * m;
        const float* Bk = B + ((size_t)sol * K + k) * n * m;
        const float* Ak = A + ((size_t)sol * K + k) * n * n;
        for (int c = lane; c < m; c += 32) {
            Acc2 acc;
            acc.add(r[((size_t)sol * K + k) * m + c]);
            for (int b = 0; b < m; ++b) acc.add_prod(Rk[c * m + b], u[b]);
            for (int b = 0; b < n; ++b) acc.add_prod(Bk[b * m + c], l[n + b]);
            w.r2[((size_t)sol * K + k) * m + c] = acc.value();
        }
        for (int a = lane; a < n; a += 32) {
            Acc2 acc;
            acc.add(e[((size_t)sol * K + k) * n + a]);
            acc.add(-x[n + a]);
            for (int b = 0; b < n; ++b) acc.add_prod(Ak[a * n + b], x[b]);
            for (int b = 0; b < m; ++b) acc.add_prod(Bk[a * m + b], u[b]);
            w.e2[((size_t)sol * K + k) * n + a] = acc.value();
        }
    }
}

__global__ void k_accumulate(Work w, float* lam, float* dX, float* dU)
{
    const int sol = blockIdx.x;
    const size_t Nn = (size_t)w.N * w.n, Km = (size_t)(w.N - 1) * w.m;
    // the correction was written densely ([M][N][n], [M][N-1][m]) by the PCG kernel
    for (size_t i = threadIdx.x; i < Nn; i += blockDim.x) {
        lam[sol * Nn + i] += w.dlam[sol * Nn + i];
        dX[sol * Nn + i] += w.ddX[sol * Nn + i];
    }
    for (size_t i = threadIdx.x; i < Km; i += blockDim.x) dU[sol * Km + i] += w.ddU[sol * Km + i];
}

}  // namespace

cudaError_t launch_kkt_residual(gato_handle* h, const float* Q, const float* R,
                                const float* q, const float* r, const float* A,
                                const float* B, const float* e, const float* s0,
                                const float* dX, const float* dU, const float* lambda,
                                cudaStream_t st)
{
    const Work& w = h->w;
    const long knots = (long)w.M * w.N;
    const int wpb = 4;
    k_kkt_residual<<<(unsigned)((knots + wpb - 1) / wpb), 32 * wpb, 0, st>>>(
        w, Q, R, q, r, A, B, e, s0, dX, dU, lambda);
    return cudaGetLastError();
}

cudaError_t launch_accumulate(gato_handle* h, float* lambda, float* dX, float* dU,
                              int32_t* iters, cudaStream_t st)
{
    (void)iters;
    k_accumulate<<<h->w.M, 256, 0, st>>>(h->w, lambda, dX, dU);
    return cudaGetLastError();
}

}  // namespace gato
