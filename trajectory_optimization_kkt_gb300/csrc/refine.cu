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

// acc += sum_{b < cnt} M[b * stride] x[b]; with NPX > 0 (cnt <= NPX) all the
// loads are issued first (unrolled, predicated), then the compensated chain
template <int NPX>
__device__ __forceinline__ void dot_acc(Acc2& acc, const float* M, int stride, const float* x,
                                        int cnt)
{
    if constexpr (NPX > 0) {
        float mv[NPX], xv[NPX];
#pragma unroll
        for (int b = 0; b < NPX; ++b) {
            mv[b] = b < cnt ? M[b * stride] : 0.f;
            xv[b] = b < cnt ? x[b] : 0.f;
        }
#pragma unroll
        for (int b = 0; b < NPX; ++b)
            if (b < cnt) acc.add_prod(mv[b], xv[b]);
    } else {
        for (int b = 0; b < cnt; ++b) acc.add_prod(M[b * stride], x[b]);
    }
}

// one warp per knot, lanes over rows, compensated sums; the correction's data
// (q2, r2, e2, s02) is written densely, like the caller's q, r, e, s0
template <int NPX>
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
        dot_acc<NPX>(acc, Qk + a * n, 1, x, n);
        if (k < N - 1) {
            const float* Ak = A + ((size_t)sol * K + k) * n * n;
            dot_acc<NPX>(acc, Ak + a, n, l + n, n);
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
            dot_acc<NPX>(acc, Rk + c * m, 1, u, m);
            dot_acc<NPX>(acc, Bk + c, m, l + n, n);
            w.r2[((size_t)sol * K + k) * m + c] = acc.value();
        }
        for (int a = lane; a < n; a += 32) {
            Acc2 acc;
            acc.add(e[((size_t)sol * K + k) * n + a]);
            acc.add(-x[n + a]);
            dot_acc<NPX>(acc, Ak + a * n, 1, x, n);
            dot_acc<NPX>(acc, Bk + a * m, 1, u, m);
            w.e2[((size_t)sol * K + k) * n + a] = acc.value();
        }
    }
}

// n, m <= 16: the same residual with one half-warp per knot (lane = row) and
// sixteen knots per block; the knot's step and multiplier vectors are staged
// in shared memory once, and each row's compensated chain adds its terms in
// the order k_kkt_residual does (bit-identical results).
__global__ void __launch_bounds__(256) k_kkt_residual_half(
    Work w, const float* __restrict__ Q, const float* __restrict__ R, const float* __restrict__ q,
    const float* __restrict__ r, const float* __restrict__ A, const float* __restrict__ B,
    const float* __restrict__ e, const float* __restrict__ s0, const float* __restrict__ dX,
    const float* __restrict__ dU, const float* __restrict__ lam)
{
    __shared__ __align__(16) float vs[16][80];  // x_k, x_{k+1}, u_k, lambda_k, lambda_{k+1}
    const int n = w.n, m = w.m, N = w.N;
    const int h = threadIdx.x >> 4, li = threadIdx.x & 15;
    const long g = (long)blockIdx.x * 16 + h;
    const bool act = g < (long)w.M * N;  // no early return: the warp syncs below
    const long gi = act ? g : 0;
    const int sol = (int)(gi / N), k = (int)(gi % N);
    const bool has_u = act && k < N - 1;
    const size_t K = (size_t)(N - 1);
    float* x = vs[h];
    float* xn = x + 16;
    float* u = x + 32;
    float* l = x + 48;
    float* l1 = x + 64;
    const float* dXk = dX + ((size_t)sol * N + k) * n;
    const float* lk = lam + ((size_t)sol * N + k) * n;
    x[li] = act && li < n ? dXk[li] : 0.f;
    xn[li] = has_u && li < n ? dXk[n + li] : 0.f;
    l[li] = act && li < n ? lk[li] : 0.f;
    l1[li] = has_u && li < n ? lk[n + li] : 0.f;
    u[li] = has_u && li < m ? dU[((size_t)sol * K + k) * m + li] : 0.f;
    __syncwarp();
    if (act && li < n) {
        const float* Qk = Q + ((size_t)sol * N + k) * n * n;
        Acc2 aq;
        aq.add(q[((size_t)sol * N + k) * n + li]);
        aq.add(-l[li]);
        if (has_u) {
            const float* Ak = A + ((size_t)sol * K + k) * n * n;
            const float* Bk = B + ((size_t)sol * K + k) * n * m;
            Acc2 ae;
            ae.add(e[((size_t)sol * K + k) * n + li]);
            ae.add(-xn[li]);
            for (int b = 0; b < n; ++b) {  // the two rows' chains side by side
                aq.add_prod(Qk[li * n + b], x[b]);
                ae.add_prod(Ak[li * n + b], x[b]);
            }
            for (int b = 0; b < n; ++b) aq.add_prod(Ak[b * n + li], l1[b]);
            for (int c = 0; c < m; ++c) ae.add_prod(Bk[li * m + c], u[c]);
            w.e2[((size_t)sol * K + k) * n + li] = ae.value();
        } else {
            for (int b = 0; b < n; ++b) aq.add_prod(Qk[li * n + b], x[b]);
        }
        w.q2[((size_t)sol * N + k) * n + li] = aq.value();
        if (k == 0) {
            Acc2 a0;
            a0.add(s0[(size_t)sol * n + li]);
            a0.add(-x[li]);
            w.s02[(size_t)sol * n + li] = a0.value();
        }
    }
    if (has_u && li < m) {
        const float* Rk = R + ((size_t)sol * K + k) * m * m;
        const float* Bk = B + ((size_t)sol * K + k) * n * m;
        Acc2 ar;
        ar.add(r[((size_t)sol * K + k) * m + li]);
        for (int c = 0; c < m; ++c) ar.add_prod(Rk[li * m + c], u[c]);
        for (int b = 0; b < n; ++b) ar.add_prod(Bk[b * m + li], l1[b]);
        w.r2[((size_t)sol * K + k) * m + li] = ar.value();
    }
}

// y += d over a dense array (the correction was written densely, [M][N][n]
// and [M][N-1][m], by the linear solve), grid-stride
__global__ void k_accumulate(float* lam, const float* dlam, float* dX, const float* ddX,
                             size_t total_x, float* dU, const float* ddU, size_t total_u)
{
    const size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_x; i += stride) {
        lam[i] += dlam[i];
        dX[i] += ddX[i];
    }
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total_u; i += stride)
        dU[i] += ddU[i];
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
    if (w.n <= 16 && w.m <= 16) {
        if (knots <= 0) return cudaSuccess;
        k_kkt_residual_half<<<(unsigned)((knots + 15) / 16), 256, 0, st>>>(w, Q, R, q, r, A, B, e,
                                                                           s0, dX, dU, lambda);
        return cudaGetLastError();
    }
    const int wpb = 4;
    // the compensated chains are the latency here, not the loads: the
    // runtime-bounded loops (fewer registers, more warps) are the faster form
    const unsigned blocks = (unsigned)((knots + wpb - 1) / wpb);
    k_kkt_residual<0><<<blocks, 32 * wpb, 0, st>>>(w, Q, R, q, r, A, B, e, s0, dX, dU, lambda);
    return cudaGetLastError();
}

cudaError_t launch_accumulate(gato_handle* h, float* lambda, float* dX, float* dU,
                              int32_t* iters, cudaStream_t st)
{
    (void)iters;
    const Work& w = h->w;
    const size_t tx = (size_t)w.M * w.N * w.n, tu = (size_t)w.M * (w.N - 1) * w.m;
    size_t blocks = (tx + 255) / 256;
    const size_t cap = (size_t)h->num_sms * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    k_accumulate<<<(unsigned)blocks, 256, 0, st>>>(lambda, w.dlam, dX, w.ddX, tx, dU, w.ddU, tu);
    return cudaGetLastError();
}

}  // namespace gato
