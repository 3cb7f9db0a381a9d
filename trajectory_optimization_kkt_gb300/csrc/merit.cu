// merit.cu -- parallel line search with the L1 merit function and the step
// update (GATO paper, Sec. III-A: the merit is evaluated over all N*M*A
// knot-candidates with block-based parallelism per timestep, then a
// block-level reduction per line-search iterate; the best iterate gives the
// update Z <- Z + alpha* dZ).
//
// k_merit         one block per (knot, candidate, solve): the knot's cost and
//                 constraint violation at x = alpha dx, u = alpha du.  Each row
//                 is summed by one thread in index order and the knot total by
//                 thread 0 in index order, so results do not depend on the
//                 block size.
// k_merit_reduce  one block per solve, one warp per candidate: knot sums in a
//                 fixed order (lane-strided partials, xor butterfly), merit =
//                 cost + mu * violation, argmin with ties to the lower index,
//                 acceptance against alpha = 0.
// k_merit_fused   (default) one block per solve: each warp streams a fixed
//                 set of knots once, lanes over the rows of a knot, and keeps
//                 the candidate-independent pieces c2 = x^T Q x + u^T R u,
//                 c1 = q^T x + r^T u and w = A x + B u - x_next of the full
//                 step; every candidate then costs 1/2 alpha^2 c2 + alpha c1
//                 + mu sum |e + alpha w| (+ mu sum |alpha x_0 - s0|), the
//                 factored form of the same merit.  Knot sums in a fixed
//                 order; the block reduction, argmin and acceptance follow.
// k_merit_knots   (the fused merit for n, m <= 16) the same factored merit
//                 with one half-warp per knot (lane = row) and sixteen knots
//                 per block, grid (ceil(N/16), M): every knot's loads are in
//                 flight at once.  Each block writes its sums (c1, c2 and the
//                 candidates' violations) to scratch; the block of a solve
//                 that arrives last (fence + counter) adds the blocks in
//                 block order, so the merits do not depend on scheduling, and
//                 takes the argmin.
// k_apply_step    X += alpha* dX, U += alpha* dU.
#include "gato_internal.cuh"

namespace gato {
namespace {

struct MeritArgs {
    Work w;
    const float *Q, *R, *q, *r, *A, *B, *e, *s0, *dX, *dU;
    int A1;      // candidates including alpha = 0
    float beta;
    int sol0;    // k_merit: first solve of the launch (grids of at most 65535 solves)
};

// alpha of candidate c: 0 for c = 0, beta^-(c-1) otherwise (repeated division)
__device__ __forceinline__ float candidate_alpha(int c, float beta)
{
    if (c == 0) return 0.f;
    float a = 1.f;
    for (int t = 1; t < c; ++t) a = a / beta;
    return a;
}

__global__ void k_merit(MeritArgs g)
{
    extern __shared__ __align__(16) float sm[];
    const int N = g.w.N, n = g.w.n, m = g.w.m;
    const int k = blockIdx.x, c = blockIdx.y, sol = g.sol0 + (int)blockIdx.z;
    const int T = blockDim.x, tid = threadIdx.x;
    const bool has_u = k < N - 1;
    const size_t K = (size_t)(N - 1);
    const float alpha = candidate_alpha(c, g.beta);

    float* x = sm;           // n
    float* xn = x + n;       // n
    float* u = xn + n;       // m
    float* tc = u + m;       // n + m  cost terms
    float* tv = tc + n + m;  // 2n     violation terms (dynamics rows, then x_0 rows)
    if (!gb_smem((size_t)(5 * n + 2 * m) * sizeof(float), g.w.status, sol) ||
        !gb_ok((long long)c * N + k, (long long)g.w.sK2, g.w.status, sol))
        return;  // block-uniform

    const float* dXs = g.dX + (size_t)sol * N * n;
    for (int i = tid; i < n; i += T) {
        x[i] = alpha * dXs[(size_t)k * n + i];
        xn[i] = has_u ? alpha * dXs[(size_t)(k + 1) * n + i] : 0.f;
    }
    for (int i = tid; i < m; i += T)
        u[i] = has_u ? alpha * g.dU[((size_t)sol * K + k) * m + i] : 0.f;
    __syncthreads();

    const float* Qk = g.Q + ((size_t)sol * N + k) * n * n;
    const float* qk = g.q + ((size_t)sol * N + k) * n;
    const float* Ak = g.A + ((size_t)sol * K + k) * n * n;
    const float* Bk = g.B + ((size_t)sol * K + k) * n * m;
    const float* ek = g.e + ((size_t)sol * K + k) * n;
    const float* s0 = g.s0 + (size_t)sol * n;
    for (int a = tid; a < n; a += T) {
        float qx = 0.f;
        for (int b = 0; b < n; ++b) qx += Qk[a * n + b] * x[b];
        tc[a] = 0.5f * x[a] * qx + qk[a] * x[a];
        float vd = 0.f;
        if (has_u) {
            float s = ek[a] - xn[a];
            for (int b = 0; b < n; ++b) s += Ak[a * n + b] * x[b];
            for (int b = 0; b < m; ++b) s += Bk[a * m + b] * u[b];
            vd = fabsf(s);
        }
        tv[a] = vd;
        tv[n + a] = (k == 0) ? fabsf(x[a] - s0[a]) : 0.f;
    }
    for (int cc = tid; cc < m; cc += T) {
        float t = 0.f;
        if (has_u) {
            const float* Rk = g.R + ((size_t)sol * K + k) * m * m;
            const float* rk = g.r + ((size_t)sol * K + k) * m;
            float ru = 0.f;
            for (int b = 0; b < m; ++b) ru += Rk[cc * m + b] * u[b];
            t = 0.5f * u[cc] * ru + rk[cc] * u[cc];
        }
        tc[n + cc] = t;
    }
    __syncthreads();
    if (tid == 0) {
        float sc = 0.f, sv = 0.f;
        for (int i = 0; i < n + m; ++i) sc += tc[i];
        for (int i = 0; i < 2 * n; ++i) sv += tv[i];
        g.w.mpart[(size_t)sol * g.w.sK2 + (size_t)c * N + k] = make_float2(sc, sv);
    }
}

__global__ void k_merit_reduce(Work w, int A1, float mu, float* merit, int32_t* best,
                               uint32_t* status)
{
    __shared__ float smer[32];
    const int sol = blockIdx.x, c = threadIdx.x >> 5, lane = lane_id();
    const int N = w.N;
    const float2* part = w.mpart + (size_t)sol * w.sK2 + (size_t)c * N;
    float sc = 0.f, sv = 0.f;
    for (int k = lane; k < N; k += 32) {
        const float2 t = part[k];
        sc += t.x;
        sv += t.y;
    }
    sc = warp_sum(sc);
    sv = warp_sum(sv);
    const float mv = sc + mu * sv;
    if (lane == 0) {
        smer[c] = mv;
        merit[(size_t)sol * A1 + c] = mv;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int b = 0;
        bool finite = isfinite(smer[0]);
        for (int i = 1; i < A1; ++i) {
            finite = finite && isfinite(smer[i]);
            if (smer[i] < smer[1 + b]) b = i - 1;
        }
        uint32_t st = 0;
        if (!finite) st |= GATO_STATUS_NONFINITE;
        if (!(smer[1 + b] < smer[0])) {
            b = -1;
            st |= GATO_STATUS_LINESEARCH_FAILED;
        }
        best[sol] = b;
        if (st) atomicOr(status + sol, st);
    }
}

constexpr int kMaxA1 = GATO_MAX_ALPHA + 1;

template <int NPX>
__global__ void __launch_bounds__(512) k_merit_fused(MeritArgs g, float mu, float* merit,
                                                     int32_t* best, uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int N = g.w.N, n = g.w.n, m = g.w.m, A1 = g.A1;
    const int sol = blockIdx.x, lane = lane_id(), warp = threadIdx.x >> 5;
    const int nw = blockDim.x >> 5;
    const size_t K = (size_t)(N - 1);
    float* xv = sm + (size_t)warp * (2 * n + m);  // x_k, x_{k+1}, u_k of this warp's knot
    float* xn = xv + n;
    float* uv = xn + n;
    float* part = sm + (size_t)nw * (2 * n + m);  // [nw][A1 + 2] warp partials
    if (!gb_smem(((size_t)nw * (2 * n + m + A1 + 2) + A1) * sizeof(float), g.w.status, sol))
        return;  // block-uniform

    float alpha[kMaxA1];
#pragma unroll
    for (int i = 0; i < kMaxA1; ++i) alpha[i] = i < A1 ? candidate_alpha(i, g.beta) : 0.f;
    float viol[kMaxA1];
#pragma unroll
    for (int i = 0; i < kMaxA1; ++i) viol[i] = 0.f;
    float c1 = 0.f, c2 = 0.f;

    const float* dXs = g.dX + (size_t)sol * N * n;
    const float* s0 = g.s0 + (size_t)sol * n;
    for (int k = warp; k < N; k += nw) {
        const bool has_u = k < N - 1;
        for (int i = lane; i < n; i += 32) {
            xv[i] = dXs[(size_t)k * n + i];
            xn[i] = has_u ? dXs[(size_t)(k + 1) * n + i] : 0.f;
        }
        for (int i = lane; i < m; i += 32)
            uv[i] = has_u ? g.dU[((size_t)sol * K + k) * m + i] : 0.f;
        __syncwarp();
        const float* Qk = g.Q + ((size_t)sol * N + k) * n * n;
        const float* qk = g.q + ((size_t)sol * N + k) * n;
        auto xs = [&](int b) { return xv[b]; };
        auto us = [&](int b) { return uv[b]; };
        for (int a = lane; a < n; a += 32) {
            const float qx = strided_dot<NPX>(Qk + a * n, 1, xs, 0, n);
            c2 += xv[a] * qx;
            c1 += qk[a] * xv[a];
            if (has_u) {
                const float* Ak = g.A + ((size_t)sol * K + k) * n * n;
                const float* Bk = g.B + ((size_t)sol * K + k) * n * m;
                const float ea = g.e[((size_t)sol * K + k) * n + a];
                float wa = -xn[a];
                wa += strided_dot<NPX>(Ak + a * n, 1, xs, 0, n);
                wa += strided_dot<NPX>(Bk + a * m, 1, us, 0, m);
#pragma unroll
                for (int i = 0; i < kMaxA1; ++i)
                    if (i < A1) viol[i] += fabsf(ea + alpha[i] * wa);
            }
            if (k == 0) {
#pragma unroll
                for (int i = 0; i < kMaxA1; ++i)
                    if (i < A1) viol[i] += fabsf(alpha[i] * xv[a] - s0[a]);
            }
        }
        if (has_u) {
            const float* Rk = g.R + ((size_t)sol * K + k) * m * m;
            const float* rk = g.r + ((size_t)sol * K + k) * m;
            for (int c = lane; c < m; c += 32) {
                const float ru = strided_dot<NPX>(Rk + c * m, 1, us, 0, m);
                c2 += uv[c] * ru;
                c1 += rk[c] * uv[c];
            }
        }
        __syncwarp();
    }
    // warp sums, then block sums in warp order
    c1 = warp_sum(c1);
    c2 = warp_sum(c2);
#pragma unroll
    for (int i = 0; i < kMaxA1; ++i)
        if (i < A1) viol[i] = warp_sum(viol[i]);
    if (lane == 0) {
        float* pw = part + (size_t)warp * (A1 + 2);
        pw[0] = c1;
        pw[1] = c2;
#pragma unroll
        for (int i = 0; i < kMaxA1; ++i)
            if (i < A1) pw[2 + i] = viol[i];
    }
    __syncthreads();
    float* smer = part + (size_t)nw * (A1 + 2);  // [A1]
    if (threadIdx.x < A1) {
        const int i = threadIdx.x;
        float C1 = 0.f, C2 = 0.f, V = 0.f;
        for (int q = 0; q < nw; ++q) {
            const float* pw = part + (size_t)q * (A1 + 2);
            C1 += pw[0];
            C2 += pw[1];
            V += pw[2 + i];
        }
        const float a = candidate_alpha(i, g.beta);
        const float mv = 0.5f * a * a * C2 + a * C1 + mu * V;
        smer[i] = mv;
        merit[(size_t)sol * A1 + i] = mv;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        int b = 0;
        bool finite = isfinite(smer[0]);
        for (int i = 1; i < A1; ++i) {
            finite = finite && isfinite(smer[i]);
            if (smer[i] < smer[1 + b]) b = i - 1;
        }
        uint32_t st = 0;
        if (!finite) st |= GATO_STATUS_NONFINITE;
        if (!(smer[1 + b] < smer[0])) {
            b = -1;
            st |= GATO_STATUS_LINESEARCH_FAILED;
        }
        best[sol] = b;
        if (st) atomicOr(status + sol, st);
    }
}

__global__ void k_apply_step(Work w, float beta, const int32_t* best, const float* dX,
                             const float* dU, float* X, float* U)
{
    const int sol = blockIdx.x;
    const int b = best[sol];
    if (b < 0) return;
    float alpha = 1.f;
    for (int t = 0; t < b; ++t) alpha = alpha / beta;
    const size_t Nn = (size_t)w.N * w.n, Km = (size_t)(w.N - 1) * w.m;
    for (size_t i = threadIdx.x; i < Nn; i += blockDim.x)
        X[sol * Nn + i] += alpha * dX[sol * Nn + i];
    for (size_t i = threadIdx.x; i < Km; i += blockDim.x)
        U[sol * Km + i] += alpha * dU[sol * Km + i];
}

// sum over the owned row li < rows of row li of M (rows x cols, row-major)
// times v (cols <= 16, from shared memory); loads issued together
__device__ __forceinline__ float row_dot16(const float* M, int cols, int li, const float* v)
{
    const float* row = M + li * cols;
    float t = 0.f;
#pragma unroll
    for (int b = 0; b < 16; ++b)
        if (b < cols) t = fmaf(row[b], v[b], t);
    return t;
}

template <int NA>
__global__ void __launch_bounds__(256) k_merit_knots(MeritArgs g, float mu, float* merit,
                                                     int32_t* best, uint32_t* status,
                                                     int* count)
{
    __shared__ __align__(16) float xs[16][48];  // per half-warp: x_k, u_k, x_{k+1}
    __shared__ float wpart[8][NA + 2];          // per warp: c1, c2, violations
    __shared__ float smer[NA];
    __shared__ int s_last;
    const int N = g.w.N, n = g.w.n, m = g.w.m, A1 = g.A1;
    const int tid = threadIdx.x, lane = lane_id(), warp = tid >> 5;
    const int h = tid >> 4, li = tid & 15;
    const int sol = blockIdx.y, nb = gridDim.x;
    const int k = blockIdx.x * 16 + h;
    const bool act = k < N;
    const bool has_u = act && k < N - 1;
    const size_t K = (size_t)(N - 1);

    float* xv = xs[h];
    float* uv = xv + 16;
    const float* dXs = g.dX + (size_t)sol * N * n;
    xv[li] = act && li < n ? dXs[(size_t)k * n + li] : 0.f;
    uv[li] = has_u && li < m ? g.dU[((size_t)sol * K + k) * m + li] : 0.f;
    const float xnext = has_u && li < n ? dXs[(size_t)(k + 1) * n + li] : 0.f;
    __syncwarp();

    float alpha[NA];
#pragma unroll
    for (int i = 0; i < NA; ++i) alpha[i] = i < A1 ? candidate_alpha(i, g.beta) : 0.f;
    float viol[NA];
#pragma unroll
    for (int i = 0; i < NA; ++i) viol[i] = 0.f;
    float c1 = 0.f, c2 = 0.f;
    if (act && li < n) {
        const float xa = xv[li];
        const float qx = row_dot16(g.Q + ((size_t)sol * N + k) * n * n, n, li, xv);
        c2 = xa * qx;
        c1 = g.q[((size_t)sol * N + k) * n + li] * xa;
        if (has_u) {
            float wa = row_dot16(g.A + ((size_t)sol * K + k) * n * n, n, li, xv);
            wa += row_dot16(g.B + ((size_t)sol * K + k) * n * m, m, li, uv);
            wa -= xnext;
            const float ea = g.e[((size_t)sol * K + k) * n + li];
#pragma unroll
            for (int i = 0; i < NA; ++i)
                if (i < A1) viol[i] = fabsf(ea + alpha[i] * wa);
        }
        if (k == 0) {
            const float s0a = g.s0[(size_t)sol * n + li];
#pragma unroll
            for (int i = 0; i < NA; ++i)
                if (i < A1) viol[i] += fabsf(alpha[i] * xa - s0a);
        }
    }
    if (has_u && li < m) {
        const float ua = uv[li];
        const float ru = row_dot16(g.R + ((size_t)sol * K + k) * m * m, m, li, uv);
        c2 = fmaf(ua, ru, c2);
        c1 = fmaf(g.r[((size_t)sol * K + k) * m + li], ua, c1);
    }
    // warp sums (two knots), then the block's sums in warp order
    c1 = warp_sum(c1);
    c2 = warp_sum(c2);
#pragma unroll
    for (int i = 0; i < NA; ++i)
        if (i < A1) viol[i] = warp_sum(viol[i]);
    if (lane == 0) {
        wpart[warp][0] = c1;
        wpart[warp][1] = c2;
#pragma unroll
        for (int i = 0; i < NA; ++i)
            if (i < A1) wpart[warp][2 + i] = viol[i];
    }
    __syncthreads();
    float* part = reinterpret_cast<float*>(g.w.mpart) + (size_t)sol * 2 * g.w.sK2;
    // the block's A1 + 2 sums, in the solve's 2 sK2 floats of scratch
    if (tid < A1 + 2 &&
        gb_ok((long long)blockIdx.x * (A1 + 2) + tid, 2 * (long long)g.w.sK2, g.w.status, sol)) {
        float t = 0.f;
        for (int q = 0; q < 8; ++q) t += wpart[q][tid];
        part[(size_t)blockIdx.x * (A1 + 2) + tid] = t;
    }
    // the last block of the solve to arrive adds all blocks in block order
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(count + sol, 1) == nb - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    if (tid < A1) {
        float C1 = 0.f, C2 = 0.f, V = 0.f;
        for (int b = 0; b < nb; ++b) {
            const float* pb = part + (size_t)b * (A1 + 2);
            C1 += __ldcg(pb);
            C2 += __ldcg(pb + 1);
            V += __ldcg(pb + 2 + tid);
        }
        const float a = candidate_alpha(tid, g.beta);
        const float mv = 0.5f * a * a * C2 + a * C1 + mu * V;
        smer[tid] = mv;
        merit[(size_t)sol * A1 + tid] = mv;
    }
    __syncthreads();
    if (tid == 0) {
        int b = 0;
        bool finite = isfinite(smer[0]);
        for (int i = 1; i < A1; ++i) {
            finite = finite && isfinite(smer[i]);
            if (smer[i] < smer[1 + b]) b = i - 1;
        }
        uint32_t st = 0;
        if (!finite) st |= GATO_STATUS_NONFINITE;
        if (!(smer[1 + b] < smer[0])) {
            b = -1;
            st |= GATO_STATUS_LINESEARCH_FAILED;
        }
        best[sol] = b;
        if (st) atomicOr(status + sol, st);
    }
}

}  // namespace

cudaError_t launch_merit(gato_handle* h, const gato_params* p, const float* Q,
                         const float* R, const float* q, const float* r, const float* A,
                         const float* B, const float* e, const float* s0, const float* dX,
                         const float* dU, float* merit, int32_t* best, uint32_t* status,
                         cudaStream_t st)
{
    const Work& w = h->w;
    MeritArgs a;
    a.w = w;
    a.Q = Q; a.R = R; a.q = q; a.r = r; a.A = A; a.B = B; a.e = e; a.s0 = s0;
    a.dX = dX; a.dU = dU;
    a.A1 = p->n_alpha + 1;
    a.beta = p->beta;
    a.sol0 = 0;
    if (p->merit_kernel == GATO_MERIT_FUSED && w.n <= 16 && w.m <= 16 && w.M <= 65535) {
        cudaError_t e = cudaMemsetAsync(w.mcount, 0, sizeof(int) * (size_t)w.M, st);
        if (e != cudaSuccess) return e;
        const dim3 grid((unsigned)((w.N + 15) / 16), (unsigned)w.M);
        if (a.A1 <= 9)
            k_merit_knots<9><<<grid, 256, 0, st>>>(a, p->mu, merit, best, status, w.mcount);
        else
            k_merit_knots<kMaxA1><<<grid, 256, 0, st>>>(a, p->mu, merit, best, status, w.mcount);
        return cudaGetLastError();
    }
    if (p->merit_kernel == GATO_MERIT_FUSED) {
        int warps = (w.N + 3) / 4;  // about four knots per warp
        if (warps > 16) warps = 16;
        if (warps < 1) warps = 1;
        const size_t smem =
            ((size_t)warps * (2 * w.n + w.m) + (size_t)warps * (a.A1 + 2) + a.A1) * sizeof(float);
        k_merit_fused<0><<<w.M, 32 * warps, smem, st>>>(a, p->mu, merit, best, status);
        return cudaGetLastError();
    }
    const size_t smem = (size_t)(5 * w.n + 2 * w.m) * sizeof(float);
    // the grid's z extent is limited to 65535: launch the solves in slices
    for (int s0 = 0; s0 < w.M; s0 += 65535) {
        a.sol0 = s0;
        const int cnt = w.M - s0 < 65535 ? w.M - s0 : 65535;
        dim3 grid(w.N, a.A1, cnt);
        k_merit<<<grid, p->merit_threads, smem, st>>>(a);
        cudaError_t e2 = cudaGetLastError();
        if (e2 != cudaSuccess) return e2;
    }
    k_merit_reduce<<<w.M, 32 * a.A1, 0, st>>>(w, a.A1, p->mu, merit, best, status);
    return cudaGetLastError();
}

cudaError_t launch_apply_step(gato_handle* h, const gato_params* p, const int32_t* best,
                              const float* dX, const float* dU, float* X, float* U,
                              cudaStream_t st)
{
    k_apply_step<<<h->w.M, 256, 0, st>>>(h->w, p->beta, best, dX, dU, X, U);
    return cudaGetLastError();
}

}  // namespace gato
