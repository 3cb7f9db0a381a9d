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
// k_apply_step    X += alpha* dX, U += alpha* dU.
#include "gato_internal.cuh"

namespace gato {
namespace {

struct MeritArgs {
    Work w;
    const float *Q, *R, *q, *r, *A, *B, *e, *s0, *dX, *dU;
    int A1;      // candidates including alpha = 0
    float beta;
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
    const int k = blockIdx.x, c = blockIdx.y, sol = blockIdx.z;
    const int T = blockDim.x, tid = threadIdx.x;
    const bool has_u = k < N - 1;
    const size_t K = (size_t)(N - 1);
    const float alpha = candidate_alpha(c, g.beta);

    float* x = sm;           // n
    float* xn = x + n;       // n
    float* u = xn + n;       // m
    float* tc = u + m;       // n + m  cost terms
    float* tv = tc + n + m;  // 2n     violation terms (dynamics rows, then x_0 rows)

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
    const size_t smem = (size_t)(5 * w.n + 2 * w.m) * sizeof(float);
    dim3 grid(w.N, a.A1, w.M);
    k_merit<<<grid, p->merit_threads, smem, st>>>(a);
    cudaError_t e2 = cudaGetLastError();
    if (e2 != cudaSuccess) return e2;
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
