// sqp.cu -- the two kernels an SQP iteration on a linear model adds around
// the KKT solve (GATO paper Sec. II: "Step 1: form the quadratic program via
// a second-order Taylor expansion ... along a nominal trajectory", "Step 3:
// apply the update step ... through the use of a merit function and a line
// search"; Sec. IV-C: rho added to the diagonal of Q_k and adjusted after
// each iteration from the status of the line search).
//
// For the linear model x_{k+1} = A_k x_k + B_k u_k + c_k the expansion is
// exact: the subproblem keeps Q, R, A, B and takes the gradients and defects
// at the nominal trajectory.  The line search then ranks
//   M(X + a dX, U + a dU) - J(X, U)
// (the merit kernel's values on the expansion's data), and the merit history
// adds J(X, U) back.
#include "gato_internal.cuh"

namespace gato {
namespace {

// One warp per knot, lanes over rows: Qd = Q + rho I, the gradients
// Q x + q and R u + r, the defects A x + B u + c - x_next and xs - x_0, and
// the knot's cost 1/2 x^T Q x + q^T x (+ 1/2 u^T R u + r^T u).
__global__ void k_sqp_linearize(Work w, const float* __restrict__ Q, const float* __restrict__ R,
                                const float* __restrict__ q, const float* __restrict__ r,
                                const float* __restrict__ A, const float* __restrict__ B,
                                const float* __restrict__ c, const float* __restrict__ xs,
                                const float* __restrict__ X, const float* __restrict__ U,
                                const float* __restrict__ rho)
{
    const int n = w.n, m = w.m, N = w.N;
    const int lane = lane_id(), wpb = blockDim.x >> 5;
    const long g = (long)blockIdx.x * wpb + (threadIdx.x >> 5);
    if (g >= (long)w.M * N) return;  // whole warps
    const int sol = (int)(g / N), k = (int)(g % N);
    const size_t kn = (size_t)sol * N + k;
    const float* x = X + kn * n;
    const float* Qk = Q + kn * n * n;
    float* Qdk = w.Qd + kn * n * n;
    const float rh = rho[sol];
    for (int t = lane; t < n * n; t += 32) Qdk[t] = Qk[t] + (t % (n + 1) == 0 ? rh : 0.f);
    float jp = 0.f;
    for (int a = lane; a < n; a += 32) {
        float s = 0.f;
        for (int b = 0; b < n; ++b) s = fmaf(Qk[a * n + b], x[b], s);
        const float qa = q[kn * n + a];
        w.qt[kn * n + a] = s + qa;
        jp = fmaf(x[a], fmaf(0.5f, s, qa), jp);
    }
    if (k < N - 1) {
        const size_t ku = (size_t)sol * (N - 1) + k;
        const float* u = U + ku * m;
        const float* Rk = R + ku * m * m;
        for (int a = lane; a < m; a += 32) {
            float s = 0.f;
            for (int b = 0; b < m; ++b) s = fmaf(Rk[a * m + b], u[b], s);
            const float ra = r[ku * m + a];
            w.rt[ku * m + a] = s + ra;
            jp = fmaf(u[a], fmaf(0.5f, s, ra), jp);
        }
        const float* Ak = A + ku * n * n;
        const float* Bk = B + ku * n * m;
        const float* xn = x + n;
        for (int a = lane; a < n; a += 32) {
            float s = c[ku * n + a] - xn[a];
            for (int b = 0; b < n; ++b) s = fmaf(Ak[a * n + b], x[b], s);
            for (int b = 0; b < m; ++b) s = fmaf(Bk[a * m + b], u[b], s);
            w.et[ku * n + a] = s;
        }
    }
    if (k == 0) {
        const size_t o = (size_t)sol * n;
        for (int a = lane; a < n; a += 32) w.s0t[o + a] = xs[o + a] - x[a];
    }
    jp = warp_sum(jp);
    if (lane == 0) w.Jk[sol * w.sN + k] = jp;
}

// One block per problem: the step (X, U) += alpha* dz when the line search
// accepted one (alpha_i = beta^-i by repeated division, as the merit kernels
// take it), the merit history, the PCG iteration count, and the damping
// update; then the problem's iteration counter advances.
__global__ void k_sqp_step(Work w, float beta, int A1, int iters, float rho_factor, float rho_min,
                           float rho_max, float* X, float* U, float* rho, float* hist,
                           int32_t* iters_hist)
{
    const int sol = blockIdx.x;
    const int N = w.N, n = w.n, m = w.m, tid = threadIdx.x, T = blockDim.x;
    const int best = w.sbest[sol];
    if (best >= 0) {
        float alpha = 1.f;
        for (int i = 0; i < best; ++i) alpha /= beta;
        const size_t xo = (size_t)sol * N * n, uo = (size_t)sol * (N - 1) * m;
        for (int i = tid; i < N * n; i += T) X[xo + i] = fmaf(alpha, w.sdX[xo + i], X[xo + i]);
        for (int i = tid; i < (N - 1) * m; i += T)
            U[uo + i] = fmaf(alpha, w.sdU[uo + i], U[uo + i]);
    }
    if (tid == 0) {
        float J = 0.f;
        for (int k = 0; k < N; ++k) J += w.Jk[sol * w.sN + k];  // fixed order
        const float* mer = w.smerit + (size_t)sol * A1;
        const int t = w.sqpt[sol];
        if (t < iters) {
            float* hs = hist + (size_t)sol * (iters + 1);
            if (t == 0) hs[0] = J + mer[0];
            hs[t + 1] = J + (best >= 0 ? mer[1 + best] : mer[0]);
            if (iters_hist) iters_hist[(size_t)sol * iters + t] = w.siters[sol];
        }
        const float rh = rho[sol];
        rho[sol] = best >= 0 ? fmaxf(rh / rho_factor, rho_min) : fminf(rh * rho_factor, rho_max);
        w.sqpt[sol] = t + 1;
    }
}

}  // namespace

cudaError_t launch_sqp_linearize(gato_handle* h, const float* Q, const float* R, const float* q,
                                 const float* r, const float* A, const float* B, const float* c,
                                 const float* xs, const float* X, const float* U,
                                 const float* rho, cudaStream_t st)
{
    const Work& w = h->w;
    const int wpb = 8;
    const long knots = (long)w.M * w.N;
    k_sqp_linearize<<<(unsigned)((knots + wpb - 1) / wpb), 32 * wpb, 0, st>>>(
        w, Q, R, q, r, A, B, c, xs, X, U, rho);
    return cudaGetLastError();
}

cudaError_t launch_sqp_step(gato_handle* h, const gato_params* p, const gato_sqp_params* sp,
                            float* X, float* U, float* rho, float* merit_hist,
                            int32_t* iters_hist, cudaStream_t st)
{
    const Work& w = h->w;
    k_sqp_step<<<w.M, 256, 0, st>>>(w, p->beta, p->n_alpha + 1, sp->iters, sp->rho_factor,
                                    sp->rho_min, sp->rho_max, X, U, rho, merit_hist, iters_hist);
    return cudaGetLastError();
}

}  // namespace gato
