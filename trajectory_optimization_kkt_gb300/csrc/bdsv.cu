// bdsv.cu -- direct solve of the block-tridiagonal Schur system S lambda =
// gamma (the "bdsv" linear solver of the GATO documentation, which measures it
// growing about linearly in the horizon and overtaking PCG from N = 256), in
// two elimination orders:
//
//   cyclic reduction   odd knots are eliminated first, then the odd knots of
//                      the reduced chain, ceil(log2 N) levels; the knots of a
//                      level are independent, so one thread block works on a
//                      whole level at once (one half-warp or warp per knot)
//   chronological      block Cholesky S = L L^T in knot order (the block
//                      Thomas algorithm, the backward pass of a Riccati
//                      recursion): N dependent steps, one warp per solve
//
// Both factor the block-Jacobi-scaled matrix S_hat = L^-1 S L^-T that the PCG
// kernels iterate on (L_j = chol(S_jj)): its diagonal blocks are identities
// and its coupling blocks are Nhat_j = L_j^-1 S_{j,j-1} L_{j-1}^-T, both
// formed with the Schur complement.  The scaled system is the better
// conditioned one, and the first level of cyclic reduction then eliminates
// identity blocks, with nothing to factor.  The solution lambda = L^-T
// lambda_hat and dz follow exactly as after PCG (eq. (4)).
//
// Cyclic reduction of the chain with diagonal blocks D_p and couplings E_p
// (block (p, p-1)): an odd knot p is factored, D_p = C C^T, F = C^-1, and
// keeps X = F E_p, Y = F E_{p+1}^T and g = F gamma_p; an even knot p then has
//     D_p   <- D_p - X_{p+1}^T X_{p+1} - Y_{p-1}^T Y_{p-1}
//     E'_p  =  -Y_{p-1}^T X_{p-1}            (its coupling to knot p - 2)
//     gamma_p <- gamma_p - X_{p+1}^T g_{p+1} - Y_{p-1}^T g_{p-1}
// and after the reduced system is solved, x_p = F^T (g - X x_{p-1} - Y x_{p+1})
// for every odd knot.  Knot 0 is never eliminated: it is the last knot left.
#include "rows16.cuh"

namespace gato {
namespace {

using namespace rows;

struct BdsvArgs {
    Work w;
    Rhs rhs;
    float* lambda;
    float* dX;
    float* dU;
    int32_t* iters;
    uint32_t* status;
    int acc_iters;
    int vec_smem;  // substitution vectors in shared memory (else Bv, Bg)
};

// per-solve block pointers
struct Blocks {
    const float* nh;  // Nhat_j at nh + (j - 1) n^2
    float* bd;
    float* be;
    float* by;
    int n2;
    __device__ Blocks(const Work& w, int sol)
        : nh(w.Nh + sol * w.sKnn),
          bd(w.Bd + sol * w.sNnn),
          be(w.Be + sol * w.sNnn),
          by(w.By + sol * w.sNnn),
          n2(w.n * w.n)
    {
    }
    __device__ const float* Nhat(int j) const { return nh + (size_t)(j - 1) * n2; }
    __device__ float* D(int j) const { return bd + (size_t)j * n2; }
    __device__ float* E(int j) const { return be + (size_t)j * n2; }
    __device__ float* Y(int j) const { return by + (size_t)j * n2; }
};

// number of odd (first) and even (second) multiples of s below N
__host__ __device__ __forceinline__ int odd_multiples(int N, int s)
{
    return s < N ? (N - 1 - s) / (2 * s) + 1 : 0;
}
__host__ __device__ __forceinline__ int even_multiples(int N, int s)
{
    return (N - 1) / (2 * s) + 1;
}

// ===========================================================================
// register kernel for cyclic reduction (n <= 16): half-warp per knot
// ===========================================================================

// row li of block idx (n x n at base + idx n^2) when valid, else the zero
// row or, with ident, the identity row
template <int P>
__device__ __forceinline__ void load_blk(float (&a)[NP], const float* base, int idx, bool valid,
                                         int n, int li, bool ident)
{
    if (valid) {
        load_row<P>(a, base + (size_t)idx * n * n, n, n, li, ident);
    } else {
#pragma unroll
        for (int j = 0; j < P; ++j) a[j] = (ident && j == li) ? 1.f : 0.f;
    }
}

template <int P>
__device__ __forceinline__ void set_row(float (&c)[NP], int li, float diag)
{
#pragma unroll
    for (int j = 0; j < P; ++j) c[j] = (j == li) ? diag : 0.f;
}

// One solve per block of 256 threads (16 half-warps).  Every phase runs in
// rounds that all half-warps take part in (uniform control flow for the
// shuffles); a half-warp without a knot in a round computes on zero or
// identity rows and stores nothing.  Rows are PN >= n columns wide (the
// columns past n are padding zeros).
template <int PN>
__global__ void __launch_bounds__(256) k_bdsv_cr_factor_rows(Work w, uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int sol = blockIdx.x;
    const int n = w.n, N = w.N;
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int half = (warp << 1) | (lane >> 4), li = lane & 15;
    const int H = blockDim.x >> 4;
    if (!gb_smem((size_t)H * 2 * NP * NP * sizeof(float), w.status, sol)) return;  // uniform
    float* S0 = sm + (size_t)half * 2 * NP * NP;
    float* S1 = S0 + NP * NP;
    const Blocks b(w, sol);
    bool ok = true;

    // level s = 1: odd knots are eliminated with identity diagonal blocks
    // (F = I, X_j = Nhat_j, Y_j = Nhat_{j+1}^T); every even knot i gets
    //   D_i = I - Nhat_i Nhat_i^T - Nhat_{i+1}^T Nhat_{i+1},  E_i = -Nhat_i Nhat_{i-1}
    {
        const int cnt = even_multiples(N, 1);
        for (int r0 = 0; r0 < cnt; r0 += H) {
            const int k = r0 + half;
            const bool act = k < cnt;
            const int i = act ? 2 * k : 0;
            float a[NP], c[NP], t[NP], tl[NP];
            // all of the round's loads first: one memory latency per round
            load_blk<PN>(a, b.nh, i - 1, act && i >= 1, n, li, false);
            load_blk<PN>(t, b.nh, i, act && i + 1 < N, n, li, false);
            load_blk<PN>(tl, b.nh, i - 2, act && i >= 2, n, li, false);
            __syncwarp();
            publish<PN>(a, S0, li);
            publish<PN>(t, S1, li);
            __syncwarp();
            set_row<PN>(c, li, 1.f);
            rows_mul_bt<PN, PN>(a, S0, n, c, -1.f);
            rows_atb<PN, PN>(S1, S1, n, li, c, -1.f);
            if (act) store_row<PN>(c, b.D(i), n, n, li);
            __syncwarp();
            publish<PN>(tl, S1, li);
            __syncwarp();
            rows_mul<PN, PN>(a, S1, n, c, -1.f);
            if (act && i >= 2) store_row<PN>(c, b.E(i), n, n, li);
        }
    }
    __syncthreads();

    for (int s = 2; s < N; s <<= 1) {
        // eliminate the odd multiples j of s
        const int cnt = odd_multiples(N, s);
        for (int r0 = 0; r0 < cnt; r0 += H) {
            const int k = r0 + half;
            const bool act = k < cnt;
            const int j = act ? (2 * k + 1) * s : 0;
            const bool right = act && j + s < N;
            float d[NP], x[NP], e[NP], er[NP], c[NP];
            load_blk<PN>(d, b.bd, j, act, n, li, true);
            load_blk<PN>(e, b.be, j, act, n, li, false);
            load_blk<PN>(er, b.be, j + s, right, n, li, false);
            __syncwarp();
            publish<PN>(e, S1, li);
            const bool okj = rows_cholesky<PN>(d, li, n, S0);
            ok = ok && (okj || !act);
            rows_lower_inverse<PN>(d, x, li, n, S0);  // x: row li of F (ends with __syncwarp)
            if (act) store_row<PN>(x, b.D(j), n, n, li);
            rows_mul<PN, PN>(x, S1, n, c, 1.f);  // X = F E_j
            if (act) store_row<PN>(c, b.E(j), n, n, li);
            __syncwarp();
            publish<PN>(er, S1, li);
            __syncwarp();
            set_row<PN>(c, li, 0.f);
            rows_mul_bt<PN, PN>(x, S1, n, c, 1.f);  // Y = F E_{j+s}^T
            if (right) store_row<PN>(c, b.Y(j), n, n, li);
        }
        __syncthreads();
        // update the even multiples i of s
        const int cnt2 = even_multiples(N, s);
        for (int r0 = 0; r0 < cnt2; r0 += H) {
            const int k = r0 + half;
            const bool act = k < cnt2;
            const int i = act ? 2 * k * s : 0;
            const bool far = act && i >= 2 * s;
            float c[NP], y[NP], t[NP], tl[NP];
            load_blk<PN>(c, b.bd, i, act, n, li, false);
            load_blk<PN>(y, b.by, i - s, act && i >= s, n, li, false);
            load_blk<PN>(t, b.be, i + s, act && i + s < N, n, li, false);
            load_blk<PN>(tl, b.be, i - s, far, n, li, false);
            __syncwarp();
            publish<PN>(y, S0, li);
            publish<PN>(t, S1, li);
            __syncwarp();
            rows_atb<PN, PN>(S0, S0, n, li, c, -1.f);  // - Y_{i-s}^T Y_{i-s}
            rows_atb<PN, PN>(S1, S1, n, li, c, -1.f);  // - X_{i+s}^T X_{i+s}
            if (act) store_row<PN>(c, b.D(i), n, n, li);
            __syncwarp();
            publish<PN>(tl, S1, li);
            __syncwarp();
            set_row<PN>(c, li, 0.f);
            rows_atb<PN, PN>(S0, S1, n, li, c, -1.f);  // E' = -Y_{i-s}^T X_{i-s}
            if (far) store_row<PN>(c, b.E(i), n, n, li);
        }
        __syncthreads();
    }

    // knot 0, the last one left: F_0 of its reduced block (warp 0 only)
    if (warp == 0) {
        const bool act = half == 0;
        float d[NP], x[NP];
        load_blk<PN>(d, b.bd, 0, act, n, li, true);
        const bool ok0 = rows_cholesky<PN>(d, li, n, S0);
        ok = ok && (ok0 || !act);
        rows_lower_inverse<PN>(d, x, li, n, S0);
        if (act) store_row<PN>(x, b.D(0), n, n, li);
    }
    if (!ok && li == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

// ===========================================================================
// shared-memory kernels (any n <= 64): one warp per knot, three n x n
// scratch matrices per warp
// ===========================================================================

__device__ __forceinline__ void warp_identity(float* T, int n)
{
    for (int t = lane_id(); t < n * n; t += 32) T[t] = (t / n == t % n) ? 1.f : 0.f;
    __syncwarp();
}

__device__ __forceinline__ void warp_load(float* dst, const float* src, int n2)
{
    warp_copy(dst, src, n2);
    __syncwarp();
}

__device__ __forceinline__ void warp_store(float* dst, const float* src, int n2)
{
    __syncwarp();
    warp_copy(dst, src, n2);
    __syncwarp();
}

__global__ void __launch_bounds__(256) k_bdsv_cr_factor_smem(Work w, uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int sol = blockIdx.x;
    const int n = w.n, N = w.N, n2 = n * n;
    const int warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (!gb_smem((size_t)nw * 3 * n2 * sizeof(float), w.status, sol)) return;  // uniform
    float* Ta = sm + (size_t)warp * 3 * n2;
    float* Tb = Ta + n2;
    float* Tc = Tb + n2;
    const Blocks b(w, sol);
    bool ok = true;

    // level s = 1 (see the register kernel)
    for (int k = warp; k < even_multiples(N, 1); k += nw) {
        const int i = 2 * k;
        warp_identity(Tc, n);
        if (i >= 1) {
            warp_load(Ta, b.Nhat(i), n2);
            warp_gemm<false, true>(n, n, n, Ta, Ta, Tc, -1.f, true);
        }
        if (i + 1 < N) {
            warp_load(Tb, b.Nhat(i + 1), n2);
            warp_gemm<true, false>(n, n, n, Tb, Tb, Tc, -1.f, true);
        }
        warp_store(b.D(i), Tc, n2);
        if (i >= 2) {
            warp_load(Tb, b.Nhat(i - 1), n2);
            warp_gemm<false, false>(n, n, n, Ta, Tb, Tc, -1.f, false);
            warp_store(b.E(i), Tc, n2);
        }
    }
    __syncthreads();

    for (int s = 2; s < N; s <<= 1) {
        for (int k = warp; k < odd_multiples(N, s); k += nw) {
            const int j = (2 * k + 1) * s;
            warp_load(Ta, b.D(j), n2);
            ok = warp_cholesky(Ta, n) && ok;
            warp_lower_inverse(Ta, Tb, n);  // F
            warp_store(b.D(j), Tb, n2);
            warp_load(Ta, b.E(j), n2);
            warp_gemm<false, false>(n, n, n, Tb, Ta, Tc, 1.f, false);  // X = F E_j
            warp_store(b.E(j), Tc, n2);
            if (j + s < N) {
                warp_load(Ta, b.E(j + s), n2);
                warp_gemm<false, true>(n, n, n, Tb, Ta, Tc, 1.f, false);  // Y = F E_{j+s}^T
                warp_store(b.Y(j), Tc, n2);
            }
        }
        __syncthreads();
        for (int k = warp; k < even_multiples(N, s); k += nw) {
            const int i = 2 * k * s;
            warp_load(Tc, b.D(i), n2);
            if (i >= s) {
                warp_load(Ta, b.Y(i - s), n2);
                warp_gemm<true, false>(n, n, n, Ta, Ta, Tc, -1.f, true);
            }
            if (i + s < N) {
                warp_load(Tb, b.E(i + s), n2);
                warp_gemm<true, false>(n, n, n, Tb, Tb, Tc, -1.f, true);
            }
            warp_store(b.D(i), Tc, n2);
            if (i >= 2 * s) {
                warp_load(Tb, b.E(i - s), n2);
                warp_gemm<true, false>(n, n, n, Ta, Tb, Tc, -1.f, false);
                warp_store(b.E(i), Tc, n2);
            }
        }
        __syncthreads();
    }

    if (warp == 0) {
        warp_load(Ta, b.D(0), n2);
        ok = warp_cholesky(Ta, n) && ok;
        warp_lower_inverse(Ta, Tb, n);
        warp_store(b.D(0), Tb, n2);
    }
    if (!ok && lane_id() == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

// Chronological block Cholesky of S_hat: C_0 = I, and for j >= 1
//   W_j = Nhat_j F_{j-1}^T,  C_j C_j^T = I - W_j W_j^T,  F_j = C_j^-1.
// One warp per solve (the steps depend on each other); F_j -> Bd, W_j -> Be.
__global__ void __launch_bounds__(128) k_bdsv_chrono_factor(Work w, uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int warp = threadIdx.x >> 5;
    const int sol = blockIdx.x * (blockDim.x >> 5) + warp;
    if (sol >= w.M) return;  // whole warps leave together
    const int n = w.n, N = w.N, n2 = n * n;
    if (!gb_smem((size_t)(warp + 1) * 3 * n2 * sizeof(float), w.status, sol)) return;  // warp
    float* Ta = sm + (size_t)warp * 3 * n2;
    float* Tf = Ta + n2;  // F_{j-1}, then F_j
    float* Tw = Tf + n2;
    const Blocks b(w, sol);
    bool ok = true;
    warp_identity(Tf, n);
    warp_store(b.D(0), Tf, n2);
    for (int j = 1; j < N; ++j) {
        warp_load(Ta, b.Nhat(j), n2);
        warp_gemm<false, true>(n, n, n, Ta, Tf, Tw, 1.f, false);  // W_j
        warp_store(b.E(j), Tw, n2);
        warp_identity(Ta, n);
        warp_gemm<false, true>(n, n, n, Tw, Tw, Ta, -1.f, true);  // I - W W^T
        ok = warp_cholesky(Ta, n) && ok;
        warp_lower_inverse(Ta, Tf, n);
        warp_store(b.D(j), Tf, n2);
    }
    if (!ok && lane_id() == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

// ===========================================================================
// substitution and recovery (one block per solve)
// ===========================================================================

// sum_b M[a][b] x[b] (T = false) or sum_b M[b][a] x[b] (T = true); Lower
// skips the zero half of a lower-triangular M (T = false: b <= a; T = true:
// b >= a).  With NPX > 0 (n <= NPX) the loop is unrolled and predicated, so
// that all of a row's loads are in flight at once.
template <bool T, bool Lower, int NPX>
__device__ __forceinline__ float rowdot(const float* M, const float* x, int a, int n)
{
    if constexpr (NPX > 0) {
        float mv[NPX], xv[NPX];
#pragma unroll
        for (int c = 0; c < NPX; ++c) {
            const bool in = c < n && (!Lower || (T ? c >= a : c <= a));
            mv[c] = in ? (T ? M[c * n + a] : M[a * n + c]) : 0.f;
            xv[c] = in ? x[c] : 0.f;
        }
        float s = 0.f;
#pragma unroll
        for (int c = 0; c < NPX; ++c) s = fmaf(mv[c], xv[c], s);
        return s;
    } else {
        float s = 0.f;
        const int lo = (Lower && T) ? a : 0;
        const int hi = (Lower && !T) ? a + 1 : n;
        for (int c = lo; c < hi; ++c) s += (T ? M[c * n + a] : M[a * n + c]) * x[c];
        return s;
    }
}

__device__ __forceinline__ void finish_solve(const BdsvArgs& g, int sol, const float* v)
{
    const int Nn = g.w.N * g.w.n;
    bool bad = false;
    for (int i = threadIdx.x; i < Nn; i += blockDim.x) bad = bad || !isfinite(v[i]);
    bad = __syncthreads_or(bad);
    if (threadIdx.x == 0) {
        if (!g.acc_iters) g.iters[sol] = 0;
        if (bad) atomicOr(g.status + sol, GATO_STATUS_NONFINITE);
    }
}

// The vectors: v holds ghat, then the reduced right-hand sides, then
// lambda_hat; G holds g = F gamma of the eliminated knots.
template <int NPX>
__global__ void __launch_bounds__(256) k_bdsv_cr_solve(BdsvArgs g)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int sol = blockIdx.x;
    const int n = w.n, N = w.N, Nn = N * n, T = blockDim.x, tid = threadIdx.x;
    if (g.vec_smem && !gb_smem(2 * (size_t)Nn * sizeof(float), w.status, sol)) return;  // uniform
    float* v = g.vec_smem ? sm : w.Bv + sol * w.sNn;
    float* G = g.vec_smem ? sm + Nn : w.Bg + sol * w.sNn;
    const Blocks b(w, sol);
    const float* gh = g.rhs.ghat + sol * w.sNn;
    for (int i = tid; i < Nn; i += T) v[i] = gh[i];
    __syncthreads();

    // forward, level 1: v_i -= Nhat_i v_{i-1} + Nhat_{i+1}^T v_{i+1} (even i;
    // the odd entries read here are not changed in this phase)
    for (int t = tid; t < even_multiples(N, 1) * n; t += T) {
        const int i = 2 * (t / n), a = t % n;
        float x = v[i * n + a];
        if (i >= 1) x -= rowdot<false, false, NPX>(b.Nhat(i), v + (i - 1) * n, a, n);
        if (i + 1 < N) x -= rowdot<true, false, NPX>(b.Nhat(i + 1), v + (i + 1) * n, a, n);
        v[i * n + a] = x;
    }
    __syncthreads();
    int smax = 1;
    for (int s = 2; s < N; s <<= 1) {
        smax = s;
        for (int t = tid; t < odd_multiples(N, s) * n; t += T) {
            const int j = (2 * (t / n) + 1) * s, a = t % n;
            G[j * n + a] = rowdot<false, true, NPX>(b.D(j), v + j * n, a, n);  // F_j v_j
        }
        __syncthreads();
        for (int t = tid; t < even_multiples(N, s) * n; t += T) {
            const int i = 2 * (t / n) * s, a = t % n;
            float x = v[i * n + a];
            if (i >= s) x -= rowdot<true, false, NPX>(b.Y(i - s), G + (i - s) * n, a, n);
            if (i + s < N) x -= rowdot<true, false, NPX>(b.E(i + s), G + (i + s) * n, a, n);
            v[i * n + a] = x;
        }
        __syncthreads();
    }
    // knot 0: v_0 = F_0^T F_0 v_0
    for (int a = tid; a < n; a += T) G[a] = rowdot<false, true, NPX>(b.D(0), v, a, n);
    __syncthreads();
    for (int a = tid; a < n; a += T) v[a] = rowdot<true, true, NPX>(b.D(0), G, a, n);
    __syncthreads();
    // backward: x_j = F_j^T (g_j - X_j x_{j-s} - Y_j x_{j+s}) for the odd
    // multiples j of s, from the last level down
    for (int s = smax; s >= 2; s >>= 1) {
        for (int t = tid; t < odd_multiples(N, s) * n; t += T) {
            const int j = (2 * (t / n) + 1) * s, a = t % n;
            float x = G[j * n + a] - rowdot<false, false, NPX>(b.E(j), v + (j - s) * n, a, n);
            if (j + s < N) x -= rowdot<false, false, NPX>(b.Y(j), v + (j + s) * n, a, n);
            G[j * n + a] = x;
        }
        __syncthreads();
        for (int t = tid; t < odd_multiples(N, s) * n; t += T) {
            const int j = (2 * (t / n) + 1) * s, a = t % n;
            v[j * n + a] = rowdot<true, true, NPX>(b.D(j), G + j * n, a, n);
        }
        __syncthreads();
    }
    // level 1: x_j = ghat_j - Nhat_j x_{j-1} - Nhat_{j+1}^T x_{j+1} (odd j;
    // v_j still holds ghat_j)
    for (int t = tid; t < odd_multiples(N, 1) * n; t += T) {
        const int j = 2 * (t / n) + 1, a = t % n;
        float x = v[j * n + a] - rowdot<false, false, NPX>(b.Nhat(j), v + (j - 1) * n, a, n);
        if (j + 1 < N) x -= rowdot<true, false, NPX>(b.Nhat(j + 1), v + (j + 1) * n, a, n);
        v[j * n + a] = x;
    }
    __syncthreads();
    finish_solve(g, sol, v);
    recover_dz<NPX>(w, g.rhs, g.lambda, g.dX, g.dU, sol,
                    [&](int j, int c) { return v[j * n + c]; }, G);
}

// Chronological substitution: y_j = F_j (ghat_j - W_j y_{j-1}), then
// x_j = F_j^T (y_j - W_{j+1}^T x_{j+1}); warp 0 walks the chain, the whole
// block recovers dz.
template <int NPX>
__global__ void __launch_bounds__(128) k_bdsv_chrono_solve(BdsvArgs g)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int sol = blockIdx.x;
    const int n = w.n, N = w.N, Nn = N * n;
    if (g.vec_smem && !gb_smem(2 * (size_t)Nn * sizeof(float), w.status, sol)) return;  // uniform
    float* v = g.vec_smem ? sm : w.Bv + sol * w.sNn;
    float* G = g.vec_smem ? sm + Nn : w.Bg + sol * w.sNn;
    const Blocks b(w, sol);
    const float* gh = g.rhs.ghat + sol * w.sNn;
    if (threadIdx.x < 32) {
        const int lane = lane_id();
        for (int j = 0; j < N; ++j) {
            for (int a = lane; a < n; a += 32) {
                float x = gh[j * n + a];
                if (j > 0) x -= rowdot<false, false, NPX>(b.E(j), v + (j - 1) * n, a, n);
                G[j * n + a] = x;
            }
            __syncwarp();
            for (int a = lane; a < n; a += 32)
                v[j * n + a] = rowdot<false, true, NPX>(b.D(j), G + j * n, a, n);
            __syncwarp();
        }
        for (int j = N - 1; j >= 0; --j) {
            for (int a = lane; a < n; a += 32) {
                float x = v[j * n + a];
                if (j + 1 < N) x -= rowdot<true, false, NPX>(b.E(j + 1), v + (j + 1) * n, a, n);
                G[j * n + a] = x;
            }
            __syncwarp();
            for (int a = lane; a < n; a += 32)
                v[j * n + a] = rowdot<true, true, NPX>(b.D(j), G + j * n, a, n);
            __syncwarp();
        }
    }
    __syncthreads();
    finish_solve(g, sol, v);
    recover_dz<NPX>(w, g.rhs, g.lambda, g.dX, g.dU, sol,
                    [&](int j, int c) { return v[j * n + c]; }, G);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

template <typename K, typename... Args>
cudaError_t launch(K kernel, unsigned grid, int T, size_t smem, cudaStream_t st, Args... args)
{
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kernel<<<grid, T, smem, st>>>(args...);
    return cudaGetLastError();
}

constexpr int kRowsThreads = 256;     // 16 half-warps
constexpr int kSmemWarps = 8;         // warps of the shared-memory factor kernel
constexpr int kChronoWarps = 4;       // solves per block of the chronological factor
constexpr int kSolveThreads = 256;
constexpr int kChronoSolveThreads = 128;

}  // namespace

cudaError_t launch_bdsv_factor(gato_handle* h, int order, uint32_t* status, cudaStream_t st)
{
    const Work& w = h->w;
    const size_t limit = (size_t)h->smem_optin;
    const size_t per_warp = 3 * (size_t)w.n * w.n * sizeof(float);
    if (order == GATO_LINSYS_BDSV_CHRONO) {
        const size_t smem = kChronoWarps * per_warp;
        if (smem > limit) return cudaErrorInvalidConfiguration;
        const unsigned grid = (unsigned)((w.M + kChronoWarps - 1) / kChronoWarps);
        return launch(k_bdsv_chrono_factor, grid, 32 * kChronoWarps, smem, st, w, status);
    }
    if (h->bdsv_kernel != GATO_BDSV_KERNEL_SHARED && w.n <= NP) {
        const size_t smem = (kRowsThreads / 16) * 2 * NP * NP * sizeof(float);  // 32 KB
        auto kernel = w.n <= 8    ? k_bdsv_cr_factor_rows<8>
                      : w.n <= 12 ? k_bdsv_cr_factor_rows<12>
                      : w.n <= 14 ? k_bdsv_cr_factor_rows<14>
                                  : k_bdsv_cr_factor_rows<16>;
        return launch(kernel, (unsigned)w.M, kRowsThreads, smem, st, w, status);
    }
    int nw = (int)(limit / per_warp);
    if (nw > kSmemWarps) nw = kSmemWarps;
    if (nw < 1) return cudaErrorInvalidConfiguration;
    return launch(k_bdsv_cr_factor_smem, (unsigned)w.M, 32 * nw, nw * per_warp, st, w, status);
}

cudaError_t launch_bdsv_solve(gato_handle* h, int order, int set, float* lambda, float* dX,
                              float* dU, int32_t* iters, int acc_iters, uint32_t* status,
                              cudaStream_t st)
{
    const Work& w = h->w;
    BdsvArgs a;
    a.w = w;
    a.rhs = w.rhs[set];
    a.lambda = lambda;
    a.dX = dX;
    a.dU = dU;
    a.iters = iters;
    a.status = status;
    a.acc_iters = acc_iters;
    const size_t vec = 2 * (size_t)w.N * w.n * sizeof(float);
    a.vec_smem = vec <= (size_t)h->smem_optin;
    // recovery needs its N n scratch in shared memory only when the vectors
    // are there too; otherwise it uses Bg in global memory
    const size_t smem = a.vec_smem ? vec : 0;
    // the row products unrolled to the state width (8, 12, 14 or 16), or
    // looped beyond 16
    const unsigned M = (unsigned)w.M;
    if (order == GATO_LINSYS_BDSV_CHRONO) {
        auto kernel = w.n <= 8    ? k_bdsv_chrono_solve<8>
                      : w.n <= 12 ? k_bdsv_chrono_solve<12>
                      : w.n <= 14 ? k_bdsv_chrono_solve<14>
                      : w.n <= NP ? k_bdsv_chrono_solve<NP>
                      : w.n <= 24 ? k_bdsv_chrono_solve<24>
                      : w.n <= 36 ? k_bdsv_chrono_solve<36>
                                  : k_bdsv_chrono_solve<0>;
        return launch(kernel, M, kChronoSolveThreads, smem, st, a);
    }
    // beyond 16 the rows are unrolled to 24 and 36 as well (the row products
    // of a substitution level are dependent global loads: unrolled, a row's
    // loads are all in flight at once; looped, they follow one another)
    auto kernel = w.n <= 8    ? k_bdsv_cr_solve<8>
                  : w.n <= 12 ? k_bdsv_cr_solve<12>
                  : w.n <= 14 ? k_bdsv_cr_solve<14>
                  : w.n <= NP ? k_bdsv_cr_solve<NP>
                  : w.n <= 24 ? k_bdsv_cr_solve<24>
                  : w.n <= 36 ? k_bdsv_cr_solve<36>
                              : k_bdsv_cr_solve<0>;
    return launch(kernel, M, kSolveThreads, smem, st, a);
}

}  // namespace gato
