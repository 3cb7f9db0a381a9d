// pcg_rows.cu -- batched PCG on S lambda = gamma with the symmetric stair
// preconditioner for larger states (17 <= n <= 64), and recovery of dz (GATO
// paper, Sec. II and eq. (4); Sec. III: one thread block per linear system,
// block-tridiagonal matrix-vector products, block reductions).
//
// The same iteration as the kernels of pcg.cu, in the block-Jacobi-scaled
// variables lambda_hat = L^T lambda, where S_hat = I + Nhat and the stair
// preconditioner is I - Nhat: both products of an iteration are products
// with the block-tridiagonal Nhat (coupling blocks Nhat_j, block (j, j-1)).
//
// k_pcg_rows<NP, R>: thread t owns rows a = q R .. q R + R - 1 of knot j
// (j = t / TPK, q = t % TPK, TPK = ceil(n / R) threads per knot) and keeps
// in registers those rows of the two coupling blocks around its knot: row a
// of Nhat_j (multiplies x_{j-1}) and row a of Nhat_{j+1}^T (column a of
// Nhat_{j+1}, multiplies x_{j+1}).  Its rows of Nhat x are then complete
// in registers: a product reads only the two neighbouring knots' vectors,
// broadcast from shared memory as 128-bit loads, and nothing else is
// exchanged.  NP is n padded to a multiple of 4 (the vectors' knot stride,
// padding slots zero), R keeps the two row tiles within 216 floats.  The
// vectors live in registers with their owners and in shared memory for the
// neighbours; a guard knot of zeros before knot 0 and after knot N-1 stands
// for the missing neighbours.
//
// Stopping rule 0 (||L r_hat|| <= eps ||gamma||) is evaluated only when the
// per-knot lower bound sum_j lambda_min-bound_j ||r_hat_j||^2 no longer rules
// convergence out, as in the kernels of pcg.cu: gated by the previous
// iteration's bound (within 1.25 of the threshold), with a fallback
// evaluation in the same iteration, so the stop is exact.
#include "pcg_common.cuh"

namespace gato {
namespace {

// rows per thread: the two tiles (2 R NP floats) within 216 registers
constexpr int rows_for(int NP) { return 216 / (2 * NP) > 0 ? 216 / (2 * NP) : 1; }

// pushed pair slots per buffer in the cluster kernel: C CTAs of nw warps each
// (C <= 8; nw <= 12 for the blocks max_threads_for allows)
constexpr int kRowsClusterSlots = 128;
// float4s before the tile chunks in the cluster kernel's shared memory: three
// block-sum buffers of 32 and three pushed-pair buffers of kRowsClusterSlots
// float2
constexpr int kRowsClusterHead = 96 + 3 * kRowsClusterSlots / 2;

// threads per block the registers allow with R rows per thread: 64K
// registers over the tiles plus about 56 for the rest, in whole warps; with
// more than one row per thread at most 256 threads, so that no SM
// sub-partition holds more than two warps and a thread may use 255 registers
// (fewer, fuller threads measured faster than more threads with spilled
// tiles)
constexpr int max_threads_raw(int NP, int R) { return (65536 / (2 * R * NP + 56)) / 32 * 32; }
constexpr int max_threads_for(int NP, int R)
{
    return R > 1 ? (max_threads_raw(NP, R) > 256 ? 256 : max_threads_raw(NP, R))
                 : (max_threads_raw(NP, R) > 1024 ? 1024 : max_threads_raw(NP, R));
}

// The registers per thread the launch bound leaves: 64K over the warps of
// the fullest SM sub-partition (a quarter of the block's warps, rounded up),
// in steps of 8.
constexpr int reg_cap_for(int NP, int R)
{
    return (16384 / (((max_threads_for(NP, R) / 32 + 3) / 4) * 32)) / 8 * 8 > 255
               ? 255
               : (16384 / (((max_threads_for(NP, R) / 32 + 3) / 4) * 32)) / 8 * 8;
}

// 128-bit column chunks of the tile rows kept in registers: as many as fit
// beside about 56 other registers; the remaining chunks live in shared
// memory (read once per product, a float4 per thread, conflict-free), so
// that nothing is spilled to local memory
constexpr int reg_chunks_for(int NP, int R)
{
    return (reg_cap_for(NP, R) - 56) / (2 * R * 4) >= NP / 4
               ? NP / 4
               : (reg_cap_for(NP, R) - 56) / (2 * R * 4);
}

template <int NP, int R>
struct RowTiles {
    static constexpr int RC = reg_chunks_for(NP, R);  // chunks in registers
    float lo[R][4 * RC];  // rows of Nhat_j        (times x_{j-1})
    float up[R][4 * RC];  // rows of Nhat_{j+1}^T  (times x_{j+1})
};

// shared-memory chunk s (the chunks from RC on) of tile k (0: lo, 1: up), row
// i of thread tid, in a block of T threads
template <int R>
__device__ __forceinline__ int ts_index(int s, int i, int k, int tid, int T)
{
    return ((s * R + i) * 2 + k) * T + tid;
}

// y[i] = (Nhat x)_a for the thread's rows; X holds the vector with knot j at
// X + (j + 1) NP (guard knots of zeros at both ends)
template <int NP, int R>
__device__ __forceinline__ void rows_matvec(const RowTiles<NP, R>& T, const float4* TS,
                                            const float* X, int j, float (&y)[R])
{
    constexpr int RC = RowTiles<NP, R>::RC;
    const float4* xm = reinterpret_cast<const float4*>(X + j * NP);        // x_{j-1}
    const float4* xp = reinterpret_cast<const float4*>(X + (j + 2) * NP);  // x_{j+1}
    const int tid = threadIdx.x, nt = blockDim.x;
    float sl[R], su[R];
#pragma unroll
    for (int i = 0; i < R; ++i) sl[i] = su[i] = 0.f;
#pragma unroll
    for (int c = 0; c < NP / 4; ++c) {
        const float4 a = xm[c], b = xp[c];
#pragma unroll
        for (int i = 0; i < R; ++i) {
            float4 l, u;
            if (c < RC) {
                l = make_float4(T.lo[i][4 * c], T.lo[i][4 * c + 1], T.lo[i][4 * c + 2],
                                T.lo[i][4 * c + 3]);
                u = make_float4(T.up[i][4 * c], T.up[i][4 * c + 1], T.up[i][4 * c + 2],
                                T.up[i][4 * c + 3]);
            } else {
                l = TS[ts_index<R>(c - RC, i, 0, tid, nt)];
                u = TS[ts_index<R>(c - RC, i, 1, tid, nt)];
            }
            sl[i] = fmaf(l.x, a.x, sl[i]);
            sl[i] = fmaf(l.y, a.y, sl[i]);
            sl[i] = fmaf(l.z, a.z, sl[i]);
            sl[i] = fmaf(l.w, a.w, sl[i]);
            su[i] = fmaf(u.x, b.x, su[i]);
            su[i] = fmaf(u.y, b.y, su[i]);
            su[i] = fmaf(u.z, b.z, su[i]);
            su[i] = fmaf(u.w, b.w, su[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < R; ++i) y[i] = sl[i] + su[i];
}

// sum over the thread's valid rows of (L_j r_hat_j)_a^2, L_j from global memory
// (read only in the iterations where the exact norm is needed)
template <int NP, int R>
__device__ __forceinline__ float rows_lnorm(const float* Lj, const float* X, int j, int a0,
                                            int n, const bool (&valid)[R])
{
    const float* xr = X + (j + 1) * NP;
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (valid[i]) {
            const int a = a0 + i;
            const float* row = Lj + (size_t)a * n;
            float t = 0.f;
            for (int b = 0; b <= a; ++b) t = fmaf(row[b], xr[b], t);
            s = fmaf(t, t, s);
        }
    }
    return s;
}

// the same from the rows of L staged in shared memory (row a of L_j at
// LS + (j n + a) NP, zero above the diagonal and past n): 128-bit products
template <int NP, int R>
__device__ __forceinline__ float rows_lnorm_smem(const float* LS, const float* X, int j, int a0,
                                                 int n, const bool (&valid)[R])
{
    const float4* xr = reinterpret_cast<const float4*>(X + (j + 1) * NP);
    float s = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        if (valid[i]) {
            const float4* row = reinterpret_cast<const float4*>(LS + ((size_t)j * n + a0 + i) * NP);
            float t = 0.f;
#pragma unroll
            for (int c = 0; c < NP / 4; ++c) {
                const float4 l = row[c], x = xr[c];
                t = fmaf(l.x, x.x, t);
                t = fmaf(l.y, x.y, t);
                t = fmaf(l.z, x.z, t);
                t = fmaf(l.w, x.w, t);
            }
            s = fmaf(t, t, s);
        }
    }
    return s;
}

template <int NP, int R>
__device__ __forceinline__ void rows_store(float* X, int j, int a0, const bool (&valid)[R],
                                           const float (&v)[R])
{
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (valid[i]) X[(j + 1) * NP + a0 + i] = v[i];
}

template <int NP, int R>
__global__ void __launch_bounds__(max_threads_for(NP, R)) k_pcg_rows(PcgArgs g)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int N = w.N, n = w.n, T = blockDim.x, tid = threadIdx.x;
    const int sol = blockIdx.x;
    const int TPK = (n + R - 1) / R;
    const int XS = (N + 2) * NP;  // one vector with its guard knots
    const bool rule0 = g.rule == GATO_STOP_RESIDUAL;

    float* XP = sm;                 // p (and lambda_hat at the end)
    float* XR = XP + XS;            // r
    float* lsm = XR + XS;           // recovery scratch, N n
    float4* redA = reinterpret_cast<float4*>(lsm + round4((size_t)N * n));
    float4* redB = redA + 32;
    float4* redC = redA + 64;
    float2* pairA = reinterpret_cast<float2*>(redA + 96);  // post2 / collect2 slots
    float2* pairB = pairA + 16;
    float2* pairC = pairB + 16;
    // the tile chunks past the registers' share, then (rule 0 with l_smem) the
    // rows of L
    constexpr int SC = NP / 4 - RowTiles<NP, R>::RC;
    float4* TS = redA + 120;
    float* LS = reinterpret_cast<float*>(TS + (size_t)SC * R * 2 * T);
    const bool l_staged_sm = g.rule == GATO_STOP_RESIDUAL && g.l_smem;
    if (!gb_smem((size_t)(LS - sm + (l_staged_sm ? (size_t)N * n * NP : 0)) * sizeof(float),
                 w.status, sol)) {
        finish(g, sol, 0, false, false);
        return;  // block-uniform
    }
    for (int i = tid; i < 2 * XS; i += T) sm[i] = 0.f;

    const int j = tid / TPK, q = tid - j * TPK;
    const int a0 = q * R;
    // the thread's rows are stored at knot j's slots (j + 1) NP + a0 .. + R - 1
    // and its products read knots j - 1 .. j + 1 of the guarded vector
    const bool owner = j < N && gb_ok((long long)(j + 2) * NP + NP - 1, XS, w.status, sol) &&
                       gb_ok(a0, n, w.status, sol);
    bool valid[R];
#pragma unroll
    for (int i = 0; i < R; ++i) valid[i] = owner && a0 + i < n;
    const int jj = owner ? j : 0;  // a safe knot for threads past the last one

    // the thread's rows of Nhat_j and Nhat_{j+1}^T (zero where there is no
    // block, no row, or no column)
    RowTiles<NP, R> tile;
    {
        const float* nh = w.Nh + sol * w.sKnn;
        const size_t nn = (size_t)n * n;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int a = a0 + i;
            const bool has_lo = valid[i] && jj >= 1;
            const bool has_up = valid[i] && jj + 1 < N;
            const float* lo = nh + (size_t)(jj >= 1 ? jj - 1 : 0) * nn + (size_t)a * n;
            const float* up = nh + (size_t)jj * nn + a;
#pragma unroll
            for (int b = 0; b < 4 * RowTiles<NP, R>::RC; ++b) {
                tile.lo[i][b] = (has_lo && b < n) ? lo[b] : 0.f;
                tile.up[i][b] = (has_up && b < n) ? up[(size_t)b * n] : 0.f;
            }
#pragma unroll
            for (int sc = 0; sc < SC; ++sc) {
                float vl[4], vu[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int b = 4 * (RowTiles<NP, R>::RC + sc) + e;
                    vl[e] = (has_lo && b < n) ? lo[b] : 0.f;
                    vu[e] = (has_up && b < n) ? up[(size_t)b * n] : 0.f;
                }
                TS[ts_index<R>(sc, i, 0, tid, T)] = make_float4(vl[0], vl[1], vl[2], vl[3]);
                TS[ts_index<R>(sc, i, 1, tid, T)] = make_float4(vu[0], vu[1], vu[2], vu[3]);
            }
        }
    }
    const float dl = owner ? w.dlow[sol * w.sN + jj] : 0.f;
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float* gL = w.L + sol * w.sNnn;
    const float* Lj = gL + (size_t)jj * n * n;
    const bool l_staged = rule0 && g.l_smem;
    if (l_staged) {  // every row padded to NP (the factor's upper part is stored as zeros)
        for (int t = tid; t < N * n * NP; t += T) {
            const int row = t / NP, b = t - row * NP;
            LS[t] = b < n ? gL[(size_t)row * n + b] : 0.f;
        }
    }

    float lam[R], r[R], p[R], y[R];
    // lambda_hat0 = L^T lambda0
#pragma unroll
    for (int i = 0; i < R; ++i) {
        lam[i] = 0.f;
        if (valid[i] && g.lambda0) {
            const int a = a0 + i;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + (size_t)jj * n;
            float x = 0.f;
            for (int b = a; b < n; ++b) x += Lj[(size_t)b * n + a] * l0[b];
            lam[i] = x;
        }
    }
    __syncthreads();  // the zeroed vectors
    rows_store<NP, R>(XP, jj, a0, valid, lam);
    __syncthreads();
    // r_hat = ghat - S_hat lambda_hat, then z = (I - Nhat) r_hat = p
    rows_matvec<NP, R>(tile, TS, XP, jj, y);
#pragma unroll
    for (int i = 0; i < R; ++i)
        r[i] = valid[i] ? ghat[jj * n + a0 + i] - lam[i] - y[i] : 0.f;
    rows_store<NP, R>(XR, jj, a0, valid, r);
    __syncthreads();
    rows_matvec<NP, R>(tile, TS, XR, jj, y);
    float red3[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < R; ++i) {
        p[i] = r[i] - y[i];
        red3[0] = fmaf(r[i], p[i], red3[0]);
        if (valid[i]) {
            const int gi = jj * n + a0 + i;
            if (rule0)
                red3[2] = fmaf(gam[gi], gam[gi], red3[2]);
            else if (g.rule == GATO_STOP_SCALED) {
                red3[1] = fmaf(r[i], r[i], red3[1]);
                red3[2] = fmaf(ghat[gi], ghat[gi], red3[2]);
            }
        }
    }
    if (rule0)
        red3[1] = l_staged ? rows_lnorm_smem<NP, R>(LS, XR, jj, a0, n, valid)
                      : rows_lnorm<NP, R>(Lj, XR, jj, a0, n, valid);
    rows_store<NP, R>(XP, jj, a0, valid, p);
    block_sum<3>(red3, redA);  // also orders the p stores before the first product
    float eta = red3[0];
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : red3[2];
    const float thr = g.eps * g.eps * ref;
    bool done = (g.rule == GATO_STOP_PRECOND ? eta : red3[1]) <= thr;
    bool nonfinite = !isfinite(eta) || !isfinite(red3[1]);
    bool exact_next = false;
    if (rule0) {
        float lb = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) lb = fmaf(dl * r[i], r[i], lb);
        float lv[1] = {lb};
        block_sum<1>(lv, redB);
        exact_next = lv[0] <= 1.25f * thr;
    }
    __syncthreads();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        // v = S_hat p, alpha = eta / p^T v; lambda and r updates
        rows_matvec<NP, R>(tile, TS, XP, jj, y);
        float pvp = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            y[i] += p[i];
            pvp = fmaf(p[i], y[i], pvp);
        }
        post2(pvp, 0.f, pairA);
        __syncthreads();
        const float pv = collect2(pairA).x;
        const float alpha = __fdividef(eta, pv);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            lam[i] = fmaf(alpha, p[i], lam[i]);
            r[i] = fmaf(-alpha, y[i], r[i]);
        }
        rows_store<NP, R>(XR, jj, a0, valid, r);
        __syncthreads();
        // z = (I - Nhat) r, eta' = r^T z; the stopping quantities
        rows_matvec<NP, R>(tile, TS, XR, jj, y);
        float red[3] = {0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < R; ++i) {
            y[i] = r[i] - y[i];
            red[0] = fmaf(r[i], y[i], red[0]);
            red[1] = fmaf(r[i], r[i], red[1]);
        }
        if (rule0) red[1] *= dl;  // the lower bound's share
        const bool exact = exact_next;
        if (exact)
            red[2] = l_staged ? rows_lnorm_smem<NP, R>(LS, XR, jj, a0, n, valid)
                         : rows_lnorm<NP, R>(Lj, XR, jj, a0, n, valid);
        post2(red[0], red[1], pairB);
        if (exact) post2(red[2], 0.f, pairC);
        __syncthreads();
        {
            const float2 sb = collect2(pairB);
            red[0] = sb.x;
            red[1] = sb.y;
            red[2] = exact ? collect2(pairC).x : 0.f;
        }
        const float eta_new = red[0];
        float lsq = red[2];
        bool have_exact = exact;
        if (rule0 && !exact && red[1] * 0.999f <= thr) {
            float lv[1] = {l_staged ? rows_lnorm_smem<NP, R>(LS, XR, jj, a0, n, valid)
                               : rows_lnorm<NP, R>(Lj, XR, jj, a0, n, valid)};
            block_sum<1>(lv, redC);
            lsq = lv[0];
            have_exact = true;
        }
        const float stopq = rule0 ? lsq : (g.rule == GATO_STOP_SCALED ? red[1] : eta_new);
        if (!isfinite(eta_new + pv + stopq + red[1])) {  // NaN and Inf propagate
            nonfinite = true;
            break;
        }
        done = (!rule0 || have_exact) && stopq <= thr;
        if (done) break;
        exact_next = rule0 && red[1] <= 1.25f * thr;
        const float beta = __fdividef(eta_new, eta);
#pragma unroll
        for (int i = 0; i < R; ++i) p[i] = fmaf(beta, p[i], y[i]);
        rows_store<NP, R>(XP, jj, a0, valid, p);
        eta = eta_new;
        __syncthreads();
    }
    __syncthreads();
    rows_store<NP, R>(XP, jj, a0, valid, lam);
    __syncthreads();
    recover_dz(g.w, g.rhs, g.lambda, g.dX, g.dU, sol,
               [&](int k, int b) { return XP[(k + 1) * NP + b]; }, lsm);
    finish(g, sol, it, done, nonfinite);
}

// ===========================================================================
// cluster form: one solve over the C CTAs of a thread-block cluster
// ===========================================================================
//
// k_pcg_rows_cluster<NP, R> runs the same iteration with a solve's knots
// split over the CTAs of a cluster (C = 2, 4 or 8, the cluster's size at
// launch): CTA c owns knots c Nc .. c Nc + Nc - 1 (Nc = ceil(N / C)) with
// their rows of the two coupling blocks, exactly as k_pcg_rows does for a
// whole solve.  A CTA's vectors keep the same guard slots, which here hold
// the neighbouring CTAs' boundary knots: the owners of a CTA's first and
// last knot also write their rows into the previous and next CTA's guards
// (distributed shared memory).  Block sums add every CTA's warp slots in rank
// order, so all CTAs hold the same scalars and take the same branches; every
// barrier is a cluster barrier.  The recovery is cluster_recover's.

// post2's pair pushed into slot rank * nw + w of every CTA of the cluster (nw
// warps a CTA; the launch keeps C nw within kRowsClusterSlots), stored before
// the cluster barrier that publishes it, so that the collect reads only local
// shared memory; every lane of a half-warp holds its half's total
__device__ __forceinline__ void rows_cluster_post2(cg::cluster_group& cl, float a, float b,
                                                   float2* buf)
{
    const int lane = lane_id();
    const bool hi = lane & 16;
    float keep = hi ? b : a;
    keep += __shfl_xor_sync(0xffffffffu, hi ? a : b, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    const int rk = lane & 15, rank = (int)cl.block_rank();
    if (rk < (int)cl.num_blocks()) {
        float2* dst = rk == rank ? buf : cl.map_shared_rank(buf, rk);
        reinterpret_cast<float*>(dst + rank * (int)(blockDim.x >> 5) +
                                 (int)(threadIdx.x >> 5))[hi ? 1 : 0] = keep;
    }
}

// the pushed pairs of every CTA, each CTA's warps in collect2's tree, the
// CTAs added in rank order (the same bits in every CTA)
__device__ __forceinline__ float2 rows_cluster_collect2(cg::cluster_group& cl, const float2* buf)
{
    float2 s = make_float2(0.f, 0.f);
    const int C = (int)cl.num_blocks(), nw = (int)(blockDim.x >> 5);
    for (int rk = 0; rk < C; ++rk) {
        const float2 v = collect2(buf + rk * nw);
        s.x += v.x;
        s.y += v.y;
    }
    return s;
}

// block_sum over the whole cluster: warp sums to this CTA's slots, a cluster
// barrier, then every thread adds all CTAs' slots in rank order
template <int K>
__device__ __forceinline__ void rows_cluster_sum(cg::cluster_group& cl, float (&v)[K],
                                                 float4* buf)
{
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = warp_sum(v[k]);
    const int wi = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane_id() == 0)
        buf[wi] = make_float4(v[0], K > 1 ? v[K > 1 ? 1 : 0] : 0.f,
                              K > 2 ? v[K > 2 ? 2 : 0] : 0.f, 0.f);
    cl.sync();
    float s[3] = {0.f, 0.f, 0.f};
    const int C = (int)cl.num_blocks();
    for (int rk = 0; rk < C; ++rk) {
        const float4* b = cl.map_shared_rank(buf, rk);
        for (int q = 0; q < nw; ++q) {
            const float4 t = b[q];
            s[0] += t.x;
            s[1] += t.y;
            s[2] += t.z;
        }
    }
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = s[k];
}

template <int NP, int R>
__global__ void __launch_bounds__(max_threads_for(NP, R)) k_pcg_rows_cluster(PcgArgs g)
{
    extern __shared__ __align__(16) float sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank(), C = (int)cl.num_blocks();
    const Work& w = g.w;
    const int N = w.N, n = w.n, T = blockDim.x, tid = threadIdx.x;
    const int sol = blockIdx.x / C;
    const int Nc = (N + C - 1) / C;
    const int k0 = rank * Nc;         // first knot of this CTA
    const int nk = min(Nc, N - k0);   // its knot count (>= 1 by the launch)
    const int TPK = (n + R - 1) / R;
    const int XS = (Nc + 2) * NP;     // one vector with its guard knots
    const bool rule0 = g.rule == GATO_STOP_RESIDUAL;

    float* XP = sm;
    float* XR = XP + XS;
    float4* redA = reinterpret_cast<float4*>(XR + XS);
    float4* redB = redA + 32;
    float4* redC = redA + 64;
    float2* pairA = reinterpret_cast<float2*>(redA + 96);  // kRowsClusterSlots each
    float2* pairB = pairA + kRowsClusterSlots;
    float2* pairC = pairB + kRowsClusterSlots;
    constexpr int SC = NP / 4 - RowTiles<NP, R>::RC;
    float4* TS = redA + kRowsClusterHead;
    float* LS = reinterpret_cast<float*>(TS + (size_t)SC * R * 2 * T);
    const bool l_staged = rule0 && g.l_smem;
    // the layout is the same in every CTA, so they all leave together
    if (!gb_smem((size_t)(LS - sm + (l_staged ? (size_t)Nc * n * NP : 0)) * sizeof(float),
                 w.status, sol)) {
        if (rank == 0) finish(g, sol, 0, false, false);
        return;
    }
    for (int i = tid; i < 2 * XS; i += T) sm[i] = 0.f;

    const int jl = tid / TPK, q = tid - jl * TPK;
    const int a0 = q * R;
    const bool owner = jl < nk && gb_ok((long long)(jl + 2) * NP + NP - 1, XS, w.status, sol) &&
                       gb_ok(a0, n, w.status, sol);
    bool valid[R];
#pragma unroll
    for (int i = 0; i < R; ++i) valid[i] = owner && a0 + i < n;
    const int jjl = owner ? jl : 0;  // a safe local knot for threads past the last one
    const int jj = k0 + jjl;         // its global index
    // the neighbours' guard slots this thread also writes: the previous CTA's
    // slot after its last knot (Nc + 1) for the CTA's first knot, the next
    // CTA's slot 0 for its last knot
    float* prevXP = (owner && jl == 0 && rank > 0) ? cl.map_shared_rank(XP, rank - 1) : nullptr;
    float* prevXR = prevXP ? cl.map_shared_rank(XR, rank - 1) : nullptr;
    float* nextXP = (owner && jl == nk - 1 && rank + 1 < C) ? cl.map_shared_rank(XP, rank + 1)
                                                             : nullptr;
    float* nextXR = nextXP ? cl.map_shared_rank(XR, rank + 1) : nullptr;
    auto store = [&](float* X, float* Xprev, float* Xnext, const float(&v)[R]) {
        rows_store<NP, R>(X, jjl, a0, valid, v);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            if (!valid[i]) continue;
            if (Xprev) Xprev[(Nc + 1) * NP + a0 + i] = v[i];
            if (Xnext) Xnext[a0 + i] = v[i];
        }
    };

    RowTiles<NP, R> tile;
    {
        const float* nh = w.Nh + sol * w.sKnn;
        const size_t nn = (size_t)n * n;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            const int a = a0 + i;
            const bool has_lo = valid[i] && jj >= 1;
            const bool has_up = valid[i] && jj + 1 < N;
            const float* lo = nh + (size_t)(jj >= 1 ? jj - 1 : 0) * nn + (size_t)a * n;
            const float* up = nh + (size_t)(jj + 1 < N ? jj : 0) * nn + a;
#pragma unroll
            for (int b = 0; b < 4 * RowTiles<NP, R>::RC; ++b) {
                tile.lo[i][b] = (has_lo && b < n) ? lo[b] : 0.f;
                tile.up[i][b] = (has_up && b < n) ? up[(size_t)b * n] : 0.f;
            }
#pragma unroll
            for (int sc = 0; sc < SC; ++sc) {
                float vl[4], vu[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int b = 4 * (RowTiles<NP, R>::RC + sc) + e;
                    vl[e] = (has_lo && b < n) ? lo[b] : 0.f;
                    vu[e] = (has_up && b < n) ? up[(size_t)b * n] : 0.f;
                }
                TS[ts_index<R>(sc, i, 0, tid, T)] = make_float4(vl[0], vl[1], vl[2], vl[3]);
                TS[ts_index<R>(sc, i, 1, tid, T)] = make_float4(vu[0], vu[1], vu[2], vu[3]);
            }
        }
    }
    const float dl = owner ? w.dlow[sol * w.sN + jj] : 0.f;
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float* gL = w.L + sol * w.sNnn;
    const float* Lj = gL + (size_t)jj * n * n;
    if (l_staged) {  // this CTA's knots' rows of L, padded to NP
        const float* gLc = gL + (size_t)k0 * n * n;
        for (int t = tid; t < nk * n * NP; t += T) {
            const int row = t / NP, b = t - row * NP;
            LS[t] = b < n ? gLc[(size_t)row * n + b] : 0.f;
        }
    }

    float lam[R], r[R], p[R], y[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        lam[i] = 0.f;
        if (valid[i] && g.lambda0) {
            const int a = a0 + i;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + (size_t)jj * n;
            float x = 0.f;
            for (int b = a; b < n; ++b) x += Lj[(size_t)b * n + a] * l0[b];
            lam[i] = x;
        }
    }
    cl.sync();  // every CTA's vectors zeroed before any guard is written
    store(XP, prevXP, nextXP, lam);
    cl.sync();
    rows_matvec<NP, R>(tile, TS, XP, jjl, y);
#pragma unroll
    for (int i = 0; i < R; ++i)
        r[i] = valid[i] ? ghat[jj * n + a0 + i] - lam[i] - y[i] : 0.f;
    store(XR, prevXR, nextXR, r);
    cl.sync();
    rows_matvec<NP, R>(tile, TS, XR, jjl, y);
    float red3[3] = {0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < R; ++i) {
        p[i] = r[i] - y[i];
        red3[0] = fmaf(r[i], p[i], red3[0]);
        if (valid[i]) {
            const int gi = jj * n + a0 + i;
            if (rule0)
                red3[2] = fmaf(gam[gi], gam[gi], red3[2]);
            else if (g.rule == GATO_STOP_SCALED) {
                red3[1] = fmaf(r[i], r[i], red3[1]);
                red3[2] = fmaf(ghat[gi], ghat[gi], red3[2]);
            }
        }
    }
    if (rule0)
        red3[1] = l_staged ? rows_lnorm_smem<NP, R>(LS, XR, jjl, a0, n, valid)
                           : rows_lnorm<NP, R>(Lj, XR, jjl, a0, n, valid);
    store(XP, prevXP, nextXP, p);
    rows_cluster_sum<3>(cl, red3, redA);  // also orders the p stores before the first product
    float eta = red3[0];
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : red3[2];
    const float thr = g.eps * g.eps * ref;
    bool done = (g.rule == GATO_STOP_PRECOND ? eta : red3[1]) <= thr;
    bool nonfinite = !isfinite(eta) || !isfinite(red3[1]);
    bool exact_next = false;
    if (rule0) {
        float lb = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) lb = fmaf(dl * r[i], r[i], lb);
        float lv[1] = {lb};
        rows_cluster_sum<1>(cl, lv, redB);
        exact_next = lv[0] <= 1.25f * thr;
    }
    cl.sync();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        rows_matvec<NP, R>(tile, TS, XP, jjl, y);
        float pvp = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i) {
            y[i] += p[i];
            pvp = fmaf(p[i], y[i], pvp);
        }
        rows_cluster_post2(cl, pvp, 0.f, pairA);
        cl.sync();
        const float pv = rows_cluster_collect2(cl, pairA).x;
        const float alpha = __fdividef(eta, pv);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            lam[i] = fmaf(alpha, p[i], lam[i]);
            r[i] = fmaf(-alpha, y[i], r[i]);
        }
        store(XR, prevXR, nextXR, r);
        cl.sync();
        rows_matvec<NP, R>(tile, TS, XR, jjl, y);
        float red[3] = {0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < R; ++i) {
            y[i] = r[i] - y[i];
            red[0] = fmaf(r[i], y[i], red[0]);
            red[1] = fmaf(r[i], r[i], red[1]);
        }
        if (rule0) red[1] *= dl;
        const bool exact = exact_next;
        if (exact)
            red[2] = l_staged ? rows_lnorm_smem<NP, R>(LS, XR, jjl, a0, n, valid)
                              : rows_lnorm<NP, R>(Lj, XR, jjl, a0, n, valid);
        rows_cluster_post2(cl, red[0], red[1], pairB);
        if (exact) rows_cluster_post2(cl, red[2], 0.f, pairC);
        cl.sync();
        {
            const float2 sb = rows_cluster_collect2(cl, pairB);
            red[0] = sb.x;
            red[1] = sb.y;
            red[2] = exact ? rows_cluster_collect2(cl, pairC).x : 0.f;
        }
        const float eta_new = red[0];
        float lsq = red[2];
        bool have_exact = exact;
        if (rule0 && !exact && red[1] * 0.999f <= thr) {
            float lv[1] = {l_staged ? rows_lnorm_smem<NP, R>(LS, XR, jjl, a0, n, valid)
                                    : rows_lnorm<NP, R>(Lj, XR, jjl, a0, n, valid)};
            rows_cluster_sum<1>(cl, lv, redC);
            lsq = lv[0];
            have_exact = true;
        }
        const float stopq = rule0 ? lsq : (g.rule == GATO_STOP_SCALED ? red[1] : eta_new);
        if (!isfinite(eta_new + pv + stopq + red[1])) {  // NaN and Inf propagate
            nonfinite = true;
            break;
        }
        done = (!rule0 || have_exact) && stopq <= thr;
        if (done) break;
        exact_next = rule0 && red[1] <= 1.25f * thr;
        const float beta = __fdividef(eta_new, eta);
#pragma unroll
        for (int i = 0; i < R; ++i) p[i] = fmaf(beta, p[i], y[i]);
        store(XP, prevXP, nextXP, p);
        eta = eta_new;
        cl.sync();
    }
    cl.sync();
    rows_store<NP, R>(XP, jjl, a0, valid, lam);
    cl.sync();
    cluster_recover<NP>(cl, g, sol, k0, nk, [&](int kl, int b) { return XP[(kl + 1) * NP + b]; });
    if (rank == 0) finish(g, sol, it, done, nonfinite);
    cl.sync();  // no CTA leaves while another may still read its shared memory
}

// one solve per cluster of C CTAs (grid M C); cudaErrorInvalidConfiguration
// when no such cluster fits on the device
template <typename K>
cudaError_t launch_rows_cluster_k(K kernel, const PcgArgs& a, int C, int T, size_t smem,
                                  cudaStream_t st)
{
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (C > 8) {
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(a.w.M * C), 1, 1);
    cfg.blockDim = dim3((unsigned)T, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    e = cudaOccupancyMaxActiveClusters(&clusters, kernel, &cfg);
    if (e != cudaSuccess || clusters < 1) {
        cudaGetLastError();
        return cudaErrorInvalidConfiguration;
    }
    e = cudaLaunchKernelEx(&cfg, kernel, a);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// the cluster form where one CTA cannot hold the solve: the smallest C in
// {2, 4, 8} whose Nc = ceil(N / C) knots fit a CTA and leave every CTA at
// least one knot
template <int NP, int R>
cudaError_t launch_rows_cluster_np(const PcgArgs& a, size_t limit, cudaStream_t st)
{
    const Work& w = a.w;
    const int TPK = (w.n + R - 1) / R;
    for (int C = 2; C <= 8; C *= 2) {
        const int Nc = (w.N + C - 1) / C;
        if ((C - 1) * Nc >= w.N) break;  // a CTA would hold no knot
        int T = ((Nc * TPK + 31) / 32) * 32;
        if (T < 64) T = 64;
        if (T > max_threads_for(NP, R)) continue;
        if (C * (T / 32) > kRowsClusterSlots) continue;  // the pushed pair slots
        constexpr int SC = NP / 4 - RowTiles<NP, R>::RC;
        size_t smem = sizeof(float) * 2 * (size_t)(Nc + 2) * NP +
                      (kRowsClusterHead + (size_t)SC * R * 2 * T) * sizeof(float4);
        if (smem > limit) return cudaErrorInvalidConfiguration;
        PcgArgs b = a;
        const size_t l_bytes = sizeof(float) * (size_t)Nc * w.n * NP;
        b.l_smem = a.rule == GATO_STOP_RESIDUAL && smem + l_bytes <= limit;
        if (b.l_smem) smem += l_bytes;
        return launch_rows_cluster_k(k_pcg_rows_cluster<NP, R>, b, C, T, smem, st);
    }
    return cudaErrorInvalidConfiguration;
}

template <int NP, int R = rows_for(NP)>
cudaError_t launch_rows_np(const PcgArgs& a, size_t limit, cudaStream_t st)
{
    const Work& w = a.w;
    const int TPK = (w.n + R - 1) / R;
    int T = ((w.N * TPK + 31) / 32) * 32;
    if (T < 64) T = 64;
    if (T > max_threads_for(NP, R)) return launch_rows_cluster_np<NP, R>(a, limit, st);
    constexpr int SC = NP / 4 - RowTiles<NP, R>::RC;
    size_t smem = sizeof(float) * (2 * (size_t)(w.N + 2) * NP + round4((size_t)w.N * w.n)) +
                  (120 + (size_t)SC * R * 2 * T) * sizeof(float4);
    if (smem > limit) return cudaErrorInvalidConfiguration;
    // rule 0: the rows of L in shared memory where they fit
    PcgArgs b = a;
    const size_t l_bytes = sizeof(float) * (size_t)w.N * w.n * NP;
    b.l_smem = a.rule == GATO_STOP_RESIDUAL && smem + l_bytes <= limit;
    if (b.l_smem) smem += l_bytes;
    auto kernel = k_pcg_rows<NP, R>;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kernel<<<w.M, T, smem, st>>>(b);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_pcg_rows(const PcgArgs& a, size_t limit, cudaStream_t st)
{
    const int n = a.w.n;
    if (n <= 20) return launch_rows_np<20>(a, limit, st);
    if (n <= 24) return launch_rows_np<24>(a, limit, st);
    if (n <= 28) return launch_rows_np<28>(a, limit, st);
    if (n <= 32) return launch_rows_np<32>(a, limit, st);
    if (n <= 36) return launch_rows_np<36>(a, limit, st);
    if (n <= 40) return launch_rows_np<40>(a, limit, st);
    if (n <= 48) return launch_rows_np<48>(a, limit, st);
    if (n <= 56) return launch_rows_np<56>(a, limit, st);
    if (n <= 64) return launch_rows_np<64>(a, limit, st);
    return cudaErrorInvalidConfiguration;
}

}  // namespace gato
