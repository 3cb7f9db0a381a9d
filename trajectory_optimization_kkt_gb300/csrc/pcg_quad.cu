// pcg_quad.cu -- batched PCG on S lambda = gamma with the symmetric stair
// preconditioner for 7 <= n <= 16, N <= 128, four threads per coupling
// block, and recovery of dz (GATO paper, Sec. II and eq. (4); Sec. III: one
// thread block per linear system, block-tridiagonal matrix-vector products,
// warp-shuffle reductions).
//
// The same iteration as k_pcg_wide (pcg.cu), in the block-Jacobi-scaled
// variables lambda_hat = L^T lambda, where S_hat = I + Nhat and the stair
// preconditioner is I - Nhat: both products of an iteration are products
// with the block-tridiagonal Nhat (coupling blocks Nhat_j, block (j, j-1)).
//
// k_pcg_quad<NN> (n = NN): the four threads of quad j (threads 4j .. 4j+3,
// lane c = t mod 4) own knot j, lane c the rows a = 4k + c (k < ceil(n/4)),
// and for j >= 1 hold those rows of Nhat_j over all n columns in registers.
// A product with Nhat then gives each lane
//   - its rows of Nhat_j x_{j-1}, complete, in registers (x_{j-1} read from
//     shared memory as four 128-bit broadcasts), and
//   - its rows' share of Nhat_j^T x_j, the column sums for knot j-1, which
//     the quad reduces and scatters with two butterfly exchanges (lane c
//     ends with the complete sums of columns c, c+4, c+8, c+12, exactly the
//     slots it writes), one 128-bit store per lane to the owners of knot j-1.
// Against k_pcg_wide (two threads per block, rows over 2H columns) a thread
// holds half the tile and does half the FMAs per product, the block has
// twice the warps to hide the latency of the shared-memory and shuffle
// dependencies, and a product needs one column-sum array instead of two.
//
// A knot's slots are ordered by lane: slot 4c + k holds row (column) 4k + c,
// so a lane's four rows are one float4.  Knot stride 16 floats: within every
// quarter-warp (two quads, knots j and j+1) the x_{j-1} broadcasts and the
// column-sum stores touch distinct banks.
#include "pcg_common.cuh"

namespace gato {
namespace {

constexpr int kQS = 16;   // knot stride of the vectors and column sums (floats)
constexpr int kQLS = 20;  // floats per staged row of L

__host__ __device__ constexpr int qrows(int nn) { return (nn + 3) / 4; }

// slot of row (column) b within a knot
__host__ __device__ constexpr int qslot(int b) { return (b & 3) * 4 + (b >> 2); }

__host__ __device__ __forceinline__ int q_knot_stride(int n)
{
    return (n * kQLS) % 32 == 0 ? n * kQLS + 8 : n * kQLS;
}

__device__ __forceinline__ float4 ld4(const float* p) { return *reinterpret_cast<const float4*>(p); }

__device__ __forceinline__ void st4(float* p, const float (&v)[4])
{
    *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float s)
{
    s = fmaf(a.x, b.x, s);
    s = fmaf(a.y, b.y, s);
    s = fmaf(a.z, b.z, s);
    return fmaf(a.w, b.w, s);
}

// Lane c keeps its tile columns in a lane-dependent order: tile column i
// holds matrix column i ^ qperm(c), so that in the quad's reduce-scatter
// every lane sends the same tile index and keeps the same one (no selects).
// With n a multiple of 4 the mask is c (both exchanges select-free), else
// c & 1 (the first exchange only); columns past n are zero.  x_{j-1} is read
// in the matching order: chunk c2 ^ qperm(c) at step c2.
template <int NN>
__host__ __device__ constexpr bool qfull() { return NN % 4 == 0; }

template <int NN>
__device__ __forceinline__ int qperm(int c) { return qfull<NN>() ? c : (c & 1); }

// tile columns: n rounded up to even (the pairs of the first exchange)
__host__ __device__ constexpr int qcols(int nn) { return (nn + 1) & ~1; }

template <int NN>
struct QuadTile {
    float t[qrows(NN)][qcols(NN)];  // rows 4k + c of Nhat_j, columns i ^ qperm(c)
};

// One product with Nhat for this lane's rows of block j: rs gets the
// complete sums of its rows of Nhat_j x_{j-1}; the column sums of Nhat_j^T
// x_j (x_j's owned part in xo) are reduced over the quad and lane c stores
// those of columns c, c+4, c+8, c+12 to yc (knot j-1's chunk c) when st.
// Returns xo^T rs, this lane's share of x^T Nhat x.  Every thread of the
// warp calls it (the exchanges are warp-wide); threads without a block hold
// a zero tile.
template <int NN>
__device__ __forceinline__ float quad_matvec(const QuadTile<NN>& T, const float* xprev,
                                             const float (&xo)[4], float (&rs)[4], float* yc,
                                             bool st, int c)
{
    constexpr int QR = qrows(NN), NI = qcols(NN);
    const int pm = qperm<NN>(c);
    float cs[NI];
#pragma unroll
    for (int i = 0; i < NI; ++i) cs[i] = 0.f;
#pragma unroll
    for (int k = 0; k < 4; ++k) rs[k] = 0.f;
#pragma unroll
    for (int c2 = 0; c2 < 4; ++c2) {
        // chunk c2 ^ pm holds columns 4 kk + (c2 ^ pm), tile columns 4 kk + c2
        const float4 v = ld4(xprev + 4 * (c2 ^ pm));
        const float xv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            const int i = 4 * kk + c2;
            if (i >= NI) continue;
#pragma unroll
            for (int k = 0; k < QR; ++k) {
                rs[k] = fmaf(T.t[k][i], xv[kk], rs[k]);
                cs[i] = fmaf(T.t[k][i], xo[k], cs[i]);
            }
        }
    }
    // reduce-scatter over the quad.  xor 1: the partner's tile index of the
    // column this lane keeps at even index 2t is 2t + 1, so every lane keeps
    // cs[2t] and sends cs[2t + 1]; u1[t] is column 2t ^ pm.  xor 2: lane c
    // keeps the columns congruent to c mod 4, u2[k] = column 4k + c
    float u1[2 * QR];
#pragma unroll
    for (int t = 0; t < 2 * QR; ++t) {
        u1[t] = 0.f;
        if (2 * t >= NI) continue;
        u1[t] = cs[2 * t] + __shfl_xor_sync(0xffffffffu, cs[2 * t + 1], 1);
    }
    float u2[4] = {0.f, 0.f, 0.f, 0.f};
    if constexpr (qfull<NN>()) {
        // u1[t] is column 2t ^ c: this lane keeps even t, the partner (mask
        // c ^ 2) holds the same column at t ^ 1
#pragma unroll
        for (int k = 0; k < QR; ++k)
            u2[k] = u1[2 * k] + __shfl_xor_sync(0xffffffffu, u1[2 * k + 1], 2);
    } else {
        // u1[t] is column 2t + (c & 1) on both partners: keep t of parity
        // c >> 1, send the other
        const bool b1 = c & 2;
#pragma unroll
        for (int k = 0; k < QR; ++k) {
            const float lo = u1[2 * k], hi = u1[2 * k + 1];
            u2[k] = (b1 ? hi : lo) + __shfl_xor_sync(0xffffffffu, b1 ? lo : hi, 2);
        }
    }
    if (st) st4(yc, u2);
    float q = 0.f;
#pragma unroll
    for (int k = 0; k < QR; ++k) q = fmaf(xo[k], rs[k], q);
    return q;
}

// (Nhat x) at the four owned slots: own row sums plus the column sums
__device__ __forceinline__ void quad_y(const float (&rs)[4], const float* yc, float (&y)[4])
{
    const float4 v = ld4(yc);
    y[0] = rs[0] + v.x;
    y[1] = rs[1] + v.y;
    y[2] = rs[2] + v.z;
    y[3] = rs[3] + v.w;
}

// Rows of L_j into LP in the slot order (zeros above the diagonal and in the
// padding): row a at LP + j KS + a kQLS, its column b at slot qslot(b).
__device__ __forceinline__ void stage_l_quad(float* LP, int KS, const float* gL, int N, int n)
{
    for (int ja = threadIdx.x; ja < N * n; ja += blockDim.x) {
        const int j = ja / n, a = ja - j * n;
        const float* src = gL + (size_t)j * n * n + a * n;
        float v[16];
#pragma unroll
        for (int s = 0; s < 16; ++s) {
            const int b = (s & 3) * 4 + (s >> 2);  // column of slot s
            v[s] = (b < n && b <= a) ? src[b] : 0.f;
        }
        float4* dst = reinterpret_cast<float4*>(LP + j * KS + a * kQLS);
#pragma unroll
        for (int s = 0; s < 4; ++s)
            dst[s] = make_float4(v[4 * s], v[4 * s + 1], v[4 * s + 2], v[4 * s + 3]);
    }
}

// sum over the owned valid rows a = 4k + c of (L_j r_hat_j)_a^2
template <int NN>
__device__ __forceinline__ float lnorm_quad(const float* LP, int KS, const float* XR, int j,
                                            int c, bool owner)
{
    constexpr int QR = qrows(NN);
    const float* xk = XR + j * kQS;
    const float4 x0 = ld4(xk), x1 = ld4(xk + 4), x2 = ld4(xk + 8), x3 = ld4(xk + 12);
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < QR; ++k) {
        const int a = 4 * k + c;
        if (!owner || a >= NN) continue;
        const float* row = LP + j * KS + a * kQLS;
        float t = dot4(ld4(row), x0, 0.f);
        t = dot4(ld4(row + 4), x1, t);
        t = dot4(ld4(row + 8), x2, t);
        t = dot4(ld4(row + 12), x3, t);
        s = fmaf(t, t, s);
    }
    return s;
}

template <int NN>
__device__ __forceinline__ void pcg_quad_solve(const PcgArgs& g, int sol)
{
    constexpr int QR = qrows(NN);
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int N = w.N, n = NN, tid = threadIdx.x;
    const int T = blockDim.x;
    const int EX = N * kQS;
    const bool rule0 = g.rule == GATO_STOP_RESIDUAL;
    const int KS = q_knot_stride(n);

    float* XP = sm;
    float* XR = XP + EX;
    float* YC = XR + EX;
    const int zero_count = 3 * EX;
    float2* redA = reinterpret_cast<float2*>(sm + zero_count);
    float2* redB = redA + 32;
    float2* redC = redA + 64;
    float2* redD = redA + 96;  // also used as float4[16] by block_sum
    float* DL = reinterpret_cast<float*>(redA + 160);
    float* LP = DL + ((N + 3) & ~3);
    if (!gb_smem((size_t)(LP - sm + (rule0 ? (size_t)N * KS : 0)) * sizeof(float), w.status,
                 sol)) {
        finish(g, sol, 0, false, false);
        return;  // block-uniform
    }

    for (int i = tid; i < zero_count; i += T) sm[i] = 0.f;
    for (int j = tid; j < N; j += T) DL[j] = w.dlow[sol * w.sN + j];
    const float* gL = w.L + sol * w.sNnn;
    if (rule0) stage_l_quad(LP, KS, gL, N, n);

    // quad j owns knot j; j >= 1 holds rows 4k + c of Nhat_j, reads x_{j-1}
    // and writes knot j-1's column sums (chunk c)
    const int c = tid & 3;
    const int j = tid >> 2;
    const bool owner = j < N && gb_ok((long long)j * kQS + 4 * c + 3, EX, w.status, sol);
    const bool has_tile = owner && j >= 1;
    const int jo = owner ? j : 0;
    const int pj = (has_tile ? j - 1 : 0) * kQS;  // knot j-1
    float* yc = YC + pj + 4 * c;
    const int xo = jo * kQS + 4 * c;  // owned slots in XP / XR / YC
    QuadTile<NN> tile;
    {
        const float* blk = w.Nh + sol * w.sKnn + (size_t)(has_tile ? j - 1 : 0) * n * n;
        const int pm = qperm<NN>(c);
#pragma unroll
        for (int k = 0; k < QR; ++k)
#pragma unroll
            for (int i = 0; i < qcols(NN); ++i) {
                const int a = 4 * k + c, b = i ^ pm;
                tile.t[k][i] = (has_tile && a < n && b < n) ? blk[a * n + b] : 0.f;
            }
    }
    bool valid[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) valid[k] = owner && k < QR && 4 * k + c < n;
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float dl = owner ? DL[jo] : 0.f;
    // slots of rows past n (and all slots of threads that own none) start at
    // zero and stay exactly zero: the tiles' padded rows are zero, so the
    // loop needs no masks
    float lam[4], r[4], p[4], y[4], rs[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) rs[k] = y[k] = 0.f;
    __syncthreads();

    // lambda_hat0 = L^T lambda0
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        lam[k] = 0.f;
        if (valid[k] && g.lambda0) {
            const int a = 4 * k + c;
            const float* Lj = gL + (size_t)jo * n * n;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + jo * n;
            float x = 0.f;
            for (int b = a; b < n; ++b) x += Lj[b * n + a] * l0[b];
            lam[k] = x;
        }
    }
    if (owner) st4(XP + xo, lam);
    __syncthreads();
    quad_matvec<NN>(tile, XP + pj, lam, rs, yc, has_tile, c);
    __syncthreads();
    // r_hat = ghat - S_hat lambda_hat
    float rr = 0.f, gg = 0.f;
    if (owner) quad_y(rs, YC + xo, y);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        r[k] = 0.f;
        if (valid[k]) {
            const int i = jo * n + 4 * k + c;
            r[k] = ghat[i] - lam[k] - y[k];
            rr += r[k] * r[k];
            gg += rule0 ? gam[i] * gam[i] : ghat[i] * ghat[i];
        }
    }
    if (owner) st4(XR + xo, r);
    post2(rr, gg, redB);
    __syncthreads();  // XR complete; the column sums of lambda are read
    float q = quad_matvec<NN>(tile, XR + pj, r, rs, yc, has_tile, c);
    float lsq = 0.f;
    if (rule0) lsq = lnorm_quad<NN>(LP, KS, XR, jo, c, owner);
    post2(q, lsq, redC);
    __syncthreads();
    float2 sB = collect2(redB), sC = collect2(redC);
    float eta = sB.x - 2.f * sC.x;  // r^T (I - Nhat) r
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : sB.y;
    const float thr = g.eps * g.eps * ref;
    float stopq = g.rule == GATO_STOP_RESIDUAL ? sC.y : (g.rule == GATO_STOP_SCALED ? sB.x : eta);
    bool done = stopq <= thr;
    bool nonfinite = !isfinite(eta) || !isfinite(stopq);
    if (owner) quad_y(rs, YC + xo, y);
#pragma unroll
    for (int k = 0; k < 4; ++k) p[k] = r[k] - y[k];  // z = (I - Nhat) r
    if (owner) st4(XP + xo, p);
    // ||L r_hat|| (stopping rule 0) is evaluated only once the per-knot lower
    // bound sum_j dlow_j ||r_hat_j||^2 no longer rules convergence out
    bool exact_next;
    {
        float lb = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) lb += dl * r[k] * r[k];
        float lbv[1] = {lb};
        block_sum<1>(lbv, reinterpret_cast<float4*>(redD));
        exact_next = rule0 && lbv[0] <= 1.25f * thr;
    }
    __syncthreads();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        // A: Nhat p: own row sums, column sums to the owners of knot j-1;
        // p^T Nhat p and p^T p partials
        q = quad_matvec<NN>(tile, XP + pj, p, rs, yc, has_tile, c);
        float pp = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) pp = fmaf(p[k], p[k], pp);
        post2(q, pp, redA);
        __syncthreads();
        // B: alpha = eta / p^T S_hat p; lambda and r updates
        const float2 sA = collect2(redA);
        const float pv = sA.y + 2.f * sA.x;
        const float alpha = __fdividef(eta, pv);
        if (owner) quad_y(rs, YC + xo, y);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float v = p[k] + y[k];
            lam[k] = fmaf(alpha, p[k], lam[k]);
            r[k] = fmaf(-alpha, v, r[k]);
        }
        if (owner) st4(XR + xo, r);
        __syncthreads();
        // C: Nhat r; r^T Nhat r and r^T r partials, the lower bound and, when
        // gated in, ||L r_hat||^2
        q = quad_matvec<NN>(tile, XR + pj, r, rs, yc, has_tile, c);
        rr = 0.f;
#pragma unroll
        for (int k = 0; k < 4; ++k) rr = fmaf(r[k], r[k], rr);
        float lsq = 0.f;
        const bool exact = exact_next;
        if (exact) lsq = lnorm_quad<NN>(LP, KS, XR, jo, c, owner);
        post4(q, rr, dl * rr, lsq, reinterpret_cast<float4*>(redB));
        __syncthreads();
        // D: eta' = r^T (I - Nhat) r, convergence, p = z + beta p
        const float4 sBC = collect4(reinterpret_cast<const float4*>(redB));
        sB = make_float2(sBC.x, sBC.y);
        sC = make_float2(sBC.z, sBC.w);
        const float eta_new = sB.y - 2.f * sB.x;
        float lsq_all = sC.y;
        bool have_exact = exact;
        if (rule0 && !exact && sC.x * 0.999f <= thr) {
            lsq = lnorm_quad<NN>(LP, KS, XR, jo, c, owner);
            float lv[1] = {lsq};
            block_sum<1>(lv, reinterpret_cast<float4*>(redD));
            lsq_all = lv[0];
            have_exact = true;
        }
        stopq = g.rule == GATO_STOP_RESIDUAL ? lsq_all
                                             : (g.rule == GATO_STOP_SCALED ? sB.y : eta_new);
        if (!isfinite(eta_new + pv + stopq + sC.x)) {  // NaN and Inf propagate
            nonfinite = true;
            break;
        }
        done = (!rule0 || have_exact) && stopq <= thr;
        if (done) break;
        exact_next = rule0 && sC.x <= 1.25f * thr;
        const float beta = __fdividef(eta_new, eta);
        if (owner) quad_y(rs, YC + xo, y);
#pragma unroll
        for (int k = 0; k < 4; ++k) p[k] = fmaf(beta, p[k], r[k] - y[k]);
        if (owner) st4(XP + xo, p);
        eta = eta_new;
        __syncthreads();
    }
    __syncthreads();
    if (owner) st4(XP + xo, lam);
    __syncthreads();
    recover_dz<16>(g.w, g.rhs, g.lambda, g.dX, g.dU, sol,
                   [&](int jj, int b) { return XP[jj * kQS + qslot(b)]; }, YC);
    finish(g, sol, it, done, nonfinite);
}

template <int NN>
__global__ void __launch_bounds__(512, 1) k_pcg_quad(PcgArgs g)
{
    __shared__ int s_sol;
    for (;;) {
        if (threadIdx.x == 0) s_sol = atomicAdd(g.queue, 1);
        __syncthreads();
        const int sol = s_sol;
        __syncthreads();
        if (sol >= g.w.M) break;
        pcg_quad_solve<NN>(g, sol);
    }
}

size_t quad_smem_bytes(int N, int n, bool l_smem)
{
    size_t f = 3 * (size_t)kQS * N;  // XP, XR, YC
    f += 5 * 32 * 2;                 // five float2[32] reduction buffers
    f += round4(N);                  // DL
    if (l_smem) f += (size_t)N * q_knot_stride(n);
    return f * sizeof(float);
}

// persistent launch: as many blocks as can be resident, at most one per solve
template <typename K>
cudaError_t launch_quad_k(K kernel, const PcgArgs& a, int T, size_t smem, int num_sms,
                          cudaStream_t st)
{
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, T, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long grid = (long)per_sm * num_sms;
    if (grid > a.w.M) grid = a.w.M;
    e = cudaMemsetAsync(a.queue, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
    kernel<<<(unsigned)grid, T, smem, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

bool pcg_quad_fits(int N, int n, int rule, size_t smem_limit)
{
    if (n < 7 || n > 16 || N < 1 || N > 128) return false;
    return quad_smem_bytes(N, n, rule == GATO_STOP_RESIDUAL) <= smem_limit;
}

cudaError_t launch_pcg_quad(const PcgArgs& a_in, size_t smem_limit, int num_sms,
                            cudaStream_t st)
{
    PcgArgs a = a_in;
    const int N = a.w.N, n = a.w.n;
    if (!pcg_quad_fits(N, n, a.rule, smem_limit)) return cudaErrorInvalidConfiguration;
    a.nh_smem = 0;
    a.l_smem = a.rule == GATO_STOP_RESIDUAL;
    const size_t smem = quad_smem_bytes(N, n, a.l_smem);
    int T = ((4 * N + 31) / 32) * 32;
    if (T < 64) T = 64;
    switch (n) {
#define GATO_QUAD_CASE(NN) \
        case NN: return launch_quad_k(k_pcg_quad<NN>, a, T, smem, num_sms, st);
        GATO_QUAD_CASE(7) GATO_QUAD_CASE(8) GATO_QUAD_CASE(9) GATO_QUAD_CASE(10)
        GATO_QUAD_CASE(11) GATO_QUAD_CASE(12) GATO_QUAD_CASE(13) GATO_QUAD_CASE(14)
        GATO_QUAD_CASE(15) GATO_QUAD_CASE(16)
#undef GATO_QUAD_CASE
        default: return cudaErrorInvalidConfiguration;
    }
}

}  // namespace gato
