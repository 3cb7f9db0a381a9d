// pcg.cu -- batched preconditioned conjugate gradient on S lambda = gamma with
// the symmetric stair preconditioner, and recovery of dz (GATO paper, Sec. II
// and eq. (4); Sec. III: one thread block per linear system, no inter-block
// coordination, block-tridiagonal matrix-vector products, warp-shuffle
// reductions).
//
// Both kernels run PCG in the block-Jacobi-scaled variables
//     lambda_hat_j = L_j^T lambda_j,   S_jj = L_j L_j^T,
// where S_hat = L^-1 S L^-T = I + Nhat with Nhat block-tridiagonal, zero
// diagonal blocks and coupling blocks Nhat_j = L_j^-1 S_{j,j-1} L_{j-1}^-T,
// and the stair preconditioner becomes L^T Phi^-1 L = I - Nhat.  PCG is
// invariant under this congruence: its iterates map one to one onto those of
// PCG on (S, Phi^-1), eta = r^T Phi^-1 r is unchanged, and the true residual
// is r = L r_hat.  Both operator applications per iteration are products with
// the one matrix Nhat.
//
// k_pcg_wide<H>  (7 <= n <= 16, N <= 128; the default there): two threads
//     per coupling block with ownership aligned to the tiles, see below.
// k_pcg_tile<H>  (7 <= n <= 16, N <= 128): every coupling block Nhat_j is
//     split into 2 x 2 tiles of H x H (H = ceil(n/2)); four threads hold one
//     block's tiles in registers for the whole solve, so a product with Nhat
//     reads only the two vector halves each tile touches from shared memory
//     and does 2 H^2 FMAs per thread (row sums for knot j, column sums for
//     knot j-1).  Vector elements are owned by threads in registers; the two
//     inner products of an iteration are folded into the barriers that the
//     products need anyway (x^T S_hat x = x^T x + 2 sum_j x_j^T Nhat_j x_{j-1}),
//     four block barriers per iteration.
// k_pcg_generic  (any n <= 64): Nhat in shared memory when it fits (else read
//     from global memory), one thread per vector element.
// k_pcg_rows<NP, R> (pcg_rows.cu; the default for 16 < n <= 64 where its
//     block fits): whole rows of the coupling blocks in registers.
#include "pcg_common.cuh"

namespace gato {
namespace {

// ===========================================================================
// generic kernel
// ===========================================================================

// (Nhat x)_i for element i = (knot j, row a):
//   sum_b Nhat_j[a][b] x_{j-1}[b] + sum_b Nhat_{j+1}[b][a] x_{j+1}[b]
__device__ __forceinline__ float nhat_row(const float* Nh, const float* x, int i, int n, int N)
{
    const int j = i / n, a = i - j * n;
    float s = 0.f;
    if (j > 0) {
        const float* blk = Nh + (size_t)(j - 1) * n * n + a * n;
        const float* xv = x + (j - 1) * n;
        for (int b = 0; b < n; ++b) s += blk[b] * xv[b];
    }
    if (j < N - 1) {
        const float* blk = Nh + (size_t)j * n * n + a;
        const float* xv = x + (j + 1) * n;
        for (int b = 0; b < n; ++b) s += blk[b * n] * xv[b];
    }
    return s;
}

// (L x)_i: packed lower rows (row a of knot j at j*tri + a(a+1)/2) or the
// full n x n factor in global memory.
__device__ __forceinline__ float lrow(const float* Lp, const float* Lg, bool packed,
                                      const float* x, int i, int n)
{
    const int j = i / n, a = i - j * n;
    const float* xv = x + j * n;
    const float* row = packed ? Lp + (size_t)j * (n * (n + 1) / 2) + a * (a + 1) / 2
                              : Lg + (size_t)j * n * n + a * n;
    float s = 0.f;
    for (int b = 0; b <= a; ++b) s += row[b] * xv[b];
    return s;
}

// All PCG vectors live in shared memory; thread t owns elements t, t + T, ...
// and is the only one to write them.
__global__ void __launch_bounds__(512) k_pcg_generic(PcgArgs g)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int N = w.N, n = w.n, Nn = N * n, T = blockDim.x, tid = threadIdx.x;
    const int sol = blockIdx.x;
    const int tri = n * (n + 1) / 2;
    const size_t nh_count = (size_t)(N - 1) * n * n;

    size_t off = 0;
    float* sNh = sm + off;
    if (g.nh_smem) off += round4(nh_count);
    float* sLp = sm + off;
    const bool lpacked = g.rule == GATO_STOP_RESIDUAL && g.l_smem;
    if (lpacked) off += round4((size_t)N * tri);
    float* lam = sm + off;
    off += round4(Nn);
    float* r = sm + off;
    off += round4(Nn);
    float* p = sm + off;
    off += round4(Nn);
    float* v = sm + off;  // S_hat p, then z
    off += round4(Nn);
    float4* redA = reinterpret_cast<float4*>(sm + off);
    float4* redB = redA + 32;
    if (!gb_smem((off + 64 * 4) * sizeof(float), w.status, sol) ||
        (nh_count > 0 && !gb_ok((long long)nh_count - 1, (long long)w.sKnn, w.status, sol)) ||
        !gb_ok((long long)Nn - 1, (long long)w.sNn, w.status, sol))
        return;  // block-uniform

    const float* gNh = w.Nh + sol * w.sKnn;
    const float* gL = w.L + sol * w.sNnn;
    if (g.nh_smem) {
        for (size_t t = tid; t < nh_count; t += T) sNh[t] = gNh[t];
    }
    if (lpacked) {
        for (int t = tid; t < Nn; t += T) {
            const int j = t / n, a = t - j * n;
            const float* src = gL + (size_t)j * n * n + a * n;
            float* dst = sLp + (size_t)j * tri + a * (a + 1) / 2;
            for (int b = 0; b <= a; ++b) dst[b] = src[b];
        }
    }
    const float* Nh = g.nh_smem ? sNh : gNh;
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;

    // initial point lambda_hat = L^T lambda0
    for (int i = tid; i < Nn; i += T) {
        float x = 0.f;
        if (g.lambda0) {
            const int j = i / n, a = i - j * n;
            const float* Lj = gL + (size_t)j * n * n;
            const float* l0 = g.lambda0 + (size_t)sol * Nn + j * n;
            for (int b = a; b < n; ++b) x += Lj[b * n + a] * l0[b];
        }
        lam[i] = x;
    }
    __syncthreads();
    for (int i = tid; i < Nn; i += T) r[i] = ghat[i] - lam[i] - nhat_row(Nh, lam, i, n, N);
    __syncthreads();
    float red3[3] = {0.f, 0.f, 0.f};
    for (int i = tid; i < Nn; i += T) {
        const float z = r[i] - nhat_row(Nh, r, i, n, N);
        p[i] = z;
        red3[0] += r[i] * z;
        if (g.rule == GATO_STOP_RESIDUAL) {
            const float t = lrow(sLp, gL, lpacked, r, i, n);
            red3[1] += t * t;
            red3[2] += gam[i] * gam[i];
        } else if (g.rule == GATO_STOP_SCALED) {
            red3[1] += r[i] * r[i];
            red3[2] += ghat[i] * ghat[i];
        }
    }
    block_sum<3>(red3, redA);
    float eta = red3[0];
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : red3[2];
    const float thr = g.eps * g.eps * ref;
    bool done = (g.rule == GATO_STOP_PRECOND ? eta : red3[1]) <= thr;
    bool nonfinite = !isfinite(eta);

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        float pv[1] = {0.f};
        for (int i = tid; i < Nn; i += T) {
            const float x = p[i] + nhat_row(Nh, p, i, n, N);
            v[i] = x;
            pv[0] += p[i] * x;
        }
        block_sum<1>(pv, redA);
        const float alpha = __fdividef(eta, pv[0]);
        for (int i = tid; i < Nn; i += T) {
            lam[i] += alpha * p[i];
            r[i] -= alpha * v[i];
        }
        __syncthreads();
        float red2[2] = {0.f, 0.f};
        for (int i = tid; i < Nn; i += T) {
            const float z = r[i] - nhat_row(Nh, r, i, n, N);
            v[i] = z;
            red2[0] += r[i] * z;
            if (g.rule == GATO_STOP_RESIDUAL) {
                const float t = lrow(sLp, gL, lpacked, r, i, n);
                red2[1] += t * t;
            } else if (g.rule == GATO_STOP_SCALED) {
                red2[1] += r[i] * r[i];
            }
        }
        block_sum<2>(red2, redB);
        const float eta_new = red2[0];
        if (!isfinite(eta_new) || !isfinite(pv[0])) {
            nonfinite = true;
            break;
        }
        done = (g.rule == GATO_STOP_PRECOND ? eta_new : red2[1]) <= thr;
        if (done) break;
        const float beta = __fdividef(eta_new, eta);
        for (int i = tid; i < Nn; i += T) p[i] = v[i] + beta * p[i];
        eta = eta_new;
        __syncthreads();
    }
    __syncthreads();
    recover_dz(g.w, g.rhs, g.lambda, g.dX, g.dU, sol,
               [&](int j, int b) { return lam[j * n + b]; }, r);
    finish(g, sol, it, done, nonfinite);
}

// ===========================================================================
// register-tiled kernel
// ===========================================================================
//
// Shared-memory layouts (floats), knot stride 16 ("padded"): element (j, a)
// sits at j*16 + (a / H)*8 + a % H, so each half of a knot's vector starts on
// a 32-byte boundary; the padding slots stay exactly zero.
//   XP, XR [N][16]          the vectors multiplied by Nhat (p, r)
//   YR0, YR1 [N][16]        row sums of block j, one copy per column tile
//   YC0, YC1 [N][16]        column sums of block j+1, one copy per row tile
//                           (each copy offset by 4 floats from the previous
//                           one so that the two tiles' stores use different
//                           banks)
//   red [5][32] float2      warp partial sums (four in use)
//   DL [N]                  1 / ||L_j^-1||_F^2 (eigenvalue lower bounds)
//   LP [N][KS]              Cholesky factors for stopping rule 0: row a of
//                           L_j at j*KS + a*LS, its entries in the padded
//                           column layout of the vectors (so that a row
//                           times r_hat_j is four float4 products); LS = 20
//                           and KS = n*LS (+8 when that is a multiple of 32)
//                           keep the owners' row loads free of bank conflicts
// Thread t owns the four padded elements 4t .. 4t+3 (one knot half, one
// float4) and keeps them in registers; the launch uses T >= 4 N threads.

template <int H>
struct Tile {
    float t[H][H];
};

// One product with Nhat for the tile (j, rt, ct) held in registers: writes
// the row and column partial sums and returns x_j^T Nhat_j(tile) x_{j-1}.
template <int H>
__device__ __forceinline__ float tile_matvec(const Tile<H>& T, int j, int rt, int ct,
                                             const float* X, float* yr_base, float* yc_base)
{
    float xc[8], xr[8];
    const float4* pc = reinterpret_cast<const float4*>(X + (j - 1) * 16 + ct * 8);
    const float4* pr = reinterpret_cast<const float4*>(X + j * 16 + rt * 8);
    {
        const float4 a0 = pc[0], a1 = pc[1], b0 = pr[0], b1 = pr[1];
        xc[0] = a0.x; xc[1] = a0.y; xc[2] = a0.z; xc[3] = a0.w;
        xc[4] = a1.x; xc[5] = a1.y; xc[6] = a1.z; xc[7] = a1.w;
        xr[0] = b0.x; xr[1] = b0.y; xr[2] = b0.z; xr[3] = b0.w;
        xr[4] = b1.x; xr[5] = b1.y; xr[6] = b1.z; xr[7] = b1.w;
    }
    float rs[8], cs[8];
#pragma unroll
    for (int a = 0; a < 8; ++a) rs[a] = cs[a] = 0.f;
#pragma unroll
    for (int a = 0; a < H; ++a)
#pragma unroll
        for (int b = 0; b < H; ++b) {
            rs[a] += T.t[a][b] * xc[b];
            cs[b] += T.t[a][b] * xr[a];
        }
    float q = 0.f;
#pragma unroll
    for (int a = 0; a < H; ++a) q += xr[a] * rs[a];
    float4* yr = reinterpret_cast<float4*>(yr_base + j * 16 + rt * 8);
    float4* yc = reinterpret_cast<float4*>(yc_base + (j - 1) * 16 + ct * 8);
    yr[0] = make_float4(rs[0], rs[1], rs[2], rs[3]);
    yr[1] = make_float4(rs[4], rs[5], rs[6], rs[7]);
    yc[0] = make_float4(cs[0], cs[1], cs[2], cs[3]);
    yc[1] = make_float4(cs[4], cs[5], cs[6], cs[7]);
    return q;
}

struct Y4 {
    const float* r0;
    const float* r1;
    const float* c0;
    const float* c1;
};

// (Nhat x) at the four padded elements e0..e0+3, partial sums in a fixed order
__device__ __forceinline__ void ysum4(const Y4& y, int e0, float (&o)[4])
{
    const float4 a = *reinterpret_cast<const float4*>(y.r0 + e0);
    const float4 b = *reinterpret_cast<const float4*>(y.r1 + e0);
    const float4 c = *reinterpret_cast<const float4*>(y.c0 + e0);
    const float4 d = *reinterpret_cast<const float4*>(y.c1 + e0);
    o[0] = a.x + b.x + c.x + d.x;
    o[1] = a.y + b.y + c.y + d.y;
    o[2] = a.z + b.z + c.z + d.z;
    o[3] = a.w + b.w + c.w + d.w;
}

__device__ __forceinline__ void store4(float* X, int e0, const float (&v)[4])
{
    *reinterpret_cast<float4*>(X + e0) = make_float4(v[0], v[1], v[2], v[3]);
}

constexpr int kLS = 20;  // floats per padded row of L in shared memory

__host__ __device__ __forceinline__ int l_knot_stride(int n)
{
    return (n * kLS) % 32 == 0 ? n * kLS + 8 : n * kLS;
}

__device__ __forceinline__ float dot4(const float4 a, const float4 b, float s)
{
    s = fmaf(a.x, b.x, s);
    s = fmaf(a.y, b.y, s);
    s = fmaf(a.z, b.z, s);
    return fmaf(a.w, b.w, s);
}

// Row a of L_j into LP in the padded column layout (zeros above the
// diagonal and in the padding), one row per thread and pass: its n loads are
// issued together and it is written as four float4.
template <int H>
__device__ __forceinline__ void stage_l_rows(float* LP, int KS, const float* gL, int N, int n)
{
    for (int ja = threadIdx.x; ja < N * n; ja += blockDim.x) {
        const int j = ja / n, a = ja - j * n;
        const float* src = gL + (size_t)j * n * n + a * n;
        float v[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int b = c < 8 ? c : H + (c - 8);
            const bool in = (c < 8 ? c < H : c - 8 < n - H) && b <= a;
            v[c] = in ? src[b] : 0.f;
        }
        float4* dst = reinterpret_cast<float4*>(LP + j * KS + a * kLS);
#pragma unroll
        for (int c = 0; c < 4; ++c)
            dst[c] = make_float4(v[4 * c], v[4 * c + 1], v[4 * c + 2], v[4 * c + 3]);
    }
}

// sum over the owned valid rows a = ao + u of (L_j r_hat_j)_a^2: from the
// padded rows in shared memory (four float4 loads per row, the second-half
// chunks only for rows that reach them), or row by row from global memory
template <int H>
__device__ __forceinline__ float lnorm_owned(const float* LP, int KS, const float* gL, bool lsm,
                                             const float* XR, int j, int ao, int n,
                                             const bool (&valid)[4])
{
    float s = 0.f;
    if (lsm) {
        const float4* xv = reinterpret_cast<const float4*>(XR + j * 16);
        const float4 x0 = xv[0], x1 = xv[1], x2 = xv[2], x3 = xv[3];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!valid[u]) continue;
            const float4* row = reinterpret_cast<const float4*>(LP + j * KS + (ao + u) * kLS);
            float t = dot4(row[0], x0, 0.f);
            t = dot4(row[1], x1, t);
            if (ao + u >= H) {  // rows of the first half end before column H
                t = dot4(row[2], x2, t);
                t = dot4(row[3], x3, t);
            }
            s = fmaf(t, t, s);
        }
    } else {
        const float* xv = XR + j * 16;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            if (!valid[u]) continue;
            const int a = ao + u;
            const float* row = gL + (size_t)j * n * n + a * n;
            float t = 0.f;
            for (int b = 0; b <= a; ++b) t += row[b] * xv[(b / H) * 8 + b % H];
            s = fmaf(t, t, s);
        }
    }
    return s;
}

template <int H>
__device__ __forceinline__ void pcg_tile_solve(const PcgArgs& g, int sol)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int N = w.N, n = w.n, T = blockDim.x, tid = threadIdx.x;
    const int E = N * 16;  // padded elements
    const bool rule0 = g.rule == GATO_STOP_RESIDUAL;
    const bool lsm = rule0 && g.l_smem;
    const int KS = l_knot_stride(n);

    float* XP = sm;
    float* XR = XP + E;
    float* YR0 = XR + E;
    float* YR1 = YR0 + E + 4;
    float* YC0 = YR1 + E + 4;
    float* YC1 = YC0 + E + 4;
    const int zero_count = 6 * E + 12;
    float2* redA = reinterpret_cast<float2*>(sm + zero_count);
    float2* redB = redA + 32;
    float2* redC = redA + 64;
    float2* redD = redA + 96;  // also used as float4[16] by block_sum
    float* DL = reinterpret_cast<float*>(redA + 160);
    float* LP = DL + ((N + 3) & ~3);
    const Y4 Y{YR0, YR1, YC0, YC1};
    if (!gb_smem((size_t)(LP - sm + (lsm ? (size_t)N * KS : 0)) * sizeof(float), w.status,
                 sol)) {
        finish(g, sol, 0, false, false);
        return;  // block-uniform
    }

    // zero vectors and partial sums (padding and missing blocks stay 0)
    for (int i = tid; i < zero_count; i += T) sm[i] = 0.f;
    for (int j = tid; j < N; j += T) DL[j] = w.dlow[sol * w.sN + j];
    const float* gL = w.L + sol * w.sNnn;
    if (lsm) stage_l_rows<H>(LP, KS, gL, N, n);

    // the tile this thread holds: block jb = 1 + tid/4, tile (rt, ct)
    const int jb = 1 + (tid >> 2), rt = (tid >> 1) & 1, ct = tid & 1;
    // a tile's row and column sums go to knot jb's and jb-1's 16 slots
    const bool has_tile = jb <= N - 1 && gb_ok((long long)jb * 16 + 15, E, w.status, sol);
    float* yr_base = ct ? YR1 : YR0;
    float* yc_base = rt ? YC1 : YC0;
    Tile<H> tile;
    {
        const float* blk = w.Nh + sol * w.sKnn + (size_t)(has_tile ? jb - 1 : 0) * n * n;
#pragma unroll
        for (int a = 0; a < H; ++a)
#pragma unroll
            for (int b = 0; b < H; ++b) {
                const int ra = rt * H + a, cb = ct * H + b;
                tile.t[a][b] = (has_tile && ra < n && cb < n) ? blk[ra * n + cb] : 0.f;
            }
    }

    // owned elements e0 + u (u < 4): knot jo, rows ao + u; valid when in range
    const int e0 = 4 * tid;
    const bool owner = e0 < E;
    const int jo = e0 >> 4, k0 = e0 & 7;
    const int ao = ((e0 >> 3) & 1) * H + k0;
    bool valid[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) valid[u] = owner && k0 + u < H && ao + u < n;
    const int gi0 = jo * n + ao;  // unpadded index of element u is gi0 + u
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float dl = owner ? DL[jo] : 0.f;
    float lam[4], r[4], p[4], y[4] = {0.f, 0.f, 0.f, 0.f};
    __syncthreads();

    // lambda_hat0 = L^T lambda0
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        lam[u] = 0.f;
        if (valid[u] && g.lambda0) {
            const int a = ao + u;
            const float* Lj = gL + (size_t)jo * n * n;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + jo * n;
            float x = 0.f;
            for (int b = a; b < n; ++b) x += Lj[b * n + a] * l0[b];
            lam[u] = x;
        }
    }
    if (owner) store4(XP, e0, lam);
    __syncthreads();
    if (has_tile) tile_matvec<H>(tile, jb, rt, ct, XP, yr_base, yc_base);
    __syncthreads();
    // r_hat = ghat - S_hat lambda_hat
    float rr = 0.f, gg = 0.f;
    if (owner) ysum4(Y, e0, y);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        r[u] = 0.f;
        if (valid[u]) {
            const int i = gi0 + u;
            r[u] = ghat[i] - lam[u] - y[u];
            rr += r[u] * r[u];
            gg += rule0 ? gam[i] * gam[i] : ghat[i] * ghat[i];
        }
    }
    if (owner) store4(XR, e0, r);
    post2(rr, gg, redB);
    __syncthreads();
    float q = has_tile ? tile_matvec<H>(tile, jb, rt, ct, XR, yr_base, yc_base) : 0.f;
    float lsq = 0.f;
    if (rule0) lsq = lnorm_owned<H>(LP, KS, gL, lsm, XR, jo, ao, n, valid);
    post2(q, lsq, redC);
    __syncthreads();
    float2 sB = collect2(redB), sC = collect2(redC);
    float eta = sB.x - 2.f * sC.x;  // r^T (I - Nhat) r
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : sB.y;
    const float thr = g.eps * g.eps * ref;
    float stopq = g.rule == GATO_STOP_RESIDUAL ? sC.y : (g.rule == GATO_STOP_SCALED ? sB.x : eta);
    bool done = stopq <= thr;
    bool nonfinite = !isfinite(eta) || !isfinite(stopq);
    if (owner) ysum4(Y, e0, y);
#pragma unroll
    for (int u = 0; u < 4; ++u) p[u] = valid[u] ? r[u] - y[u] : 0.f;  // z = (I - Nhat) r
    if (owner) store4(XP, e0, p);
    // exact ||L r_hat|| is evaluated in phase C when the previous iteration's
    // lower bound was within a factor 1.25 of the threshold (the residual
    // shrinks by about 1-2 % per iteration here); should the bound of
    // the current residual fall below the threshold without the exact value,
    // phase D evaluates it there (one extra barrier), so the stopping test is
    // exact in every iteration.
    bool exact_next;
    {
        float lb = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) lb += dl * r[u] * r[u];
        float lbv[1] = {lb};
        block_sum<1>(lbv, reinterpret_cast<float4*>(redD));
        exact_next = rule0 && lbv[0] <= 1.25f * thr;
    }
    __syncthreads();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        // A: Nhat p (tiles) with its partial p^T Nhat p, and p^T p (owners)
        q = has_tile ? tile_matvec<H>(tile, jb, rt, ct, XP, yr_base, yc_base) : 0.f;
        float pp = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) pp += p[u] * p[u];
        post2(q, pp, redA);
        __syncthreads();
        // B: alpha = eta / p^T S_hat p; lambda and r updates (owners)
        const float2 sA = collect2(redA);  // (sum_j p_j^T Nhat_j p_{j-1}, p^T p)
        const float pv = sA.y + 2.f * sA.x;
        const float alpha = __fdividef(eta, pv);
        if (owner) ysum4(Y, e0, y);
#pragma unroll
        for (int u = 0; u < 4; ++u) {
            const float v = p[u] + y[u];
            lam[u] += alpha * p[u];
            r[u] = valid[u] ? r[u] - alpha * v : 0.f;
        }
        if (owner) store4(XR, e0, r);
        __syncthreads();
        // C: Nhat r (tiles) with r^T Nhat r partials; r^T r, the lower bound
        // sum_j lambda_min-bound_j ||r_hat_j||^2 <= ||L r_hat||^2 and, when
        // gated in, ||L r_hat||^2 (owners)
        q = has_tile ? tile_matvec<H>(tile, jb, rt, ct, XR, yr_base, yc_base) : 0.f;
        rr = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) rr += r[u] * r[u];
        float lsq = 0.f;
        const bool exact = exact_next;
        if (exact) lsq = lnorm_owned<H>(LP, KS, gL, lsm, XR, jo, ao, n, valid);
        post4(q, rr, dl * rr, lsq, reinterpret_cast<float4*>(redB));
        __syncthreads();
        // D: eta' = r^T (I - Nhat) r, convergence, p = z + beta p (owners)
        const float4 sBC = collect4(reinterpret_cast<const float4*>(redB));
        sB = make_float2(sBC.x, sBC.y);
        sC = make_float2(sBC.z, sBC.w);
        const float eta_new = sB.y - 2.f * sB.x;
        float lsq_all = sC.y;
        bool have_exact = exact;
        if (rule0 && !exact && sC.x * 0.999f <= thr) {
            // the bound no longer rules convergence out: evaluate ||L r_hat||
            lsq = lnorm_owned<H>(LP, KS, gL, lsm, XR, jo, ao, n, valid);
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
        if (owner) ysum4(Y, e0, y);
#pragma unroll
        for (int u = 0; u < 4; ++u) p[u] = valid[u] ? (r[u] - y[u]) + beta * p[u] : 0.f;
        if (owner) store4(XP, e0, p);
        eta = eta_new;
        __syncthreads();
    }
    __syncthreads();
    if (owner) store4(XP, e0, lam);
    __syncthreads();
    recover_dz<16>(g.w, g.rhs, g.lambda, g.dX, g.dU, sol,
                   [&](int j, int b) { return XP[j * 16 + (b / H) * 8 + b % H]; }, YR0);
    finish(g, sol, it, done, nonfinite);
}

// Persistent: each block takes the next unsolved system from g.queue until
// none is left, so the batch is balanced over the resident blocks instead of
// running in waves that each last as long as their slowest solve.  Every
// solve's arithmetic is independent of which block runs it.
template <int H>
__global__ void __launch_bounds__(512, 1) k_pcg_tile(PcgArgs g)
{
    __shared__ int s_sol;
    for (;;) {
        if (threadIdx.x == 0) s_sol = atomicAdd(g.queue, 1);
        __syncthreads();
        const int sol = s_sol;
        __syncthreads();
        if (sol >= g.w.M) break;
        pcg_tile_solve<H>(g, sol);
    }
}

// ===========================================================================
// wide-tile kernel: two threads per coupling block, ownership aligned with
// the tiles
// ===========================================================================
//
// k_pcg_wide<H> (7 <= n <= 16, N <= 128) runs the same iteration as
// k_pcg_tile<H> with half the threads and about half its shared-memory
// traffic.  Thread t < 2(N-1) holds rows rt*H .. rt*H+H-1 of Nhat_j over all
// 2H columns (j = 1 + t/2, rt = t mod 2) and owns the same rows of knot j:
// its row sums (Nhat_j x_{j-1})_rows are complete and stay in registers, and
// its own part of x never has to be read back.  Only the transposed
// products (Nhat_j^T x_j, partial over the two row halves) go through shared
// memory, to the owners of knot j-1.  Threads 2(N-1) and 2(N-1)+1 own knot 0.
//
// Shared memory (floats): XP, XR [N][24] (a knot's first half at +0, its
// second at +12), YC0, YC1 [N][24] (same layout; YC1 offset by 4 more
// floats), the reduction slots, the eigenvalue bounds and the padded L.
// These strides keep every 128-bit access of an iteration free of bank
// conflicts for N = 16 .. 128.

constexpr int kWS = 24;  // knot stride of the vectors and column sums
constexpr int kWH = 12;  // offset of a knot's second half

template <int H>
struct WideTile {
    float t[H][2 * H];
};

// logical padded position of unpadded column b (< 2H): halves of 8 slots
template <int H>
__host__ __device__ constexpr int pcol(int b)
{
    return b < H ? b : 8 + (b - H);
}

// physical offset of logical slot p within a knot
__host__ __device__ constexpr int wphys(int p) { return p < 8 ? p : kWH + (p - 8); }

// the 16 logical slots of a knot (four float4 chunks at +0, +4, +12, +16)
__device__ __forceinline__ void wload16(const float* X, float (&x)[16])
{
#pragma unroll
    for (int c = 0; c < 4; ++c) {
        const float4 v = *reinterpret_cast<const float4*>(X + wphys(4 * c));
        x[4 * c] = v.x;
        x[4 * c + 1] = v.y;
        x[4 * c + 2] = v.z;
        x[4 * c + 3] = v.w;
    }
}

__device__ __forceinline__ void wload8(const float* X, float (&x)[8])
{
    const float4 a = *reinterpret_cast<const float4*>(X);
    const float4 b = *reinterpret_cast<const float4*>(X + 4);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}

__device__ __forceinline__ void wstore8(float* X, const float (&v)[8])
{
    *reinterpret_cast<float4*>(X) = make_float4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<float4*>(X + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// One product with Nhat for the rows (j, rt) held by this thread: rs gets the
// complete row sums of those rows, the column sums (partial over the row
// halves) go to yc (knot j-1's slots); returns xr^T rs, this thread's share
// of x^T Nhat x.  xprev holds x_{j-1}, xr is the thread's own part of x_j.
template <int H>
__device__ __forceinline__ float wide_matvec(const WideTile<H>& T, const float* xprev,
                                             const float (&xr)[8], float (&rs)[8], float* yc)
{
    float xc[16];
    wload16(xprev, xc);
    float cs[16];
#pragma unroll
    for (int a = 0; a < 8; ++a) rs[a] = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) cs[c] = 0.f;
#pragma unroll
    for (int a = 0; a < H; ++a)
#pragma unroll
        for (int b = 0; b < 2 * H; ++b) {
            const float v = T.t[a][b];
            rs[a] = fmaf(v, xc[pcol<H>(b)], rs[a]);
            cs[pcol<H>(b)] = fmaf(v, xr[a], cs[pcol<H>(b)]);
        }
    float q = 0.f;
#pragma unroll
    for (int a = 0; a < H; ++a) q = fmaf(xr[a], rs[a], q);
#pragma unroll
    for (int c = 0; c < 4; ++c)
        *reinterpret_cast<float4*>(yc + wphys(4 * c)) =
            make_float4(cs[4 * c], cs[4 * c + 1], cs[4 * c + 2], cs[4 * c + 3]);
    return q;
}

// (Nhat x) at the eight owned slots: own row sums plus the two column parts
__device__ __forceinline__ void wide_y(const float (&rs)[8], const float* YC0, const float* YC1,
                                       int off, float (&y)[8])
{
    float c0[8], c1[8];
    wload8(YC0 + off, c0);
    wload8(YC1 + off, c1);
#pragma unroll
    for (int k = 0; k < 8; ++k) y[k] = rs[k] + c0[k] + c1[k];
}

// sum over the owned rows a = half*H + k < n (k < H) of (L_j r_hat_j)_a^2
template <int H>
__device__ __forceinline__ float lnorm_half(const float* LP, int KS, const float* gL, bool lsm,
                                            const float* XR, int j, int half, int n, int owner)
{
    float s = 0.f;
    const float* xk = XR + j * kWS;
    if (lsm) {
        const float4 x0 = *reinterpret_cast<const float4*>(xk);
        const float4 x1 = *reinterpret_cast<const float4*>(xk + 4);
        const float4 x2 = half ? *reinterpret_cast<const float4*>(xk + kWH)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 x3 = half ? *reinterpret_cast<const float4*>(xk + kWH + 4)
                               : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < H; ++k) {
            if (!owner || half * H + k >= n) continue;
            const float4* row =
                reinterpret_cast<const float4*>(LP + j * KS + (half * H + k) * kLS);
            float t = dot4(row[0], x0, 0.f);
            t = dot4(row[1], x1, t);
            if (half) {  // rows of the first half end before column H
                t = dot4(row[2], x2, t);
                t = dot4(row[3], x3, t);
            }
            s = fmaf(t, t, s);
        }
    } else {
        // rows from global memory: the loads of a row are independent, the x
        // values come from the knot's four float4 chunks
        float xs[16];
        wload16(xk, xs);
        const float* Lj = gL + (size_t)j * n * n;
#pragma unroll
        for (int k = 0; k < H; ++k) {
            const int a = half * H + k;
            if (!owner || a >= n) continue;
            const float* row = Lj + a * n;
            float t = 0.f;
#pragma unroll
            for (int b = 0; b < 2 * H; ++b)
                if (b <= a) t = fmaf(row[b], xs[pcol<H>(b)], t);
            s = fmaf(t, t, s);
        }
    }
    return s;
}

template <int H>
__device__ __forceinline__ void pcg_wide_solve(const PcgArgs& g, int sol)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int N = w.N, n = w.n, T = blockDim.x, tid = threadIdx.x;
    const int EX = N * kWS;
    const bool rule0 = g.rule == GATO_STOP_RESIDUAL;
    const bool lsm = rule0 && g.l_smem;
    const int KS = l_knot_stride(n);

    float* XP = sm;
    float* XR = XP + EX;
    float* YC0 = XR + EX;
    float* YC1 = YC0 + EX + 4;
    const int zero_count = 4 * EX + 8;
    float2* redA = reinterpret_cast<float2*>(sm + zero_count);
    float2* redB = redA + 32;
    float2* redC = redA + 64;
    float2* redD = redA + 96;  // also used as float4[16] by block_sum
    float* DL = reinterpret_cast<float*>(redA + 160);
    float* LP = DL + ((N + 3) & ~3);
    if (!gb_smem((size_t)(LP - sm + (lsm ? (size_t)N * KS : 0)) * sizeof(float), w.status,
                 sol)) {
        finish(g, sol, 0, false, false);
        return;  // block-uniform
    }

    for (int i = tid; i < zero_count; i += T) sm[i] = 0.f;
    for (int j = tid; j < N; j += T) DL[j] = w.dlow[sol * w.sN + j];
    const float* gL = w.L + sol * w.sNnn;
    if (lsm) stage_l_rows<H>(LP, KS, gL, N, n);

    // tile rows (block jb, half rt) and the owned slots (knot jo, same half);
    // the tile reads x_{j-1} (knot jb-1's 20 floats) and writes its column
    // sums there, the owner its 8 slots of knot jo
    const int rt = tid & 1;
    const int jb = 1 + (tid >> 1);
    const bool has_tile =
        tid < 2 * (N - 1) && gb_ok((long long)(jb - 1) * kWS + 19, EX, w.status, sol);
    const bool owner =
        tid < 2 * N && gb_ok((long long)(tid < 2 * (N - 1) ? jb : 0) * kWS + (tid & 1) * kWH + 7,
                             EX, w.status, sol);
    const int jo = has_tile ? jb : 0;
    const int half = rt;
    float* yc_base = rt ? YC1 : YC0;
    WideTile<H> tile;
    {
        const float* blk = w.Nh + sol * w.sKnn + (size_t)(has_tile ? jb - 1 : 0) * n * n;
#pragma unroll
        for (int a = 0; a < H; ++a)
#pragma unroll
            for (int b = 0; b < 2 * H; ++b) {
                const int ra = rt * H + a;
                tile.t[a][b] = (has_tile && ra < n && b < n) ? blk[ra * n + b] : 0.f;
            }
    }
    const int xo = jo * kWS + half * kWH;  // owned slots in XP / XR / YC
    const int pj = (has_tile ? jb - 1 : 0) * kWS;  // knot j-1 of the tile rows
    float* yc = yc_base + pj;
    bool valid[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) valid[k] = owner && k < H && half * H + k < n;
    const int gi0 = jo * n + half * H;  // unpadded index of owned slot k is gi0 + k
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float dl = owner ? DL[jo] : 0.f;
    // slots past n (and all slots of a thread that owns none) start at zero
    // and stay exactly zero: the padded rows and columns of the tiles are
    // zero, so the loop needs no masks
    float lam[8], r[8], p[8], y[8], rs[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) rs[k] = y[k] = 0.f;
    __syncthreads();

    // lambda_hat0 = L^T lambda0
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        lam[k] = 0.f;
        if (valid[k] && g.lambda0) {
            const int a = half * H + k;
            const float* Lj = gL + (size_t)jo * n * n;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + jo * n;
            float x = 0.f;
            for (int b = a; b < n; ++b) x += Lj[b * n + a] * l0[b];
            lam[k] = x;
        }
    }
    if (owner) wstore8(XP + xo, lam);
    __syncthreads();
    if (has_tile) wide_matvec<H>(tile, XP + pj, lam, rs, yc);
    __syncthreads();
    // r_hat = ghat - S_hat lambda_hat
    float rr = 0.f, gg = 0.f;
    if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        r[k] = 0.f;
        if (valid[k]) {
            const int i = gi0 + k;
            r[k] = ghat[i] - lam[k] - y[k];
            rr += r[k] * r[k];
            gg += rule0 ? gam[i] * gam[i] : ghat[i] * ghat[i];
        }
    }
    if (owner) wstore8(XR + xo, r);
    post2(rr, gg, redB);
    __syncthreads();  // XR complete; the column sums of lambda are read
    float q = has_tile ? wide_matvec<H>(tile, XR + pj, r, rs, yc) : 0.f;
    float lsq = 0.f;
    if (rule0) lsq = lnorm_half<H>(LP, KS, gL, lsm, XR, jo, half, n, owner);
    post2(q, lsq, redC);
    __syncthreads();
    float2 sB = collect2(redB), sC = collect2(redC);
    float eta = sB.x - 2.f * sC.x;  // r^T (I - Nhat) r
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : sB.y;
    const float thr = g.eps * g.eps * ref;
    float stopq = g.rule == GATO_STOP_RESIDUAL ? sC.y : (g.rule == GATO_STOP_SCALED ? sB.x : eta);
    bool done = stopq <= thr;
    bool nonfinite = !isfinite(eta) || !isfinite(stopq);
    if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k] = r[k] - y[k];  // z = (I - Nhat) r
    if (owner) wstore8(XP + xo, p);
    // the exact ||L r_hat|| is gated as in k_pcg_tile
    bool exact_next;
    {
        float lb = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) lb += dl * r[k] * r[k];
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
        q = has_tile ? wide_matvec<H>(tile, XP + pj, p, rs, yc) : 0.f;
        float pp = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) pp = fmaf(p[k], p[k], pp);
        post2(q, pp, redA);
        __syncthreads();
        // B: alpha = eta / p^T S_hat p; lambda and r updates
        const float2 sA = collect2(redA);
        const float pv = sA.y + 2.f * sA.x;
        const float alpha = __fdividef(eta, pv);
        if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float v = p[k] + y[k];
            lam[k] = fmaf(alpha, p[k], lam[k]);
            r[k] = fmaf(-alpha, v, r[k]);
        }
        if (owner) wstore8(XR + xo, r);
        __syncthreads();
        // C: Nhat r; r^T Nhat r and r^T r partials, the lower bound and, when
        // gated in, ||L r_hat||^2
        q = has_tile ? wide_matvec<H>(tile, XR + pj, r, rs, yc) : 0.f;
        rr = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) rr = fmaf(r[k], r[k], rr);
        float lsq = 0.f;
        const bool exact = exact_next;
        if (exact) lsq = lnorm_half<H>(LP, KS, gL, lsm, XR, jo, half, n, owner);
        // two post2 calls: one post4 (the same sums) measured about 1% slower here
        post2(q, rr, redB);
        post2(dl * rr, lsq, redC);
        __syncthreads();
        // D: eta' = r^T (I - Nhat) r, convergence, p = z + beta p
        sB = collect2(redB);
        sC = collect2(redC);
        const float eta_new = sB.y - 2.f * sB.x;
        float lsq_all = sC.y;
        bool have_exact = exact;
        if (rule0 && !exact && sC.x * 0.999f <= thr) {
            lsq = lnorm_half<H>(LP, KS, gL, lsm, XR, jo, half, n, owner);
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
        if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
        for (int k = 0; k < 8; ++k) p[k] = fmaf(beta, p[k], r[k] - y[k]);
        if (owner) wstore8(XP + xo, p);
        eta = eta_new;
        __syncthreads();
    }
    __syncthreads();
    if (owner) wstore8(XP + xo, lam);
    __syncthreads();
    recover_dz<16>(g.w, g.rhs, g.lambda, g.dX, g.dU, sol,
                   [&](int j, int b) { return XP[j * kWS + wphys(pcol<H>(b))]; }, YC0);
    finish(g, sol, it, done, nonfinite);
}

template <int H>
__global__ void __launch_bounds__(256, 1) k_pcg_wide(PcgArgs g)
{
    __shared__ int s_sol;
    for (;;) {
        if (threadIdx.x == 0) s_sol = atomicAdd(g.queue, 1);
        __syncthreads();
        const int sol = s_sol;
        __syncthreads();
        if (sol >= g.w.M) break;
        pcg_wide_solve<H>(g, sol);
    }
}

// ===========================================================================
// cluster kernel: one solve across the CTAs of a thread-block cluster
// ===========================================================================
//
// k_pcg_cluster<H, C> (7 <= n <= 16, 128 < N <= 128 C) runs the wide-tile
// iteration with a solve's knots split over the C CTAs of a cluster: CTA c
// holds knots c*Nc .. c*Nc+Nc-1 (Nc = ceil(N / C)), their rows of Nhat and
// the owned vector slots, exactly as k_pcg_wide does for a whole solve.  Only
// a CTA's first block (j = c*Nc, c >= 1) reaches across: it reads x_{j-1}
// from CTA c-1's shared memory and writes its transposed product there
// (distributed shared memory).  Block sums add every CTA's warp slots in rank
// order, so all CTAs hold the same scalars and take the same branches; every
// phase barrier is a cluster barrier.

// post2's pair pushed into slot rank * 8 + w of every CTA of the cluster (at
// most eight warps a CTA and four CTAs: the 32 slots of a buffer), stored
// before the cluster barrier that publishes it, so that the collect reads
// only local shared memory; every lane of a half-warp holds its half's total
template <int C>
__device__ __forceinline__ void cluster_post2(cg::cluster_group& cl, float a, float b,
                                              float2* buf)
{
    static_assert(C <= 4, "32 slots hold four CTAs of at most eight warps");
    const int lane = lane_id();
    const bool hi = lane & 16;
    float keep = hi ? b : a;
    keep += __shfl_xor_sync(0xffffffffu, hi ? a : b, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    const int rk = lane & 15, rank = (int)cl.block_rank();
    if (rk < C) {
        float2* dst = rk == rank ? buf : cl.map_shared_rank(buf, rk);
        reinterpret_cast<float*>(dst + rank * 8 + (int)(threadIdx.x >> 5))[hi ? 1 : 0] = keep;
    }
}

// the pushed pairs of every CTA, each CTA's warps in collect2's tree, the
// CTAs added in rank order (the same bits in every CTA)
template <int C>
__device__ __forceinline__ float2 cluster_collect2(const float2* buf)
{
    float2 s = make_float2(0.f, 0.f);
#pragma unroll
    for (int rk = 0; rk < C; ++rk) {
        const float2 v = collect2(buf + rk * 8);
        s.x += v.x;
        s.y += v.y;
    }
    return s;
}

template <int H, int C>
__device__ __forceinline__ void pcg_cluster_solve(const PcgArgs& g)
{
    extern __shared__ __align__(16) float sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int sol = blockIdx.x / C;
    const Work& w = g.w;
    const int N = w.N, n = w.n, T = blockDim.x, tid = threadIdx.x;
    const int Nc = (N + C - 1) / C;
    const int k0 = rank * Nc;          // first knot of this CTA
    const int nk = min(Nc, N - k0);    // its knot count (>= 1)
    const int EX = Nc * kWS;
    const bool rule0 = g.rule == GATO_STOP_RESIDUAL;
    const bool lsm = rule0 && g.l_smem;
    const int KS = l_knot_stride(n);

    float* XP = sm;
    float* XR = XP + EX;
    float* YC0 = XR + EX;
    float* YC1 = YC0 + EX + 4;
    const int zero_count = 4 * EX + 8;
    float2* redA = reinterpret_cast<float2*>(sm + zero_count);
    float2* redB = redA + 32;
    float2* redC = redA + 64;
    float2* redD = redA + 96;
    float* DL = reinterpret_cast<float*>(redA + 160);
    float* LP = DL + ((Nc + 3) & ~3);
    // the layout is the same in every CTA of the cluster, so they all leave
    // together (no cluster barrier is left waiting)
    if (!gb_smem((size_t)(LP - sm + (lsm ? (size_t)Nc * KS : 0)) * sizeof(float), w.status,
                 sol)) {
        if (rank == 0) finish(g, sol, 0, false, false);
        return;
    }

    for (int i = tid; i < zero_count; i += T) sm[i] = 0.f;
    for (int jl = tid; jl < nk; jl += T) DL[jl] = w.dlow[sol * w.sN + k0 + jl];
    const float* gL = w.L + sol * w.sNnn;
    if (lsm) stage_l_rows<H>(LP, KS, gL + (size_t)k0 * n * n, nk, n);

    // thread: local knot jl, row half rt; block j = k0 + jl when j >= 1
    const int jl = tid >> 1, rt = tid & 1, half = rt;
    const bool owner = jl < nk && gb_ok((long long)jl * kWS + half * kWH + 7, EX, w.status, sol);
    const int j = k0 + jl;
    const bool has_tile = owner && j >= 1;
    float* yc_base = rt ? YC1 : YC0;
    WideTile<H> tile;
    {
        const float* blk = w.Nh + sol * w.sKnn + (size_t)(has_tile ? j - 1 : 0) * n * n;
#pragma unroll
        for (int a = 0; a < H; ++a)
#pragma unroll
            for (int b = 0; b < 2 * H; ++b) {
                const int ra = rt * H + a;
                tile.t[a][b] = (has_tile && ra < n && b < n) ? blk[ra * n + b] : 0.f;
            }
    }
    // x_{j-1} and the slots for block j's column sums: local knot jl-1, or
    // the last knot of CTA rank-1 for the CTA's first block
    const bool edge = has_tile && jl == 0;
    const int pj = edge ? (Nc - 1) * kWS : (has_tile ? (jl - 1) * kWS : 0);
    const float* xpp = (edge ? cl.map_shared_rank(XP, rank - 1) : XP) + pj;
    const float* xrp = (edge ? cl.map_shared_rank(XR, rank - 1) : XR) + pj;
    float* yc = (edge ? cl.map_shared_rank(yc_base, rank - 1) : yc_base) + pj;

    const int xo = (owner ? jl : 0) * kWS + half * kWH;
    bool valid[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) valid[k] = owner && k < H && half * H + k < n;
    const int gi0 = (owner ? j : 0) * n + half * H;
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float dl = owner ? DL[jl] : 0.f;
    // slots past n (and all slots of a thread that owns none) start at zero
    // and stay exactly zero, as in k_pcg_wide
    float lam[8], r[8], p[8], y[8], rs[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) rs[k] = y[k] = 0.f;
    cl.sync();

    // lambda_hat0 = L^T lambda0
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        lam[k] = 0.f;
        if (valid[k] && g.lambda0) {
            const int a = half * H + k;
            const float* Lj = gL + (size_t)j * n * n;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + (size_t)j * n;
            float x = 0.f;
            for (int b = a; b < n; ++b) x += Lj[b * n + a] * l0[b];
            lam[k] = x;
        }
    }
    if (owner) wstore8(XP + xo, lam);
    cl.sync();
    if (has_tile) wide_matvec<H>(tile, xpp, lam, rs, yc);
    cl.sync();
    float rr = 0.f, gg = 0.f;
    if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        r[k] = 0.f;
        if (valid[k]) {
            const int i = gi0 + k;
            r[k] = ghat[i] - lam[k] - y[k];
            rr += r[k] * r[k];
            gg += rule0 ? gam[i] * gam[i] : ghat[i] * ghat[i];
        }
    }
    if (owner) wstore8(XR + xo, r);
    cluster_post2<C>(cl, rr, gg, redB);
    cl.sync();
    float q = has_tile ? wide_matvec<H>(tile, xrp, r, rs, yc) : 0.f;
    float lsq = 0.f;
    if (rule0 && owner) lsq = lnorm_half<H>(LP, KS, gL + (size_t)k0 * n * n, lsm, XR, jl, half, n,
                                            owner);
    cluster_post2<C>(cl, q, lsq, redC);
    cl.sync();
    float2 sB = cluster_collect2<C>(redB), sC = cluster_collect2<C>(redC);
    float eta = sB.x - 2.f * sC.x;
    const float ref = g.rule == GATO_STOP_PRECOND ? eta : sB.y;
    const float thr = g.eps * g.eps * ref;
    float stopq = g.rule == GATO_STOP_RESIDUAL ? sC.y : (g.rule == GATO_STOP_SCALED ? sB.x : eta);
    bool done = stopq <= thr;
    bool nonfinite = !isfinite(eta) || !isfinite(stopq);
    if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
    for (int k = 0; k < 8; ++k) p[k] = r[k] - y[k];
    if (owner) wstore8(XP + xo, p);
    bool exact_next;
    {
        float lb = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) lb += dl * r[k] * r[k];
        cluster_post2<C>(cl, lb, 0.f, redD);
        cl.sync();
        exact_next = rule0 && cluster_collect2<C>(redD).x <= 1.25f * thr;
    }
    cl.sync();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        // A: Nhat p, p^T Nhat p and p^T p partials
        q = has_tile ? wide_matvec<H>(tile, xpp, p, rs, yc) : 0.f;
        float pp = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) pp = fmaf(p[k], p[k], pp);
        cluster_post2<C>(cl, q, pp, redA);
        cl.sync();
        // B: alpha; lambda and r updates
        const float2 sA = cluster_collect2<C>(redA);
        const float pv = sA.y + 2.f * sA.x;
        const float alpha = __fdividef(eta, pv);
        if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float v = p[k] + y[k];
            lam[k] = fmaf(alpha, p[k], lam[k]);
            r[k] = fmaf(-alpha, v, r[k]);
        }
        if (owner) wstore8(XR + xo, r);
        cl.sync();
        // C: Nhat r; r^T Nhat r, r^T r, the bound and (gated) ||L r_hat||^2
        q = has_tile ? wide_matvec<H>(tile, xrp, r, rs, yc) : 0.f;
        rr = 0.f;
#pragma unroll
        for (int k = 0; k < 8; ++k) rr = fmaf(r[k], r[k], rr);
        float lsq = 0.f;
        const bool exact = exact_next;
        if (exact && owner)
            lsq = lnorm_half<H>(LP, KS, gL + (size_t)k0 * n * n, lsm, XR, jl, half, n, owner);
        cluster_post2<C>(cl, q, rr, redB);
        cluster_post2<C>(cl, dl * rr, lsq, redC);
        cl.sync();
        // D: eta', convergence, p = z + beta p
        sB = cluster_collect2<C>(redB);
        sC = cluster_collect2<C>(redC);
        const float eta_new = sB.y - 2.f * sB.x;
        float lsq_all = sC.y;
        bool have_exact = exact;
        if (rule0 && !exact && sC.x * 0.999f <= thr) {
            lsq = owner ? lnorm_half<H>(LP, KS, gL + (size_t)k0 * n * n, lsm, XR, jl, half, n,
                                        owner)
                        : 0.f;
            cluster_post2<C>(cl, lsq, 0.f, redD);
            cl.sync();
            lsq_all = cluster_collect2<C>(redD).x;
            have_exact = true;
        }
        stopq = g.rule == GATO_STOP_RESIDUAL ? lsq_all
                                             : (g.rule == GATO_STOP_SCALED ? sB.y : eta_new);
        if (!isfinite(eta_new + pv + stopq + sC.x)) {
            nonfinite = true;
            break;
        }
        done = (!rule0 || have_exact) && stopq <= thr;
        if (done) break;
        exact_next = rule0 && sC.x <= 1.25f * thr;
        const float beta = __fdividef(eta_new, eta);
        if (owner) wide_y(rs, YC0, YC1, xo, y);
#pragma unroll
        for (int k = 0; k < 8; ++k) p[k] = fmaf(beta, p[k], r[k] - y[k]);
        if (owner) wstore8(XP + xo, p);
        eta = eta_new;
        cl.sync();
    }
    cl.sync();
    if (owner) wstore8(XP + xo, lam);
    cl.sync();
    cluster_recover(cl, g, sol, k0, nk,
                    [&](int kl, int b) { return XP[kl * kWS + wphys(pcol<H>(b))]; });
    if (rank == 0) finish(g, sol, it, done, nonfinite);
}

template <int H, int C>
__global__ void __launch_bounds__(256, 1) k_pcg_cluster(PcgArgs g)
{
    pcg_cluster_solve<H, C>(g);
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------

size_t generic_smem_bytes(const Work& w, int nh_smem, int l_smem)
{
    const size_t n = w.n, N = w.N;
    size_t f = 0;
    if (nh_smem) f += round4((N - 1) * n * n);
    if (l_smem) f += round4(N * (n * (n + 1) / 2));
    f += 4 * round4(N * n);  // lambda_hat, r_hat, p, v
    f += 64 * 4;             // two float4[32] reduction buffers
    return f * sizeof(float);
}

size_t wide_smem_bytes(const Work& w, int l_smem, int knots = 0)
{
    const size_t n = w.n, N = knots ? knots : w.N;
    size_t f = 4 * kWS * N + 8;  // XP, XR, YC0/1
    f += 5 * 32 * 2;            // five float2[32] reduction buffers
    f += round4(N);             // DL
    if (l_smem) f += N * (size_t)l_knot_stride((int)n);
    return f * sizeof(float);
}

size_t tile_smem_bytes(const Work& w, int l_smem)
{
    const size_t n = w.n, N = w.N;
    size_t f = 6 * 16 * N + 12;  // XP, XR, YR0/1, YC0/1
    f += 5 * 32 * 2;        // five float2[32] reduction buffers
    f += round4(N);         // DL
    if (l_smem) f += N * (size_t)l_knot_stride((int)n);
    return f * sizeof(float);
}

template <typename K>
cudaError_t launch_k(K kernel, const PcgArgs& a, int T, size_t smem, cudaStream_t st)
{
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kernel<<<a.w.M, T, smem, st>>>(a);
    return cudaGetLastError();
}

// persistent launch: as many blocks as can be resident, at most one per solve
template <typename K>
cudaError_t launch_persistent(K kernel, const PcgArgs& a, int T, size_t smem, int num_sms,
                              cudaStream_t st)
{
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    int per_sm = 0;
    cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, T, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorInvalidConfiguration;
    long grid = (long)per_sm * num_sms;
    if (grid > a.w.M) grid = a.w.M;
    e = cudaMemsetAsync(a.queue, 0, sizeof(int), st);
    if (e != cudaSuccess) return e;
    kernel<<<(unsigned)grid, T, smem, st>>>(a);
    return cudaGetLastError();
}

// one solve per cluster of C CTAs (grid M C); cudaErrorInvalidConfiguration
// when no such cluster fits on the device
template <typename K>
cudaError_t launch_cluster(K kernel, const PcgArgs& a, int C, int T, size_t smem,
                           cudaStream_t st)
{
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
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

}  // namespace

namespace {

// blocks of a kernel an SM can hold with T threads and smem bytes of dynamic
// shared memory; 0 on error.  Above 48 KB the opt-in is raised first, as for
// a launch; it is never set below 48 KB, which every launch of at most 48 KB
// relies on without setting it
template <typename K>
int blocks_per_sm(K kernel, int T, size_t smem)
{
    int per_sm = 0;
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, T, smem);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return per_sm;
}

int wide_blocks_per_sm(int H, int T, size_t smem)
{
    switch (H) {
        case 4: return blocks_per_sm(k_pcg_wide<4>, T, smem);
        case 5: return blocks_per_sm(k_pcg_wide<5>, T, smem);
        case 6: return blocks_per_sm(k_pcg_wide<6>, T, smem);
        case 7: return blocks_per_sm(k_pcg_wide<7>, T, smem);
        case 8: return blocks_per_sm(k_pcg_wide<8>, T, smem);
        default: return 0;
    }
}

// The automatic choice between the wide-tile and the quad kernel: the quad
// kernel where the wide one would leave each SM at most four working warps
// (a solve's 2N threads, times the solves an SM holds: those of the whole
// concurrent batch per SM, at most the wide kernel's occupancy).  There the
// quad's twice as many warps hide latency that the few wide warps leave
// exposed (3 to 42 % less time per PCG solve measured for n = 12, 14, 16 and
// N = 16 .. 64); with eight or more working warps per SM the quad's 1.5 times
// as many instructions make it up to 13 % slower.
bool quad_preferred(const gato_handle* h, int H, int Tw, size_t smem_wide)
{
    const Work& w = h->w;
    // at n = 12 (three unpadded rows per lane, both exchanges select-free) the
    // quad kernel measured faster at every horizon and batch swept (N = 16 ..
    // 128, 16 .. 1024 solves: 0.5 to 30 % less time)
    if (w.n == 12) return true;
    const int conc = h->batch_M > 0 ? h->batch_M : w.M;
    int per_sm = (conc + h->num_sms - 1) / h->num_sms;
    const int occ = wide_blocks_per_sm(H, Tw, smem_wide);
    if (occ < 1) return false;
    if (per_sm > occ) per_sm = occ;
    const int warps_per_solve = (2 * w.N + 31) / 32;
    return warps_per_solve * per_sm <= 4;
}

}  // namespace

// Solves a PCG launch over the handle's whole batch holds at once: for the
// fp32 kernels at 7 <= n <= 16, N <= 128 the wide-tile kernel's resident
// blocks per SM times the SMs (the quad kernel the automatic rule may take
// instead holds at least as many), otherwise one solve per SM (the
// register-row, double-float and generic kernels hold one at the sizes they
// serve).
int pcg_solves_per_wave(const gato_handle* h, const gato_params* p)
{
    const Work& w = h->w;
    const int kind = h->pcg_kernel;
    if (p && p->pcg_precision != GATO_PCG_PRECISION_FF && w.n >= 7 && w.n <= 16 &&
        w.N <= 128 &&
        (kind == GATO_PCG_AUTO || kind == GATO_PCG_WIDE || kind == GATO_PCG_QUAD)) {
        int Tw = ((2 * w.N + 31) / 32) * 32;
        if (Tw < 64) Tw = 64;
        const size_t limit = (size_t)h->smem_optin;
        size_t smem = wide_smem_bytes(w, p->stop_rule == GATO_STOP_RESIDUAL);
        if (smem > limit) smem = wide_smem_bytes(w, 0);
        if (Tw <= 256 && smem <= limit) {
            const int occ = wide_blocks_per_sm((w.n + 1) / 2, Tw, smem);
            if (occ > 0) return occ * h->num_sms;
        }
    }
    return h->num_sms;
}

// launches the PCG kernel for these sizes and parameters; ran gets its
// GATO_PCG_* value
static cudaError_t launch_pcg_pick(gato_handle* h, const gato_params* p, int set,
                                   const float* lambda0, float* lambda, float* dX, float* dU,
                                   int32_t* iters, int acc_iters, uint32_t* status,
                                   cudaStream_t st, int& ran)
{
    const Work& w = h->w;
    PcgArgs a;
    a.w = w;
    a.rhs = w.rhs[set];
    a.lambda0 = lambda0;
    a.lambda = lambda;
    a.dX = dX;
    a.dU = dU;
    a.iters = iters;
    a.status = status;
    a.eps = p->pcg_eps;
    a.max_iters = p->pcg_max_iters;
    a.rule = p->stop_rule;
    a.acc_iters = acc_iters;
    a.queue = w.queue;
    const size_t limit = (size_t)h->smem_optin;
    const int want_l = p->stop_rule == GATO_STOP_RESIDUAL;

    // double-float arithmetic (pcg_ff.cu) when asked for; sizes beyond that
    // kernel are rejected rather than solved at a lower precision
    if (p->pcg_precision == GATO_PCG_PRECISION_FF) {
        a.nh_smem = 0;
        a.l_smem = 0;
        ran = GATO_PCG_DOUBLE_FLOAT;
        return launch_pcg_ff(a, limit, h->num_sms, st);
    }

    const int H = (w.n + 1) / 2;
    const bool tiled_n = w.n >= 7 && w.n <= 16;

    // wide-tile kernel: two threads per coupling block
    int Tw = ((2 * w.N + 31) / 32) * 32;
    if (Tw < 64) Tw = 64;
    int kind = h->pcg_kernel;
    // register-row kernel (pcg_rows.cu): the default for 16 < n <= 64 where its
    // block fits, any n <= 64 when chosen; where it does not fit, as AUTO
    if (kind == GATO_PCG_ROWS || (kind == GATO_PCG_AUTO && w.n > 16)) {
        ran = GATO_PCG_ROWS;
        cudaError_t e = launch_pcg_rows(a, limit, st);
        if (e != cudaErrorInvalidConfiguration) return e;
        kind = GATO_PCG_AUTO;
    }
    if ((kind == GATO_PCG_AUTO || kind == GATO_PCG_WIDE || kind == GATO_PCG_QUAD) && tiled_n &&
        Tw <= 256) {
        a.nh_smem = 0;
        a.l_smem = want_l;
        size_t smem = wide_smem_bytes(w, a.l_smem);
        if (smem > limit) {
            a.l_smem = 0;
            smem = wide_smem_bytes(w, 0);
        }
        // quad kernel (pcg_quad.cu): four threads per coupling block, when
        // chosen or by the automatic rule above
        if (kind == GATO_PCG_QUAD ||
            (kind == GATO_PCG_AUTO && smem <= limit && quad_preferred(h, H, Tw, smem))) {
            ran = GATO_PCG_QUAD;
            cudaError_t e = launch_pcg_quad(a, limit, h->num_sms, st);
            if (e != cudaErrorInvalidConfiguration) return e;
        }
        ran = GATO_PCG_WIDE;
        if (smem <= limit) {
            switch (H) {
                case 4: return launch_persistent(k_pcg_wide<4>, a, Tw, smem, h->num_sms, st);
                case 5: return launch_persistent(k_pcg_wide<5>, a, Tw, smem, h->num_sms, st);
                case 6: return launch_persistent(k_pcg_wide<6>, a, Tw, smem, h->num_sms, st);
                case 7: return launch_persistent(k_pcg_wide<7>, a, Tw, smem, h->num_sms, st);
                case 8: return launch_persistent(k_pcg_wide<8>, a, Tw, smem, h->num_sms, st);
                default: break;
            }
        }
    }

    // cluster kernel: 128 < N <= 512, the solve split over 2 or 4 CTAs
    if ((kind == GATO_PCG_AUTO || kind == GATO_PCG_WIDE) && tiled_n && w.N > 128 &&
        w.N <= 512) {
        const int C = w.N <= 256 ? 2 : 4;
        const int Nc = (w.N + C - 1) / C;
        int Tc = ((2 * Nc + 31) / 32) * 32;
        if (Tc < 64) Tc = 64;
        a.nh_smem = 0;
        a.l_smem = want_l;
        size_t smem = wide_smem_bytes(w, a.l_smem, Nc);
        if (smem > limit) {
            a.l_smem = 0;
            smem = wide_smem_bytes(w, 0, Nc);
        }
        if (smem <= limit) {
            ran = GATO_PCG_CLUSTER;
            cudaError_t e = cudaErrorInvalidConfiguration;
            switch (H * 8 + C) {
#define GATO_CLUSTER_CASE(HH, CC)                                                    \
                case HH * 8 + CC:                                                    \
                    e = launch_cluster(k_pcg_cluster<HH, CC>, a, CC, Tc, smem, st); \
                    break;
                GATO_CLUSTER_CASE(4, 2) GATO_CLUSTER_CASE(4, 4)
                GATO_CLUSTER_CASE(5, 2) GATO_CLUSTER_CASE(5, 4)
                GATO_CLUSTER_CASE(6, 2) GATO_CLUSTER_CASE(6, 4)
                GATO_CLUSTER_CASE(7, 2) GATO_CLUSTER_CASE(7, 4)
                GATO_CLUSTER_CASE(8, 2) GATO_CLUSTER_CASE(8, 4)
#undef GATO_CLUSTER_CASE
                default: break;
            }
            // a cluster that cannot be placed falls through to the generic kernel
            if (e != cudaErrorInvalidConfiguration) return e;
        }
    }

    // register-tiled kernel: 7 <= n <= 16, four threads per coupling block
    int T = ((4 * w.N + 31) / 32) * 32;
    if (T < 64) T = 64;
    if (kind != GATO_PCG_GENERIC && tiled_n && T <= 512) {
        a.nh_smem = 0;
        a.l_smem = want_l;
        size_t smem = tile_smem_bytes(w, a.l_smem);
        if (smem > limit) {
            a.l_smem = 0;
            smem = tile_smem_bytes(w, 0);
        }
        if (smem <= limit) {
            ran = GATO_PCG_TILE;
            switch (H) {
                case 4: return launch_persistent(k_pcg_tile<4>, a, T, smem, h->num_sms, st);
                case 5: return launch_persistent(k_pcg_tile<5>, a, T, smem, h->num_sms, st);
                case 6: return launch_persistent(k_pcg_tile<6>, a, T, smem, h->num_sms, st);
                case 7: return launch_persistent(k_pcg_tile<7>, a, T, smem, h->num_sms, st);
                case 8: return launch_persistent(k_pcg_tile<8>, a, T, smem, h->num_sms, st);
                default: break;
            }
        }
    }

    // generic kernel
    a.nh_smem = 1;
    a.l_smem = want_l;
    size_t smem = generic_smem_bytes(w, a.nh_smem, a.l_smem);
    if (smem > limit && want_l) {
        a.l_smem = 0;
        smem = generic_smem_bytes(w, a.nh_smem, a.l_smem);
    }
    if (smem > limit) {
        a.nh_smem = 0;
        smem = generic_smem_bytes(w, a.nh_smem, a.l_smem);
    }
    if (smem > limit) return cudaErrorInvalidConfiguration;
    ran = GATO_PCG_GENERIC;
    const int Nn = w.N * w.n;
    T = ((Nn + 1) / 2 + 31) / 32 * 32;
    if (T < 64) T = 64;
    if (T > 512) T = 512;
    return launch_k(k_pcg_generic, a, T, smem, st);
}

// the kernel is recorded for gato_stats: pcg_kernel for a main solve (set 0),
// refine_kernel for a correction (set 1)
cudaError_t launch_pcg_ex(gato_handle* h, const gato_params* p, int set, const float* lambda0,
                          float* lambda, float* dX, float* dU, int32_t* iters, int acc_iters,
                          uint32_t* status, cudaStream_t st)
{
    int ran = 0;
    const cudaError_t e = launch_pcg_pick(h, p, set, lambda0, lambda, dX, dU, iters, acc_iters,
                                          status, st, ran);
    if (e == cudaSuccess) (set == 0 ? h->pcg_ran : h->refine_ran) = ran;
    return e;
}

cudaError_t launch_pcg(gato_handle* h, const gato_params* p, const float* lambda0,
                       float* lambda, float* dX, float* dU, int32_t* iters,
                       uint32_t* status, cudaStream_t st)
{
    return launch_pcg_ex(h, p, 0, lambda0, lambda, dX, dU, iters, 0, status, st);
}

}  // namespace gato
