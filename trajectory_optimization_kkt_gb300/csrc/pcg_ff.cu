// pcg_ff.cu -- batched PCG on S lambda = gamma with the symmetric stair
// preconditioner in double-float arithmetic, and recovery of dz (GATO paper,
// Sec. II and eq. (4): PCG refines lambda up to the tolerance eps; Sec. III:
// one thread block per linear system, block-tridiagonal products, block
// reductions).
//
// Why: the iteration count of CG in finite precision grows as the rounding
// unit grows (the computed residuals lose their orthogonality and the
// method re-explores converged directions).  On the horizons and conditioning
// of the benchmark problems with stated iteration caps, fp32 PCG needs
// 3-25 % more iterations than fp64 PCG to reach a relative residual of 1e-6,
// and every fp32 rounding in the iteration (the product's input, its
// accumulation, its output, the vector updates and the inner products)
// contributes on its own: the count falls by about one iteration per extra
// significand bit.  This kernel carries the vectors, the products' sums, the
// inner products and the CG scalars as double-float values (about 48 bits);
// the operator (the scaled coupling blocks Nhat_j, formed in fp32) and the
// right-hand side stay as formed.  Its iterates are those of the fp32
// kernels' iteration (same variables, same recurrence, same stopping rules),
// computed more accurately.
//
// The iteration runs in the block-Jacobi-scaled variables lambda_hat =
// L^T lambda, where S_hat = I + Nhat and the stair preconditioner is I - Nhat
// (see pcg.cu).  Thread t owns the rows t, t + T, ... (R of them) of the
// solve's N n rows; row a of knot j needs row a of Nhat_j (times x_{j-1}) and
// column a of Nhat_{j+1} (times x_{j+1}), read from one copy of the blocks in
// shared memory framed by two zero blocks, so that the first and last knot
// need no branch.  The vectors p and r live in shared memory as high and low
// arrays with a guard knot of zeros at each end.  Four block barriers per
// iteration, as in the fp32 kernels; every block reduction sums the warps'
// double-float partials in a fixed order, so results do not depend on
// scheduling.
#include "ff.cuh"
#include "pcg_common.cuh"

namespace gato {
namespace {

constexpr int kFFMaxThreads = 1024;
// rows per CTA from which a solve is split over a cluster of two CTAs: measured
// on workload 2's sizes (448 rows per CTA) the split saves a quarter of the
// solve, with 56 rows per CTA (four CTAs at N = 16, n = 14) it costs 14 %
constexpr int kFFClusterRows = 256;

// (Nhat x)_a for row a of knot j: row a of Nhat_j times x_{j-1} plus column a
// of Nhat_{j+1} times x_{j+1}, two compensated chains.  NB holds the blocks
// (block j at NB + j n^2: zero, Nhat_1 .. Nhat_{N-1}, zero), XH / XL the
// vector with knot j at (j + 1) NP.
template <int NP>
__device__ __forceinline__ ff ff_row(const float* NB, int n, int nn, int j, int a,
                                     const float* XH, const float* XL)
{
    const float* lo = NB + (size_t)j * nn + a * n;
    const float* up = NB + (size_t)(j + 1) * nn + a;
    const float4* mh = reinterpret_cast<const float4*>(XH + j * NP);
    const float4* ml = reinterpret_cast<const float4*>(XL + j * NP);
    const float4* ph = reinterpret_cast<const float4*>(XH + (j + 2) * NP);
    const float4* pl = reinterpret_cast<const float4*>(XL + (j + 2) * NP);
    Dot2 c1, c2;
#pragma unroll
    for (int q = 0; q < NP / 4; ++q) {
        const float4 a4 = mh[q], b4 = ml[q], c4 = ph[q], d4 = pl[q];
        const float xmh[4] = {a4.x, a4.y, a4.z, a4.w};
        const float xml[4] = {b4.x, b4.y, b4.z, b4.w};
        const float xph[4] = {c4.x, c4.y, c4.z, c4.w};
        const float xpl[4] = {d4.x, d4.y, d4.z, d4.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int b = 4 * q + e;
            if (b < n) {
                c1.add(lo[b], xmh[e], xml[e]);
                c2.add(up[b * n], xph[e], xpl[e]);
            }
        }
    }
    return ff_add(c1.value(), c2.value());
}

// sum over the block of one double-float and two floats per thread; every
// thread returns the totals (fixed order: the warps' butterflies, then one
// butterfly over the warp slots)
__device__ __forceinline__ void ff_warp_reduce(ff& v, float& f1, float& f2)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const ff u{__shfl_xor_sync(0xffffffffu, v.h, o), __shfl_xor_sync(0xffffffffu, v.l, o)};
        v = ff_add(v, u);
        f1 += __shfl_xor_sync(0xffffffffu, f1, o);
        f2 += __shfl_xor_sync(0xffffffffu, f2, o);
    }
}

__device__ __forceinline__ void ff_post(ff v, float f1, float f2, float4* slots)
{
    ff_warp_reduce(v, f1, f2);
    if (lane_id() == 0) slots[threadIdx.x >> 5] = make_float4(v.h, v.l, f1, f2);
}

__device__ __forceinline__ void ff_collect(const float4* slots, ff& v, float& f1, float& f2)
{
    const int lane = lane_id();
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < (int)(blockDim.x >> 5)) t = slots[lane];
    v = ff{t.x, t.y};
    f1 = t.z;
    f2 = t.w;
    ff_warp_reduce(v, f1, f2);
}

// (L_j r_hat_j)_a^2 from the high parts of r (fp32: only the stopping test
// reads it); L_j lower triangular, full n x n in global memory
__device__ __forceinline__ float ff_lrow_sq(const float* Lj, const float* RH, int NP, int j, int a,
                                            int n)
{
    const float* row = Lj + (size_t)a * n;
    const float* x = RH + (j + 1) * NP;
    float t = 0.f;
    for (int b = 0; b <= a; ++b) t = fmaf(row[b], x[b], t);
    return t * t;
}

template <int NP, int R>
__global__ void __launch_bounds__(kFFMaxThreads, 1) k_pcg_ff(PcgArgs g)
{
    extern __shared__ __align__(16) float sm[];
    const Work& w = g.w;
    const int N = w.N, n = w.n, nn = n * n, T = blockDim.x, tid = threadIdx.x;
    const int sol = blockIdx.x;
    const int XS = (N + 2) * NP;
    const int rule = g.rule;
    const bool rule0 = rule == GATO_STOP_RESIDUAL;

    float* PH = sm;
    float* PL = PH + XS;
    float* RH = PL + XS;
    float* RL = RH + XS;
    float4* slotA = reinterpret_cast<float4*>(RL + XS);
    float4* slotC = slotA + 32;
    float4* slotD = slotA + 64;
    float* NB = reinterpret_cast<float*>(slotA + 96);
    {
        const size_t blocks = (size_t)(N + 1) * nn, scratch = (size_t)N * n;
        if (!gb_smem((size_t)(NB - sm + round4(blocks > scratch ? blocks : scratch)) *
                         sizeof(float),
                     w.status, sol)) {
            finish(g, sol, 0, false, false);
            return;  // block-uniform
        }
    }

    for (int i = tid; i < 4 * XS; i += T) sm[i] = 0.f;
    {
        const float* gN = w.Nh + sol * w.sKnn;
        const int nb = (N - 1) * nn;
        for (int i = tid; i < nn; i += T) {
            NB[i] = 0.f;
            NB[(size_t)N * nn + i] = 0.f;
        }
        for (int i = tid; i < nb; i += T) NB[nn + i] = gN[i];
    }

    // the thread's rows
    int jr[R], ar[R];
    bool valid[R];
#pragma unroll
    for (int i = 0; i < R; ++i) {
        const int row = tid + i * T;
        // a row's products read knots j - 1 .. j + 1 (the guarded vectors)
        // and blocks j, j + 1 (the framed copy of Nhat)
        valid[i] = row < N * n && gb_ok((long long)(row / n + 2) * NP + NP - 1, XS, w.status, sol) &&
                   gb_ok((long long)(row / n + 2) * nn - 1, (long long)(N + 1) * nn, w.status, sol);
        jr[i] = valid[i] ? row / n : 0;
        ar[i] = valid[i] ? row - jr[i] * n : 0;
    }
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float* gL = w.L + sol * w.sNnn;
    const float* dlow = w.dlow + sol * w.sN;

    ff lam[R], r[R], p[R], v[R];
    // lambda_hat0 = L^T lambda0 (compensated)
#pragma unroll
    for (int i = 0; i < R; ++i) {
        lam[i] = ff_of(0.f);
        if (valid[i] && g.lambda0) {
            const int j = jr[i], a = ar[i];
            const float* Lj = gL + (size_t)j * nn;
            const float* l0 = g.lambda0 + (size_t)sol * N * n + (size_t)j * n;
            Dot2 d;
            for (int b = a; b < n; ++b) d.add(Lj[(size_t)b * n + a], l0[b], 0.f);
            lam[i] = d.value();
        }
    }
    __syncthreads();  // zeroed vectors and copied blocks
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (valid[i]) {
            PH[(jr[i] + 1) * NP + ar[i]] = lam[i].h;
            PL[(jr[i] + 1) * NP + ar[i]] = lam[i].l;
        }
    __syncthreads();
    // r_hat = ghat - lambda_hat - Nhat lambda_hat
#pragma unroll
    for (int i = 0; i < R; ++i) {
        r[i] = ff_of(0.f);
        if (valid[i]) {
            const ff y = ff_row<NP>(NB, n, nn, jr[i], ar[i], PH, PL);
            r[i] = ff_sub(ff_sub(ff_of(ghat[jr[i] * n + ar[i]]), lam[i]), y);
            RH[(jr[i] + 1) * NP + ar[i]] = r[i].h;
            RL[(jr[i] + 1) * NP + ar[i]] = r[i].l;
        }
    }
    __syncthreads();
    // z = (I - Nhat) r = p; eta = r^T z; the stopping reference and quantity
    ff eta_part = ff_of(0.f);
    float ref_part = 0.f, q_part = 0.f;
#pragma unroll
    for (int i = 0; i < R; ++i) {
        p[i] = ff_of(0.f);
        if (valid[i]) {
            const int j = jr[i], a = ar[i], gi = j * n + a;
            const ff y = ff_row<NP>(NB, n, nn, j, a, RH, RL);
            p[i] = ff_sub(r[i], y);
            eta_part = ff_add(eta_part, ff_mul(r[i], p[i]));
            if (rule0) {
                ref_part = fmaf(gam[gi], gam[gi], ref_part);
                q_part += ff_lrow_sq(gL + (size_t)j * nn, RH, NP, j, a, n);
            } else if (rule == GATO_STOP_SCALED) {
                ref_part = fmaf(ghat[gi], ghat[gi], ref_part);
                q_part = fmaf(r[i].h, r[i].h, q_part);
            }
        }
    }
    ff_post(eta_part, ref_part, q_part, slotA);
    __syncthreads();
    ff eta;
    float ref, stopq;
    ff_collect(slotA, eta, ref, stopq);
    if (rule == GATO_STOP_PRECOND) {
        ref = eta.h;
        stopq = eta.h;
    }
    const float thr = g.eps * g.eps * ref;
    bool done = stopq <= thr;
    bool nonfinite = !isfinite(eta.h) || !isfinite(stopq);
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (valid[i]) {
            PH[(jr[i] + 1) * NP + ar[i]] = p[i].h;
            PL[(jr[i] + 1) * NP + ar[i]] = p[i].l;
        }
    // the exact ||L r_hat|| of rule 0 is evaluated only once the per-knot
    // lower bound sum_j dlow_j ||r_hat_j||^2 comes within 1.25 of the
    // threshold (as in the fp32 kernels); a fallback evaluates it in the
    // iteration where the bound drops below the threshold without it
    bool exact_next = false;
    if (rule0) {
        float lb = 0.f;
#pragma unroll
        for (int i = 0; i < R; ++i)
            if (valid[i]) lb = fmaf(dlow[jr[i]] * r[i].h, r[i].h, lb);
        float z0 = 0.f;
        ff zf = ff_of(0.f);
        ff_post(zf, lb, z0, slotC);
        __syncthreads();
        ff_collect(slotC, zf, lb, z0);
        exact_next = lb <= 1.25f * thr;
    }
    __syncthreads();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        // A: v = S_hat p = p + Nhat p, p^T v
        ff pv_part = ff_of(0.f);
#pragma unroll
        for (int i = 0; i < R; ++i) {
            v[i] = ff_of(0.f);
            if (valid[i]) {
                v[i] = ff_add(p[i], ff_row<NP>(NB, n, nn, jr[i], ar[i], PH, PL));
                pv_part = ff_add(pv_part, ff_mul(p[i], v[i]));
            }
        }
        ff_post(pv_part, 0.f, 0.f, slotA);
        __syncthreads();
        // B: alpha = eta / p^T v; lambda and r updates
        ff pv;
        float u1, u2;
        ff_collect(slotA, pv, u1, u2);
        const ff alpha = ff_div(eta, pv);
#pragma unroll
        for (int i = 0; i < R; ++i)
            if (valid[i]) {
                lam[i] = ff_add(lam[i], ff_mul(alpha, p[i]));
                r[i] = ff_sub(r[i], ff_mul(alpha, v[i]));
                RH[(jr[i] + 1) * NP + ar[i]] = r[i].h;
                RL[(jr[i] + 1) * NP + ar[i]] = r[i].l;
            }
        __syncthreads();
        // C: z = (I - Nhat) r (kept in v), eta' = r^T z; the lower bound's
        // and (gated in) the exact norm's shares
        ff eta_part2 = ff_of(0.f);
        float lb_part = 0.f, lsq_part = 0.f;
        const bool exact = exact_next;
#pragma unroll
        for (int i = 0; i < R; ++i)
            if (valid[i]) {
                const int j = jr[i], a = ar[i];
                v[i] = ff_sub(r[i], ff_row<NP>(NB, n, nn, j, a, RH, RL));
                eta_part2 = ff_add(eta_part2, ff_mul(r[i], v[i]));
                if (rule0) {
                    lb_part = fmaf(dlow[j] * r[i].h, r[i].h, lb_part);
                    if (exact) lsq_part += ff_lrow_sq(gL + (size_t)j * nn, RH, NP, j, a, n);
                } else if (rule == GATO_STOP_SCALED) {
                    lb_part = fmaf(r[i].h, r[i].h, lb_part);
                }
            }
        ff_post(eta_part2, lb_part, lsq_part, slotC);
        __syncthreads();
        // D: convergence, beta = eta' / eta, p = z + beta p
        ff eta_new;
        float lb, lsq;
        ff_collect(slotC, eta_new, lb, lsq);
        bool have_exact = exact;
        if (rule0 && !exact && lb * 0.999f <= thr) {
            float part = 0.f, z0 = 0.f;
#pragma unroll
            for (int i = 0; i < R; ++i)
                if (valid[i]) part += ff_lrow_sq(gL + (size_t)jr[i] * nn, RH, NP, jr[i], ar[i], n);
            ff zf = ff_of(0.f);
            ff_post(zf, part, z0, slotD);
            __syncthreads();
            ff_collect(slotD, zf, lsq, z0);
            have_exact = true;
        }
        stopq = rule0 ? lsq : (rule == GATO_STOP_SCALED ? lb : eta_new.h);
        if (!isfinite(eta_new.h + pv.h + stopq + lb)) {  // NaN and Inf propagate
            nonfinite = true;
            break;
        }
        done = (!rule0 || have_exact) && stopq <= thr;
        if (done) break;
        exact_next = rule0 && lb <= 1.25f * thr;
        const ff beta = ff_div(eta_new, eta);
#pragma unroll
        for (int i = 0; i < R; ++i)
            if (valid[i]) {
                p[i] = ff_add(v[i], ff_mul(beta, p[i]));
                PH[(jr[i] + 1) * NP + ar[i]] = p[i].h;
                PL[(jr[i] + 1) * NP + ar[i]] = p[i].l;
            }
        eta = eta_new;
        __syncthreads();
    }
    __syncthreads();
    // lambda_hat to fp32 (h is the rounded sum of h + l), then lambda and dz;
    // the recovery's scratch reuses the blocks' space
#pragma unroll
    for (int i = 0; i < R; ++i)
        if (valid[i]) PH[(jr[i] + 1) * NP + ar[i]] = lam[i].h;
    __syncthreads();
    recover_dz(g.w, g.rhs, g.lambda, g.dX, g.dU, sol,
               [&](int k, int b) { return PH[(k + 1) * NP + b]; }, NB);
    finish(g, sol, it, done, nonfinite);
}

// ---------------------------------------------------------------------------
// The same solve split over a cluster of C CTAs (when the batch leaves SMs
// idle and the CTAs keep enough rows): CTA c owns knots c Nc .. c Nc + nk - 1 (Nc = ceil(N / C)) with one
// row per thread, and holds the coupling blocks of its knots plus the one
// that couples its last knot to the next CTA's first.  A vector update
// writes the CTA's first and last knots also into the guard slots of the
// neighbouring CTAs (distributed shared memory), so the products read only
// local memory.  Every barrier is a cluster barrier; a block reduction adds
// all CTAs' warp slots in rank order, so every CTA holds the same scalars and
// takes the same branches.
// ---------------------------------------------------------------------------

// A warp's partial sums go into slot rank * nw + w of every CTA of the cluster
// (distributed shared memory, stored before the barrier that publishes them),
// so the collect after it reads only local shared memory: no remote load on
// the critical path.  Every lane holds the warp's total after the butterfly.
template <int C>
__device__ __forceinline__ void ff_post_cluster(cg::cluster_group& cl, ff v, float f1, float f2,
                                                float4* slots)
{
    ff_warp_reduce(v, f1, f2);
    const int lane = lane_id(), rank = (int)cl.block_rank();
    if (lane < C) {
        float4* dst = lane == rank ? slots : cl.map_shared_rank(slots, lane);
        dst[rank * (int)(blockDim.x >> 5) + (int)(threadIdx.x >> 5)] =
            make_float4(v.h, v.l, f1, f2);
    }
}

// the double-float totals of the C CTAs' warp slots (C nw <= 32 slots), added
// in rank-major order, the same in every CTA
template <int C>
__device__ __forceinline__ void ff_collect_cluster(const float4* slots, ff& v, float& f1,
                                                   float& f2)
{
    const int lane = lane_id(), nw = (int)(blockDim.x >> 5);
    float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
    if (lane < C * nw) t = slots[lane];
    v = ff{t.x, t.y};
    f1 = t.z;
    f2 = t.w;
    ff_warp_reduce(v, f1, f2);
}

// a CTA of a cluster has at most 1024 / C threads (its warp slots and the
// other CTAs' fit one 32-lane butterfly), which leaves more registers
template <int NP, int C>
__global__ void __launch_bounds__(kFFMaxThreads / C, 1) k_pcg_ff_cluster(PcgArgs g)
{
    extern __shared__ __align__(16) float sm[];
    cg::cluster_group cl = cg::this_cluster();
    const int rank = (int)cl.block_rank();
    const int sol = (int)(blockIdx.x / C);
    const Work& w = g.w;
    const int N = w.N, n = w.n, nn = n * n, T = blockDim.x, tid = threadIdx.x;
    const int Nc = (N + C - 1) / C;
    const int k0 = rank * Nc;        // first knot of this CTA
    const int nk = min(Nc, N - k0);  // its knots (>= 1: the launcher checks)
    const int XS = (Nc + 2) * NP;
    const int rule = g.rule;
    const bool rule0 = rule == GATO_STOP_RESIDUAL;

    float* PH = sm;
    float* PL = PH + XS;
    float* RH = PL + XS;
    float* RL = RH + XS;
    float4* slotA = reinterpret_cast<float4*>(RL + XS);
    float4* slotC = slotA + 32;
    float4* slotD = slotA + 64;
    float* NB = reinterpret_cast<float*>(slotA + 96);
    {
        const size_t blocks = (size_t)(Nc + 1) * nn, scratch = (size_t)Nc * n;
        // the same layout in every CTA: all leave together
        if (!gb_smem((size_t)(NB - sm + round4(blocks > scratch ? blocks : scratch)) *
                         sizeof(float),
                     w.status, sol)) {
            if (rank == 0) finish(g, sol, 0, false, false);
            return;
        }
    }
    // the neighbours' vectors (for the guard-slot writes)
    float* nPH[2] = {nullptr, nullptr};
    float* nPL[2] = {nullptr, nullptr};
    float* nRH[2] = {nullptr, nullptr};
    float* nRL[2] = {nullptr, nullptr};
    if (rank > 0) {
        nPH[0] = cl.map_shared_rank(PH, rank - 1);
        nPL[0] = cl.map_shared_rank(PL, rank - 1);
        nRH[0] = cl.map_shared_rank(RH, rank - 1);
        nRL[0] = cl.map_shared_rank(RL, rank - 1);
    }
    if (rank < C - 1) {
        nPH[1] = cl.map_shared_rank(PH, rank + 1);
        nPL[1] = cl.map_shared_rank(PL, rank + 1);
        nRH[1] = cl.map_shared_rank(RH, rank + 1);
        nRL[1] = cl.map_shared_rank(RL, rank + 1);
    }

    for (int i = tid; i < 4 * XS; i += T) sm[i] = 0.f;
    {
        // block jl (jl = 0 .. Nc) is Nhat_{k0 + jl} where it exists, else zero
        const float* gN = w.Nh + sol * w.sKnn;
        for (int i = tid; i < (Nc + 1) * nn; i += T) {
            const int jl = i / nn, j = k0 + jl;
            NB[i] = (jl <= nk && j >= 1 && j <= N - 1) ? gN[(size_t)(j - 1) * nn + (i - jl * nn)]
                                                       : 0.f;
        }
    }
    const int row = tid;
    const bool valid = row < nk * n && gb_ok((long long)(row / n + 2) * NP + NP - 1, XS,
                                             w.status, sol);
    const int jl = valid ? row / n : 0, a = valid ? row - jl * n : 0, j = k0 + jl;
    // a value of this thread's row into p or r, and into a neighbour's guard
    // slot when the row is a boundary knot's
    auto put = [&](float* XH, float* XL, float* const (&nH)[2], float* const (&nL)[2], ff v) {
        if (!valid) return;
        XH[(jl + 1) * NP + a] = v.h;
        XL[(jl + 1) * NP + a] = v.l;
        if (jl == 0 && rank > 0) {
            nH[0][(Nc + 1) * NP + a] = v.h;
            nL[0][(Nc + 1) * NP + a] = v.l;
        }
        if (jl == nk - 1 && rank < C - 1) {
            nH[1][a] = v.h;
            nL[1][a] = v.l;
        }
    };
    const float* ghat = g.rhs.ghat + sol * w.sNn;
    const float* gam = g.rhs.gamma + sol * w.sNn;
    const float* gL = w.L + sol * w.sNnn;
    const float* dlow = w.dlow + sol * w.sN;
    const float dl = valid ? dlow[j] : 0.f;

    ff lam = ff_of(0.f), r = ff_of(0.f), p = ff_of(0.f), v = ff_of(0.f);
    if (valid && g.lambda0) {
        const float* Lj = gL + (size_t)j * nn;
        const float* l0 = g.lambda0 + (size_t)sol * N * n + (size_t)j * n;
        Dot2 d;
        for (int b = a; b < n; ++b) d.add(Lj[(size_t)b * n + a], l0[b], 0.f);
        lam = d.value();
    }
    cl.sync();  // zeroed vectors and blocks in every CTA
    put(PH, PL, nPH, nPL, lam);
    cl.sync();
    if (valid) {
        r = ff_sub(ff_sub(ff_of(ghat[j * n + a]), lam), ff_row<NP>(NB, n, nn, jl, a, PH, PL));
        put(RH, RL, nRH, nRL, r);
    }
    cl.sync();
    ff eta_part = ff_of(0.f);
    float ref_part = 0.f, q_part = 0.f;
    if (valid) {
        const int gi = j * n + a;
        p = ff_sub(r, ff_row<NP>(NB, n, nn, jl, a, RH, RL));
        eta_part = ff_mul(r, p);
        if (rule0) {
            ref_part = gam[gi] * gam[gi];
            q_part = ff_lrow_sq(gL + (size_t)j * nn, RH, NP, jl, a, n);
        } else if (rule == GATO_STOP_SCALED) {
            ref_part = ghat[gi] * ghat[gi];
            q_part = r.h * r.h;
        }
    }
    ff_post_cluster<C>(cl, eta_part, ref_part, q_part, slotA);
    cl.sync();
    ff eta;
    float ref, stopq;
    ff_collect_cluster<C>(slotA, eta, ref, stopq);
    if (rule == GATO_STOP_PRECOND) {
        ref = eta.h;
        stopq = eta.h;
    }
    const float thr = g.eps * g.eps * ref;
    bool done = stopq <= thr;
    bool nonfinite = !isfinite(eta.h) || !isfinite(stopq);
    put(PH, PL, nPH, nPL, p);
    bool exact_next = false;
    if (rule0) {
        float lb = valid ? dl * r.h * r.h : 0.f, z0 = 0.f;
        ff zf = ff_of(0.f);
        ff_post_cluster<C>(cl, zf, lb, z0, slotC);
        cl.sync();
        ff_collect_cluster<C>(slotC, zf, lb, z0);
        exact_next = lb <= 1.25f * thr;
    }
    cl.sync();

    int it = 0;
    while (!done && !nonfinite && it < g.max_iters) {
        ++it;
        // A: v = p + Nhat p, p^T v
        ff pv_part = ff_of(0.f);
        if (valid) {
            v = ff_add(p, ff_row<NP>(NB, n, nn, jl, a, PH, PL));
            pv_part = ff_mul(p, v);
        }
        ff_post_cluster<C>(cl, pv_part, 0.f, 0.f, slotA);
        cl.sync();
        // B: alpha; lambda and r
        ff pv;
        float u1, u2;
        ff_collect_cluster<C>(slotA, pv, u1, u2);
        const ff alpha = ff_div(eta, pv);
        if (valid) {
            lam = ff_add(lam, ff_mul(alpha, p));
            r = ff_sub(r, ff_mul(alpha, v));
            put(RH, RL, nRH, nRL, r);
        }
        cl.sync();
        // C: z = r - Nhat r, eta' = r^T z, the bound's and the exact norm's shares
        ff eta_part2 = ff_of(0.f);
        float lb_part = 0.f, lsq_part = 0.f;
        const bool exact = exact_next;
        if (valid) {
            v = ff_sub(r, ff_row<NP>(NB, n, nn, jl, a, RH, RL));
            eta_part2 = ff_mul(r, v);
            if (rule0) {
                lb_part = dl * r.h * r.h;
                if (exact) lsq_part = ff_lrow_sq(gL + (size_t)j * nn, RH, NP, jl, a, n);
            } else if (rule == GATO_STOP_SCALED) {
                lb_part = r.h * r.h;
            }
        }
        ff_post_cluster<C>(cl, eta_part2, lb_part, lsq_part, slotC);
        cl.sync();
        // D: convergence, beta, p
        ff eta_new;
        float lb, lsq;
        ff_collect_cluster<C>(slotC, eta_new, lb, lsq);
        bool have_exact = exact;
        if (rule0 && !exact && lb * 0.999f <= thr) {
            float part = valid ? ff_lrow_sq(gL + (size_t)j * nn, RH, NP, jl, a, n) : 0.f, z0 = 0.f;
            ff zf = ff_of(0.f);
            ff_post_cluster<C>(cl, zf, part, z0, slotD);
            cl.sync();
            ff_collect_cluster<C>(slotD, zf, lsq, z0);
            have_exact = true;
        }
        stopq = rule0 ? lsq : (rule == GATO_STOP_SCALED ? lb : eta_new.h);
        if (!isfinite(eta_new.h + pv.h + stopq + lb)) {  // NaN and Inf propagate
            nonfinite = true;
            break;
        }
        done = (!rule0 || have_exact) && stopq <= thr;
        if (done) break;
        exact_next = rule0 && lb <= 1.25f * thr;
        const ff beta = ff_div(eta_new, eta);
        if (valid) {
            p = ff_add(v, ff_mul(beta, p));
            put(PH, PL, nPH, nPL, p);
        }
        eta = eta_new;
        cl.sync();
    }
    cl.sync();
    if (valid) PH[(jl + 1) * NP + a] = lam.h;
    cl.sync();
    cluster_recover(cl, g, sol, k0, nk, [&](int kl, int b) { return PH[(kl + 1) * NP + b]; });
    if (rank == 0) finish(g, sol, it, done, nonfinite);
}

// row width of the vectors: n padded to a multiple of 4 (the instantiations)
int ff_np(int n)
{
    static const int widths[] = {4, 8, 12, 16, 20, 24, 28, 32, 36, 40, 48, 56, 64};
    for (int v : widths)
        if (n <= v) return v;
    return 0;
}

// shared memory of one block: p and r (high and low) with guard knots, the
// reduction slots, and the N + 1 coupling blocks (which the recovery reuses
// as its N n scratch)
size_t ff_smem_bytes(int N, int n, int NP)
{
    const size_t blocks = (size_t)(N + 1) * n * n;
    const size_t scratch = (size_t)N * n;
    return sizeof(float) *
           (4 * (size_t)(N + 2) * NP + 96 * 4 + round4(blocks > scratch ? blocks : scratch));
}

// rows per thread: 1 up to 1024 rows, 2 up to 2048 when n <= 16; 0 beyond
int ff_rows_per_thread(int N, int n)
{
    const long rows = (long)N * n;
    if (rows <= kFFMaxThreads) return 1;
    if (rows <= 2 * kFFMaxThreads && n <= 16) return 2;
    return 0;
}

template <int NP, int R>
cudaError_t launch_ff(const PcgArgs& a, int T, size_t limit, cudaStream_t st)
{
    const Work& w = a.w;
    const size_t smem = ff_smem_bytes(w.N, w.n, NP);
    if (smem > limit) return cudaErrorInvalidConfiguration;
    auto kernel = k_pcg_ff<NP, R>;
    if (smem > 48 * 1024) {
        cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    kernel<<<w.M, T, smem, st>>>(a);
    return cudaGetLastError();
}

// one solve per cluster of C CTAs (grid M C); cudaErrorInvalidConfiguration
// when the split does not apply or no such cluster fits
template <int NP, int C>
cudaError_t launch_ff_cluster(const PcgArgs& a, size_t limit, cudaStream_t st)
{
    const Work& w = a.w;
    const int Nc = (w.N + C - 1) / C;
    if ((C - 1) * Nc >= w.N) return cudaErrorInvalidConfiguration;  // a CTA without knots
    const int rows = Nc * w.n;
    int T = (rows + 31) / 32 * 32;
    if (T < 32) T = 32;
    if (T > kFFMaxThreads || C * (T / 32) > 32) return cudaErrorInvalidConfiguration;
    const size_t smem = ff_smem_bytes(Nc, w.n, NP);
    if (smem > limit) return cudaErrorInvalidConfiguration;
    auto kernel = k_pcg_ff_cluster<NP, C>;
    cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(w.M * C), 1, 1);
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

template <int NP>
cudaError_t launch_ff_np(const PcgArgs& a, size_t limit, int num_sms, cudaStream_t st)
{
    // a batch of at most half the SMs: each solve over two CTAs (n <= 16),
    // when each keeps at least kFFClusterRows rows; below that the cluster
    // barriers and the remote reductions cost more than the halved work
    if constexpr (NP <= 16) {
        const int Nc = (a.w.N + 1) / 2;
        if (a.w.M * 2 <= num_sms && Nc * a.w.n >= kFFClusterRows) {
            const cudaError_t e = launch_ff_cluster<NP, 2>(a, limit, st);
            if (e != cudaErrorInvalidConfiguration) return e;
        }
    }
    const int rows = a.w.N * a.w.n;
    const int R = ff_rows_per_thread(a.w.N, a.w.n);
    if (R == 0) return cudaErrorInvalidConfiguration;
    int T = ((rows + R - 1) / R + 31) / 32 * 32;
    if (T < 32) T = 32;
    if (R == 1) return launch_ff<NP, 1>(a, T, limit, st);
    if constexpr (NP <= 16) return launch_ff<NP, 2>(a, T, limit, st);
    return cudaErrorInvalidConfiguration;
}

}  // namespace

bool pcg_ff_fits(int N, int n, size_t smem_limit)
{
    const int NP = ff_np(n);
    return NP > 0 && ff_rows_per_thread(N, n) > 0 && ff_smem_bytes(N, n, NP) <= smem_limit;
}

cudaError_t launch_pcg_ff(const PcgArgs& a, size_t limit, int num_sms, cudaStream_t st)
{
    const int n = a.w.n;
    if (n <= 4) return launch_ff_np<4>(a, limit, num_sms, st);
    if (n <= 8) return launch_ff_np<8>(a, limit, num_sms, st);
    if (n <= 12) return launch_ff_np<12>(a, limit, num_sms, st);
    if (n <= 16) return launch_ff_np<16>(a, limit, num_sms, st);
    if (n <= 20) return launch_ff_np<20>(a, limit, num_sms, st);
    if (n <= 24) return launch_ff_np<24>(a, limit, num_sms, st);
    if (n <= 28) return launch_ff_np<28>(a, limit, num_sms, st);
    if (n <= 32) return launch_ff_np<32>(a, limit, num_sms, st);
    if (n <= 36) return launch_ff_np<36>(a, limit, num_sms, st);
    if (n <= 40) return launch_ff_np<40>(a, limit, num_sms, st);
    if (n <= 48) return launch_ff_np<48>(a, limit, num_sms, st);
    if (n <= 56) return launch_ff_np<56>(a, limit, num_sms, st);
    if (n <= 64) return launch_ff_np<64>(a, limit, num_sms, st);
    return cudaErrorInvalidConfiguration;
}

}  // namespace gato
