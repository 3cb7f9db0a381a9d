// form_schur.cu -- Schur complement S, gamma and the symmetric stair
// preconditioner (GATO paper, Sec. II eqs. (4)-(6); Sec. III: block-local
// formation with one grid-wide synchronisation before Phi^-1 is final).
//
// One warp per knot; each warp keeps its knot's small matrices in its own
// slice of shared memory.  Three launches, whose boundaries are the grid-wide
// synchronisations the block-local formation needs:
//   k_form_inv   knot k:  Q_k^-1, R_k^-1, S_{k+1,k} = -A_k Q_k^-1, V_k = B_k R_k^-1
//   k_form_diag  row j:   S_jj = Q_j^-1 + A_{j-1} Q_{j-1}^-1 A_{j-1}^T + V_{j-1} B_{j-1}^T,
//                         its Cholesky factor L_j, L_j^-1 and the eigenvalue
//                         bound 1 / ||L_j^-1||_F^2
//   k_form_off   row j:   Nhat_j = L_j^-1 S_{j,j-1} L_{j-1}^-T
// The solve applies Phi^-1 in that factored form; the explicit blocks
// S_jj^-1 and -S_jj^-1 S_{j,j-1} S_{j-1,j-1}^-1 are formed only for export
// (k_form_phi_diag, k_form_phi_off, launched by gato_get_schur).
// and a fourth for the right-hand side (also used by iterative refinement):
//   k_form_rhs   row j:   gamma_j, L_j^-1 gamma_j, -Q_j^-1 q_j, -R_j^-1 r_j
#include "gato_internal.cuh"

namespace gato {
namespace {

// floats per warp of k_form_inv: sQ (n x n) and a second slice that holds
// L^-1, later the R part (3 m^2 + n m) and A (n^2)
__host__ __device__ __forceinline__ int form_inv_floats(int n, int m)
{
    const int rest = 3 * m * m + n * m > n * n ? 3 * m * m + n * m : n * n;
    return (n * n + rest + 3) & ~3;
}

__global__ void k_form_inv(Work w, const float* __restrict__ Q, const float* __restrict__ R,
                           const float* __restrict__ A, const float* __restrict__ B,
                           uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, m = w.m, N = w.N;
    const int nn = n * n, mm = m * m, nm = n * m;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    const long g = (long)blockIdx.x * wpb + warp;
    if (g >= (long)w.M * N) return;
    const int sol = (int)(g / N), k = (int)(g % N);
    if (!gb_smem((size_t)(warp + 1) * form_inv_floats(n, m) * sizeof(float), w.status, sol))
        return;  // the warp's slice (warp-uniform)
    // two n x n slices per warp (more warps per SM): L and then Q^-1 in sQ;
    // L^-1 in sT, then the R part (R's factor, R^-1 rows, R^-1, B), then A
    float* sQ = sm + (size_t)warp * form_inv_floats(n, m);
    float* sT = sQ + nn;
    float* sR = sT;
    float* sRt = sR + mm;
    float* sRi = sRt + mm;
    float* sB = sRi + mm;

    warp_copy(sQ, Q + ((size_t)sol * N + k) * nn, nn);
    bool ok = warp_cholesky(sQ, n);
    warp_lower_inverse(sQ, sT, n);
    warp_gram_lower(sT, sQ, n);  // Q^-1 over L (read no more)
    float* sQi = sQ;
    warp_copy(w.Qinv + sol * w.sNnn + (size_t)k * nn, sQi, nn);
    if (k < N - 1) {
        const size_t K = (size_t)(N - 1);
        warp_copy(sR, R + ((size_t)sol * K + k) * mm, mm);
        ok = warp_cholesky(sR, m) && ok;
        warp_lower_inverse(sR, sRt, m);
        warp_gram_lower(sRt, sRi, m);
        warp_copy(w.Rinv + sol * w.sKmm + (size_t)k * mm, sRi, mm);
        warp_copy(sB, B + ((size_t)sol * K + k) * nm, nm);
        __syncwarp();
        warp_gemm<false, false>(n, m, m, sB, sRi, w.V + sol * w.sKnm + (size_t)k * nm, 1.f, false);
        warp_copy(sT, A + ((size_t)sol * K + k) * nn, nn);  // the R part is done: A_k
        __syncwarp();
        warp_gemm<false, false>(n, n, n, sT, sQi, w.O + sol * w.sKnn + (size_t)k * nn, -1.f, false);
    }
    if (!ok && lane_id() == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

__global__ void k_form_diag(Work w, const float* __restrict__ A, const float* __restrict__ B,
                            uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, m = w.m, N = w.N;
    const int nn = n * n, nm = n * m;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    const long g = (long)blockIdx.x * wpb + warp;
    if (g >= (long)w.M * N) return;
    const int sol = (int)(g / N), j = (int)(g % N);
    if (!gb_smem((size_t)(warp + 1) * (4 * nn + 2 * nm) * sizeof(float), w.status, sol))
        return;  // the warp's slice (warp-uniform)
    float* sD = sm + (size_t)warp * (4 * nn + 2 * nm);
    float* sO = sD + nn;
    float* sA = sO + nn;
    float* sL = sA + nn;
    float* sV = sL + nn;
    float* sB = sV + nm;

    warp_copy(sD, w.Qinv + sol * w.sNnn + (size_t)j * nn, nn);
    if (j > 0) {
        const size_t K = (size_t)(N - 1);
        warp_copy(sO, w.O + sol * w.sKnn + (size_t)(j - 1) * nn, nn);
        warp_copy(sA, A + ((size_t)sol * K + (j - 1)) * nn, nn);
        warp_copy(sV, w.V + sol * w.sKnm + (size_t)(j - 1) * nm, nm);
        warp_copy(sB, B + ((size_t)sol * K + (j - 1)) * nm, nm);
        __syncwarp();
        // theta: A Q^-1 A^T = -S_{j,j-1} A^T, plus B R^-1 B^T = V B^T; A^T (and
        // B^T where m <= n, so that it fits) is staged in sL (free until the
        // factorisation) so that the products take warp_gemm's 128-bit path
        // (the transposed operand's strided reads would conflict on the
        // banks); the sums are the same
        warp_transpose(sA, n, n, sL);
        warp_gemm<false, false>(n, n, n, sO, sL, sD, -1.f, true);
        if (m <= n) {
            warp_transpose(sB, n, m, sL);
            warp_gemm<false, false>(n, n, m, sV, sL, sD, 1.f, true);
        } else {
            warp_gemm<false, true>(n, n, m, sV, sB, sD, 1.f, true);
        }
    }
    __syncwarp();
    const size_t off = sol * w.sNnn + (size_t)j * nn;
    warp_copy(w.D + off, sD, nn);
    warp_copy(sL, sD, nn);
    const bool ok = warp_cholesky(sL, n);
    warp_copy(w.L + off, sL, nn);
    warp_lower_inverse(sL, sA, n);
    warp_copy(w.Linv + off, sA, nn);
    {
        // ||L_j^-1||_F^2 = trace(S_jj^-1) >= 1 / lambda_min(S_jj)
        float f = 0.f;
        for (int t = lane_id(); t < nn; t += 32) f += sA[t] * sA[t];
        f = warp_sum(f);
        if (lane_id() == 0) w.dlow[sol * w.sN + j] = 1.f / f;
    }
    if (!ok && lane_id() == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

__global__ void k_form_off(Work w)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N, K = N - 1;
    const int nn = n * n;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    const long g = (long)blockIdx.x * wpb + warp;
    if (K < 1 || g >= (long)w.M * K) return;
    const int sol = (int)(g / K), j = 1 + (int)(g % K);
    if (!gb_smem((size_t)(warp + 1) * 3 * nn * sizeof(float), w.status, sol))
        return;  // the warp's slice (warp-uniform)
    float* s1 = sm + (size_t)warp * 3 * nn;
    float* s2 = s1 + nn;
    float* s4 = s2 + nn;
    const size_t dj = sol * w.sNnn + (size_t)j * nn, dp = dj - nn;
    const size_t oj = sol * w.sKnn + (size_t)(j - 1) * nn;

    warp_copy(s1, w.Linv + dj, nn);
    warp_copy(s2, w.O + oj, nn);
    __syncwarp();
    warp_gemm<false, false>(n, n, n, s1, s2, s4, 1.f, false);
    warp_copy(s1, w.Linv + dp, nn);  // L_j^-1 is read no more: L_{j-1}^-1
    __syncwarp();
    // L_{j-1}^-T staged in s2 (O is read no more) for warp_gemm's 128-bit path
    warp_transpose(s1, n, n, s2);
    warp_gemm<false, false>(n, n, n, s4, s2, w.Nh + oj, 1.f, false);
}

// The explicit Phi^-1 blocks for export: S_jj^-1 = L_j^-T L_j^-1 ...
__global__ void k_form_phi_diag(Work w)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N, nn = n * n;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    const long g = (long)blockIdx.x * wpb + warp;
    if (g >= (long)w.M * N) return;
    const int sol = (int)(g / N), j = (int)(g % N);
    if (!gb_smem((size_t)(warp + 1) * 2 * nn * sizeof(float), w.status, sol))
        return;  // the warp's slice (warp-uniform)
    float* sA = sm + (size_t)warp * 2 * nn;
    float* sO = sA + nn;
    const size_t off = sol * w.sNnn + (size_t)j * nn;
    warp_copy(sA, w.Linv + off, nn);
    __syncwarp();
    warp_gram_lower(sA, sO, n);
    warp_copy(w.Pd + off, sO, nn);
}

// ... and -S_jj^-1 S_{j,j-1} S_{j-1,j-1}^-1
__global__ void k_form_phi_off(Work w)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N, K = N - 1, nn = n * n;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5;
    const long g = (long)blockIdx.x * wpb + warp;
    if (K < 1 || g >= (long)w.M * K) return;
    const int sol = (int)(g / K), j = 1 + (int)(g % K);
    if (!gb_smem((size_t)(warp + 1) * 4 * nn * sizeof(float), w.status, sol))
        return;  // the warp's slice (warp-uniform)
    float* s1 = sm + (size_t)warp * 4 * nn;
    float* s2 = s1 + nn;
    float* s3 = s2 + nn;
    float* s4 = s3 + nn;
    const size_t dj = sol * w.sNnn + (size_t)j * nn, dp = dj - nn;
    const size_t oj = sol * w.sKnn + (size_t)(j - 1) * nn;
    warp_copy(s1, w.Pd + dj, nn);
    warp_copy(s2, w.O + oj, nn);
    warp_copy(s3, w.Pd + dp, nn);
    __syncwarp();
    warp_gemm<false, false>(n, n, n, s1, s2, s4, 1.f, false);
    warp_gemm<false, false>(n, n, n, s4, s3, w.Po + oj, -1.f, false);
}

// n, m <= 16: the same right-hand side with one half-warp per knot (lane =
// row) and sixteen knots per block, every row product unrolled; the row
// sums are those of k_form_rhs, in the same order.
__global__ void __launch_bounds__(256) k_form_rhs_half(Work w, Rhs out, const float* __restrict__ q,
                                                       const float* __restrict__ r,
                                                       const float* __restrict__ e,
                                                       const float* __restrict__ s0,
                                                       size_t s0_stride)
{
    __shared__ __align__(16) float sgs[16][16];
    const int n = w.n, m = w.m, N = w.N;
    const int nn = n * n;
    const int h = threadIdx.x >> 4, li = threadIdx.x & 15;
    const long g = (long)blockIdx.x * 16 + h;
    const bool act = g < (long)w.M * N;  // no early return: the warp syncs below
    const long gi = act ? g : 0;
    const int sol = (int)(gi / N), j = (int)(gi % N);
    const size_t K = (size_t)(N - 1);
    float* sg = sgs[h];
    auto at = [](const float* v) { return [v](int b) { return v[b]; }; };
    if (act && li < n) {
        const float* Qi = w.Qinv + sol * w.sNnn + (size_t)j * nn;
        const float* qj = q + ((size_t)sol * N + j) * n;
        const float t = strided_dot<16>(Qi + li * n, 1, at(qj), 0, n);  // (Q_j^-1 q_j)_li
        float gv;
        if (j == 0) {
            gv = s0[sol * s0_stride + li] + t;
        } else {
            const float* qp = q + ((size_t)sol * N + (j - 1)) * n;
            const float* rp = r + ((size_t)sol * K + (j - 1)) * m;
            const float* Op = w.O + sol * w.sKnn + (size_t)(j - 1) * nn;
            const float* Vp = w.V + sol * w.sKnm + (size_t)(j - 1) * n * m;
            gv = e[((size_t)sol * K + (j - 1)) * n + li];
            gv += strided_dot<16>(Op + li * n, 1, at(qp), 0, n);
            gv -= strided_dot<16>(Vp + li * m, 1, at(rp), 0, m);
            gv += t;
        }
        sg[li] = gv;
        out.gamma[sol * w.sNn + (size_t)j * n + li] = gv;
        out.avec[sol * w.sNn + (size_t)j * n + li] = -t;
    }
    __syncwarp();
    if (act && li < n) {
        const float* Li = w.Linv + sol * w.sNnn + (size_t)j * nn;
        out.ghat[sol * w.sNn + (size_t)j * n + li] =
            strided_dot<16>(Li + li * n, 1, at(sg), 0, li + 1);
    }
    if (act && j < N - 1 && li < m) {
        const float* Ri = w.Rinv + sol * w.sKmm + (size_t)j * m * m;
        const float* rj = r + ((size_t)sol * K + j) * m;
        out.bvec[sol * w.sKm + (size_t)j * m + li] =
            -strided_dot<16>(Ri + li * m, 1, at(rj), 0, m);
    }
}

// Right-hand side for (q, r, e, s0); s0 of solve i starts at s0 + i * s0_stride.
// One warp per knot, lanes over rows; with NPX > 0 (n, m <= NPX) every row
// product is unrolled and predicated so that its loads are in flight at once.
template <int NPX>
__global__ void k_form_rhs(Work w, Rhs out, const float* __restrict__ q,
                           const float* __restrict__ r, const float* __restrict__ e,
                           const float* __restrict__ s0, size_t s0_stride)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, m = w.m, N = w.N;
    const int nn = n * n;
    const int warp = threadIdx.x >> 5, wpb = blockDim.x >> 5, lane = lane_id();
    const long g = (long)blockIdx.x * wpb + warp;
    if (g >= (long)w.M * N) return;
    const int sol = (int)(g / N), j = (int)(g % N);
    const size_t K = (size_t)(N - 1);
    if (!gb_smem((size_t)(warp + 1) * n * sizeof(float), w.status, sol)) return;
    float* sg = sm + (size_t)warp * n;
    const float* Qi = w.Qinv + sol * w.sNnn + (size_t)j * nn;
    const float* qj = q + ((size_t)sol * N + j) * n;
    const float* qp = q + ((size_t)sol * N + (j > 0 ? j - 1 : 0)) * n;
    const float* rp = r + ((size_t)sol * K + (j > 0 ? j - 1 : 0)) * m;
    const float* Op = w.O + sol * w.sKnn + (size_t)(j > 0 ? j - 1 : 0) * nn;
    const float* Vp = w.V + sol * w.sKnm + (size_t)(j > 0 ? j - 1 : 0) * n * m;
    auto at = [](const float* v) { return [v](int b) { return v[b]; }; };
    for (int a = lane; a < n; a += 32) {
        const float t = strided_dot<NPX>(Qi + a * n, 1, at(qj), 0, n);  // (Q_j^-1 q_j)_a
        float gv;
        if (j == 0) {
            gv = s0[sol * s0_stride + a] + t;
        } else {
            gv = e[((size_t)sol * K + (j - 1)) * n + a];
            gv += strided_dot<NPX>(Op + a * n, 1, at(qp), 0, n);
            gv -= strided_dot<NPX>(Vp + a * m, 1, at(rp), 0, m);
            gv += t;
        }
        sg[a] = gv;
        out.gamma[sol * w.sNn + (size_t)j * n + a] = gv;
        out.avec[sol * w.sNn + (size_t)j * n + a] = -t;
    }
    __syncwarp();
    const float* Li = w.Linv + sol * w.sNnn + (size_t)j * nn;
    for (int a = lane; a < n; a += 32)
        out.ghat[sol * w.sNn + (size_t)j * n + a] =
            strided_dot<NPX>(Li + a * n, 1, at(sg), 0, a + 1);
    if (j < N - 1) {
        const float* Ri = w.Rinv + sol * w.sKmm + (size_t)j * m * m;
        const float* rj = r + ((size_t)sol * K + j) * m;
        for (int c = lane; c < m; c += 32)
            out.bvec[sol * w.sKm + (size_t)j * m + c] =
                -strided_dot<NPX>(Ri + c * m, 1, at(rj), 0, m);
    }
}

// warps per block so that the per-warp slices fit in `budget` bytes
int warps_for(size_t per_warp_bytes, size_t budget)
{
    size_t w = per_warp_bytes ? budget / per_warp_bytes : 8;
    if (w > 8) w = 8;
    if (w < 1) w = 1;
    return (int)w;
}

template <typename K, typename... Args>
cudaError_t launch_warp_per_item(K kernel, long items, size_t per_warp_bytes,
                                 const gato_handle* h, cudaStream_t st, Args... args)
{
    if (items <= 0) return cudaSuccess;
    const int wpb = warps_for(per_warp_bytes, 48 * 1024);
    const size_t smem = (size_t)wpb * per_warp_bytes;
    if (smem > (size_t)h->smem_optin) return cudaErrorInvalidConfiguration;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)smem);
        if (e != cudaSuccess) return e;
    }
    const long blocks = (items + wpb - 1) / wpb;
    kernel<<<(unsigned)blocks, wpb * 32, smem, st>>>(args...);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_form_matrices(gato_handle* h, const float* Q, const float* R,
                                 const float* A, const float* B, uint32_t* status,
                                 cudaStream_t st)
{
    const Work& w = h->w;
    h->phi_pending = 1;  // formed on demand by gato_get_schur
    h->phi_smem = 0;
    if (!h->force_smem_form && rows_formation_supported(w))
        return launch_form_rows(h, Q, R, A, B, status, st);
    h->phi_smem = 1;
    const size_t n = w.n, m = w.m, f = sizeof(float);
    const long knots = (long)w.M * w.N;
    cudaError_t e;
    e = launch_warp_per_item(k_form_inv, knots, form_inv_floats((int)n, (int)m) * f, h, st, w,
                             Q, R, A, B, status);
    if (e != cudaSuccess) return e;
    e = launch_warp_per_item(k_form_diag, knots, (4 * n * n + 2 * n * m) * f, h, st, w, A, B,
                             status);
    if (e != cudaSuccess) return e;
    return launch_warp_per_item(k_form_off, (long)w.M * (w.N - 1), 3 * n * n * f, h, st, w);
}

cudaError_t launch_form_phi_smem(gato_handle* h, cudaStream_t st)
{
    const Work& w = h->w;
    const size_t nn = (size_t)w.n * w.n * sizeof(float);
    cudaError_t e = launch_warp_per_item(k_form_phi_diag, (long)w.M * w.N, 2 * nn, h, st, w);
    if (e != cudaSuccess) return e;
    return launch_warp_per_item(k_form_phi_off, (long)w.M * (w.N - 1), 4 * nn, h, st, w);
}

cudaError_t launch_form_rhs(gato_handle* h, int set, const float* q, const float* r,
                            const float* e, const float* s0, size_t s0_stride, cudaStream_t st)
{
    const Work& w = h->w;
    const long knots = (long)w.M * w.N;
    const size_t per_warp = (size_t)w.n * sizeof(float);
    if (w.n <= 16 && w.m <= 16) {
        if (knots <= 0) return cudaSuccess;
        k_form_rhs_half<<<(unsigned)((knots + 15) / 16), 256, 0, st>>>(w, w.rhs[set], q, r, e, s0,
                                                                       s0_stride);
        return cudaGetLastError();
    }
    return launch_warp_per_item(k_form_rhs<0>, knots, per_warp, h, st, w, w.rhs[set], q, r, e,
                                s0, s0_stride);
}

}  // namespace gato
