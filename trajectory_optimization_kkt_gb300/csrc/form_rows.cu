// form_rows.cu -- Schur complement and stair preconditioner formation for
// n, m <= 16 with the small matrices held in registers (GATO paper, Sec. II
// eqs. (4)-(6); Sec. III block-local formation with a grid-wide sync before
// Phi^-1 is final).
//
// Each half-warp (16 lanes) works on one knot; lane l holds row l of the
// current matrix (16 floats, rows >= n are identity rows so that every
// factorisation acts on diag(M, I)).  Cholesky runs right-looking with
// half-warp shuffles; finished rows are published to a 16 x 16 scratch in
// shared memory, from which the other lanes read them with 128-bit loads for
// the triangular inverse and the small products.  Three launches, as in the
// shared-memory kernels, with the same outputs:
//   k_rows_knot  knot k:  Q_k^-1, R_k^-1, S_{k+1,k} = -A_k Q_k^-1,
//                         V_k = B_k R_k^-1, and theta_k = A_k Q_k^-1 A_k^T +
//                         V_k B_k^T (stored where S_{k+1,k+1} goes)
//   k_rows_diag  row j:   S_jj = Q_j^-1 + theta_{j-1}, L_j, L_j^-1 and the
//                         eigenvalue bound 1 / ||L_j^-1||_F^2
//   k_rows_off   row j:   Nhat_j = L_j^-1 S_{j,j-1} L_{j-1}^-T
// The solve applies Phi^-1 in that factored form; the explicit blocks
// S_jj^-1 and -S_jj^-1 S_{j,j-1} S_{j-1,j-1}^-1 are formed only for export
// (k_rows_phi_diag, k_rows_phi_off, launched by gato_get_schur).
//
// Every kernel is compiled for column widths PN >= n (8, 12, 14 or 16) and
// PM >= m (8 or 16), and its row routines touch only that many columns.  The
// columns from n (or m) up to the width are padding zeros, whose products add
// exact zeros, so the results equal those of 16-wide rows with fewer
// operations.
#include "rows16.cuh"

namespace gato {
namespace {

using namespace rows;

constexpr int kKnotsPerBlock = 16;  // 8 warps, two knots each

struct Half {
    int li;        // lane within the half-warp (row index)
    long item;     // knot (or block row) index over the batch
    bool active;
    float* S0;
    float* S1;
    float* S2;
};

// a half's scratch: nmat 16 x 16 matrices (S0, S1, S2 as far as nmat goes)
__device__ __forceinline__ Half half_setup(long items, float* sm, int nmat)
{
    Half h;
    const int lane = lane_id(), warp = threadIdx.x >> 5;
    const int half = (warp << 1) | (lane >> 4);
    h.li = lane & 15;
    h.item = (long)blockIdx.x * kKnotsPerBlock + half;
    h.active = h.item < items;
    h.S0 = sm + (size_t)half * nmat * NP * NP;
    h.S1 = nmat > 1 ? h.S0 + NP * NP : nullptr;
    h.S2 = nmat > 2 ? h.S0 + 2 * NP * NP : nullptr;
    return h;
}

// debug build: the block's sixteen scratches fit its dynamic shared memory
// (the same for every half, so a failed check returns the whole block)
__device__ __forceinline__ bool rows_scratch_ok(int nmat, const Work& w, int sol)
{
    return gb_smem((size_t)kKnotsPerBlock * nmat * NP * NP * sizeof(float), w.status, sol);
}

// three blocks per SM at 80 registers (no spills at PN = 14, PM = 8; a few at
// 16 x 16)
template <int PN, int PM>
__global__ void __launch_bounds__(256, 3) k_rows_knot(Work w, const float* __restrict__ Q,
                                                   const float* __restrict__ R,
                                                   const float* __restrict__ A,
                                                   const float* __restrict__ B, uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, m = w.m, N = w.N;
    const Half h = half_setup((long)w.M * N, sm, 3);
    // inactive halves run the same code on identity data so that every lane
    // of the warp takes part in the shuffles and barriers; they store nothing
    const long item = h.active ? h.item : 0;
    const int sol = (int)(item / N), k = (int)(item % N);
    if (!rows_scratch_ok(3, w, sol)) return;
    const size_t K = (size_t)(N - 1);
    // the last knot has no control: its half still runs the control part (on
    // knot 0's data of the same solve, when there is one) so that the warp's
    // shuffles and barriers stay uniform, but stores nothing from it
    const bool has_u = k < N - 1;
    const bool store_u = h.active && has_u && N > 1;
    const int ku = has_u ? k : 0;
    const int li = h.li;

    // R_k^-1 and V = B_k R_k^-1 first, with B's rows set aside in S2 for
    // theta, then Q_k^-1 and O: at most four rows of registers are live
    float a[NP], x[NP], c[NP];
    const bool dyn = N > 1;  // a single-knot problem has no A, B, R
    if (dyn) {
        load_row<PM>(a, R + ((size_t)sol * K + ku) * m * m, m, m, li, true);
    } else {
#pragma unroll
        for (int j = 0; j < PM; ++j) a[j] = (j == li) ? 1.f : 0.f;
    }
    const bool okr = rows_cholesky<PM>(a, li, m, h.S0);
    __syncwarp();
    rows_lower_inverse<PM>(a, x, li, m, h.S0);
    rows_gram_lower<PM>(h.S0, c, li, m);  // row li of R_k^-1
    if (store_u) store_row<PM>(c, w.Rinv + sol * w.sKmm + (size_t)k * m * m, m, m, li);
    __syncwarp();
    publish<PM>(c, h.S1, li);  // R_k^-1 rows
    __syncwarp();
    float v[NP];
    {
        float brow[NP];
        if (dyn) {
            load_row<PM>(brow, B + ((size_t)sol * K + ku) * n * m, n, m, li, false);
        } else {
#pragma unroll
            for (int j = 0; j < PM; ++j) brow[j] = 0.f;
        }
        rows_mul<PM, PM>(brow, h.S1, m, v, 1.f);
        publish<PM>(brow, h.S2, li);  // B_k rows, for theta
    }
    if (store_u) store_row<PM>(v, w.V + sol * w.sKnm + (size_t)k * n * m, n, m, li);
    // Q_k^-1
    load_row<PN>(a, Q + ((size_t)sol * N + k) * n * n, n, n, li, true);
    bool ok = rows_cholesky<PN>(a, li, n, h.S0);
    if (has_u) ok = ok && okr;
    __syncwarp();
    rows_lower_inverse<PN>(a, x, li, n, h.S0);
    rows_gram_lower<PN>(h.S0, c, li, n);  // row li of Q_k^-1
    if (h.active) store_row<PN>(c, w.Qinv + sol * w.sNnn + (size_t)k * n * n, n, n, li);
    __syncwarp();
    publish<PN>(c, h.S1, li);  // Q_k^-1 rows
    __syncwarp();
    // O = S_{k+1,k} = -A_k Q_k^-1
    float o[NP];
    {
        float arow[NP];
        if (dyn) {
            load_row<PN>(arow, A + ((size_t)sol * K + ku) * n * n, n, n, li, false);
        } else {
#pragma unroll
            for (int j = 0; j < PN; ++j) arow[j] = 0.f;
        }
        rows_mul<PN, PN>(arow, h.S1, n, o, -1.f);
        publish<PN>(arow, h.S0, li);  // A_k rows, for theta
    }
    if (store_u) store_row<PN>(o, w.O + sol * w.sKnn + (size_t)k * n * n, n, n, li);
    // theta_k = A Q^-1 A^T + V B^T = -O A^T + V B^T  (into S_{k+1,k+1}'s slot)
    __syncwarp();
    float t[NP];
#pragma unroll
    for (int j = 0; j < PN; ++j) t[j] = 0.f;
    rows_mul_bt<PN, PN>(o, h.S0, n, t, -1.f);
    rows_mul_bt<PM, PN>(v, h.S2, n, t, 1.f);
    if (store_u) store_row<PN>(t, w.D + sol * w.sNnn + (size_t)(k + 1) * n * n, n, n, li);
    if (h.active && !ok && li == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

template <int PN>
__global__ void __launch_bounds__(256) k_rows_diag(Work w, uint32_t* status)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N;
    const Half h = half_setup((long)w.M * N, sm, 1);
    const long item = h.active ? h.item : 0;
    const int sol = (int)(item / N), j = (int)(item % N);
    if (!rows_scratch_ok(1, w, sol)) return;
    const int li = h.li;
    const size_t off = sol * w.sNnn + (size_t)j * n * n;

    float d[NP], q[NP];
    load_row<PN>(q, w.Qinv + off, n, n, li, false);
    if (j > 0) {
        load_row<PN>(d, w.D + off, n, n, li, false);  // theta_{j-1}
#pragma unroll
        for (int c = 0; c < PN; ++c) d[c] += q[c];
    } else {
#pragma unroll
        for (int c = 0; c < PN; ++c) d[c] = q[c];
    }
    __syncwarp();
    if (h.active) store_row<PN>(d, w.D + off, n, n, li);
    if (li >= n) {
#pragma unroll
        for (int c = 0; c < PN; ++c) d[c] = (c == li) ? 1.f : 0.f;
    }
    const bool ok = rows_cholesky<PN>(d, li, n, h.S0);
    if (h.active) store_row<PN>(d, w.L + off, n, n, li);
    float x[NP];
    rows_lower_inverse<PN>(d, x, li, n, h.S0);
    if (h.active) store_row<PN>(x, w.Linv + off, n, n, li);
    // ||L_j^-1||_F^2 = trace(S_jj^-1) >= 1 / lambda_min(S_jj)
    float f = 0.f;
#pragma unroll
    for (int k = 0; k < PN; ++k) f += (li < n) ? x[k] * x[k] : 0.f;
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) f += __shfl_xor_sync(0xffffffffu, f, o, 16);
    if (h.active && li == 0) w.dlow[sol * w.sN + j] = 1.f / f;
    if (h.active && !ok && li == 0) atomicOr(status + sol, GATO_STATUS_NONPOSITIVE_PIVOT);
}

template <int PN>
__global__ void __launch_bounds__(256) k_rows_off(Work w)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N, K = N - 1;
    const Half h = half_setup((long)w.M * K, sm, 2);
    const long item = h.active ? h.item : 0;
    const int sol = (int)(item / K), j = 1 + (int)(item % K);
    if (!rows_scratch_ok(2, w, sol)) return;
    const int li = h.li;
    const size_t dj = sol * w.sNnn + (size_t)j * n * n, dp = dj - (size_t)n * n;
    const size_t oj = sol * w.sKnn + (size_t)(j - 1) * n * n;

    float a[NP], t[NP], r[NP];
    // Nhat_j = (L_j^-1 S_{j,j-1}) L_{j-1}^-T
    load_row<PN>(a, w.O + oj, n, n, li, false);
    publish<PN>(a, h.S0, li);  // S_{j,j-1} rows
    load_row<PN>(a, w.Linv + dp, n, n, li, false);
    publish<PN>(a, h.S1, li);  // L_{j-1}^-1 rows
    __syncwarp();
    load_row<PN>(a, w.Linv + dj, n, n, li, false);
    rows_mul<PN, PN>(a, h.S0, n, t, 1.f);
#pragma unroll
    for (int c = 0; c < PN; ++c) r[c] = 0.f;
    rows_mul_bt<PN, PN>(t, h.S1, n, r, 1.f);
    if (h.active) store_row<PN>(r, w.Nh + oj, n, n, li);
}

// The explicit blocks of Phi^-1 for export (the solve applies Phi^-1 in the
// factored form L^-T (I - Nhat) L^-1): diagonal S_jj^-1 = L_j^-T L_j^-1 ...
template <int PN>
__global__ void __launch_bounds__(256) k_rows_phi_diag(Work w)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N;
    const Half h = half_setup((long)w.M * N, sm, 1);
    const long item = h.active ? h.item : 0;
    const int sol = (int)(item / N), j = (int)(item % N);
    if (!rows_scratch_ok(1, w, sol)) return;
    const int li = h.li;
    const size_t off = sol * w.sNnn + (size_t)j * n * n;
    float x[NP], c[NP];
    load_row<PN>(x, w.Linv + off, n, n, li, false);
    __syncwarp();
    publish<PN>(x, h.S0, li);
    __syncwarp();
    rows_gram_lower<PN>(h.S0, c, li, n);
    if (h.active) store_row<PN>(c, w.Pd + off, n, n, li);
}

// ... and off-diagonal -S_jj^-1 S_{j,j-1} S_{j-1,j-1}^-1
template <int PN>
__global__ void __launch_bounds__(256) k_rows_phi_off(Work w)
{
    extern __shared__ __align__(16) float sm[];
    const int n = w.n, N = w.N, K = N - 1;
    const Half h = half_setup((long)w.M * K, sm, 2);
    const long item = h.active ? h.item : 0;
    const int sol = (int)(item / K), j = 1 + (int)(item % K);
    if (!rows_scratch_ok(2, w, sol)) return;
    const int li = h.li;
    const size_t dj = sol * w.sNnn + (size_t)j * n * n, dp = dj - (size_t)n * n;
    const size_t oj = sol * w.sKnn + (size_t)(j - 1) * n * n;
    float a[NP], t[NP], r[NP];
    load_row<PN>(a, w.O + oj, n, n, li, false);
    publish<PN>(a, h.S0, li);  // S_{j,j-1} rows
    load_row<PN>(a, w.Pd + dp, n, n, li, false);
    publish<PN>(a, h.S1, li);  // S_{j-1,j-1}^-1 rows
    __syncwarp();
    load_row<PN>(a, w.Pd + dj, n, n, li, false);
    rows_mul<PN, PN>(a, h.S0, n, t, 1.f);
    // (T S_{j-1,j-1}^-1) row li: sum_k T[li][k] Pd_{j-1}[k][:]
    rows_mul<PN, PN>(t, h.S1, n, r, -1.f);
    if (h.active) store_row<PN>(r, w.Po + oj, n, n, li);
}

// nmat: the kernel's scratch matrices per half-warp (16 KB per block each)
template <typename K, typename... Args>
cudaError_t launch_rows(K kernel, int nmat, long items, cudaStream_t st, Args... args)
{
    if (items <= 0) return cudaSuccess;
    const size_t smem = (size_t)kKnotsPerBlock * nmat * NP * NP * sizeof(float);
    const long blocks = (items + kKnotsPerBlock - 1) / kKnotsPerBlock;
    kernel<<<(unsigned)blocks, 256, smem, st>>>(args...);
    return cudaGetLastError();
}

}  // namespace

bool rows_formation_supported(const Work& w) { return w.n <= NP && w.m <= NP; }

namespace {

template <int PN>
cudaError_t form_phi_w(const Work& w, cudaStream_t st)
{
    cudaError_t e = launch_rows(k_rows_phi_diag<PN>, 1, (long)w.M * w.N, st, w);
    if (e != cudaSuccess) return e;
    return launch_rows(k_rows_phi_off<PN>, 2, (long)w.M * (w.N - 1), st, w);
}

template <int PN, int PM>
cudaError_t form_rows_w(const Work& w, const float* Q, const float* R, const float* A,
                        const float* B, uint32_t* status, cudaStream_t st)
{
    const long knots = (long)w.M * w.N;
    cudaError_t e = launch_rows(k_rows_knot<PN, PM>, 3, knots, st, w, Q, R, A, B, status);
    if (e != cudaSuccess) return e;
    e = launch_rows(k_rows_diag<PN>, 1, knots, st, w, status);
    if (e != cudaSuccess) return e;
    return launch_rows(k_rows_off<PN>, 2, (long)w.M * (w.N - 1), st, w);
}

template <int PN>
cudaError_t form_rows_m(const Work& w, const float* Q, const float* R, const float* A,
                        const float* B, uint32_t* status, cudaStream_t st)
{
    return w.m <= 8 ? form_rows_w<PN, 8>(w, Q, R, A, B, status, st)
                    : form_rows_w<PN, 16>(w, Q, R, A, B, status, st);
}

}  // namespace

cudaError_t launch_form_phi(gato_handle* h, cudaStream_t st)
{
    const Work& w = h->w;
    if (h->phi_smem) return launch_form_phi_smem(h, st);
    if (w.n <= 8) return form_phi_w<8>(w, st);
    if (w.n <= 12) return form_phi_w<12>(w, st);
    if (w.n <= 14) return form_phi_w<14>(w, st);
    return form_phi_w<16>(w, st);
}

cudaError_t launch_form_rows(gato_handle* h, const float* Q, const float* R, const float* A,
                             const float* B, uint32_t* status, cudaStream_t st)
{
    const Work& w = h->w;
    if (w.n <= 8) return form_rows_m<8>(w, Q, R, A, B, status, st);
    if (w.n <= 12) return form_rows_m<12>(w, Q, R, A, B, status, st);
    if (w.n <= 14) return form_rows_m<14>(w, Q, R, A, B, status, st);
    return form_rows_m<16>(w, Q, R, A, B, status, st);
}

}  // namespace gato
