// pcg_common.cuh -- what the PCG kernels of pcg.cu and pcg_rows.cu share: the
// kernel arguments, the block reduction and the per-solve epilogue (iteration
// count and status bits).
#pragma once

#include <cooperative_groups.h>

#include "gato_internal.cuh"

namespace gato {

namespace cg = cooperative_groups;

struct PcgArgs {
    Work w;
    Rhs rhs;
    const float* lambda0;  // original variables, [M][N][n], may be NULL
    float* lambda;
    float* dX;
    float* dU;
    int32_t* iters;
    uint32_t* status;
    float eps;
    int max_iters;
    int rule;
    int nh_smem;     // generic kernel: Nhat staged in shared memory
    int l_smem;      // packed L staged in shared memory (rule 0 only)
    int acc_iters;   // add to iters instead of storing
    int* queue;      // tiled kernel: next-solve counter, zero at launch
};

__host__ __device__ __forceinline__ size_t round4(size_t x) { return (x + 3) & ~(size_t)3; }

template <int K>
__device__ __forceinline__ void block_sum(float (&v)[K], float4* buf)
{
    static_assert(K >= 1 && K <= 3, "block_sum reduces up to three values");
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = warp_sum(v[k]);
    const int w = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (lane_id() == 0) {
        float4 t = make_float4(v[0], 0.f, 0.f, 0.f);
        if (K > 1) t.y = v[K > 1 ? 1 : 0];
        if (K > 2) t.z = v[K > 2 ? 2 : 0];
        buf[w] = t;
    }
    __syncthreads();
    float s[3] = {0.f, 0.f, 0.f};
    for (int q = 0; q < nw; ++q) {
        const float4 t = buf[q];
        s[0] += t.x;
        s[1] += t.y;
        s[2] += t.z;
    }
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = s[k];
}

// Warp partial sums written before a barrier and summed by every thread after
// it, in a fixed order (deterministic).  buf holds up to 16 float2 (one per
// warp).  post2 reduces two values at the cost of one: the first exchange
// leaves the pair sums of a in the low half-warp and those of b in the high
// half, the remaining four steps run on one value per lane.
__device__ __forceinline__ void post2(float a, float b, float2* buf)
{
    const int lane = lane_id();
    const bool hi = lane & 16;
    float keep = hi ? b : a;
    keep += __shfl_xor_sync(0xffffffffu, hi ? a : b, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    float* slot = reinterpret_cast<float*>(buf + (threadIdx.x >> 5));
    if ((lane & 15) == 0) slot[hi ? 1 : 0] = keep;
}

__device__ __forceinline__ float2 collect2(const float2* buf)
{
    // the low half-warp sums the .x fields of the (at most 16) warp slots,
    // the high half the .y fields; the full butterfly leaves every lane of a
    // half with that half's total (each level adds the same pair in both
    // lanes, so all lanes agree bit for bit), and one exchange across the
    // halves gives every lane both totals
    const int lane = lane_id(), q = lane & 15;
    const bool hi = lane & 16;
    float v = 0.f;
    if (q < (int)(blockDim.x >> 5)) {
        const float2 t = buf[q];
        v = hi ? t.y : t.x;
    }
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const float other = __shfl_xor_sync(0xffffffffu, v, 16);
    return hi ? make_float2(other, v) : make_float2(v, other);
}

// Four values at the cost of six exchanges (two post2 calls take ten): the
// exchange across the halves keeps (a, b) in the low half-warp and (c, d) in
// the high one, the next across the quarters one value per quarter, three
// more finish it.  Every value is summed in post2's tree, so a pair of post2
// slots and one post4 slot hold the same bits.  buf holds up to 16 float4.
__device__ __forceinline__ void post4(float a, float b, float c, float d, float4* buf)
{
    const int lane = lane_id();
    const bool hi = lane & 16, odd = lane & 8;
    float k0 = hi ? c : a, k1 = hi ? d : b;
    k0 += __shfl_xor_sync(0xffffffffu, hi ? a : c, 16);
    k1 += __shfl_xor_sync(0xffffffffu, hi ? b : d, 16);
    float keep = odd ? k1 : k0;
    keep += __shfl_xor_sync(0xffffffffu, odd ? k0 : k1, 8);
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) keep += __shfl_xor_sync(0xffffffffu, keep, o);
    float* slot = reinterpret_cast<float*>(buf + (threadIdx.x >> 5));
    if ((lane & 7) == 0) slot[lane >> 3] = keep;
}

// The four totals of post4's slots, in collect2's order: the eight lanes of
// quarter k sum field k, lane q adding warps q and q + 8 (collect2's first
// level) before the butterfly over the quarter; three independent exchanges
// then give every lane the other quarters' totals (one shuffle level fewer
// than collect2).
__device__ __forceinline__ float4 collect4(const float4* buf)
{
    const int lane = lane_id(), q = lane & 7, k = lane >> 3;
    const int nw = blockDim.x >> 5;
    const float* f = reinterpret_cast<const float*>(buf);
    float v = q < nw ? f[4 * q + k] : 0.f;
    v += q + 8 < nw ? f[4 * (q + 8) + k] : 0.f;
#pragma unroll
    for (int o = 4; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    const float v1 = __shfl_xor_sync(0xffffffffu, v, 8);   // field k ^ 1
    const float v2 = __shfl_xor_sync(0xffffffffu, v, 16);  // field k ^ 2
    const float v3 = __shfl_xor_sync(0xffffffffu, v, 24);  // field k ^ 3
    const bool b0 = k & 1, b1 = k & 2;
    const float lo0 = b0 ? v1 : v, lo1 = b0 ? v : v1;   // fields (k & 2), (k & 2) + 1
    const float hi0 = b0 ? v3 : v2, hi1 = b0 ? v2 : v3;  // the other pair
    return b1 ? make_float4(hi0, hi1, lo0, lo1) : make_float4(lo0, lo1, hi0, hi1);
}

__device__ __forceinline__ void finish(const PcgArgs& g, int sol, int it, bool done,
                                       bool nonfinite)
{
    if (threadIdx.x == 0) {
        if (g.acc_iters)
            g.iters[sol] += it;
        else
            g.iters[sol] = it;
        uint32_t st = 0;
        if (!done && !nonfinite) st |= GATO_STATUS_PCG_MAX_ITERS;
        if (nonfinite) st |= GATO_STATUS_NONFINITE;
        if (st) atomicOr(g.status + sol, st);
    }
}

// lambda = L^-T lambda_hat for this CTA's knots, then (after a cluster
// barrier, with the neighbours' lambda in global memory) dz by eq. (4); the
// dot products unrolled to NPX >= n (0: loops for any n)
template <int NPX = 16, typename LhatFn>
__device__ __forceinline__ void cluster_recover(cg::cluster_group& cl, const PcgArgs& g, int sol,
                                                int k0, int nk, LhatFn lhat)
{
    const Work& w = g.w;
    const int N = w.N, n = w.n, m = w.m, T = blockDim.x, tid = threadIdx.x;
    const size_t Nn = (size_t)N * n;
    float* lam = g.lambda + (size_t)sol * Nn;
    const float* gLi = w.Linv + sol * w.sNnn;
    for (int i = tid; i < nk * n; i += T) {
        const int jl = i / n, a = i - jl * n, j = k0 + jl;
        lam[(size_t)j * n + a] = strided_dot<NPX>(gLi + (size_t)j * n * n + a, n,
                                                 [&](int b) { return lhat(jl, b); }, a, n);
    }
    cl.sync();
    const float* Qi = w.Qinv + sol * w.sNnn;
    const float* Ob = w.O + sol * w.sKnn;
    const float* av = g.rhs.avec + sol * w.sNn;
    auto at = [](const float* v) { return [v](int b) { return v[b]; }; };
    for (int i = tid; i < nk * n; i += T) {
        const int kl = i / n, a = i - kl * n, k = k0 + kl;
        float x = av[(size_t)k * n + a];
        x += strided_dot<NPX>(Qi + (size_t)k * n * n + a * n, 1, at(lam + (size_t)k * n), 0, n);
        if (k < N - 1)
            x += strided_dot<NPX>(Ob + (size_t)k * n * n + a, n, at(lam + (size_t)(k + 1) * n), 0,
                                 n);
        g.dX[(size_t)sol * Nn + (size_t)k * n + a] = x;
    }
    const int ku = min(nk, N - 1 - k0);  // this CTA's knots that have a control
    const float* Vb = w.V + sol * w.sKnm;
    const float* bv = g.rhs.bvec + sol * w.sKm;
    for (int t = tid; t < ku * m; t += T) {
        const int kl = t / m, c = t - kl * m, k = k0 + kl;
        const float u = strided_dot<NPX>(Vb + (size_t)k * n * m + c, m,
                                        at(lam + (size_t)(k + 1) * n), 0, n);
        g.dU[(size_t)sol * (N - 1) * m + (size_t)k * m + c] = bv[(size_t)k * m + c] - u;
    }
}

// the register-row kernel (pcg_rows.cu): launched when it applies to the
// sizes, else cudaErrorInvalidConfiguration (the caller then takes another
// kernel)
cudaError_t launch_pcg_rows(const PcgArgs& a, size_t smem_limit, cudaStream_t st);

// the double-float kernel (pcg_ff.cu): cudaErrorInvalidConfiguration when the
// sizes are beyond it (more than 2048 rows N n, more than 1024 when n > 16, or
// its shared memory above smem_limit); a batch of at most half the SM count
// runs each solve over a cluster of two CTAs when each keeps enough rows
cudaError_t launch_pcg_ff(const PcgArgs& a, size_t smem_limit, int num_sms, cudaStream_t st);

// the four-thread quad kernel (pcg_quad.cu): 7 <= n <= 16 and N <= 128 with
// its shared memory within smem_limit, else cudaErrorInvalidConfiguration
bool pcg_quad_fits(int N, int n, int rule, size_t smem_limit);
cudaError_t launch_pcg_quad(const PcgArgs& a, size_t smem_limit, int num_sms, cudaStream_t st);

}  // namespace gato
