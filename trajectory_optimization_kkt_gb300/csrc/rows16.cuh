// rows16.cuh -- register-row kernels for small dense matrices (order <= 16):
// a half-warp holds one matrix, lane l keeps row l in 16 registers.  Rows of
// another lane are read through a 16 x 16 scratch in shared memory (128-bit
// loads) or with 16-wide shuffles.  Matrices of order n < 16 are padded with
// identity rows (factorisations) or zero rows (products), so every routine
// acts on diag(M, I) or on M padded with zeros.
//
// All routines use full-warp shuffles and __syncwarp: both half-warps of a
// warp must call them in the same order (uniform control flow); a half with
// nothing to do runs them on dummy data and skips its stores.
#pragma once

#include "gato_internal.cuh"

namespace gato {
namespace rows {

constexpr int NP = 16;  // padded order

// 128-bit chunks that hold the first P columns of a row
template <int P>
__host__ __device__ constexpr int chunks() { return (P + 3) / 4; }

__device__ __forceinline__ float shfl16(float v, int src)
{
    return __shfl_sync(0xffffffffu, v, src, 16);
}

// a[li] (runtime li) without dynamic register indexing
template <int P = NP>
__device__ __forceinline__ float pick(const float (&a)[NP], int li)
{
    float v = 0.f;
#pragma unroll
    for (int j = 0; j < P; ++j) v = (j == li) ? a[j] : v;
    return v;
}

// Row li of a rows x cols row-major global matrix into a (zero beyond cols);
// rows >= `rows` become identity rows when `ident`, zero rows otherwise.
template <int P = NP>
__device__ __forceinline__ void load_row(float (&a)[NP], const float* M, int rows, int cols,
                                         int li, bool ident)
{
#pragma unroll
    for (int j = 0; j < P; ++j) {
        float v = 0.f;
        if (li < rows) {
            if (j < cols) v = M[li * cols + j];
        } else if (ident && j == li) {
            v = 1.f;
        }
        a[j] = v;
    }
}

template <int P = NP>
__device__ __forceinline__ void store_row(const float (&a)[NP], float* M, int rows, int cols,
                                          int li, float s = 1.f)
{
    if (li < rows) {
#pragma unroll
        for (int j = 0; j < P; ++j)
            if (j < cols) M[li * cols + j] = s * a[j];
    }
}

// publish the first P columns of row li into the 16 x 16 scratch S (row
// stride 16; the rest of the last 128-bit chunk written as zeros)
template <int P = NP>
__device__ __forceinline__ void publish(const float (&a)[NP], float* S, int li)
{
    float4* d = reinterpret_cast<float4*>(S + li * NP);
#pragma unroll
    for (int c = 0; c < chunks<P>(); ++c)
        d[c] = make_float4(4 * c < P ? a[4 * c] : 0.f, 4 * c + 1 < P ? a[4 * c + 1] : 0.f,
                           4 * c + 2 < P ? a[4 * c + 2] : 0.f, 4 * c + 3 < P ? a[4 * c + 3] : 0.f);
}

template <int P = NP>
__device__ __forceinline__ void fetch(float (&b)[NP], const float* S, int k)
{
    const float4* s = reinterpret_cast<const float4*>(S + k * NP);
#pragma unroll
    for (int c = 0; c < chunks<P>(); ++c) {
        const float4 t = s[c];
        b[4 * c] = t.x;
        b[4 * c + 1] = t.y;
        b[4 * c + 2] = t.z;
        b[4 * c + 3] = t.w;
    }
}

// In-register Cholesky of diag(M, I) (M of order n <= P): a becomes row li of
// L, strict upper part zeroed.  A pivot <= 0 or not finite is flagged (false)
// and replaced by 1.  Column k of L reaches the other lanes through the
// 32-float scratch col (two alternating 16-float buffers): one store per lane
// and broadcast 128-bit loads per step.
template <int P = NP>
__device__ inline bool rows_cholesky(float (&a)[NP], int li, int n, float* col)
{
    bool ok = true;
#pragma unroll
    for (int k = 0; k < P; ++k) {
        if (k < n) {
            const float d = shfl16(a[k], k);
            const bool bad = !(d > 0.f) || !isfinite(d);
            ok = ok && !bad;
            const float s = bad ? 1.f : sqrtf(d);
            const float inv = 1.f / s;
            a[k] = (li == k) ? s : (li > k ? a[k] * inv : a[k]);
            float* ck = col + (k & 1) * NP;
            ck[li] = a[k];
            __syncwarp();
            float lk[NP];
            fetch<P>(lk, ck, 0);
#pragma unroll
            for (int j = k + 1; j < P; ++j)
                if (j < n && li >= j) a[j] -= a[k] * lk[j];
        }
    }
#pragma unroll
    for (int j = 0; j < P; ++j)
        if (j > li) a[j] = 0.f;
    return ok;
}

// x = row li of L^-1 (L lower of order n <= P, rows in a); the finished rows
// of L^-1 end up in the scratch S.
template <int P = NP>
__device__ inline void rows_lower_inverse(const float (&a)[NP], float (&x)[NP], int li, int n,
                                          float* S)
{
    __syncwarp();  // S may still be read by the routine before (rows_cholesky's column)
#pragma unroll
    for (int j = 0; j < P; ++j) x[j] = (j == li) ? 1.f : 0.f;
    const float inv_diag = 1.f / pick<P>(a, li);
#pragma unroll
    for (int k = 0; k < P; ++k) {
        if (k < n) {
            if (li == k) {
#pragma unroll
                for (int j = 0; j < P; ++j) x[j] *= inv_diag;
                publish<P>(x, S, k);
            }
            __syncwarp();
            if (li > k) {
                float xk[NP];
                fetch<P>(xk, S, k);
                const float lik = a[k];
#pragma unroll
                for (int j = 0; j < P; ++j) x[j] -= lik * xk[j];
            }
        }
    }
    if (li >= n) publish<P>(x, S, li);  // identity rows, so S holds all of diag(L^-1, I)
    __syncwarp();
}

// c = row li of X^T X, the rows of X in the scratch S (X lower triangular of
// order n <= P)
template <int P = NP>
__device__ __forceinline__ void rows_gram_lower(const float* S, float (&c)[NP], int li, int n)
{
#pragma unroll
    for (int j = 0; j < P; ++j) c[j] = 0.f;
#pragma unroll
    for (int k = 0; k < P; ++k) {
        if (k < n && k >= li) {
            float xk[NP];
            fetch<P>(xk, S, k);
            const float xki = S[k * NP + li];
#pragma unroll
            for (int j = 0; j < P; ++j) c[j] += xki * xk[j];
        }
    }
}

// c = s * (row li of A) * B, B's rows (kk <= PK of them, PJ columns) in the
// scratch S
template <int PK = NP, int PJ = NP>
__device__ __forceinline__ void rows_mul(const float (&a)[NP], const float* S, int kk,
                                         float (&c)[NP], float s)
{
#pragma unroll
    for (int j = 0; j < PJ; ++j) c[j] = 0.f;
#pragma unroll
    for (int k = 0; k < PK; ++k) {
        if (k < kk) {
            float bk[NP];
            fetch<PJ>(bk, S, k);
            const float ak = s * a[k];
#pragma unroll
            for (int j = 0; j < PJ; ++j) c[j] += ak * bk[j];
        }
    }
}

// c[j] += s * dot(row li of A, row j of B), B's rows (count <= PJ of them, PK
// columns) in S
template <int PK = NP, int PJ = NP>
__device__ __forceinline__ void rows_mul_bt(const float (&a)[NP], const float* S, int count,
                                            float (&c)[NP], float s)
{
#pragma unroll
    for (int j = 0; j < PJ; ++j) {
        if (j < count) {
            float bj[NP];
            fetch<PK>(bj, S, j);
            float d = 0.f;
#pragma unroll
            for (int k = 0; k < PK; ++k) d += a[k] * bj[k];
            c[j] += s * d;
        }
    }
}

// c += s * (A^T B)[li][:] = s * sum_k A[k][li] * (row k of B), the rows of A
// in SA and those of B in SB (kk <= PK rows each, PJ columns of B)
template <int PK = NP, int PJ = NP>
__device__ __forceinline__ void rows_atb(const float* SA, const float* SB, int kk, int li,
                                         float (&c)[NP], float s)
{
#pragma unroll
    for (int k = 0; k < PK; ++k) {
        if (k < kk) {
            float bk[NP];
            fetch<PJ>(bk, SB, k);
            // rows of SA were published PJ columns wide: lanes past that hold
            // padding rows of the result
            const float a = li < PJ ? s * SA[k * NP + li] : 0.f;
#pragma unroll
            for (int j = 0; j < PJ; ++j) c[j] += a * bk[j];
        }
    }
}

}  // namespace rows
}  // namespace gato
