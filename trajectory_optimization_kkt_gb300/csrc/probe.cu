// probe.cu -- fp32 arithmetic throughput probe.  Not part of the method:
// the PCG kernels keep their operator on chip, so their roofline is the SM's
// fp32 FMA issue rate, and this probe measures that rate on the GPU at hand
// instead of assuming the nominal unit count.  Every thread runs independent
// FMA chains (enough of them to cover the FMA latency), either as scalar
// fma.rn.f32 or as the packed two-lane fma.rn.f32x2; the result is written
// only under a condition that never holds (every chain stays positive), so
// nothing is optimised away.
#include "gato_internal.cuh"

namespace {

constexpr int kChains = 8;   // independent accumulators per thread (scalar form)
constexpr int kUnroll = 16;  // FMAs per chain per loop trip

__global__ void __launch_bounds__(1024) k_probe_ffma(float* sink, int trips, float a, float b)
{
    float x[kChains];
#pragma unroll
    for (int k = 0; k < kChains; ++k) x[k] = 1e-3f * (float)(threadIdx.x + k);
    for (int i = 0; i < trips; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int k = 0; k < kChains; ++k) x[k] = fmaf(x[k], a, b);
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains; ++k) s += x[k];
    if (s < -1.f) sink[blockIdx.x] = s;  // never: every chain stays positive
}

__device__ __forceinline__ unsigned long long pack2(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

// the same number of FMAs per thread as k_probe_ffma, in half the instructions
__global__ void __launch_bounds__(1024) k_probe_ffma2(float* sink, int trips, float a, float b)
{
    unsigned long long x[kChains / 2];
    const unsigned long long av = pack2(a, a), bv = pack2(b, b);
#pragma unroll
    for (int k = 0; k < kChains / 2; ++k)
        x[k] = pack2(1e-3f * (float)(threadIdx.x + 2 * k), 1e-3f * (float)(threadIdx.x + 2 * k + 1));
    for (int i = 0; i < trips; ++i) {
#pragma unroll
        for (int u = 0; u < kUnroll; ++u)
#pragma unroll
            for (int k = 0; k < kChains / 2; ++k)
                asm volatile("fma.rn.f32x2 %0, %0, %1, %2;" : "+l"(x[k]) : "l"(av), "l"(bv));
    }
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < kChains / 2; ++k) {
        float lo, hi;
        asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(x[k]));
        s += lo + hi;
    }
    if (s < -1.f) sink[blockIdx.x] = s;  // never: every chain stays positive
}

}  // namespace

extern "C" {

long long gato_probe_fp32(int packed, int blocks, int threads, int trips, float* sink,
                          void* stream)
{
    if (blocks < 1 || threads < 32 || threads > 1024 || threads % 32 || trips < 1 || !sink)
        return GATO_ERR_INVALID_ARG;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // a = 1 - 2^-20 and b = 2^-12 keep every chain finite and away from
    // subnormals for any trip count
    const float a = 1.f - 9.5367431640625e-7f, b = 2.44140625e-4f;
    if (packed)
        k_probe_ffma2<<<blocks, threads, 0, st>>>(sink, trips, a, b);
    else
        k_probe_ffma<<<blocks, threads, 0, st>>>(sink, trips, a, b);
    if (cudaGetLastError() != cudaSuccess) return GATO_ERR_CUDA;
    return 2LL * blocks * threads * (long long)trips * kUnroll * kChains;
}

}  // extern "C"
