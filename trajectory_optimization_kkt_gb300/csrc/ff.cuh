// ff.cuh -- double-float arithmetic: a value is the unevaluated sum h + l of
// two floats with |l| <= ulp(h) / 2, which carries about 48 significand bits
// at fp32 instruction speed (this GPU's fp64 rate is a small fraction of its
// fp32 rate).  Built from error-free transformations:
//   TwoSum      s + e == a + b exactly, for any a, b (Knuth, TAOCP vol. 2,
//               sec. 4.2.2, Theorem B)
//   FastTwoSum  the same in three operations when |a| >= |b| (Dekker, "A
//               floating-point technique for extending the available
//               precision", Numer. Math. 18, 1971)
//   TwoProduct  p + e == a * b exactly, the error by one FMA
// and the double-length addition and multiplication of Dekker's paper (the
// addition in its "sloppy" form: the low parts are added after the error-free
// sum of the high parts, so the absolute error stays within about
// u^2 (|a| + |b|), u = 2^-24).  The __f*_rn intrinsics keep the compiler from
// contracting or reassociating the transformations.
#pragma once

#include <cuda_runtime.h>

namespace gato {

struct ff {
    float h, l;
};

__device__ __forceinline__ ff ff_of(float x) { return ff{x, 0.f}; }

__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e)
{
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// exact when |a| >= |b| or a == 0
__device__ __forceinline__ ff fast_two_sum(float a, float b)
{
    const float s = __fadd_rn(a, b);
    return ff{s, __fsub_rn(b, __fsub_rn(s, a))};
}

// a + b; commutative bit for bit (the TwoSum error is exact, so it does not
// depend on the operand order), which keeps butterfly reductions identical
// on every lane
__device__ __forceinline__ ff ff_add(ff a, ff b)
{
    float s, e;
    two_sum(a.h, b.h, s, e);
    e = __fadd_rn(e, __fadd_rn(a.l, b.l));
    return fast_two_sum(s, e);
}

__device__ __forceinline__ ff ff_neg(ff a) { return ff{-a.h, -a.l}; }

__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff_neg(b)); }

__device__ __forceinline__ ff ff_mul(ff a, ff b)
{
    const float p = __fmul_rn(a.h, b.h);
    float e = __fmaf_rn(a.h, b.h, -p);
    e = __fmaf_rn(a.h, b.l, e);
    e = __fmaf_rn(a.l, b.h, e);
    return fast_two_sum(p, e);
}

// a / b: the quotient of the high parts, corrected by the remainder
__device__ __forceinline__ ff ff_div(ff a, ff b)
{
    const float q1 = __fdiv_rn(a.h, b.h);
    const ff rem = ff_sub(a, ff_mul(b, ff_of(q1)));
    const float q2 = __fdiv_rn(rem.h, b.h);
    return fast_two_sum(q1, q2);
}

// sum_b a_b x_b for fp32 a_b and double-float x_b: the compensated dot
// product of Ogita, Rump & Oishi ("Accurate sum and dot product", SIAM J.
// Sci. Comput. 26(6), 2005, Algorithm Dot2) extended by the low parts of x:
// the products of the high parts are split exactly (TwoProduct), their sum
// is carried by TwoSum, and every rounding error plus a_b x_b.l accumulates
// in c; the result is as accurate as a sum computed in twice the working
// precision.
struct Dot2 {
    float s = 0.f, c = 0.f;
    __device__ __forceinline__ void add(float a, float xh, float xl)
    {
        const float p = __fmul_rn(a, xh);
        const float pe = __fmaf_rn(a, xh, -p);
        float t, e;
        two_sum(s, p, t, e);
        s = t;
        c = __fmaf_rn(a, xl, __fadd_rn(c, __fadd_rn(pe, e)));
    }
    __device__ __forceinline__ ff value() const
    {
        float h, l;
        two_sum(s, c, h, l);
        return ff{h, l};
    }
};

}  // namespace gato
