// exp2_poly.cuh -- 2^x on the FMA pipes, to take part of the softmax
// exponentials off the MUFU unit.
//
// Source: "FlashAttention-4: Algorithm and Kernel Pipelining Co-Design for
// Asymmetric Hardware Scaling" (gist.science/nl), Technische samenvatting,
// Methodologie §2: exp is emulated in software by a polynomial on the FMA
// units (degree 3 or 5), used for a subset of the values while the rest go
// to MUFU; bf16 rounding of P dominates the approximation error.
//
// Reduction: x = n + f with n = rint(x) and f in [-1/2, 1/2].  rint is taken
// by adding 1.5*2^23, which leaves n in the low mantissa bits of the sum; the
// same bits, shifted by 23, add n to the exponent field of p(f) ~ 2^f.  The
// coefficients are a relative-error minimax fit made by fit_exp2_poly.py.
#pragma once
#include "exp2_poly_coeffs.h"
#include "sm100_ptx.cuh"

namespace fa {

template <int DEG>
__device__ __forceinline__ float exp2_poly_core(float f) {
    if constexpr (DEG == 5) {
        float p = FA_EXP2_P5_C5;
        p = fmaf(p, f, FA_EXP2_P5_C4);
        p = fmaf(p, f, FA_EXP2_P5_C3);
        p = fmaf(p, f, FA_EXP2_P5_C2);
        p = fmaf(p, f, FA_EXP2_P5_C1);
        return fmaf(p, f, FA_EXP2_P5_C0);
    } else {
        float p = FA_EXP2_P3_C3;
        p = fmaf(p, f, FA_EXP2_P3_C2);
        p = fmaf(p, f, FA_EXP2_P3_C1);
        return fmaf(p, f, FA_EXP2_P3_C0);
    }
}

// Kernel variant.  Valid (relative error of the fit) for x in [-125, 64];
// inputs below -125 (including -inf) are clamped and return a value in
// (0, 2^-124], which is negligible next to the row sum (>= 1) it joins.
template <int DEG = 3>
__device__ __forceinline__ float exp2_poly(float x) {
    constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
    x = fmaxf(x, -125.0f);
    const float t = __fadd_rn(x, kShift);
    const float n = __fsub_rn(t, kShift);  // rint(x)
    const float f = __fsub_rn(x, n);       // in [-1/2, 1/2]
    const float p = exp2_poly_core<DEG>(f);
    return __int_as_float(__float_as_int(p) + (__float_as_int(t) << 23));
}

// Full-range variant for [-127, 64]: 2^n is applied in two steps (2^(n+64),
// then an IEEE multiply by 2^-64) so results in the subnormal range are
// rounded correctly instead of wrapping the exponent field.
template <int DEG = 3>
__device__ __forceinline__ float exp2_poly_full(float x) {
    constexpr float kShift = 12582912.0f;
    x = fmaxf(x, -127.0f);
    const float t = __fadd_rn(x, kShift);
    const float n = __fsub_rn(t, kShift);
    const float f = __fsub_rn(x, n);
    const float p = exp2_poly_core<DEG>(f);
    const float big = __int_as_float(__float_as_int(p) + ((__float_as_int(t) + 64) << 23));
    return __fmul_rn(big, 5.42101086242752217e-20f);  // * 2^-64
}

// Two lanes at once, the kernel variant's arithmetic with two-lane fp32
// instructions (same rounding, same results as exp2_poly<DEG> per lane).
template <int DEG>
__device__ __forceinline__ float2 exp2_poly_x2(float2 x) {
    const float2 kShift = make_float2(12582912.0f, 12582912.0f);
    x.x = fmaxf(x.x, -125.0f);
    x.y = fmaxf(x.y, -125.0f);
    const float2 t = add2(x, kShift);
    const float2 n = add2(t, make_float2(-12582912.0f, -12582912.0f));
    const float2 f = fma2(n, make_float2(-1.0f, -1.0f), x);
    float2 p;
    if constexpr (DEG == 5) {
        p = fma2(make_float2(FA_EXP2_P5_C5, FA_EXP2_P5_C5), f,
                 make_float2(FA_EXP2_P5_C4, FA_EXP2_P5_C4));
        p = fma2(p, f, make_float2(FA_EXP2_P5_C3, FA_EXP2_P5_C3));
        p = fma2(p, f, make_float2(FA_EXP2_P5_C2, FA_EXP2_P5_C2));
        p = fma2(p, f, make_float2(FA_EXP2_P5_C1, FA_EXP2_P5_C1));
        p = fma2(p, f, make_float2(FA_EXP2_P5_C0, FA_EXP2_P5_C0));
    } else {
        static_assert(DEG == 3, "degree 3 or 5");
        p = fma2(make_float2(FA_EXP2_P3_C3, FA_EXP2_P3_C3), f,
                 make_float2(FA_EXP2_P3_C2, FA_EXP2_P3_C2));
        p = fma2(p, f, make_float2(FA_EXP2_P3_C1, FA_EXP2_P3_C1));
        p = fma2(p, f, make_float2(FA_EXP2_P3_C0, FA_EXP2_P3_C0));
    }
    return make_float2(__int_as_float(__float_as_int(p.x) + (__float_as_int(t.x) << 23)),
                       __int_as_float(__float_as_int(p.y) + (__float_as_int(t.y) << 23)));
}

__device__ __forceinline__ float2 exp2_poly3_x2(float2 x) { return exp2_poly_x2<3>(x); }

}  // namespace fa
