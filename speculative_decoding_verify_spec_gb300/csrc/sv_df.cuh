// sv_df.cuh -- double-float ("float-float") arithmetic on the FP32 pipes, for the rare
// re-draws that must reproduce the fp64 definition of the sampler.
//
// A value is hi + lo with |lo| <= ulp(hi) / 2, about 48 significant bits.  The error-free
// transformations are Knuth's TwoSum (TAOCP vol. 2, 4.2.2), Dekker's FastTwoSum and the
// FMA-based TwoProd; addition follows the "accurate double-word plus double-word" scheme of
// Joldes, Muller and Popescu (ACM TOMS 2017), division is Newton-style long division on
// the hi parts (Dekker 1971).  Every operation is written with explicitly rounded
// intrinsics so the compiler can neither contract nor reassociate them.
//
// exp_df: exp(y) for y <= 0 by Cody-Waite range reduction to sixteenths of ln2,
// y = (16 n + j) ln2 / 16 + r with ln2 / 16 split into three floats (13 + 24 + 24
// significant bits, so kk * C1 is exact for |kk| < 2^11), |r| <= ln2 / 32; then
// exp(r) = 1 + r + r^2/2 + r^3/6 in double-float plus the remaining Taylor terms
// (r^4/24 + ... + r^7/5040 < 1e-8, truncation below 2e-18) in float, times the table value
// 2^(j/16) in double-float, times 2^n exactly.  The coefficients and the table are exact
// values rounded to double-float.  y below -87 gives 0 (under the smallest normal float;
// such terms are < 1e-37 of a row's largest term).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace sv {

struct df {
    float hi, lo;
};

__device__ __forceinline__ df two_sum(float a, float b) {
    const float s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    const float err = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
    return df{s, err};
}
__device__ __forceinline__ df fast_two_sum(float a, float b) {  // requires |a| >= |b| (or a = 0)
    const float s = __fadd_rn(a, b);
    return df{s, __fsub_rn(b, __fsub_rn(s, a))};
}
__device__ __forceinline__ df two_prod(float a, float b) {
    const float p = __fmul_rn(a, b);
    return df{p, __fmaf_rn(a, b, -p)};
}
__device__ __forceinline__ df df_from(float a) { return df{a, 0.f}; }
__device__ __forceinline__ df df_neg(df x) { return df{-x.hi, -x.lo}; }

__device__ __forceinline__ df df_add(df x, df y) {
    df s = two_sum(x.hi, y.hi);
    const df t = two_sum(x.lo, y.lo);
    s = fast_two_sum(s.hi, __fadd_rn(s.lo, t.hi));
    return fast_two_sum(s.hi, __fadd_rn(s.lo, t.lo));
}
__device__ __forceinline__ df df_sub(df x, df y) { return df_add(x, df_neg(y)); }

__device__ __forceinline__ df df_mul(df x, df y) {
    df p = two_prod(x.hi, y.hi);
    float e = __fmaf_rn(x.hi, y.lo, p.lo);
    e = __fmaf_rn(x.lo, y.hi, e);
    return fast_two_sum(p.hi, e);
}
__device__ __forceinline__ df df_mul_f(df x, float f) {
    df p = two_prod(x.hi, f);
    return fast_two_sum(p.hi, __fmaf_rn(x.lo, f, p.lo));
}
// x / y: three quotient digits from the hi parts, each remainder formed exactly enough.
__device__ __forceinline__ df df_div(df x, df y) {
    const float q1 = __fdiv_rn(x.hi, y.hi);
    df r = df_sub(x, df_mul_f(y, q1));
    const float q2 = __fdiv_rn(r.hi, y.hi);
    r = df_sub(r, df_mul_f(y, q2));
    const float q3 = __fdiv_rn(r.hi, y.hi);
    const df q = fast_two_sum(q1, q2);
    return df_add(q, df_from(q3));
}
__device__ __forceinline__ df df_div_f(df x, float y) { return df_div(x, df_from(y)); }

// A running sum of fp32 terms kept as an unevaluated pair (hi, lo): TwoSum on the high
// parts, the errors gathered in lo -- ~2^-48 relative at the lengths the draws sum.
struct PairSum {
    float hi = 0.f, lo = 0.f;
    __device__ __forceinline__ void add(float x) {
        const df s = two_sum(hi, x);
        hi = s.hi;
        lo = __fadd_rn(lo, s.lo);
    }
    __device__ __forceinline__ df value() const { return fast_two_sum(hi, lo); }
};

// A running sum of double-float terms: TwoSum on the high parts, the low parts and the
// rounding errors gathered in one float -- about 2^-48 relative for sums of a few tens of
// terms of one sign, at half the cost of df_add.
struct DfSum {
    float hi = 0.f, lo = 0.f;
    __device__ __forceinline__ void add(df x) {
        const df s = two_sum(hi, x.hi);
        hi = s.hi;
        lo = __fadd_rn(lo, __fadd_rn(s.lo, x.lo));
    }
    __device__ __forceinline__ df value() const { return fast_two_sum(hi, lo); }
};

// x < y and x > y on double-float values (both normalised).
__device__ __forceinline__ bool df_lt(df x, df y) { return x.hi < y.hi || (x.hi == y.hi && x.lo < y.lo); }
__device__ __forceinline__ bool df_gt(df x, df y) { return df_lt(y, x); }
__device__ __forceinline__ bool df_pos(df x) { return x.hi > 0.f || (x.hi == 0.f && x.lo > 0.f); }

__device__ __forceinline__ df df_shfl_xor(df x, int o) {
    return df{__shfl_xor_sync(0xFFFFFFFFu, x.hi, o), __shfl_xor_sync(0xFFFFFFFFu, x.lo, o)};
}
__device__ __forceinline__ df df_shfl_up(df x, int o) {
    return df{__shfl_up_sync(0xFFFFFFFFu, x.hi, o), __shfl_up_sync(0xFFFFFFFFu, x.lo, o)};
}
__device__ __forceinline__ df df_shfl(df x, int l) {
    return df{__shfl_sync(0xFFFFFFFFu, x.hi, l), __shfl_sync(0xFFFFFFFFu, x.lo, l)};
}
// Warp sum in a fixed butterfly order (every lane gets the same value).
__device__ __forceinline__ df df_warp_sum(df x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = df_add(x, df_shfl_xor(x, o));
    return x;
}
// Inclusive warp scan in lane order.
__device__ __forceinline__ df df_warp_scan(df x, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const df w = df_shfl_up(x, o);
        if (lane >= o) x = df_add(w, x);
    }
    return x;
}

// 2^(j/16), j = 0..15, rounded to double-float (hi, lo).
static __constant__ float2 kExp2Sixteenths[16] = {
    {0x1.p+0f, 0.f},
    {0x1.0b5586p+0f, 0x1.9f3122p-25f},
    {0x1.172b84p+0f, -0x1.c15742p-27f},
    {0x1.2387a6p+0f, 0x1.ceac48p-25f},
    {0x1.306fe0p+0f, 0x1.4636e2p-25f},
    {0x1.3dea64p+0f, 0x1.824684p-25f},
    {0x1.4bfdaep+0f, -0x1.593abcp-25f},
    {0x1.5ab07ep+0f, -0x1.5bd5ecp-27f},
    {0x1.6a09e6p+0f, 0x1.9fcef4p-26f},
    {0x1.7a1148p+0f, -0x1.829fd0p-25f},
    {0x1.8ace54p+0f, 0x1.15506ep-27f},
    {0x1.9c4918p+0f, 0x1.51f848p-27f},
    {0x1.ae89fap+0f, -0x1.a94b14p-26f},
    {0x1.c199bep+0f, -0x1.3d56b2p-27f},
    {0x1.d5818ep+0f, -0x1.822dbcp-27f},
    {0x1.ea4afap+0f, 0x1.52486cp-27f},
};

// exp(y) for -87 <= y <= 0 (see the header comment); 0 below -87.  Branch-free (the argument
// is clamped and the result selected at the end), so the independent exponentials of a
// thread interleave in the instruction stream.  tab(j) returns 2^(j/16) as (hi, lo).
template <class Tab>
__device__ __forceinline__ df exp_df_core(df y, Tab tab) {
    const bool live = y.hi >= -87.f;
    if (!live) y = df{-87.f, 0.f};
    constexpr float k16InvLn2 = 0x1.715476p+4f;
    // ln2 / 16 = C1 + C2 + C3; C1 has 13 significant bits and |kk| < 2^11, so kk * C1 is exact
    constexpr float kC1 = 0x1.62ep-5f, kC2 = 0x1.0bfbe8p-19f, kC3 = 0x1.cf79acp-44f;
    const float kk = rintf(__fmul_rn(y.hi, k16InvLn2));
    df r = df_add(y, df_from(-__fmul_rn(kk, kC1)));
    r = df_sub(r, two_prod(kk, kC2));
    r = df_sub(r, df_from(__fmul_rn(kk, kC3)));  // |r| <= ln2 / 32
    // exp(r) = 1 + r + r^2/2 + r^3/6 in double-float, the rest (< 1e-8) in float
    const df r2 = df_mul(r, r);
    const df r3 = df_mul(r2, r);
    const float h = r.hi;
    float tail = __fmaf_rn(h, 0x1.a01a02p-13f, 0x1.6c16c2p-10f);  // 1/5040, 1/720
    tail = __fmaf_rn(h, tail, 0x1.111112p-7f);                    // 1/120
    tail = __fmaf_rn(h, tail, 0x1.555556p-5f);                    // 1/24
    tail = __fmul_rn(tail, __fmul_rn(r2.hi, r2.hi));
    df e = df_add(df_mul(r3, df{0x1.555556p-3f, -0x1.555556p-28f}), df_from(tail));  // r^3/6 + tail
    e = df_add(df{__fmul_rn(r2.hi, 0.5f), __fmul_rn(r2.lo, 0.5f)}, e);
    e = df_add(r, e);
    e = df_add(df_from(1.f), e);
    const int ki = int(kk);
    const float2 tj = tab(ki & 15);
    e = df_mul(e, df{tj.x, tj.y});
    const float scale = __int_as_float(((ki >> 4) + 127) << 23);  // 2^floor(kk/16) >= 2^-126
    return live ? df{__fmul_rn(e.hi, scale), __fmul_rn(e.lo, scale)} : df{0.f, 0.f};
}
__device__ __forceinline__ df exp_df(df y) {
    return exp_df_core(y, [](int j) { return kExp2Sixteenths[j]; });
}
// The same value with the table fetched by warp shuffles instead of divergent constant
// loads: every lane of the warp calls it together; tj = kExp2Sixteenths[lane & 15].
__device__ __forceinline__ df exp_df_warp(df y, float2 tj) {
    return exp_df_core(y, [&](int j) {
        return make_float2(__shfl_sync(0xFFFFFFFFu, tj.x, j), __shfl_sync(0xFFFFFFFFu, tj.y, j));
    });
}

// exp((x - M) / T) for a logit x <= M (inv_t = 1 / T): x - M exactly (TwoSum), the product
// and the exponential in double-float; a -inf logit gives 0.
__device__ __forceinline__ df weight_df(float x, float M, df inv_t) {
    const bool masked = !(x > -__int_as_float(0x7f800000));
    const df e = exp_df(df_mul(two_sum(masked ? M : x, -M), inv_t));
    return masked ? df{0.f, 0.f} : e;
}
// weight_df for a whole warp at once (see exp_df_warp).
__device__ __forceinline__ df weight_df_warp(float x, float M, df inv_t, float2 tj) {
    const bool masked = !(x > -__int_as_float(0x7f800000));
    const df e = exp_df_warp(df_mul(two_sum(masked ? M : x, -M), inv_t), tj);
    return masked ? df{0.f, 0.f} : e;
}

}  // namespace sv
