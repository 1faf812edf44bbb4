// Device-side building blocks of the verify step: Philox4x32-10 uniforms, float-float arithmetic
// and the precise base-2 exponential the sampler runs on. Written for sm_103a.
//
// Sources: Philox4x32-10 follows Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3" (SC'11). The float-float operations are the classic error-free transformations (Knuth's
// TwoSum, Dekker's product via fused multiply-add). The exponential is Tang's table method:
// 2^t = 2^n * 2^(j/64) * e^y with |y| <= ln(2)/128, the table built on the host from exp2() in
// double and the remainder by its Taylor series (written from the series, no library constants).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

namespace sv {

// ------------------------------------------------------------------------------------------------
// Philox4x32-10: 10 rounds of the 4x32 S-box; between rounds the key advances by the Weyl
// constants (the golden ratio and sqrt(3) - 1 in 32-bit fixed point).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t m0 = 0xD2511F53u, m1 = 0xCD9E8D57u;
        const uint32_t hi0 = __umulhi(m0, c.x), lo0 = m0 * c.x;
        const uint32_t hi1 = __umulhi(m1, c.z), lo1 = m1 * c.z;
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// Uniform of one draw: the top 24 bits of word 0, scaled by 2^-24 (exact in float and double).
// purpose 0: accept test of `slot`; purpose 1: the residual / bonus draw at the emitting slot.
__device__ __forceinline__ double philox_uniform(uint64_t seed, uint64_t step, uint32_t seq,
                                                uint32_t slot, uint32_t purpose) {
    const uint4 ctr = make_uint4((uint32_t)step, (uint32_t)(step >> 32), seq, (slot << 8) | (purpose & 0xFFu));
    const uint2 key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
    return (double)(philox4x32_10(ctr, key).x >> 8) * (1.0 / 16777216.0);
}

// ------------------------------------------------------------------------------------------------
// float-float helpers
// ------------------------------------------------------------------------------------------------
struct ff {
    float hi, lo;
};

// s + e == a + b exactly (Knuth TwoSum, no precondition on magnitudes).
__device__ __forceinline__ void two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    const float bb = __fsub_rn(s, a);
    e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
}

// s + e == a + b exactly, valid when |a| >= |b| or a == 0 (Dekker's Fast2Sum).
__device__ __forceinline__ void fast_two_sum(float a, float b, float& s, float& e) {
    s = __fadd_rn(a, b);
    e = __fsub_rn(b, __fsub_rn(s, a));
}

// Running float-float sum: hi carries the bulk, lo collects exact rounding errors and small parts.
struct ffacc {
    float hi = 0.f, lo = 0.f;
    __device__ __forceinline__ void add(float h, float l) {
        float s, e;
        two_sum(hi, h, s, e);
        hi = s;
        lo = __fadd_rn(lo, __fadd_rn(e, l));
    }
    __device__ __forceinline__ double value() const { return (double)hi + (double)lo; }
};

// ------------------------------------------------------------------------------------------------
// Precise 2^t for t = d * K <= 0, d = d_hi + d_lo, K = K_hi + K_lo (float-float).
// Returns a float-float value (|lo| a few ulp(hi) at most) with relative error below about 1e-9
// (the fp32 roundings of r, y and e^y - 1, each ~3e-10 of a quantity below 0.0055); values below
// 2^-125 return 0 (they are below any weight the draw can see).
// `tab` holds 2^(j/64), j = 0..63, as (hi, lo) pairs.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ ff exp2_ff(float d_hi, float d_lo, float K_hi, float K_lo, const float2* tab) {
    const float t_hi = __fmul_rn(d_hi, K_hi);
    float t_lo = __fmaf_rn(d_hi, K_hi, -t_hi);  // exact rounding error of the product
    t_lo = __fmaf_rn(d_hi, K_lo, t_lo);
    t_lo = __fmaf_rn(d_lo, K_hi, t_lo);
    if (!(t_hi > -125.5f)) return ff{0.f, 0.f};  // also catches -inf and NaN
    const float jf = rintf(__fmul_rn(t_hi, 64.f));
    const int j = (int)jf;
    // t_hi - j/64 is exact: both are multiples of ulp(t_hi) and |difference| <= 1/128
    const float r = __fadd_rn(__fmaf_rn(jf, -0.015625f, t_hi), t_lo);
    // y = r * ln 2 with ln 2 split in two floats (hi = 0.693145751953125 exactly, 12 bits)
    const float y = __fmaf_rn(r, 0.693145751953125f, __fmul_rn(r, 1.42860682030941723212e-6f));
    // e^y - 1 = y + y^2 (1/2 + y/6 + y^2/24) + O(y^5), |y| <= 0.0055
    float c = __fmaf_rn(y, 1.0f / 24.0f, 1.0f / 6.0f);
    c = __fmaf_rn(c, y, 0.5f);
    const float em1 = __fmaf_rn(__fmul_rn(c, y), y, y);
    const float2 T = tab[j & 63];
    // 2^(j/64) * e^y = T.x + T.x*em1 + T.y*(1 + em1); the middle product is split exactly
    const float p = __fmul_rn(T.x, em1);
    const float pe = __fmaf_rn(T.x, em1, -p);
    float h, l;
    fast_two_sum(T.x, p, h, l);
    l = __fadd_rn(l, __fadd_rn(pe, __fmaf_rn(T.y, em1, T.y)));
    // scale by 2^(j >> 6): exact power-of-two multiply while the result stays normal
    const int n = j >> 6;  // floor(j / 64)
    const float sc = __int_as_float((n + 127) << 23);
    return ff{__fmul_rn(h, sc), __fmul_rn(l, sc)};
}

// ------------------------------------------------------------------------------------------------
// Fast (MUFU) 2^x for the statistics pass: relative error about 2^-22, ex2(-inf) = 0.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Streaming 16-byte load that does not allocate in L1 (each logit is read once by the stats pass).
__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

}  // namespace sv
