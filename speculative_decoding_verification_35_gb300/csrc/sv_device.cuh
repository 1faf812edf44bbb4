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
// Packed forms: two independent float-float values per register pair, so every floating-point step
// issues once for two columns (Blackwell's f32x2 add / mul / fma).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __fadd2_rn(a, make_float2(-b.x, -b.y)); }
__device__ __forceinline__ float2 mul2(float2 a, float2 b) { return __fmul2_rn(a, b); }
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) { return __ffma2_rn(a, b, c); }

struct ff2 {
    float2 hi, lo;
};

// Running sums of two independent float-float streams.
struct ffacc2 {
    float2 hi = make_float2(0.f, 0.f), lo = make_float2(0.f, 0.f);
    __device__ __forceinline__ void add(float2 h, float2 l) {
        const float2 s = add2(hi, h);
        const float2 bb = sub2(s, hi);
        const float2 e = add2(sub2(hi, sub2(s, bb)), sub2(h, bb));  // exact error of hi + h
        hi = s;
        lo = add2(lo, add2(e, l));
    }
    // sum of both streams as one float-float value (exact split of the two hi parts)
    __device__ __forceinline__ ffacc fold() const {
        ffacc r;
        float s, e;
        two_sum(hi.x, hi.y, s, e);
        r.hi = s;
        r.lo = __fadd_rn(__fadd_rn(lo.x, lo.y), e);
        return r;
    }
};

// 2^((l - m) K) for two columns, precise as exp2_ff: the subtraction split exactly (TwoSum), the
// argument carried as float-float, Tang's table step and the e^y - 1 series on |y| <= ln2/128.
// Columns whose argument is below -125.5 (including -inf logits) give exactly 0.
__device__ __forceinline__ ff2 exp2_ff2(float2 l, float2 m, float K_hi, float K_lo, const float2* tab) {
    const float2 Kh = f2(K_hi), Kl = f2(K_lo);
    // d = l - m exactly as d_hi + d_lo
    const float2 d_hi = sub2(l, m);
    const float2 bb = sub2(d_hi, l);
    const float2 d_lo = add2(sub2(l, sub2(d_hi, bb)), sub2(make_float2(-m.x, -m.y), bb));
    // t = d * K as t_hi + t_lo
    const float2 t_hi = mul2(d_hi, Kh);
    float2 t_lo = fma2(d_hi, Kh, make_float2(-t_hi.x, -t_hi.y));
    t_lo = fma2(d_hi, Kl, t_lo);
    t_lo = fma2(d_lo, Kh, t_lo);
    const bool ok0 = t_hi.x > -125.5f, ok1 = t_hi.y > -125.5f;  // false for -inf and NaN as well
    // columns that are not ok run on a harmless argument and are zeroed at the end
    const float2 tc = make_float2(ok0 ? t_hi.x : 0.f, ok1 ? t_hi.y : 0.f);
    t_lo = make_float2(ok0 ? t_lo.x : 0.f, ok1 ? t_lo.y : 0.f);
    // j = rint(64 t): adding 1.5 * 2^23 rounds to an integer held in the low mantissa bits
    const float2 jm = fma2(tc, f2(64.f), f2(12582912.f));
    const int j0 = __float_as_int(jm.x) - 0x4B400000, j1 = __float_as_int(jm.y) - 0x4B400000;
    const float2 jf = sub2(jm, f2(12582912.f));
    const float2 r = add2(fma2(jf, f2(-0.015625f), tc), t_lo);  // |r| <= 1/128 (+ rounding)
    const float2 y = fma2(r, f2(0.693145751953125f), mul2(r, f2(1.42860682030941723212e-6f)));
    float2 c = fma2(y, f2(1.0f / 24.0f), f2(1.0f / 6.0f));
    c = fma2(c, y, f2(0.5f));
    const float2 em1 = fma2(mul2(c, y), y, y);
    const float2 T0 = tab[j0 & 63], T1 = tab[j1 & 63];
    const float2 Tx = make_float2(T0.x, T1.x), Ty = make_float2(T0.y, T1.y);
    const float2 p = mul2(Tx, em1);
    const float2 pe = fma2(Tx, em1, make_float2(-p.x, -p.y));
    const float2 h = add2(Tx, p);
    float2 lo = sub2(p, sub2(h, Tx));
    lo = add2(lo, add2(pe, fma2(Ty, em1, Ty)));
    const float2 sc = make_float2(__int_as_float(((j0 >> 6) + 127) << 23), __int_as_float(((j1 >> 6) + 127) << 23));
    const float2 vh = mul2(h, sc), vl = mul2(lo, sc);
    return ff2{make_float2(ok0 ? vh.x : 0.f, ok1 ? vh.y : 0.f), make_float2(ok0 ? vl.x : 0.f, ok1 ? vl.y : 0.f)};
}

// ------------------------------------------------------------------------------------------------
// Fast (MUFU) 2^x for the statistics pass: relative error about 2^-22, ex2(-inf) = 0.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// ------------------------------------------------------------------------------------------------
// Bulk asynchronous copies (TMA, 1-D) into shared memory, completed on an mbarrier.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}
// make initialised barriers visible to the asynchronous (TMA) proxy
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// order this thread's earlier shared-memory accesses before later asynchronous-proxy writes
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}
// global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned)
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}
// Wait for phase `parity` of the barrier to complete, giving up after `limit` polls. Returns false on
// time-out.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint32_t limit) {
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(smem_addr(bar)), "r"(parity)
            : "memory");
        if (done) return true;
    }
    return false;
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
