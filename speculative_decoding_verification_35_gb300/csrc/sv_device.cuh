// Device-side building blocks of the verify step: Philox4x32-10 uniforms, float-float arithmetic
// and the precise base-2 exponential the sampler runs on. Written for sm_103a.
//
// Sources: Philox4x32-10 follows Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as
// 1, 2, 3" (SC'11). The float-float operations are the classic error-free transformations (Knuth's
// TwoSum, Dekker's product via fused multiply-add). The exponential is Tang's table method:
// 2^t = 2^n * 2^(j/128) * e^y with |y| <= ln(2)/256, the table built on the host from exp2() in
// double and the remainder by its Taylor series (written from the series, no library constants).
#pragma once
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "sv_internal.h"

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

// ------------------------------------------------------------------------------------------------
// Arithmetic on the FMA and integer pipes only. The statistics pass keeps the multi-function unit
// (MUFU: ex2, reciprocal, conversions) saturated; a warp on the critical path (a decision, a sampler
// task, a find) that needs that unit waits behind it, so those warps use these instead.
// ------------------------------------------------------------------------------------------------
// float(v), exact for v < 2^24: the low 23 bits through the 2^23 mantissa trick, bit 23 added after.
__device__ __forceinline__ float u24_to_float(uint32_t v) {
    const float lo = __fsub_rn(__uint_as_float(0x4B000000u | (v & 0x7FFFFFu)), 8388608.f);
    return (v & 0x800000u) ? __fadd_rn(lo, 8388608.f) : lo;
}

// 2^x for x <= 0 (fp32 accuracy, a few ulp): x = n + f with n = rint(x), |f| <= 1/2, and 2^f = e^(f ln 2)
// by its Taylor series to degree 7 (truncation below 5e-9 for |f ln 2| <= 0.35). 0 below -126.
__device__ __forceinline__ float exp2_fma(float x) {
    x = fmaxf(x, -127.f);
    const float jm = __fadd_rn(x, 12582912.f);  // rint(x) in the low mantissa bits
    const int n = __float_as_int(jm) - 0x4B400000;
    const float y = __fmul_rn(__fsub_rn(x, __fsub_rn(jm, 12582912.f)), 0.693147180559945309f);
    float p = __fmaf_rn(y, 1.f / 5040.f, 1.f / 720.f);
    p = __fmaf_rn(p, y, 1.f / 120.f);
    p = __fmaf_rn(p, y, 1.f / 24.f);
    p = __fmaf_rn(p, y, 1.f / 6.f);
    p = __fmaf_rn(p, y, 0.5f);
    p = __fmaf_rn(p, y, 1.f);
    p = __fmaf_rn(p, y, 1.f);
    return n >= -126 ? __fmul_rn(p, __int_as_float((n + 127) << 23)) : 0.f;
}

// a / b for finite a and b in [2^-125, 2^125] (within an ulp or so): reciprocal by Newton's iteration
// r <- r (2 - b r) from the seed with bits 0x7F000000 - bits(b), which is 2^(-e-1) (3 - m) for
// b = 2^e m, 1 <= m < 2, i.e. within 1/8 of 1/b (four steps reach float precision); then one residual
// correction of the quotient.
__device__ __forceinline__ float div_fma(float a, float b) {
    float r = __int_as_float(0x7F000000 - __float_as_int(b));
#pragma unroll
    for (int k = 0; k < 4; ++k) r = __fmul_rn(r, __fmaf_rn(-b, r, 2.f));
    const float q = __fmul_rn(a, r);
    return __fmaf_rn(r, __fmaf_rn(-b, q, a), q);
}

// Uniform of one draw: the top 24 bits of word 0, scaled by 2^-24 (exact in float).
// purpose 0: accept test of `slot`; purpose 1: the residual / bonus draw at the emitting slot.
__device__ __forceinline__ float philox_uniform(uint64_t seed, uint64_t step, uint32_t seq, uint32_t slot,
                                                uint32_t purpose) {
    const uint4 ctr = make_uint4((uint32_t)step, (uint32_t)(step >> 32), seq, (slot << 8) | (purpose & 0xFFu));
    const uint2 key = make_uint2((uint32_t)seed, (uint32_t)(seed >> 32));
    return u24_to_float(philox4x32_10(ctr, key).x >> 8) * 5.9604644775390625e-8f;  // 2^-24
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
};

// Normalised float-float arithmetic (hi = RN(hi + lo)); about 2^-44 relative accuracy, which is all
// the inverse CDF needs. Normalised values compare lexicographically.
__device__ __forceinline__ ff ff_norm(float hi, float lo) {
    ff r;
    fast_two_sum(hi, lo, r.hi, r.lo);
    return r;
}
__device__ __forceinline__ ff ff_add(ff a, ff b) {
    float s, e;
    two_sum(a.hi, b.hi, s, e);
    return ff_norm(s, __fadd_rn(e, __fadd_rn(a.lo, b.lo)));
}
__device__ __forceinline__ ff ff_sub(ff a, ff b) { return ff_add(a, ff{-b.hi, -b.lo}); }
__device__ __forceinline__ ff ff_mul(ff a, ff b) {
    const float p = __fmul_rn(a.hi, b.hi);
    float e = __fmaf_rn(a.hi, b.hi, -p);  // exact rounding error of the leading product
    e = __fmaf_rn(a.hi, b.lo, e);
    e = __fmaf_rn(a.lo, b.hi, e);
    return ff_norm(p, e);
}
// a / b: one correction step on the float quotient
__device__ __forceinline__ ff ff_div(ff a, ff b) {
    const float q1 = div_fma(a.hi, b.hi);
    const ff r = ff_sub(a, ff_mul(ff{q1, 0.f}, b));
    return ff_norm(q1, div_fma(r.hi, b.hi));
}
__device__ __forceinline__ bool ff_gt(ff a, ff b) { return a.hi > b.hi || (a.hi == b.hi && a.lo > b.lo); }

// ------------------------------------------------------------------------------------------------
// Packed forms: two independent float-float values per register pair, so every floating-point step
// issues once for two columns (Blackwell's f32x2 add / mul / fma).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float2 f2(float a) { return make_float2(a, a); }
__device__ __forceinline__ float2 add2(float2 a, float2 b) { return __fadd2_rn(a, b); }
// a - b as one packed fused multiply-add (b * -1 is exact, so this rounds exactly like a - b)
__device__ __forceinline__ float2 sub2(float2 a, float2 b) { return __ffma2_rn(b, make_float2(-1.f, -1.f), a); }
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
    // sum of both streams as one normalised float-float value (exact split of the two hi parts)
    __device__ __forceinline__ ff fold() const {
        float s, e;
        two_sum(hi.x, hi.y, s, e);
        return ff_norm(s, __fadd_rn(__fadd_rn(lo.x, lo.y), e));
    }
};

// Constants of the precise exponential: K = log2(e) / T as float-float, and the clamp of l - m that
// maps every argument at or below it (and -inf logits) to exactly 0.
struct ExpConst {
    float K_hi, K_lo;         // log2(e) / T as float-float
    float d_min;              // about -126.5 / K: 2^(d_min K) would be subnormal
};

// 2^((l - m) K) for two columns, m the row maximum (so the argument is <= 0), as float-float with
// relative error below about 4e-10. Tang's method with a 128-entry table: t = d K, j = rint(128 t),
// 2^t = 2^(j >> 7) * 2^((j & 127) / 128) * e^y, y = (t - j/128) ln 2, |y| <= ln2/256, and e^y - 1 from
// its Taylor series to degree 3 (the next term is below 3e-12).
// tab holds 2^(i/128) split in floats: tab[i] (high part) and tab[128 + i] (low part), i = 0..127.
// TWOSUM: l - m is carried as float-float. For bf16 logits l - m rounds in float only when the two
// exponents are more than 16 apart; with |m| >= 2^-4 that needs |l| >= 2^12 (a zero weight) or a
// logit within 2^-16 |m| of zero (a single rare column, error below 1e-7 of its weight), so callers
// may drop the correction for such rows (kNeedTwoSum); rows whose maximum is near zero (log-softmax
// inputs) need it for every column.
// Arguments at or below d_min K, including -inf logits, give exactly 0 (2^-126 and below only).
constexpr float kNeedTwoSum = 0.0625f;
constexpr int kExpTab = 128;
template <bool TWOSUM = true>
__device__ __forceinline__ ff2 exp2_ff2(float2 l, float2 m, const ExpConst& C, const float* tab) {
    float2 d = sub2(l, m);
    float2 dl = make_float2(0.f, 0.f);
    if (TWOSUM) {
        const float2 bb = sub2(d, l);
        dl = add2(sub2(l, sub2(d, bb)), sub2(make_float2(-m.x, -m.y), bb));
        // zero where the clamp below applies (including -inf logits, whose TwoSum error is NaN)
        dl = make_float2(d.x > C.d_min ? dl.x : 0.f, d.y > C.d_min ? dl.y : 0.f);
    }
    d = make_float2(fmaxf(d.x, C.d_min), fmaxf(d.y, C.d_min));
    // adding 1.5 * 2^16 rounds d K_hi (exact inside the fused product-add) to a multiple of 1/128: the
    // sum's unit in the last place; j lands in the low mantissa bits of jm
    const float2 jm = fma2(d, f2(C.K_hi), f2(98304.f));
    const uint32_t b0 = __float_as_uint(jm.x), b1 = __float_as_uint(jm.y);
    const float2 njf = sub2(f2(98304.f), jm);  // -j/128, exact
    // r = t - j/128 = (d K_hi - j/128) + d K_lo: |r| <= 1/256 + 2^-17, each step rounds once (<= 2^-33)
    float2 r = fma2(d, f2(C.K_hi), njf);
    r = fma2(d, f2(C.K_lo), r);
    if (TWOSUM) r = fma2(dl, f2(C.K_hi), r);
    // e^(r ln2) - 1 = r ln2 + r^2 (ln2)^2 / 2 + r^3 (ln2)^3 / 6, ln2 = L_hi + L_lo: the leading product
    // r L_hi is exact inside the last fused product-add, so em1 rounds once
    float2 c = fma2(r, f2(0.05550410866482158f), f2(0.2402265069591007f));
    c = fma2(c, r, f2(-1.904654299957768e-09f));
    const float2 em1 = fma2(r, f2(0.693147182464599609375f), mul2(c, r));
    const uint32_t i0 = b0 & (kExpTab - 1), i1 = b1 & (kExpTab - 1);
    const float2 Th = make_float2(tab[i0], tab[i1]), Tl = make_float2(tab[kExpTab + i0], tab[kExpTab + i1]);
    // Th (1 + em1) + Tl (1 + em1) as h + lo: Th - h is exact, and the fused product-add recovers
    // the rounding error of h
    const float2 h = fma2(Th, em1, Th);
    const float2 lo = add2(fma2(Th, em1, sub2(Th, h)), fma2(Tl, em1, Tl));
    // 2^n, n = floor(j / 128): (j - (j & 127)) << 16 is n in the exponent field; n = -127 gives exactly 0
    const float2 sc = make_float2(__uint_as_float(((b0 - i0) << 16) + 0x3F800000u),
                                  __uint_as_float(((b1 - i1) << 16) + 0x3F800000u));
    return ff2{mul2(h, sc), mul2(lo, sc)};
}

// 1.0f where a > b, else 0.0f (one instruction; false for NaN operands, like a > b)
__device__ __forceinline__ float gt_mask(float a, float b) {
    float r;
    asm("set.gt.f32.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

// Split of a weight w in [0, 2^E] into a part on the 2^(E-20) grid (hi) and the rest (lo, |lo| <= 2^(E-21)),
// G = 1.5 * 2^(E+3) (G = 12 for weights in [0, 1]): w + G rounds w to the grid (the unit in the last place
// of G), and sums of up to 16 grid parts (at most 2^(E+4), on a grid of 2^(E-20)) are exact in float, so
// an accumulator only needs plain adds.
__device__ __forceinline__ float2 grid_hi(float2 w, float G) { return add2(add2(w, f2(G)), f2(-G)); }
__device__ __forceinline__ float2 grid_hi(float2 w) { return grid_hi(w, 12.f); }

// The grid constant for weights below 2^(floor(e) + 1), e = the log2 of the largest weight (|e| <= 100).
__device__ __forceinline__ float grid_const(float e) {
    const int E = (int)floorf(e) + 1;
    return 3.f * __int_as_float((E + 2 + 127) << 23);  // 1.5 * 2^(E + 3)
}

// Weights of the two columns of a bf16 pair word from the value table in shared memory (see kTabCodeLo):
// both magnitudes clamped to the table's range by one bf16x2 max and one min (exact), their offsets from
// the range's start scaled by the entry size in one shift, the sign bit of each column selecting the
// table's half. x: the low column, y: the high column.
__device__ __forceinline__ ff2 tab_pair(uint32_t w, const char* vt) {
    const uint32_t a = w & 0x7FFF7FFFu;
    __nv_bfloat162 v = __hmax2(*reinterpret_cast<const __nv_bfloat162*>(&a),
                               __halves2bfloat162(__ushort_as_bfloat16((unsigned short)kTabCodeLo),
                                                  __ushort_as_bfloat16((unsigned short)kTabCodeLo)));
    v = __hmin2(v, __halves2bfloat162(__ushort_as_bfloat16((unsigned short)kTabCodeHi),
                                      __ushort_as_bfloat16((unsigned short)kTabCodeHi)));
    const uint32_t d3 = (*reinterpret_cast<const uint32_t*>(&v) - (kTabCodeLo | kTabCodeLo << 16)) << 3;
    const uint32_t o0 = (d3 & 0x7FF8u) | (w & 0x8000u);  // 8 (i + 4096 s) of the low column
    const uint32_t o1 = (d3 | (w & 0x80000000u)) >> 16;  // and of the high column
    const float2 t0 = *reinterpret_cast<const float2*>(vt + o0);
    const float2 t1 = *reinterpret_cast<const float2*>(vt + o1);
    return ff2{make_float2(t0.x, t1.x), make_float2(t0.y, t1.y)};
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
// 16-byte asynchronous copy global -> shared through L2 only (cp.async.cg), and its commit groups
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_addr(smem)), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

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
// L2 policy of the streamed logits: evicted first, so the kernel's code, the words handed between warps
// and the small index arrays stay in L2 while hundreds of megabytes stream through it.
__device__ __forceinline__ uint64_t l2_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}
// global -> shared bulk copy of `bytes` (multiple of 16, both addresses 16-byte aligned), evict-first
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(l2_evict_first())
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
