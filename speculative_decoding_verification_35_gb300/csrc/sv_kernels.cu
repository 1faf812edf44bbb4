// The verify step as one persistent kernel (sm_103a).
//
// The method, per sequence of a CSR-packed batch (velog "6-1편. Speculative Decoding", §2 steps 3-4,
// §2-1 accept/reject rule, §2-2 corrected distribution and sampling; greedy: "All About Transformer
// Inference", App. D steps 1-3; bonus token: "Accelerating Sonar through speculation",
// §"Speculative decoding"):
//   p_i = softmax(l_target_i / T), q_i = softmax(l_draft_i / T); accept x_i while u_i q_i(x_i) < p_i(x_i);
//   draw the first rejected slot from norm(max(0, p - q)), or a bonus token from p_gamma.
//
// Every warp of the grid is an independent worker that repeatedly takes one task:
//   statistics task (row r, 4096-column chunk c), in sequence-major order, statically strided over the
//     warps: one streaming pass over the logits (16 x 16-byte loads in flight per lane) computing the
//     raw max, the fp32 sum of exp((l - max) / T) and, greedy, the first argmax. This pass moves almost
//     all HBM traffic. The warp that finishes the last statistics task of a sequence runs its decision.
//   decision (one warp, one sequence): merge the chunk partials of each row, evaluate
//     u_i * q_i(x_i) < p_i(x_i) in fp64 for every slot, find the first rejection with a ballot, write
//     the accepted tokens and publish the sequence's sampler work (a per-sequence ready flag).
//   sampler task (sequence b, 2048 columns), claimed in sequence order in preference to statistics work:
//     the draw's weights (max(0, p - q), or p for a bonus) in float-float precision, summed per
//     512-column sub-chunk. The rows were streamed moments earlier, so these reads hit L2. The warp that
//     finishes the last sampler task of a sequence runs its find.
//   find (one warp, one sequence): exact normalisers, then the inverse CDF in fp64 over the sub-chunk
//     sums and over the 512 columns of the crossing sub-chunk.
// Precision: the accept test tolerates fp32 statistics (its decision moves by ~1e-7 of p/q); the
// inverse CDF over ~1e5 tokens does not, hence the float-float sampler with exact normalisers.
// Waits: a warp out of statistics work waits for published sampler work with a bounded spin; the launch
// is cooperative, so every CTA is resident and every awaited task is held by a running warp.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

constexpr uint32_t kSpinLimit = 1u << 21;  // polls before a wait gives up (about 1-4 s with back-off)

// ------------------------------------------------------------------------------------------------
// Memory-model helpers for data written by other warps during this launch (never through L1's
// non-coherent path).
// ------------------------------------------------------------------------------------------------
// Relaxed polling loads (no acquire on every poll: an acquire load discards the SM's L1 contents,
// which the other warps' cached data and spills would then miss). A poll that succeeds is followed by
// one fence before the published data is read.
__device__ __forceinline__ uint32_t ld_relaxed(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
// Lane 0 waits (bounded, exponential back-off) until *p >= target, then fences so the data published
// before the flag is visible. Returns false on time-out (the status word gets SV_ERR_TIMEOUT).
__device__ __forceinline__ bool wait_geq(const uint32_t* p, uint32_t target, uint32_t* status) {
    uint32_t spins = 0, ns = 64;
    while (*(const volatile uint32_t*)p < target) {
        if (++spins > (1u << 21)) {
            atomicOr(status, 1u << SV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(ns);
        ns = ns < 2048 ? 2 * ns : 2048;
    }
    __threadfence();
    return true;
}
__device__ __forceinline__ void st_release(uint32_t* p, uint32_t v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ PartialWord ld_word(const PartialWord* p) {
    return *(const volatile PartialWord*)p;
}
__device__ __forceinline__ void st_word(PartialWord* p, PartialWord v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ SeqTask ld_task(const SeqTask* p) {
    static_assert(sizeof(SeqTask) == 48 && alignof(SeqTask) == 16, "SeqTask layout");
    const int4 a = __ldcg((const int4*)p);
    const int4 c = __ldcg((const int4*)p + 1);
    const double u = __ldcg((const double*)p + 4);
    SeqTask t;
    t.mode = a.x; t.n = a.y; t.prow = a.z; t.qrow = a.w;
    t.m_p = __int_as_float(c.x); t.m_q = __int_as_float(c.y); t.rho = __int_as_float(c.z); t.out_pos = c.w;
    t.u = u;
    return t;
}

// ------------------------------------------------------------------------------------------------
// Warp reductions
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ float warp_sumf(float v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ double warp_sumd(double v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ uint32_t warp_or(uint32_t v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v |= __shfl_xor_sync(0xFFFFFFFFu, v, o);
    return v;
}
__device__ __forceinline__ int warp_min_i(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
__device__ __forceinline__ int warp_max_i(int v) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = max(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    return v;
}
// float-float butterfly: every lane ends with the same total (the pairwise steps are symmetric)
__device__ __forceinline__ double warp_sum_ff(ffacc a) {
    float hi = a.hi, lo = a.lo;
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        const float oh = __shfl_xor_sync(0xFFFFFFFFu, hi, o);
        const float ol = __shfl_xor_sync(0xFFFFFFFFu, lo, o);
        float s, e;
        two_sum(hi, oh, s, e);
        hi = s;
        lo = __fadd_rn(__fadd_rn(lo, ol), e);
    }
    return (double)hi + (double)lo;
}
// Exclusive prefix over the warp (fp64).
__device__ __forceinline__ double warp_exscan(double v, int lane) {
    double incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += y;
    }
    return incl - v;
}

// ------------------------------------------------------------------------------------------------
// CSR helpers (the offsets are validated by every CTA before any row is read).
// ------------------------------------------------------------------------------------------------
template <bool GREEDY>
__device__ __forceinline__ int32_t stat_rows(int32_t g) { return GREEDY ? g + 1 : 2 * g + 1; }

template <bool GREEDY>
__device__ __forceinline__ int32_t stat_base(const Params& P, int32_t b) {
    const int32_t o = __ldg(P.offs + b);
    return GREEDY ? o + b : 2 * o + b;
}

template <int DT>
__device__ __forceinline__ float logit_at(const void* base, size_t idx) {
    if (DT == SV_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)base + idx) << 16);
    return __ldg((const float*)base + idx);
}

// Table of 2^(j/64), j = 0..63, as float-float, from the fp64 exp2 of the CUDA math library.
__device__ __forceinline__ void fill_exp2_table(float2* tab) {
    if (threadIdx.x < 64) {
        const double v = exp2((double)threadIdx.x * (1.0 / 64.0));
        const float hi = (float)v;
        tab[threadIdx.x] = make_float2(hi, (float)(v - (double)hi));
    }
}

// ------------------------------------------------------------------------------------------------
// Statistics of one row segment [0, len) of up to 4096 columns, one warp. Result on every lane:
// m (raw max), s (sum of 2^((l - m) K), fp32; NaN when a NaN or +inf logit was seen), arg (first
// argmax, greedy), bad (greedy: NaN or +inf seen).
// ------------------------------------------------------------------------------------------------
struct SegStats {
    float m, s;
    int arg;
    uint32_t bad;
};

// Merge two partial (m, s) pairs of the same row (online softmax rescaling in fp32).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float K) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    s = (m == -INFINITY ? 0.f : s * ex2_approx((m - M) * K)) + (m2 == -INFINITY ? 0.f : s2 * ex2_approx((m2 - M) * K));
    m = M;
}

// Sampling-mode statistics of 16 x 8 bf16 values per lane (4096 columns per warp): bf16x2 max, then the
// fp32 sum of 2^((l - m) K) with packed FMA/ADD and one MUFU ex2 per value.
__device__ __forceinline__ SegStats stats_bf16(const uint4 (&v)[16], float K) {
    SegStats r{-INFINITY, 0.f, 0x7FFFFFFF, 0u};
    __nv_bfloat162 mx = __halves2bfloat162(__ushort_as_bfloat16(0xFF80), __ushort_as_bfloat16(0xFF80));
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].x));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].y));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].z));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].w));
    }
    const float m = warp_max(fmaxf(__low2float(mx), __high2float(mx)));
    float s = 0.f;
    if (m != -INFINITY) {
        const float2 K2 = make_float2(K, K);
        const float2 nmK2 = make_float2(-m * K, -m * K);
        float2 acc = make_float2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const float2 x = make_float2(bf16lo_to_f32(w[h]), bf16hi_to_f32(w[h]));
                const float2 t = __ffma2_rn(x, K2, nmK2);
                acc = __fadd2_rn(acc, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
            }
        }
        s = acc.x + acc.y;
    } else {
        // no finite maximum: only a NaN can still hide among -inf entries
        uint32_t nan = 0;
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
            for (int h = 0; h < 4; ++h)
                nan |= ((w[h] & 0x7F80u) == 0x7F80u && (w[h] & 0x7Fu)) ||
                       ((w[h] & 0x7F800000u) == 0x7F800000u && (w[h] & 0x7F0000u));
        }
        s = nan ? __int_as_float(0x7FC00000) : 0.f;
    }
    r.m = m;
    r.s = warp_sumf(s);  // a NaN or +inf logit makes this NaN (flagged by the caller)
    return r;
}

// The same statistics from a bulk-copied shared-memory stage of `len` columns.
__device__ __forceinline__ SegStats stats_bf16_smem(const unsigned char* buf, int len, int lane, float K) {
    uint4 v[16];
    const uint4* b4 = reinterpret_cast<const uint4*>(buf);
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        const int e0 = (q * 32 + lane) * 8;
        v[q] = e0 < len ? b4[q * 32 + lane] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
    }
    return stats_bf16(v, K);
}

template <int DT, bool VEC, bool GREEDY>
__device__ __forceinline__ SegStats seg_stats(const char* rowp, int len, int lane, float K) {
    SegStats r{-INFINITY, 0.f, 0x7FFFFFFF, 0u};
    if (VEC && DT == SV_BF16) {
        // 4096 columns: 16 loads of 8 bf16 per lane, all in flight before any arithmetic
        uint4 v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int e0 = (q * 32 + lane) * 8;
            v[q] = e0 < len ? ldg_stream((const uint4*)rowp + q * 32 + lane)
                            : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
        if (GREEDY) {
            float m = -INFINITY;
            int a = 0x7FFFFFFF;
            uint32_t bad = 0;
#pragma unroll
            for (int q = 0; q < 16; ++q) {
                const uint32_t w[4] = {v[q].x, v[q].y, v[q].z, v[q].w};
#pragma unroll
                for (int h = 0; h < 8; ++h) {
                    const float x = (h & 1) ? bf16hi_to_f32(w[h >> 1]) : bf16lo_to_f32(w[h >> 1]);
                    bad |= x != x;
                    if (x > m) { m = x; a = (q * 32 + lane) * 8 + h; }
                }
            }
            const float M = warp_max(m);
            r.arg = warp_min_i(m == M ? a : 0x7FFFFFFF);
            r.m = M;
            r.bad = warp_or(bad) | (M == INFINITY);
        } else {
            r = stats_bf16(v, K);
        }
        return r;
    }
    // fp32 rows (vectorised) and unaligned rows (scalar): 64 columns per lane per pass, merged online
    constexpr int kPerLane = 64;
    for (int base = 0; base < len; base += 32 * kPerLane) {
        float x[kPerLane];
        if (VEC) {
#pragma unroll
            for (int q = 0; q < kPerLane / 4; ++q) {
                const int e0 = base + (q * 32 + lane) * 4;
                const uint4 v = e0 < len ? ldg_stream((const uint4*)(rowp + (size_t)base * 4) + q * 32 + lane)
                                         : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
                x[q * 4 + 0] = __uint_as_float(v.x); x[q * 4 + 1] = __uint_as_float(v.y);
                x[q * 4 + 2] = __uint_as_float(v.z); x[q * 4 + 3] = __uint_as_float(v.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < kPerLane; ++i) {
                const int e = base + i * 32 + lane;
                x[i] = e < len ? logit_at<DT>(rowp, (size_t)e) : -INFINITY;
            }
        }
        float m = -INFINITY;
        int a = 0x7FFFFFFF;
        uint32_t bad = 0;
#pragma unroll
        for (int i = 0; i < kPerLane; ++i) {
            if (GREEDY) {
                bad |= x[i] != x[i];
                const int col = VEC ? base + ((i / 4) * 32 + lane) * 4 + (i % 4) : base + i * 32 + lane;
                if (x[i] > m) { m = x[i]; a = col; }
            } else {
                m = fmaxf(m, x[i]);
            }
        }
        const float M = warp_max(m);
        if (GREEDY) {
            const int A = warp_min_i(m == M ? a : 0x7FFFFFFF);
            bad = warp_or(bad) | (M == INFINITY);
            if (M > r.m) { r.m = M; r.arg = A; }
            r.bad |= bad;
        } else {
            float s = 0.f;
            if (M != -INFINITY) {
                const float nmK = -M * K;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) s += ex2_approx(__fmaf_rn(x[i], K, nmK));
            } else {
                bool nan = false;
#pragma unroll
                for (int i = 0; i < kPerLane; ++i) nan |= x[i] != x[i];
                s = nan ? __int_as_float(0x7FC00000) : 0.f;
            }
            s = warp_sumf(s);
            if (s != s) {
                r.s = s;
                r.m = fmaxf(r.m, M);
            } else if (r.s == r.s) {
                merge_ms(r.m, r.s, M, s, K);
            }
        }
    }
    return r;
}

// ------------------------------------------------------------------------------------------------
// Decision for sequence b (one warp): merge partials, accept tests, first rejection, outputs.
// ------------------------------------------------------------------------------------------------
template <int DT, bool GREEDY>
__device__ __noinline__ void decide(const Params& P, int32_t b, int32_t g, int32_t o0, int lane, const float2* tab) {
    const int32_t t0 = o0 + b;
    const int nrows = stat_rows<GREEDY>(g);
    const int32_t sbase = stat_base<GREEDY>(P, b);
    const int nch = P.nchA;
    const float K = P.K_hi;
    float my_m[2] = {-INFINITY, -INFINITY};
    float my_s[2] = {0.f, 0.f};
    int my_a[2] = {-1, -1};
    uint32_t err = 0;
    for (int j0 = 0; j0 < nrows; j0 += 8) {
        // lanes over chunks, 8 rows per batch with their loads in flight together
        float lm[8], ls[8];
        int la[8];
        uint32_t lf[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) { lm[k] = -INFINITY; ls[k] = 0.f; la[k] = 0x7FFFFFFF; lf[k] = 0u; }
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int c = c0 + lane;
            PartialWord q[8];
#pragma unroll
            for (int k = 0; k < 8; ++k)
                q[k] = (j0 + k < nrows && c < nch) ? ld_word(P.partials + (size_t)(sbase + j0 + k) * nch + c) : 1ull;
            // words still 0 are statistics tasks in flight: poll them (bounded back-off)
            uint32_t spins = 0, ns = 64;
            while (__any_sync(0xFFFFFFFFu, q[0] == 0 || q[1] == 0 || q[2] == 0 || q[3] == 0 || q[4] == 0 ||
                                               q[5] == 0 || q[6] == 0 || q[7] == 0)) {
                if (++spins > (1u << 21)) {
                    if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                    err |= 1u << SV_ERR_TIMEOUT;
                    break;
                }
                __nanosleep(ns);
                ns = ns < 2048 ? 2 * ns : 2048;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (q[k] == 0) q[k] = ld_word(P.partials + (size_t)(sbase + j0 + k) * nch + c);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (j0 + k >= nrows || c >= nch) continue;
                const float qm = __uint_as_float((uint32_t)q[k]);
                const uint32_t qh = (uint32_t)(q[k] >> 32);
                if (GREEDY) {
                    if (qh >> 31) lf[k] |= 1u << SV_ERR_NONFINITE;
                    if (qm > lm[k]) { lm[k] = qm; la[k] = (int)(qh & 0x7FFFFFFFu) - 1; }
                } else {
                    const float qs = __uint_as_float(qh);
                    if (qs != qs) {
                        ls[k] = qs;
                        lm[k] = fmaxf(lm[k], qm);
                    } else if (ls[k] == ls[k]) {
                        merge_ms(lm[k], ls[k], qm, qs, K);
                    }
                }
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int jr = j0 + k;
            if (jr >= nrows) break;
            const float M = warp_max(lm[k]);
            float v = 0.f;
            int a = 0x7FFFFFFF;
            if (GREEDY) {
                a = warp_min_i(lm[k] == M ? la[k] : 0x7FFFFFFF);
            } else {
                v = ls[k] != ls[k] ? ls[k] : (lm[k] == -INFINITY ? 0.f : ls[k] * ex2_approx((lm[k] - M) * K));
                v = warp_sumf(v);
            }
            // a row with a NaN or +inf is reported as such, not as empty (both fail the sequence)
            const uint32_t rf = warp_or(lf[k]) | (v != v ? 1u << SV_ERR_NONFINITE : 0u);
            err |= rf;
            if (M == -INFINITY && !rf) err |= 1u << SV_ERR_EMPTY_ROW;
            if (lane == (jr & 31)) {
                my_m[jr >> 5] = M;
                my_s[jr >> 5] = v;
                my_a[jr >> 5] = a;
            }
        }
    }
    int32_t x = 0;
    if (lane < g) {
        x = __ldg(P.tokens + o0 + lane);
        if (x < 0 || x >= P.V) err |= 1u << SV_ERR_BAD_TOKEN;
    }
    err = warp_or(err);
    if (err) {
        if (lane == 0) {
            atomicOr(P.status, err);
            P.out_n[b] = -1;
            if (!GREEDY) {
                SeqTask tk{};
                tk.mode = kModeNone;
                P.tasks[b] = tk;
            }
        }
        for (int32_t j = lane; j <= g; j += 32) P.out_tokens[t0 + j] = -1;
        return;
    }
    if (GREEDY) {
        const int a = my_a[0];  // argmax of target row `lane` (lane <= g <= 31)
        if (lane <= g && P.dbg.row_argmax) P.dbg.row_argmax[t0 + lane] = a;
        const uint32_t mism = __ballot_sync(0xFFFFFFFFu, lane < g && x != a);
        const int n = mism ? __ffs(mism) - 1 : g;
        if (lane <= g) P.out_tokens[t0 + lane] = lane < n ? x : (lane == n ? a : -1);
        if (lane == 0) P.out_n[b] = n;
        return;
    }
    // the draft row of slot `lane` is statistics row g + 1 + lane: lane (g+1+lane) & 31, register >> 5
    const int jd = g + 1 + lane;
    const float dm0 = __shfl_sync(0xFFFFFFFFu, my_m[0], jd & 31), dm1 = __shfl_sync(0xFFFFFFFFu, my_m[1], jd & 31);
    const float ds0 = __shfl_sync(0xFFFFFFFFu, my_s[0], jd & 31), ds1 = __shfl_sync(0xFFFFFFFFu, my_s[1], jd & 31);
    const float dm = (jd >> 5) ? dm1 : dm0, ds = (jd >> 5) ? ds1 : ds0;
    bool acc = true;
    if (lane < g) {
        // p(x) and q(x) from the precise exponential of the exact logit gaps, over the fp32 normalisers
        const float lt = logit_at<DT>(P.target, (size_t)(t0 + lane) * P.V + x);
        const float ld = logit_at<DT>(P.draft, (size_t)(o0 + lane) * P.V + x);
        const ff2 e = exp2_ff2(make_float2(lt, ld), make_float2(my_m[0], dm), P.K_hi, P.K_lo, tab);
        const float px = __fdiv_rn(e.hi.x + e.lo.x, my_s[0]);
        const float qx = __fdiv_rn(e.hi.y + e.lo.y, ds);
        const float u = (float)philox_uniform(P.seed, P.step, (uint32_t)b, (uint32_t)lane, 0);  // exact
        acc = u * qx < px;
        if (P.dbg.p_x) P.dbg.p_x[o0 + lane] = (double)px;
        if (P.dbg.q_x) P.dbg.q_x[o0 + lane] = (double)qx;
    }
    if (P.dbg.row_lse) {
        const int32_t R_t = __ldg(P.offs + P.B) + P.B;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int jr = lane + 32 * h;
            if (jr < nrows) {
                const double lse = (double)my_m[h] * P.invT64 + log((double)my_s[h]);
                P.dbg.row_lse[jr <= g ? t0 + jr : R_t + o0 + (jr - g - 1)] = lse;
            }
        }
    }
    const uint32_t rej = __ballot_sync(0xFFFFFFFFu, lane < g && !acc);
    const int n = rej ? __ffs(rej) - 1 : g;
    if (lane <= g && lane != n) P.out_tokens[t0 + lane] = lane < n ? x : -1;
    // statistics of the emitting slot's rows
    const float pm = __shfl_sync(0xFFFFFFFFu, my_m[0], n), ps = __shfl_sync(0xFFFFFFFFu, my_s[0], n);
    const float qm = __shfl_sync(0xFFFFFFFFu, dm, n), qs = __shfl_sync(0xFFFFFFFFu, ds, n);
    if (lane == 0) {
        SeqTask tk;
        tk.mode = n < g ? kModeResidual : kModeBonus;
        tk.n = n;
        tk.prow = t0 + n;
        tk.qrow = n < g ? o0 + n : -1;
        tk.m_p = pm;
        tk.m_q = n < g ? qm : 0.f;
        tk.rho = n < g ? (float)((double)ps / (double)qs) : 1.f;
        tk.out_pos = t0 + n;
        tk.u = philox_uniform(P.seed, P.step, (uint32_t)b, (uint32_t)n, 1);
        P.tasks[b] = tk;
        P.out_n[b] = n;
    }
}

// Publish sequence b's sampler work: lane 0 wrote the task record, and its release store orders that
// write before the flag.
__device__ __forceinline__ void publish(const Params& P, int32_t b, int lane) {
    if (lane == 0) st_release(P.seq_ready + (size_t)b * kFlagStride, 1u);
}

// ------------------------------------------------------------------------------------------------
// Sampler weights
// ------------------------------------------------------------------------------------------------
// 16 consecutive columns k0 .. k0 + 15 of `row`, kept packed (bf16: 8 words; fp32: 16 words); -inf
// past V.
struct Cols16 {
    uint32_t w[16];
};

template <int DT, bool VEC>
__device__ __forceinline__ Cols16 load_cols16(const void* base, size_t row, int32_t V, int32_t k0) {
    Cols16 c;
    const size_t off = row * (size_t)V + (size_t)k0;
    if (VEC && k0 + 16 <= V) {
        if (DT == SV_BF16) {
            const uint4* p = (const uint4*)((const unsigned short*)base + off);
            const uint4 a = __ldg(p), d = __ldg(p + 1);
            c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
            c.w[4] = d.x; c.w[5] = d.y; c.w[6] = d.z; c.w[7] = d.w;
        } else {
            const uint4* p = (const uint4*)((const float*)base + off);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint4 v = __ldg(p + i);
                c.w[4 * i] = v.x; c.w[4 * i + 1] = v.y; c.w[4 * i + 2] = v.z; c.w[4 * i + 3] = v.w;
            }
        }
    } else if (DT == SV_BF16) {
        const unsigned short* p = (const unsigned short*)base + off;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t lo = k0 + 2 * i < V ? __ldg(p + 2 * i) : 0xFF80u;
            const uint32_t hi = k0 + 2 * i + 1 < V ? __ldg(p + 2 * i + 1) : 0xFF80u;
            c.w[i] = lo | (hi << 16);
        }
    } else {
        const float* p = (const float*)base + off;
#pragma unroll
        for (int i = 0; i < 16; ++i) c.w[i] = k0 + i < V ? __float_as_uint(__ldg(p + i)) : 0xFF800000u;
    }
    return c;
}

template <int DT>
__device__ __forceinline__ float col(const Cols16& c, int e) {
    if (DT == SV_BF16) return (e & 1) ? bf16hi_to_f32(c.w[e >> 1]) : bf16lo_to_f32(c.w[e >> 1]);
    return __uint_as_float(c.w[e]);
}

// columns 2e and 2e + 1 as a float2
template <int DT>
__device__ __forceinline__ float2 col2(const Cols16& c, int e) {
    if (DT == SV_BF16) return make_float2(bf16lo_to_f32(c.w[e]), bf16hi_to_f32(c.w[e]));
    return make_float2(__uint_as_float(c.w[2 * e]), __uint_as_float(c.w[2 * e + 1]));
}

// Residual selection of two columns: p > q, judged on the approximate normaliser ratio rho. The same
// rule (same float operations) is applied by every step that sums or scans the residual.
__device__ __forceinline__ float2 sel_mask(const ff2& ep, const ff2& eq, float rho) {
    return make_float2(ep.hi.x > rho * eq.hi.x ? 1.f : 0.f, ep.hi.y > rho * eq.hi.y ? 1.f : 0.f);
}

// Inverse-CDF search over the columns [k_lo, k_hi) for the remaining target `rem`, in blocks of 512
// columns with fp64 running sums. Returns the token, or the last column of positive weight when the
// crossing is lost to rounding (or `tail_rule` asks for exactly that).
template <int DT, bool VEC>
__device__ int32_t scan_elements(const Params& P, const SeqTask& tk, bool resid, double rho, int32_t k_lo,
                                 int32_t k_hi, double rem, bool tail_rule, const float2* tab, int lane) {
    int32_t last_pos = -1;
    for (int32_t base = k_lo; base < k_hi; base += kSub) {
        const int32_t k0 = base + lane * kSubPerLane;
        const Cols16 cp = load_cols16<DT, VEC>(P.target, (size_t)tk.prow, P.V, k0);
        Cols16 cq;
        if (resid) cq = load_cols16<DT, VEC>(P.draft, (size_t)tk.qrow, P.V, k0);
        double w[16];
        double tot = 0.0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const ff2 ep = exp2_ff2(col2<DT>(cp, e), f2(tk.m_p), P.K_hi, P.K_lo, tab);
            double w0 = (double)ep.hi.x + (double)ep.lo.x, w1 = (double)ep.hi.y + (double)ep.lo.y;
            if (resid) {
                const ff2 eq = exp2_ff2(col2<DT>(cq, e), f2(tk.m_q), P.K_hi, P.K_lo, tab);
                const float2 mk = sel_mask(ep, eq, tk.rho);
                w0 = mk.x != 0.f ? fmax(0.0, w0 - rho * ((double)eq.hi.x + (double)eq.lo.x)) : 0.0;
                w1 = mk.y != 0.f ? fmax(0.0, w1 - rho * ((double)eq.hi.y + (double)eq.lo.y)) : 0.0;
            }
            if (k0 + 2 * e >= k_hi) w0 = 0.0;
            if (k0 + 2 * e + 1 >= k_hi) w1 = 0.0;
            w[2 * e] = w0;
            w[2 * e + 1] = w1;
            tot += w0 + w1;
        }
        int lastp = -1;
#pragma unroll
        for (int e = 0; e < 16; ++e)
            if (w[e] > 0.0) lastp = k0 + e;
        lastp = warp_max_i(lastp);
        if (lastp >= 0) last_pos = lastp;
        const double lpre = warp_exscan(tot, lane);
        const double btot = __shfl_sync(0xFFFFFFFFu, lpre + tot, 31);
        if (!tail_rule && btot > rem) {
            int my_k = -1;
            if (lpre + tot > rem) {
                double c = lpre;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    if (my_k < 0 && w[e] > 0.0 && c + w[e] > rem) my_k = k0 + e;
                    c += w[e];
                }
            }
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, my_k >= 0);
            if (hit) return __shfl_sync(0xFFFFFFFFu, my_k, __ffs(hit) - 1);
            return last_pos;
        }
        rem -= btot;
    }
    return last_pos;
}

// Find for sequence b (one warp): normalisers, sub-chunk search, element search, output.
template <int DT, bool VEC>
__device__ __noinline__ void find(const Params& P, int32_t b, const float2* tab, int lane) {
    const SeqTask tk = ld_task(P.tasks + b);
    if (tk.mode == kModeNone) return;
    const double2* ss = P.subs + (size_t)b * P.nsub;
    const double2* st = P.stot + (size_t)b * P.nS;
    const int nsub = P.nsub, nS = P.nS;
    double sp = 0.0, sq = 0.0;
    for (int i = lane; i < nS; i += 32) {
        const double2 v = __ldcg(st + i);
        sp += v.x;
        sq += v.y;
    }
    sp = warp_sumd(sp);
    sq = warp_sumd(sq);
    bool resid = tk.mode == kModeResidual;
    const double rho = resid ? sp / sq : 0.0;

    // level 1: units (sub-chunks, or sampler tasks for the p-only fallback); lane owns [s0, s1)
    int units = nsub;
    bool by_task = false;
    auto unit_w = [&](int i) -> double {
        if (by_task) return __ldcg(st + i).x;
        const double2 v = __ldcg(ss + i);
        return resid ? v.x - rho * v.y : v.x;
    };
    // the loads of a lane's range are issued 8 at a time, not one dependent round trip each
    auto range_sum = [&](int s0, int s1) -> double {
        double sum = 0.0;
        for (int i0 = s0; i0 < s1; i0 += 8) {
            double v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) v[k] = i0 + k < s1 ? unit_w(i0 + k) : 0.0;
#pragma unroll
            for (int k = 0; k < 8; ++k) sum += v[k];
        }
        return sum;
    };
    int per = (units + 31) / 32;
    int s0 = min(units, lane * per), s1 = min(units, s0 + per);
    double lsum = range_sum(s0, s1);
    double S = warp_sumd(lsum);
    if (resid && !(S > 0.0)) {  // residual mass 0 (only through rounding): draw from p
        resid = false;
        by_task = true;
        units = nS;
        per = (units + 31) / 32;
        s0 = min(units, lane * per);
        s1 = min(units, s0 + per);
        lsum = range_sum(s0, s1);
        S = warp_sumd(lsum);
    }
    const double target = tk.u * S;
    const double pre = warp_exscan(lsum, lane);
    int unit = -1;
    double before = 0.0;
    {
        int my_u = -1;
        double my_before = 0.0;
        if (pre + lsum > target) {
            double c = pre;
            for (int i0 = s0; i0 < s1 && my_u < 0; i0 += 8) {
                double v[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) v[k] = i0 + k < s1 ? unit_w(i0 + k) : 0.0;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    if (my_u < 0 && v[k] > 0.0 && c + v[k] > target) { my_u = i0 + k; my_before = c; }
                    c += v[k];
                }
            }
        }
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, my_u >= 0);
        if (hit) {
            const int L = __ffs(hit) - 1;
            unit = __shfl_sync(0xFFFFFFFFu, my_u, L);
            before = __shfl_sync(0xFFFFFFFFu, my_before, L);
        }
    }
    bool tail_rule = false;
    if (unit < 0) {  // rounding left no crossing: the last unit with positive weight
        int last = -1;
        for (int i = s0; i < s1; ++i)
            if (unit_w(i) > 0.0) last = i;
        unit = warp_max_i(last);
        tail_rule = true;
    }
    int32_t token = -1;
    if (unit >= 0) {
        const int32_t span = by_task ? kSTask : kSub;
        const int32_t k_lo = unit * span, k_hi = min(P.V, k_lo + span);
        token = scan_elements<DT, VEC>(P, tk, resid, rho, k_lo, k_hi, target - before, tail_rule, tab, lane);
    }
    if (lane == 0) {
        P.out_tokens[tk.out_pos] = token;
        if (P.dbg.seq_mass) P.dbg.seq_mass[b] = S / sp;
    }
}

// 8 consecutive columns k0 .. k0 + 7 of `row`, packed (bf16: 4 words; fp32: 8 words); -inf past V.
struct Cols8 {
    uint32_t w[8];
};

template <int DT, bool VEC>
__device__ __forceinline__ Cols8 load_cols8(const void* base, size_t row, int32_t V, int32_t k0) {
    Cols8 c;
    const size_t off = row * (size_t)V + (size_t)k0;
    if (VEC && k0 + 8 <= V) {
        if (DT == SV_BF16) {
            const uint4 a = __ldg((const uint4*)((const unsigned short*)base + off));
            c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
        } else {
            const uint4* q = (const uint4*)((const float*)base + off);
            const uint4 a = __ldg(q), d = __ldg(q + 1);
            c.w[0] = a.x; c.w[1] = a.y; c.w[2] = a.z; c.w[3] = a.w;
            c.w[4] = d.x; c.w[5] = d.y; c.w[6] = d.z; c.w[7] = d.w;
        }
    } else if (DT == SV_BF16) {
        const unsigned short* q = (const unsigned short*)base + off;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = k0 + 2 * i < V ? __ldg(q + 2 * i) : 0xFF80u;
            const uint32_t hi = k0 + 2 * i + 1 < V ? __ldg(q + 2 * i + 1) : 0xFF80u;
            c.w[i] = lo | (hi << 16);
        }
    } else {
        const float* q = (const float*)base + off;
#pragma unroll
        for (int i = 0; i < 8; ++i) c.w[i] = k0 + i < V ? __float_as_uint(__ldg(q + i)) : 0xFF800000u;
    }
    return c;
}

template <int DT>
__device__ __forceinline__ float2 pair8(const Cols8& c, int e) {
    if (DT == SV_BF16) return make_float2(bf16lo_to_f32(c.w[e]), bf16hi_to_f32(c.w[e]));
    return make_float2(__uint_as_float(c.w[2 * e]), __uint_as_float(c.w[2 * e + 1]));
}

// Sampler task c: sequence b = c / nS, columns [i * 2048, (i + 1) * 2048) for i = c % nS. The warp walks
// the task in 8 steps of 256 columns (8 consecutive columns per lane, one 16-byte load per row,
// prefetched one step ahead); every 2 steps close a 512-column sub-chunk, whose selected sums are
// reduced over the warp and stored.
template <int DT, bool VEC>
__device__ void s_task(const Params& P, uint32_t c, const float2* tab, int lane) {
    const int32_t b = (int32_t)(c / (uint32_t)P.nS);
    const int i = (int)(c % (uint32_t)P.nS);
    uint32_t ok = 1;
    if (lane == 0) ok = wait_geq(P.seq_ready + (size_t)b * kFlagStride, 1u, P.status);  // back-off wait
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    __syncwarp();
    if (!ok) return;
    const SeqTask tk = ld_task(P.tasks + b);
    if (tk.mode != kModeNone) {
        const bool resid = tk.mode == kModeResidual;
        const float2 mp = f2(tk.m_p), mq = f2(tk.m_q);
        const int32_t cbase = i * kSTask;
        const int steps = min(kSTask / 256, (P.V - cbase + 255) / 256);
        ffacc2 Pp, Qq, A, Bq;
        Cols8 np = load_cols8<DT, VEC>(P.target, (size_t)tk.prow, P.V, cbase + 8 * lane);
        Cols8 nq;
        if (resid) nq = load_cols8<DT, VEC>(P.draft, (size_t)tk.qrow, P.V, cbase + 8 * lane);
#pragma unroll 1
        for (int e = 0; e < steps; ++e) {
            const Cols8 cp = np, cq = nq;
            if (e + 1 < steps) {
                const int32_t k1 = cbase + 256 * (e + 1) + 8 * lane;
                np = load_cols8<DT, VEC>(P.target, (size_t)tk.prow, P.V, k1);
                if (resid) nq = load_cols8<DT, VEC>(P.draft, (size_t)tk.qrow, P.V, k1);
            }
            if (resid) {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const ff2 ep = exp2_ff2(pair8<DT>(cp, h), mp, P.K_hi, P.K_lo, tab);
                    const ff2 eq = exp2_ff2(pair8<DT>(cq, h), mq, P.K_hi, P.K_lo, tab);
                    Pp.add(ep.hi, ep.lo);
                    Qq.add(eq.hi, eq.lo);
                    const float2 mk = sel_mask(ep, eq, tk.rho);
                    A.add(mul2(ep.hi, mk), mul2(ep.lo, mk));
                    Bq.add(mul2(eq.hi, mk), mul2(eq.lo, mk));
                }
            } else {
#pragma unroll
                for (int h = 0; h < 4; ++h) {
                    const ff2 ep = exp2_ff2(pair8<DT>(cp, h), mp, P.K_hi, P.K_lo, tab);
                    A.add(ep.hi, ep.lo);
                }
            }
            if ((e & 1) || e + 1 == steps) {  // a 512-column sub-chunk is complete
                const int sc = i * kSubPerTask + (e >> 1);
                const double sa = warp_sum_ff(A.fold());
                const double sb = resid ? warp_sum_ff(Bq.fold()) : 0.0;
                if (lane == 0) P.subs[(size_t)b * P.nsub + sc] = make_double2(sa, sb);
                if (!resid) {  // the p total of a bonus draw is the sum of its sub-chunk sums
                    const float hs = (float)sa;
                    Pp.add(make_float2(hs, 0.f), make_float2((float)(sa - (double)hs), 0.f));
                }
                A = ffacc2();
                Bq = ffacc2();
            }
        }
        const double sp = resid ? warp_sum_ff(Pp.fold()) : Pp.fold().value();
        const double sq = resid ? warp_sum_ff(Qq.fold()) : 0.0;
        if (lane == 0) P.stot[(size_t)b * P.nS + i] = make_double2(sp, sq);
    }
    uint32_t last = 0;
    if (lane == 0) {
        __threadfence();
        last = atomicAdd(P.s_done + b, 1u) == (uint32_t)P.nS - 1u;
    }
    last = __shfl_sync(0xFFFFFFFFu, last, 0);
    if (last) {
        __threadfence();
        find<DT, VEC>(P, b, tab, lane);
    }
}

// ------------------------------------------------------------------------------------------------
// Statistics tasks
// ------------------------------------------------------------------------------------------------
struct ATask {
    int32_t r, ch, b, g, o0;
    const char* rowp;
    int len;
};

// Row, chunk and sequence of statistics task t (sequence-major order). `cur` is a sequence cursor that
// only moves forward: a warp visits its tasks in increasing order, so the owning sequence is found
// with a couple of cached offset reads instead of a search.
template <int DT, bool GREEDY>
__device__ __forceinline__ ATask a_task_at(const Params& P, long long t, int32_t& cur, const int32_t* bases) {
    ATask at;
    at.r = (int32_t)(t / P.nchA);
    at.ch = (int32_t)(t % P.nchA);
    // bases: the sequences' first statistics rows in shared memory (small batches), else from offsets
    while (cur + 1 < P.B && (bases ? bases[cur + 1] : stat_base<GREEDY>(P, cur + 1)) <= at.r) ++cur;
    at.b = cur;
    at.o0 = __ldg(P.offs + at.b);
    at.g = __ldg(P.gammas + at.b);
    const int32_t j = at.r - (GREEDY ? at.o0 + at.b : 2 * at.o0 + at.b);
    const size_t row = j <= at.g ? (size_t)(at.o0 + at.b + j) : (size_t)(at.o0 + j - at.g - 1);
    const size_t esz = DT == SV_BF16 ? 2 : 4;
    at.rowp = (const char*)(j <= at.g ? P.target : P.draft) + (row * (size_t)P.V + (size_t)at.ch * kAChunk) * esz;
    at.len = min(kAChunk, P.V - at.ch * kAChunk);
    return at;
}

// Store the task's partial word (one 64-bit store; no fence, no counter: the decision polls the words).
template <bool GREEDY>
__device__ __forceinline__ void a_finish(const Params& P, const ATask& at, const SegStats& st, int lane) {
    if (lane == 0) {
        uint32_t hi;
        if (GREEDY) {
            const int arg = st.arg == 0x7FFFFFFF ? -1 : at.ch * kAChunk + st.arg;
            hi = (uint32_t)(arg + 1) | (st.bad ? 0x80000000u : 0u);
        } else {
            hi = __float_as_uint(st.s);
        }
        st_word(P.partials + (size_t)at.r * P.nchA + at.ch, ((PartialWord)hi << 32) | __float_as_uint(st.m));
    }
}

// Decision of sequence b, run by the warp holding its first ticket; it waits for the partials itself.
template <int DT, bool GREEDY>
__device__ void lead_decide(const Params& P, int32_t b, const float2* tab, int lane) {
    const int32_t o0 = __ldg(P.offs + b), g = __ldg(P.gammas + b);
    decide<DT, GREEDY>(P, b, g, o0, lane, tab);  // polls the sequence's partial words
    if (!GREEDY) publish(P, b, lane);
}

// A streamer warp on the bulk-copy path: its statistics tasks (statically strided over all streamers)
// arrive through a ring of kStages shared-memory stages filled by 1-D bulk copies, so up to
// kStages - 1 tasks stay in flight while one is reduced, without holding registers.
__device__ void stream_bulk(const Params& P, long long nA, unsigned char* dsmem, const int32_t* bases, int warp,
                            int lane) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(dsmem + kStreamWarps * kStages * kStageBytes) + warp * kStages;
    unsigned char* bufs = dsmem + (size_t)warp * kStages * kStageBytes;
    const long long SW = (long long)gridDim.x * kStreamWarps;
    const long long sw = (long long)blockIdx.x * kStreamWarps + warp;
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    int32_t cur_issue = 0, cur_proc = 0;
    auto issue = [&](long long t, int s) {  // lane 0
        const ATask at = a_task_at<SV_BF16, false>(P, t, cur_issue, bases);
        const uint32_t bytes = (uint32_t)at.len * 2u;
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_g2s(bufs + (size_t)s * kStageBytes, at.rowp, bytes, &bars[s]);
    };
    if (lane == 0)
        for (int s = 0; s < kStages; ++s)
            if (sw + s * SW < nA) issue(sw + s * SW, s);
    uint32_t parity = 0;  // bit s: parity of stage s's next completion
    int k = 0;
    for (long long t = sw; t < nA; t += SW, ++k) {
        const int s = k % kStages;
        const bool ok = mbar_wait(&bars[s], (parity >> s) & 1u, kSpinLimit);
        parity ^= 1u << s;
        if (!ok) {
            // a copy that never lands: report, let the copies still in flight land, stop streaming
            if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
            for (int q = 1; q < kStages; ++q) {
                const int s2 = (k + q) % kStages;
                if (t + q * SW < nA) mbar_wait(&bars[s2], (parity >> s2) & 1u, kSpinLimit);
            }
            return;
        }
        const ATask at = a_task_at<SV_BF16, false>(P, t, cur_proc, bases);
        const SegStats st = stats_bf16_smem(bufs + (size_t)s * kStageBytes, at.len, lane, P.K_hi);
        __syncwarp();
        if (lane == 0 && t + kStages * SW < nA) {
            fence_proxy_async_smem();  // this stage's reads come before the copy that overwrites it
            issue(t + kStages * SW, s);
        }
        a_finish<false>(P, at, st, lane);
    }
}

// ------------------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------------------
template <int DT, bool VEC, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 2) k_verify(const Params P) {
    constexpr bool kBulk = DT == SV_BF16 && VEC && !GREEDY;
    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ float2 tab[64];
    __shared__ int s_bad;
    __shared__ int32_t s_base[kBaseCache];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!GREEDY) fill_exp2_table(tab);
    if (tid == 0) s_bad = __ldg(P.offs) != 0;
    __syncthreads();
    // every CTA checks the whole CSR structure before any row is read (and caches small batches' row
    // bases for the statistics tasks)
    int bad = 0;
    const bool cache = P.B <= kBaseCache;
    for (int32_t b = tid; b < P.B; b += kThreads) {
        const int32_t o0 = __ldg(P.offs + b), o1 = __ldg(P.offs + b + 1), g = __ldg(P.gammas + b);
        bad |= !(g >= 0 && g <= P.max_gamma && o0 >= 0 && o1 - o0 == g);
        if (cache) s_base[b] = GREEDY ? o0 + b : 2 * o0 + b;
    }
    const int32_t* bases = cache ? s_base : nullptr;
    if (__syncthreads_or(bad) || s_bad) {
        if (blockIdx.x == 0) {
            for (int32_t b = tid; b < P.B; b += kThreads) P.out_n[b] = -1;
            if (tid == 0) atomicOr(P.status, 1u << SV_ERR_BAD_OFFSETS);
        }
        return;
    }
    const int32_t oB = __ldg(P.offs + P.B);
    const long long nA = (long long)(GREEDY ? oB + P.B : 2 * oB + P.B) * P.nchA;
    const uint32_t nStot = GREEDY ? 0u : (uint32_t)P.B * (uint32_t)P.nS;

    // Statistics. Bulk-copy path: kStreamWarps warps per CTA stream while the others start sampling at
    // once. Other paths: every warp streams its strided tasks from registers first.
    if (kBulk) {
        if (warp < kStreamWarps) stream_bulk(P, nA, dsmem, bases, warp, lane);
    } else {
        const long long W = (long long)gridDim.x * kWarps;
        int32_t cur = 0;
        for (long long a = (long long)blockIdx.x * kWarps + warp; a < nA; a += W) {
            const ATask at = a_task_at<DT, GREEDY>(P, a, cur, bases);
            const SegStats st = seg_stats<DT, VEC, GREEDY>(at.rowp, at.len, lane, P.K_hi);
            a_finish<GREEDY>(P, at, st, lane);
        }
    }
    // Tickets in sequence order. Greedy: one ticket per sequence, its decision. Sampling: nS sampler
    // tasks per sequence; the holder of a sequence's first ticket first waits for the sequence's
    // statistics, decides and publishes it; the others wait for that ready flag. Waits are bounded.
    // Only warps whose statistics tasks are done ever wait, so every awaited count is completed by warps
    // that never wait.
    const uint32_t ntick = GREEDY ? (uint32_t)P.B : nStot;
    while (true) {
        uint32_t cl = 0;
        if (lane == 0) cl = atomicAdd(&P.ctr->claim, 1u);
        cl = __shfl_sync(0xFFFFFFFFu, cl, 0);
        if (cl >= ntick) break;
        if (GREEDY) {
            lead_decide<DT, true>(P, (int32_t)cl, tab, lane);
            continue;
        }
        if (cl % (uint32_t)P.nS == 0u) lead_decide<DT, false>(P, (int32_t)(cl / (uint32_t)P.nS), tab, lane);
        s_task<DT, VEC>(P, cl, tab, lane);
    }
}

// ------------------------------------------------------------------------------------------------
// Launch
// ------------------------------------------------------------------------------------------------
template <int DT, bool VEC, bool GREEDY>
static cudaError_t launch_typed(const Params& P, cudaStream_t st) {
    constexpr bool kBulk = DT == SV_BF16 && VEC && !GREEDY;
    constexpr int smem = kBulk ? kTmaSmemBytes : 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (kBulk) {
        e = cudaFuncSetAttribute(k_verify<DT, VEC, GREEDY>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
        if (e != cudaSuccess) return e;
    }
    int sms = 0, per_sm = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_verify<DT, VEC, GREEDY>, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1 || sms < 1) return cudaErrorInvalidConfiguration;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(per_sm * sms));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_verify<DT, VEC, GREEDY>, P);
}

cudaError_t launch_verify(const Params& P, const Layout& L, void* ws, int dtype, bool vec, bool greedy,
                          cudaStream_t st) {
    if (P.B == 0) return cudaSuccess;
    const cudaError_t e = cudaMemsetAsync((char*)ws + L.zero_begin, 0, L.zero_end - L.zero_begin, st);
    if (e != cudaSuccess) return e;
    if (dtype == SV_BF16) {
        if (vec) return greedy ? launch_typed<SV_BF16, true, true>(P, st) : launch_typed<SV_BF16, true, false>(P, st);
        return greedy ? launch_typed<SV_BF16, false, true>(P, st) : launch_typed<SV_BF16, false, false>(P, st);
    }
    if (vec) return greedy ? launch_typed<SV_F32, true, true>(P, st) : launch_typed<SV_F32, true, false>(P, st);
    return greedy ? launch_typed<SV_F32, false, true>(P, st) : launch_typed<SV_F32, false, false>(P, st);
}

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t nchA = ((size_t)V + kAChunk - 1) / kAChunk;
    const size_t nsub = ((size_t)V + kSub - 1) / kSub;
    const size_t nS = ((size_t)V + kSTask - 1) / kSTask;
    Layout L;
    // the first four regions are cleared before every call, with one memset
    L.counters = 0;
    L.s_done = up(L.counters + sizeof(Counters));
    L.seq_ready = up(L.s_done + (size_t)B * sizeof(uint32_t));
    L.partials = up(L.seq_ready + (size_t)B * kFlagStride * sizeof(uint32_t));
    L.tasks = up(L.partials + (size_t)B * (2 * (size_t)max_gamma + 1) * nchA * sizeof(PartialWord));
    L.zero_begin = 0;
    L.zero_end = L.tasks;
    L.subs = up(L.tasks + (size_t)B * sizeof(SeqTask));
    L.stot = up(L.subs + (size_t)B * nsub * sizeof(double2));
    L.status = up(L.stot + (size_t)B * nS * sizeof(double2));
    L.total = up(L.status + sizeof(uint32_t));
    return L;
}

}  // namespace sv
