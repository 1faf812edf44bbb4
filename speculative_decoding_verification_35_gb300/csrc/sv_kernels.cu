// The verify step as one persistent kernel (sm_103a).
//
// The method, per sequence of a CSR-packed batch (velog "6-1편. Speculative Decoding", §2 steps 3-4,
// §2-1 accept/reject rule, §2-2 corrected distribution and sampling; greedy: "All About Transformer
// Inference", App. D steps 1-3; bonus token: "Accelerating Sonar through speculation",
// §"Speculative decoding"):
//   p_i = softmax(l_target_i / T), q_i = softmax(l_draft_i / T); accept x_i while u_i q_i(x_i) < p_i(x_i);
//   draw the first rejected slot from norm(max(0, p - q)), or a bonus token from p_gamma.
//
// Work items and who runs them (bf16 rows with 16-byte alignment take the bulk-copy path):
//   statistics task (row r, 4096-column chunk c), in sequence-major order, statically strided over the
//     streamer warps (the upper 4 warps of every CTA; every warp on the other paths): the chunk arrives
//     by a 1-D bulk copy into a shared-memory ring (two stages per streamer, evict-first in L2), and
//     the warp reduces it to the raw max and the fp32 sum of 2^((l - max) K) (greedy: first argmax).
//     One 64-bit partial word per task. This pass moves all the algorithmic HBM traffic.
//   decision (bulk-copy path with no more sequences than CTAs: CTA b's four non-streaming warps share
//     sequence b's rows, warp 0 finishing; otherwise one warp per sequence, the lower warps of the CTAs
//     by static slot): polls the sequence's partial words, merges each row (fp32 online rescaling),
//     evaluates u q(x) < p(x) for every slot with a float-float exponential of the exact logit gap,
//     takes the first rejection with a ballot, writes the accepted tokens and publishes the draw (mode,
//     slot, row maxima, approximate normaliser ratio, uniform) as self-validating task words.
//   sampler task (sequence b, 1024 columns), claimed from a counter in sequence-major order by any free
//     warp: the draw's weights max(0, p - q) (or p for a bonus) in float-float precision, stored as four
//     per-task sums and per-128-column group sums.
//   find (run by the warp that claimed the sequence's last sampler task): exact normalisers from the
//     task sums, the crossing task, the crossing group from its group sums, then the crossing column among
//     the group's 128 columns recomputed with the same float-float weights.
// Handoff: every word passed between warps is written once per call with one relaxed store into a
// region zeroed before the call and is non-zero once written, so readers poll the words themselves
// (bounded back-off); no fences, flags or counters order them.
// Precision: the accept test tolerates fp32 statistics (its decision moves by ~1e-7 of p/q, inside the
// 1e-6 band); the inverse CDF over ~1e5 tokens does not: a token boundary shifted by e is hit by the
// uniform with probability ~(tokens of positive weight) x e, so every weight carries ~1e-9 relative
// precision and the normalisers are exact sums of them.
// Waits: every wait is bounded (then SV_ERR_TIMEOUT); the launch is cooperative, so every awaited word is
// produced by a resident warp that is not waiting on the waiter.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

// ------------------------------------------------------------------------------------------------
// Words handed between warps during the launch (never read through L1's non-coherent path)
// ------------------------------------------------------------------------------------------------
// Relaxed 64-bit accesses to the words handed between warps (see Word): a word is written once per
// call with one store and is single-copy atomic, so a reader sees either 0 or the final value.
__device__ __forceinline__ Word ld_word(const Word* p) {
    Word v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_word(Word* p, Word v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_u32(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ Word pack_words(uint32_t hi32, uint32_t lo32) { return ((Word)hi32 << 32) | lo32; }
// a non-negative float-float value with the marker bit in its high part's sign
__device__ __forceinline__ Word pack_ff(ff v) { return pack_words(__float_as_uint(v.lo), __float_as_uint(v.hi) | kWordMark); }
__device__ __forceinline__ ff unpack_ff(Word w) {
    return ff{__uint_as_float((uint32_t)w & 0x7FFFFFFFu), __uint_as_float((uint32_t)(w >> 32))};
}
__device__ __forceinline__ Word shfl_word(Word v, int src) {
    return pack_words(__shfl_sync(0xFFFFFFFFu, (uint32_t)(v >> 32), src), __shfl_sync(0xFFFFFFFFu, (uint32_t)v, src));
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
// A lane's grid-split accumulator pair (two streams each) as one normalised float-float value; the two
// grid parts are combined by TwoSum, so nothing is lost when their sum leaves the grid's exact range.
__device__ __forceinline__ ff lane_ff(float2 h, float2 l) {
    float s, e;
    two_sum(h.x, h.y, s, e);
    return ff_norm(s, __fadd_rn(e, __fadd_rn(l.x, l.y)));
}
// float-float butterfly: every lane ends with the same total (ff_add is symmetric in its operands)
__device__ __forceinline__ ff warp_sum_ff(ff a) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        a = ff_add(a, ff{__shfl_xor_sync(0xFFFFFFFFu, a.hi, o), __shfl_xor_sync(0xFFFFFFFFu, a.lo, o)});
    return a;
}
// The butterfly's remaining levels o0, 2 o0, ..., 16 (a sum already complete over groups of o0 lanes).
__device__ __forceinline__ ff warp_sum_ff_from(ff a, int o0) {
#pragma unroll
    for (int o = o0; o < 32; o <<= 1)
        a = ff_add(a, ff{__shfl_xor_sync(0xFFFFFFFFu, a.hi, o), __shfl_xor_sync(0xFFFFFFFFu, a.lo, o)});
    return a;
}
// Two float-float values carried lane-wise in packed pairs (x: the first value, y: the second), so that
// two sums share each f32x2 instruction; every component takes exactly the scalar ff_add's steps.
struct ffp {
    float2 hi, lo;
};
__device__ __forceinline__ ffp ffp_add(ffp a, ffp b) {
    const float2 s = add2(a.hi, b.hi);  // TwoSum of the high parts
    const float2 bb = sub2(s, a.hi);
    const float2 e = add2(sub2(a.hi, sub2(s, bb)), sub2(b.hi, bb));
    const float2 l = add2(e, add2(a.lo, b.lo));
    const float2 h = add2(s, l);  // Fast2Sum normalisation
    return ffp{h, sub2(l, sub2(h, s))};
}
__device__ __forceinline__ ffp shfl_xor_ffp(ffp v, int o) {
    return ffp{make_float2(__shfl_xor_sync(0xFFFFFFFFu, v.hi.x, o), __shfl_xor_sync(0xFFFFFFFFu, v.hi.y, o)),
               make_float2(__shfl_xor_sync(0xFFFFFFFFu, v.lo.x, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo.y, o))};
}
// lane_ff of two accumulator pairs at once: x from (ha, la), y from (hb, lb)
__device__ __forceinline__ ffp lane_ffp(float2 ha, float2 la, float2 hb, float2 lb) {
    return ffp_add(ffp{make_float2(ha.x, hb.x), make_float2(la.x, lb.x)},
                   ffp{make_float2(ha.y, hb.y), make_float2(la.y, lb.y)});
}

// Inclusive float-float prefix over the warp.
__device__ __forceinline__ ff warp_inscan_ff(ff v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff y{__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
        if (lane >= o) v = ff_add(y, v);
    }
    return v;
}
__device__ __forceinline__ ff shfl_ff(ff v, int src) {
    return ff{__shfl_sync(0xFFFFFFFFu, v.hi, src), __shfl_sync(0xFFFFFFFFu, v.lo, src)};
}
// exclusive prefix from an inclusive one (lane 0 gets 0)
__device__ __forceinline__ ff exclusive_of(ff incl, int lane) {
    const ff y{__shfl_up_sync(0xFFFFFFFFu, incl.hi, 1), __shfl_up_sync(0xFFFFFFFFu, incl.lo, 1)};
    return lane ? y : ff{0.f, 0.f};
}

// ------------------------------------------------------------------------------------------------
// CSR helpers (the offsets are validated by every CTA before any row is read).
// ------------------------------------------------------------------------------------------------
template <bool GREEDY>
__device__ __forceinline__ int32_t stat_rows(const Params& P, int32_t g) { return GREEDY || P.pm ? g + 1 : 2 * g + 1; }

template <bool GREEDY>
__device__ __forceinline__ int32_t stat_base(const Params& P, int32_t b) {
    const int32_t o = __ldg(P.offs + b);
    return GREEDY || P.pm ? o + b : 2 * o + b;
}

template <int DT>
__device__ __forceinline__ float logit_at(const void* base, size_t idx) {
    if (DT == SV_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)base + idx) << 16);
    return __ldg((const float*)base + idx);
}

// Shared-memory copy of the table of 2^(j/128), j = 0..127 (built on the host): high parts in
// tab[0..127], low parts in tab[128..255].
__device__ __forceinline__ void fill_exp2_table(const Params& P, float* tab) {
    if (threadIdx.x < kExpTab) {
        tab[threadIdx.x] = P.exp2_tab[threadIdx.x].x;
        tab[kExpTab + threadIdx.x] = P.exp2_tab[threadIdx.x].y;
    }
}
__device__ __forceinline__ ExpConst exp_const(const Params& P) { return ExpConst{P.K_hi, P.K_lo, P.d_min}; }

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

// Merge two partial (m, s) pairs of the same row (online softmax rescaling in fp32). FMA_EXP: 2^x on the
// FMA pipe (critical-path warps) instead of the MUFU.
template <bool FMA_EXP = false>
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2, float K) {
    const float M = fmaxf(m, m2);
    if (M == -INFINITY) return;
    auto e2 = [](float x) { return FMA_EXP ? exp2_fma(x) : ex2_approx(x); };
    s = (m == -INFINITY ? 0.f : s * e2((m - M) * K)) + (m2 == -INFINITY ? 0.f : s2 * e2((m2 - M) * K));
    m = M;
}

// Sampling-mode statistics of 16 x 8 bf16 values per lane (4096 columns per warp): bf16x2 max, then the
// fp32 sum of 2^((l - m) K) with packed FMA/ADD and one MUFU ex2 per value. In two parts: the lane's
// maximum (which reads every value, so the values are in registers once it is done), then the rest.
__device__ __forceinline__ float lane_max_bf16(const uint4 (&v)[16]) {
    __nv_bfloat162 mx = __halves2bfloat162(__ushort_as_bfloat16(0xFF80), __ushort_as_bfloat16(0xFF80));
#pragma unroll
    for (int q = 0; q < 16; ++q) {
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].x));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].y));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].z));
        mx = __hmax2(mx, *reinterpret_cast<const __nv_bfloat162*>(&v[q].w));
    }
    return fmaxf(__low2float(mx), __high2float(mx));
}
__device__ __forceinline__ SegStats stats_bf16_finish(const uint4 (&v)[16], float mlane, float K) {
    SegStats r{-INFINITY, 0.f, 0x7FFFFFFF, 0u};
    const float m = warp_max(mlane);
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
__device__ __forceinline__ SegStats stats_bf16(const uint4 (&v)[16], float K) {
    return stats_bf16_finish(v, lane_max_bf16(v), K);
}

// A bulk-copied shared-memory stage of `len` columns into registers (-inf past len).
__device__ __forceinline__ void load_stage(const unsigned char* buf, int len, int lane, uint4 (&v)[16]) {
    const uint4* b4 = reinterpret_cast<const uint4*>(buf);
    if (len == kAChunk) {  // a full task (all but a row's last): no per-read guard
#pragma unroll
        for (int q = 0; q < 16; ++q) v[q] = b4[q * 32 + lane];
    } else {
#pragma unroll
        for (int q = 0; q < 16; ++q) {
            const int e0 = (q * 32 + lane) * 8;
            v[q] = e0 < len ? b4[q * 32 + lane] : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
        }
    }
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
// Fused post-verify update (spec_verify_fused; "Accelerating Sonar through speculation",
// §"MTP scheduling"): run by the one warp that writes a sequence's final token, after writing it. It
// appends the n accepted drafts (acc, lane j < n holding slot j's) and the drawn token to the sequence's
// history at its length, advances the length and writes the next input token; a failed sequence (n < 0)
// gets next token -1, and one whose history would overflow is left as it is with next token -1 and
// SV_ERR_CAPACITY.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ void commit_seq(const Params& P, int32_t b, int32_t n, int32_t acc, int32_t drawn, int lane) {
    if (!P.hist) return;
    const int32_t L = n >= 0 ? P.lens[b] : 0;
    if (n < 0 || L < 0 || (int64_t)L + n + 1 > P.cap) {
        if (lane == 0) {
            P.next[b] = -1;
            if (n >= 0) atomicOr(P.status, 1u << SV_ERR_CAPACITY);
        }
        return;
    }
    int32_t* h = P.hist + (size_t)b * (size_t)P.cap + (size_t)L;
    if (lane < n) h[lane] = acc;  // the accepted drafts
    if (lane == n) h[n] = drawn;
    if (lane == 0) {
        P.lens[b] = L + n + 1;
        P.next[b] = drawn;
    }
}

// Outputs of a failed sequence: n = -1, every slot -1, no accepted path; with the fused update, next
// token -1 and the history and length untouched.
__device__ __noinline__ void fail_outputs(const Params& P, int32_t b, int lane) {
    const int32_t o0 = __ldg(P.offs + b), g = __ldg(P.offs + b + 1) - o0;  // validated by every CTA
    for (int32_t j = lane; j <= g; j += 32) P.out_tokens[o0 + b + j] = -1;
    if (P.out_path)
        for (int32_t j = lane; j < g; j += 32) P.out_path[o0 + j] = -1;
    if (lane == 0) {
        P.out_n[b] = -1;
        if (P.hist) P.next[b] = -1;
    }
}

// A sampled sequence's outputs have one writer: its find, or a warp whose wait on the sequence gave up.
// Each claims the sequence's state word (0 -> 1 for the find, 0 -> 2 for a failure); the loser writes
// nothing. Returns the word's previous value, on every lane.
__device__ __forceinline__ uint32_t claim_seq(const Params& P, int32_t b, uint32_t who, int lane) {
    uint32_t old = 0;
    if (lane == 0) old = atomicCAS(P.seqstate + b, 0u, who);
    return __shfl_sync(0xFFFFFFFFu, old, 0);
}

// A wait on sequence b's words gave up (SV_ERR_TIMEOUT already set): fail the sequence unless its find
// holds it (the find then fails it itself, when its own wait on the missing words gives up).
__device__ __noinline__ void give_up_seq(const Params& P, int32_t b, int lane) {
    if (claim_seq(P, b, 2u, lane) == 0u) fail_outputs(P, b, lane);
}

// ------------------------------------------------------------------------------------------------
// Sampler work of a sequence (see kTaskWords)
// ------------------------------------------------------------------------------------------------
// Whether a draw's weights come from the value table (bf16 rows with 16-byte alignment, both maxima in the
// table's range; see kTabCodeLo): decided from the draw's words alone, so its decision, every sampler task
// and its find agree.
template <int DT, bool VEC>
__device__ __forceinline__ bool draw_uses_table(const Params& P, int32_t mode, float m_p, float m_q) {
    if (!(DT == SV_BF16 && VEC) || !P.use_tab) return false;
    auto ok = [&](float m) { return m >= P.tab_mlo && m <= P.tab_mhi; };
    return ok(m_p) && (mode != kModeResidual || ok(m_q));
}

// The value table in shared memory: entry (s << 12) | i = 2^(l K) as (hi, lo) for the bf16 value l of sign
// s and magnitude code kTabCodeLo + i; entry i = 0 holds l = 0 and the last negative entry 0 (see
// kTabCodeLo). Built by threads t = 0 .. nt - 1 of the CTA, two entries per exponential, with the precise
// exponential of the sampler's fallback path (l - m with m = 0 is exact). Entries whose 2^(l K) would
// leave the float range hold 2^126 and are never read by a draw that uses the table.
__device__ __noinline__ void build_value_table(const Params& P, float2* vt, const float* tab, int t, int nt) {
    const ExpConst EC{P.K_hi, P.K_lo, P.d_min};
    const float lmax = 126.f / P.K_hi;
    for (int j = 2 * t; j < 2 * kTabHalf; j += 2 * nt) {  // j, j + 1: one sign, consecutive codes
        const uint32_t sgn = (uint32_t)j >> 12, i = (uint32_t)j & (kTabHalf - 1);
        auto val = [&](uint32_t ii) {
            return ii ? fminf(__uint_as_float(((sgn << 15) | (kTabCodeLo + ii)) << 16), lmax) : 0.f;
        };
        const ff2 e = exp2_ff2<false>(make_float2(val(i), val(i + 1)), f2(0.f), EC, tab);
        vt[j] = make_float2(e.hi.x, e.lo.x);
        vt[j + 1] = sgn && i + 1 == kTabHalf - 1 ? make_float2(0.f, 0.f) : make_float2(e.hi.y, e.lo.y);
    }
}

struct TaskInfo {
    int32_t mode, n;  // n: the node (slot) whose target row the draw takes
    int32_t npos;     // the output slot of the drawn token (n itself, except in a token tree)
    float m_p, m_q, rho, u;  // rho: the selection ratio (s_p / s_q approximately; for a draw that uses the
                             // value table, in table units: times 2^((m_p - m_q) K))
    int32_t xcl;  // kModeResidualPM: the column the draw removes (the draft token); else -1
    int32_t nrm;  // tokens the draw removes: 1 (kModeResidualPM), k (kModeResidualSet), else 0
};

// Written by the decision (lanes 0-2 store one word each).
__device__ __forceinline__ void put_task(const Params& P, int32_t b, int lane, int32_t mode, int32_t n, float m_p,
                                         float m_q, float rho, float u, int32_t npos) {
    Word w = 0;
    if (lane == 0) w = pack_words(kWordMark | (uint32_t)mode << 8 | (uint32_t)n, __float_as_uint(m_p));
    if (lane == 1) w = pack_words(__float_as_uint(rho), __float_as_uint(m_q));
    if (lane == 2) w = pack_words(kWordMark | (uint32_t)npos, __float_as_uint(u));
    if (lane < 3) st_word(P.taskw + (size_t)b * kTaskWords + lane, w);
}

// Read by each sampler task: lanes 0-2 poll one word each (bounded back-off). False on time-out.
__device__ __forceinline__ bool get_task(const Params& P, int32_t b, int lane, TaskInfo& t) {
    const Word* w = P.taskw + (size_t)b * kTaskWords;
    Word v = lane < 3 ? ld_word(w + lane) : 1ull;
    uint32_t spins = 0, ns = 32;
    while (__any_sync(0xFFFFFFFFu, v == 0)) {
        if (++spins > P.spin) {
            if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(ns);
        ns = ns < 256 ? 2 * ns : 256;
        if (v == 0) v = ld_word(w + lane);
    }
    const Word w0 = shfl_word(v, 0), w1 = shfl_word(v, 1), w2 = shfl_word(v, 2);
    t.mode = (int32_t)((w0 >> 40) & 0xFF);
    t.n = (int32_t)((w0 >> 32) & 0xFF);
    t.m_p = __uint_as_float((uint32_t)w0);
    t.m_q = __uint_as_float((uint32_t)w1);
    t.rho = __uint_as_float((uint32_t)(w1 >> 32));
    t.u = __uint_as_float((uint32_t)w2);
    t.npos = (int32_t)((w2 >> 32) & 0xFFu);
    t.xcl = -1;
    t.nrm = 0;
    if (t.mode == kModeResidualPM) {
        t.xcl = (int32_t)(w1 >> 32) - 1;
        t.nrm = 1;
        t.rho = 1.f;
    } else if (t.mode == kModeResidualSet) {
        t.nrm = (int32_t)(w1 >> 32);
        t.rho = 1.f;
    }
    return true;
}

// The tokens a draw removes, one per lane (lanes 0 .. tk.nrm - 1, -1 elsewhere): the draft token of a
// point-mass residual, or a tree draw's removed-token words (polled, bounded). False on time-out.
__device__ __forceinline__ bool removed_tokens(const Params& P, int32_t b, const TaskInfo& tk, int lane, int32_t& tok) {
    tok = -1;
    if (tk.mode == kModeResidualPM) {
        tok = lane == 0 ? tk.xcl : -1;
        return true;
    }
    if (tk.mode != kModeResidualSet) return true;
    const Word* w = P.remw + (size_t)b * kMaxRemoved;
    Word v = lane < tk.nrm ? ld_word(w + lane) : (Word)kWordMark << 32;
    uint32_t spins = 0, ns = 32;
    while (__any_sync(0xFFFFFFFFu, v == 0)) {
        if (++spins > P.spin) {
            if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
            return false;
        }
        __nanosleep(ns);
        ns = ns < 256 ? 2 * ns : 256;
        if (v == 0) v = ld_word(w + lane);
    }
    if (lane < tk.nrm) tok = (int32_t)(uint32_t)v;
    return true;
}

// Bits of the columns [base, base + width) (width <= 32, base per lane) that are among the removed
// tokens held by lanes 0 .. nrm - 1 (nrm warp-uniform).
__device__ __forceinline__ uint32_t removed_bits(int32_t tok, int32_t nrm, int32_t base, int width) {
    uint32_t bits = 0;
    for (int i = 0; i < nrm; ++i) {
        const int32_t d = __shfl_sync(0xFFFFFFFFu, tok, i) - base;
        if (d >= 0 && d < width) bits |= 1u << d;
    }
    return bits;
}

// ------------------------------------------------------------------------------------------------
// Token trees (spec_verify_tree): the walk from the root, after the decision has the row statistics.
// Slot i of sequence b is node i + 1, with token x and parent par (per lane); a tree's rows are its nodes
// (at most 32), so row j's statistics sit on lane j.
// ------------------------------------------------------------------------------------------------
// Greedy: at node cur, the first child whose token is cur's argmax (a: the argmax of row `lane`).
__device__ __noinline__ void tree_greedy(const Params& P, int32_t b, int32_t g, int32_t o0, int32_t x, int32_t par,
                                         int32_t a, int lane) {
    const int32_t t0 = o0 + b;
    const int apar = __shfl_sync(0xFFFFFFFFu, a, par & 31);
    int cur = 0, n = 0, mytok = -1, mynode = -1;
    while (true) {
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, lane < g && par == cur && x == apar);
        if (!hit) break;
        const int c = __ffs(hit) - 1;
        const int xc = __shfl_sync(0xFFFFFFFFu, x, c);
        if (lane == n) { mytok = xc; mynode = c + 1; }
        ++n;
        cur = c + 1;
    }
    const int ac = __shfl_sync(0xFFFFFFFFu, a, cur);
    if (lane <= g) P.out_tokens[t0 + lane] = lane < n ? mytok : (lane == n ? ac : -1);
    if (P.out_path && lane < g) P.out_path[o0 + lane] = lane < n ? mynode : -1;
    if (lane == 0) P.out_n[b] = n;
}

// Sampled, point-mass candidates: at node cur, its children (slots whose parent is cur) are tried in
// slot order, each accepted iff u (1 - P_E) < p_cur(x), P_E the p mass of the distinct tokens rejected
// before it (a repeated token is rejected outright). The first accepted child is emitted and becomes cur;
// if none is, the draw takes p_cur without those tokens (their words written before the sampler work).
// px: p_par(x) of slot `lane`; m_row: the raw maximum of row `lane`.
__device__ __noinline__ void tree_sampled(const Params& P, int32_t b, int32_t g, int32_t o0, int32_t x, int32_t par,
                                          float px, float u_acc, float u_draw, float m_row, int lane) {
    int cur = 0, n = 0, mytok = -1, mynode = -1;
    uint32_t removed = 0;  // slots holding the tokens the final draw removes
    while (true) {
        const bool child = lane < g && par == cur;
        const uint32_t cm = __ballot_sync(0xFFFFFFFFu, child);
        if (!cm) break;  // a leaf: the draw takes p_cur
        const uint32_t same = __match_any_sync(0xFFFFFFFFu, child ? x : -1 - lane);
        const bool first = child && !(same & cm & ((1u << lane) - 1u));
        const float pv = first ? px : 0.f;
        float incl = pv;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const float y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
            if (lane >= o) incl += y;
        }
        const bool accept = first && u_acc * (1.f - (incl - pv)) < px;
        const uint32_t am = __ballot_sync(0xFFFFFFFFu, accept);
        if (!am) {
            removed = __ballot_sync(0xFFFFFFFFu, first);
            break;
        }
        const int c = __ffs(am) - 1;
        const int xc = __shfl_sync(0xFFFFFFFFu, x, c);
        if (lane == n) { mytok = xc; mynode = c + 1; }
        ++n;
        cur = c + 1;
    }
    // the accepted path, for the find (the sequence's one output writer)
    if (lane < n) st_word(P.pathw + (size_t)b * kMaxRemoved + lane, pack_words(kWordMark | (uint32_t)mynode, (uint32_t)mytok));
    const int nrm = __popc(removed);
    if ((removed >> lane) & 1u)
        st_word(P.remw + (size_t)b * kMaxRemoved + __popc(removed & ((1u << lane) - 1u)),
                pack_words(kWordMark, (uint32_t)x));
    const float pm = __shfl_sync(0xFFFFFFFFu, m_row, cur);
    const float un = __shfl_sync(0xFFFFFFFFu, u_draw, cur);
    put_task(P, b, lane, nrm ? kModeResidualSet : kModeBonus, cur, pm, 0.f, nrm ? __int_as_float(nrm) : 1.f, un, n);
}

// ------------------------------------------------------------------------------------------------
// Decision for sequence b (one warp): merge partials, accept tests, first rejection, outputs.
// Everything that does not depend on the statistics (the draft tokens, the two logits at each token,
// both uniforms of every slot) is fetched before the partials are polled. Rows are reduced 8 at a
// time without control flow between them, so their shuffle trees overlap.
// ------------------------------------------------------------------------------------------------
// Order key of a failing statistics row jr of a sequence with g drafts (code in the low 4 bits): the rule
// reads target row i, then draft row i (rows 0..g are the target rows, g + 1 + i draft row i)
__device__ __forceinline__ uint32_t row_key(int jr, int g, uint32_t code) {
    const uint32_t ord = jr <= g ? 2u * (uint32_t)jr : 2u * (uint32_t)(jr - g - 1) + 1u;
    return ord << 4 | code;
}

// Row statistics shared by the warps of a cooperative decision: (max, sum) per statistics row, and
// the error bits of the rows; two sets, used by alternate decisions of the CTA.
struct CoopRows {
    float2 rs[2][2 * 32];
    uint32_t err[2];  // time-outs (OR)
    uint32_t key[2];  // the first failing row (minimum of row_key; ~0: none)
};

// nsub > 1: a cooperative decision. Warp wsub of the nsub deciding warps of the CTA reduces the rows
// wsub, wsub + nsub, ...; the row statistics meet in shared memory (set `set` of `co`) behind a named
// barrier over the deciding warps, and warp 0 goes on alone (the others return after the barrier).
// nsub == 1: the warp reduces every row itself.
template <int DT, bool VEC, bool GREEDY>
__device__ __noinline__ void decide(const Params& P, int32_t b, int32_t g, int32_t o0, int lane, const float* tab,
                                    int wsub, int nsub, CoopRows* co, int set) {
    const int32_t t0 = o0 + b;
    const int nrows_all = stat_rows<GREEDY>(P, g);
    // this warp's rows: jr = wsub + nsub * j, j = 0 .. nrows - 1
    const int nrows = nrows_all > wsub ? (nrows_all - wsub + nsub - 1) / nsub : 0;
    auto row_of = [&](int j) { return wsub + nsub * j; };
    const int32_t sbase = GREEDY || P.pm ? o0 + b : 2 * o0 + b;
    const int nch = P.nchA;
    const float K = P.K_hi;
    // Partial words of a block (8 rows from j0, the 32 chunks from c0), one row per register; rows past
    // the sequence and chunks past the row read as 1 (never polled). The first block's loads are issued
    // before anything else, and each next block's right after the current block's words are in.
    auto load_block = [&](int j0, int c0, PartialWord (&q)[8]) {
#pragma unroll
        for (int k = 0; k < 8; ++k)
            q[k] = j0 + k < nrows && c0 + lane < nch
                       ? ld_word(P.partials + (size_t)(sbase + row_of(j0 + k)) * nch + c0 + lane) : 1ull;
    };
    PartialWord qn[8];
    load_block(0, 0, qn);
    int32_t x = 0;
    uint32_t err = 0;    // time-outs
    uint32_t tcode = 0;  // this slot's draft error: a bad token, else (token tree) a bad parent
    uint32_t rkey = ~0u; // the first failing row of this warp's rows, as row_key
    float lt = 0.f, ld = 0.f, u_acc = 0.f, u_draw = 0.f;
    // the node whose target row tests slot `lane`: its parent in a token tree, the slot itself otherwise
    int32_t par = lane;
    if (wsub == 0 && lane < g) {
        x = __ldg(P.tokens + o0 + lane);
        if (P.parents) {
            par = __ldg(P.parents + o0 + lane);
            if (par < 0 || par > lane) {
                tcode = SV_ERR_BAD_OFFSETS;
                par = lane;
            }
        }
        if (x < 0 || x >= P.V) tcode = SV_ERR_BAD_TOKEN;
        else if (!GREEDY) {
            lt = logit_at<DT>(P.target, (size_t)(t0 + par) * P.V + x);
            if (!P.pm) ld = logit_at<DT>(P.draft, (size_t)(o0 + lane) * P.V + x);
        }
    }
    if (!GREEDY && wsub == 0) {
        if (lane < g) u_acc = philox_uniform(P.seed, P.step, P.seq_base + (uint32_t)b, (uint32_t)lane, 0);
        if (lane <= g) u_draw = philox_uniform(P.seed, P.step, P.seq_base + (uint32_t)b, (uint32_t)lane, 1);
    }
    // row statistics: row jr's (max, sum) or (max, argmax) ends on lane jr & 31, register jr >> 5
    float my_m0 = -INFINITY, my_m1 = -INFINITY, my_s0 = 0.f, my_s1 = 0.f;
    int my_a0 = -1;
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
            bool v[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                v[k] = j0 + k < nrows && c < nch;
                q[k] = qn[k];
            }
            // words still 0 are statistics tasks in flight: poll them (bounded back-off)
            uint32_t spins = 0, ns = 64;
            while (__any_sync(0xFFFFFFFFu, q[0] == 0 || q[1] == 0 || q[2] == 0 || q[3] == 0 || q[4] == 0 ||
                                               q[5] == 0 || q[6] == 0 || q[7] == 0)) {
                if (++spins > P.spin) {
                    if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                    err |= 1u << SV_ERR_TIMEOUT;
                    break;
                }
                __nanosleep(ns);
                ns = ns < 256 ? 2 * ns : 256;
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    if (q[k] == 0) q[k] = ld_word(P.partials + (size_t)(sbase + row_of(j0 + k)) * nch + c);
            }
            {  // the next block's loads, in flight while this block is merged and reduced
                const int nc0 = c0 + 32 < nch ? c0 + 32 : 0, nj0 = c0 + 32 < nch ? j0 : j0 + 8;
                if (nj0 < nrows) load_block(nj0, nc0, qn);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float qm = v[k] ? __uint_as_float((uint32_t)q[k]) : -INFINITY;
                const uint32_t qh = (uint32_t)(q[k] >> 32);
                if (GREEDY) {
                    lf[k] |= v[k] && (qh >> 31) ? 1u << SV_ERR_NONFINITE : 0u;
                    const bool take = qm > lm[k];
                    la[k] = take ? (int)(qh & 0x7FFFFFFFu) - 1 : la[k];
                    lm[k] = take ? qm : lm[k];
                } else {
                    const float qs = v[k] ? __uint_as_float(qh) : 0.f;
                    if (c0 == 0) {  // first chunk of the lane: nothing to merge with
                        lm[k] = qm;
                        ls[k] = qs;
                    } else if (qs != qs) {
                        ls[k] = qs;
                        lm[k] = fmaxf(lm[k], qm);
                    } else if (ls[k] == ls[k]) {
                        merge_ms<true>(lm[k], ls[k], qm, qs, K);
                    }
                }
            }
        }
        // the 8 rows' lane reductions, interleaved
        float M[8], S[8];
        int A[8];
        uint32_t F[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) M[k] = lm[k];
#pragma unroll
        for (int o = 16; o; o >>= 1)
#pragma unroll
            for (int k = 0; k < 8; ++k) M[k] = fmaxf(M[k], __shfl_xor_sync(0xFFFFFFFFu, M[k], o));
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            if (GREEDY) {
                A[k] = lm[k] == M[k] ? la[k] : 0x7FFFFFFF;
                F[k] = lf[k];
            } else {
                S[k] = ls[k] != ls[k] ? ls[k] : (lm[k] == -INFINITY ? 0.f : ls[k] * exp2_fma((lm[k] - M[k]) * K));
            }
        }
#pragma unroll
        for (int o = 16; o; o >>= 1)
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                if (GREEDY) {
                    A[k] = min(A[k], __shfl_xor_sync(0xFFFFFFFFu, A[k], o));
                    F[k] |= __shfl_xor_sync(0xFFFFFFFFu, F[k], o);
                } else {
                    S[k] += __shfl_xor_sync(0xFFFFFFFFu, S[k], o);
                }
            }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const bool in = j0 + k < nrows;
            const int jr = row_of(j0 + k);
            // a row with a NaN or +inf is reported as such, not as empty (both fail the sequence)
            const uint32_t rf = GREEDY ? (F[k] | (M[k] == INFINITY ? 1u << SV_ERR_NONFINITE : 0u))
                                       : (S[k] != S[k] ? 1u << SV_ERR_NONFINITE : 0u);
            const uint32_t rc = rf ? SV_ERR_NONFINITE : (M[k] == -INFINITY ? SV_ERR_EMPTY_ROW : 0u);
            if (in && rc) rkey = min(rkey, row_key(jr, g, rc));
            if (nsub > 1) {
                if (in && lane == 0) co->rs[set][jr] = make_float2(M[k], GREEDY ? 0.f : S[k]);
            } else {
                if (in && lane == jr) { my_m0 = M[k]; my_s0 = GREEDY ? 0.f : S[k]; my_a0 = GREEDY ? A[k] : -1; }
                if (in && lane == jr - 32) { my_m1 = M[k]; my_s1 = GREEDY ? 0.f : S[k]; }
            }
        }
    }
    err = warp_or(err);
    rkey = __reduce_min_sync(0xFFFFFFFFu, rkey);
    if (nsub > 1) {  // meet the other deciding warps; warp 0 continues with every row's statistics
        if (lane == 0 && err) atomicOr(&co->err[set], err);
        if (lane == 0 && rkey != ~0u) atomicMin(&co->key[set], rkey);
        asm volatile("bar.sync 1, %0;" ::"r"(32 * nsub) : "memory");
        if (wsub != 0) return;
        err = co->err[set];
        rkey = co->key[set];
        if (lane < nrows_all) {
            const float2 r0 = co->rs[set][lane];
            my_m0 = r0.x;
            my_s0 = r0.y;
        }
        if (lane + 32 < nrows_all) {
            const float2 r1 = co->rs[set][lane + 32];
            my_m1 = r1.x;
            my_s1 = r1.y;
        }
        __syncwarp();
        if (lane == 0) {  // read by every lane above; cleared for the set's next use
            co->err[set] = 0u;
            co->key[set] = ~0u;
        }
    }
    // the failing sequence's code, in the rule's order: the first slot with a bad draft token (a token tree:
    // or a bad parent), else the first failing row (target row i, then draft row i); time-outs added
    {
        const uint32_t tb = __ballot_sync(0xFFFFFFFFu, tcode != 0u);
        const uint32_t tc = tb ? __shfl_sync(0xFFFFFFFFu, tcode, __ffs(tb) - 1) : 0u;
        err |= tc ? 1u << tc : (rkey != ~0u ? 1u << (rkey & 15u) : 0u);
    }
    if (err) {
        if (lane == 0) {
            atomicOr(P.status, err);
            P.out_n[b] = -1;
        }
        if (!GREEDY) put_task(P, b, lane, kModeNone, 0, 0.f, 0.f, 1.f, 0.f, 0);
        for (int32_t j = lane; j <= g; j += 32) P.out_tokens[t0 + j] = -1;
        if (P.out_path && lane < g) P.out_path[o0 + lane] = -1;
        commit_seq(P, b, -1, -1, -1, lane);
        return;
    }
    if (GREEDY) {
        const int a = my_a0;  // argmax of target row `lane` (lane <= g <= 31)
        if (lane <= g && P.dbg.row_argmax) P.dbg.row_argmax[t0 + lane] = a;
        if (P.parents) {  // token tree (out of line: the linear path's code stays small)
            tree_greedy(P, b, g, o0, x, par, a, lane);
            return;
        }
        const uint32_t mism = __ballot_sync(0xFFFFFFFFu, lane < g && x != a);
        const int n = mism ? __ffs(mism) - 1 : g;
        if (lane <= g) P.out_tokens[t0 + lane] = lane < n ? x : (lane == n ? a : -1);
        if (lane == 0) P.out_n[b] = n;
        commit_seq(P, b, n, x, __shfl_sync(0xFFFFFFFFu, a, n), lane);
        return;
    }
    // the draft row of slot `lane` is statistics row g + 1 + lane: lane (g+1+lane) & 31, register >> 5
    // (point-mass drafts have no draft rows: q(x) = 1)
    const int jd = g + 1 + lane;
    const float dm0 = __shfl_sync(0xFFFFFFFFu, my_m0, jd & 31), dm1 = __shfl_sync(0xFFFFFFFFu, my_m1, jd & 31);
    const float ds0 = __shfl_sync(0xFFFFFFFFu, my_s0, jd & 31), ds1 = __shfl_sync(0xFFFFFFFFu, my_s1, jd & 31);
    const float dm = P.pm ? 0.f : (jd >> 5) ? dm1 : dm0, ds = P.pm ? 1.f : (jd >> 5) ? ds1 : ds0;
    bool acc = true;
    float px = 0.f;
    // the statistics of the row that tests slot `lane` (rows 0..31 sit on lanes 0..31 here: a tree's
    // rows are its nodes, at most 32)
    const float mpar = __shfl_sync(0xFFFFFFFFu, my_m0, par & 31), spar = __shfl_sync(0xFFFFFFFFu, my_s0, par & 31);
    if (lane < g) {
        // p(x) and q(x) from the precise exponential of the exact logit gaps, over the fp32 normalisers
        const ff2 e = exp2_ff2(make_float2(lt, ld), make_float2(mpar, dm), exp_const(P), tab);
        px = div_fma(e.hi.x + e.lo.x, spar);
        const float qx = P.pm ? 1.f : div_fma(e.hi.y + e.lo.y, ds);
        acc = u_acc * qx < px;
        if (P.dbg.p_x) P.dbg.p_x[o0 + lane] = (double)px;
        if (P.dbg.q_x) P.dbg.q_x[o0 + lane] = (double)qx;
    }
    if (P.dbg.row_lse) {
        const int32_t R_t = __ldg(P.offs + P.B) + P.B;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int jr = lane + 32 * h;
            if (jr < nrows_all) {
                const float m = h ? my_m1 : my_m0, sum = h ? my_s1 : my_s0;
                const double lse = (double)m * P.invT64 + log((double)sum);
                P.dbg.row_lse[jr <= g ? t0 + jr : R_t + o0 + (jr - g - 1)] = lse;
            }
        }
    }
    if (P.parents) {  // token tree (out of line: the linear path's code stays small)
        tree_sampled(P, b, g, o0, x, par, px, u_acc, u_draw, my_m0, lane);
        return;
    }
    // the sequence's outputs are written by its find, once the draw is known (one writer per sequence)
    const uint32_t rej = __ballot_sync(0xFFFFFFFFu, lane < g && !acc);
    const int n = rej ? __ffs(rej) - 1 : g;
    // statistics of the emitting slot's rows
    const float pm = __shfl_sync(0xFFFFFFFFu, my_m0, n), ps = __shfl_sync(0xFFFFFFFFu, my_s0, n);
    const float qm = __shfl_sync(0xFFFFFFFFu, dm, n), qs = __shfl_sync(0xFFFFFFFFu, ds, n);
    const float un = __shfl_sync(0xFFFFFFFFu, u_draw, n);
    const int32_t xn = __shfl_sync(0xFFFFFFFFu, x, n < g ? n : 0);
    if (P.pm)  // the residual of a point-mass draft removes column x_n; rho's word carries x_n + 1
        put_task(P, b, lane, n < g ? kModeResidualPM : kModeBonus, n, pm, 0.f,
                 n < g ? __int_as_float(xn + 1) : 1.f, un, n);
    else {
        // the selection ratio s_p / s_q, in table units (times 2^((m_p - m_q) K)) for a draw the table serves
        float rho = 1.f;
        if (n < g) {
            rho = div_fma(ps, qs);
            if (draw_uses_table<DT, VEC>(P, kModeResidual, pm, qm)) rho *= exp2_fma((pm - qm) * K);
        }
        put_task(P, b, lane, n < g ? kModeResidual : kModeBonus, n, pm, n < g ? qm : 0.f, rho, un, n);
    }
}

// Slot order (P.prog, batches with draft rows): the statistics rows are numbered by slot, q = 2 B s + k:
// k = b for the target row of slot s of sequence b, k = B + b for its draft row; the last slot
// (s = max_gamma) holds target rows only. A q that sequence b does not have (s > gamma_b, or the draft row
// of slot gamma_b) is a hole. The partial words are indexed by q; the CTA's row map holds, per q, the
// logits row (bits 0-11), the sequence (bits 12-21), the slot (bits 22-26) and the draft flag (bit 31),
// or kProgHole.
constexpr uint32_t kProgHole = 0x7FFFFFFFu;
__device__ __forceinline__ uint32_t prog_rows(const Params& P) {
    return (2u * (uint32_t)P.max_gamma + 1u) * (uint32_t)P.B;
}
__device__ __forceinline__ int32_t prog_q(const Params& P, int32_t b, int32_t s, bool draft) {
    return (2 * s + (draft ? 1 : 0)) * P.B + b;
}

// Slot order: a published decision takes the next position of the decision-order queue, from which the
// sampler tasks are claimed (so that no warp waits on a sequence decided late while decided ones wait).
// A position a claimer gave up waiting for (kOrderLost, SV_ERR_TIMEOUT set) fails its sequence here.
__device__ __noinline__ void enqueue_decided(const Params& P, int32_t b, int lane) {
    uint32_t lost = 0;
    if (lane == 0) {
        const uint32_t p = atomicAdd(&P.ctr->decided, 1u);
        lost = atomicCAS(P.order + p, 0u, (uint32_t)b + 1u) != 0u;
    }
    if (__shfl_sync(0xFFFFFFFFu, lost, 0)) give_up_seq(P, b, lane);
}

// Decision in slot order (P.prog, linear sampled drafts with draft rows; one warp): slot s is tested as soon as its rows'
// statistics are in (target row s and draft row s, which the slot-order stream delivers together), and
// the first rejection ends the decision: the rows of later slots are not waited for. Errors follow the
// order of the rule: a bad draft token first, then the rows slot by slot (target before draft); a row of a
// later slot is checked by the sequence's find. The draw's words are those of decide().
template <int DT, bool VEC>
__device__ __noinline__ void decide_prog(const Params& P, int32_t b, int32_t g, int32_t o0, int lane, const float* tab) {
    const int32_t t0 = o0 + b;
    const int nch = P.nchA;
    const float K = P.K_hi;
    int32_t x = 0;
    uint32_t err = 0;
    float lt = 0.f, ld = 0.f, u_acc = 0.f, u_draw = 0.f;
    if (lane < g) {
        x = __ldg(P.tokens + o0 + lane);
        if (x < 0 || x >= P.V) {
            err = 1u << SV_ERR_BAD_TOKEN;
        } else {
            lt = logit_at<DT>(P.target, (size_t)(t0 + lane) * P.V + x);
            ld = logit_at<DT>(P.draft, (size_t)(o0 + lane) * P.V + x);
        }
        u_acc = philox_uniform(P.seed, P.step, P.seq_base + (uint32_t)b, (uint32_t)lane, 0);
    }
    if (lane <= g) u_draw = philox_uniform(P.seed, P.step, P.seq_base + (uint32_t)b, (uint32_t)lane, 1);
    err = warp_or(err);
    // rows (max, sum) of the current slot; the loads of slot s + 1 are issued once slot s's words are in
    float Mt = -INFINITY, St = 0.f, Md = 0.f, Sd = 1.f;
    int n = g;
    auto word_at = [&](int32_t r, int c) { return ld_word(P.partials + (size_t)r * nch + c); };
    for (int s = 0; s <= g && !err; ++s) {
        const bool hd = s < g;
        const int32_t rt = prog_q(P, b, s, false), rd = prog_q(P, b, s, true);
        float mt = -INFINITY, st = 0.f, md = -INFINITY, sd = 0.f;
        for (int c0 = 0; c0 < nch; c0 += 32) {
            const int c = c0 + lane;
            const bool in = c < nch;
            PartialWord wt = in ? word_at(rt, c) : 1ull, wd = in && hd ? word_at(rd, c) : 1ull;
            uint32_t spins = 0, nsl = 64;
            while (__any_sync(0xFFFFFFFFu, wt == 0 || wd == 0)) {
                if (++spins > P.spin) {
                    if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                    err = 1u << SV_ERR_TIMEOUT;
                    break;
                }
                __nanosleep(nsl);
                nsl = nsl < 256 ? 2 * nsl : 256;
                if (wt == 0) wt = word_at(rt, c);
                if (wd == 0) wd = word_at(rd, c);
            }
            if (err) break;
            if (in) {  // merge the lane's chunks (online rescaling; a NaN sum stays NaN)
                const float qm = __uint_as_float((uint32_t)wt), qs = __uint_as_float((uint32_t)(wt >> 32));
                if (c0 == 0) { mt = qm; st = qs; }
                else if (qs != qs) { st = qs; mt = fmaxf(mt, qm); }
                else if (st == st) merge_ms<true>(mt, st, qm, qs, K);
                if (hd) {
                    const float rm = __uint_as_float((uint32_t)wd), rs = __uint_as_float((uint32_t)(wd >> 32));
                    if (c0 == 0) { md = rm; sd = rs; }
                    else if (rs != rs) { sd = rs; md = fmaxf(md, rm); }
                    else if (sd == sd) merge_ms<true>(md, sd, rm, rs, K);
                }
            }
        }
        if (err) break;
        // the two rows' reductions, interleaved
        float MT = mt, MD = md;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            MT = fmaxf(MT, __shfl_xor_sync(0xFFFFFFFFu, MT, o));
            MD = fmaxf(MD, __shfl_xor_sync(0xFFFFFFFFu, MD, o));
        }
        float ST = st != st ? st : (mt == -INFINITY ? 0.f : st * exp2_fma((mt - MT) * K));
        float SD = sd != sd ? sd : (md == -INFINITY ? 0.f : sd * exp2_fma((md - MD) * K));
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            ST += __shfl_xor_sync(0xFFFFFFFFu, ST, o);
            SD += __shfl_xor_sync(0xFFFFFFFFu, SD, o);
        }
        // the first failing row in order: target before draft (a NaN or +inf row is reported as such)
        if (ST != ST) err = 1u << SV_ERR_NONFINITE;
        else if (MT == -INFINITY) err = 1u << SV_ERR_EMPTY_ROW;
        else if (hd && SD != SD) err = 1u << SV_ERR_NONFINITE;
        else if (hd && MD == -INFINITY) err = 1u << SV_ERR_EMPTY_ROW;
        if (err) break;
        Mt = MT;
        St = ST;
        if (hd) {
            Md = MD;
            Sd = SD;
        }
        if (s == g) break;  // every draft accepted: the bonus draw from target row g
        // the accept test of slot s: p(x) and q(x) from the precise exponential of the exact logit gaps
        const float lts = __shfl_sync(0xFFFFFFFFu, lt, s), lds = __shfl_sync(0xFFFFFFFFu, ld, s);
        const float us = __shfl_sync(0xFFFFFFFFu, u_acc, s);
        const ff2 e = exp2_ff2(make_float2(lts, lds), make_float2(Mt, Md), exp_const(P), tab);
        const float px = div_fma(e.hi.x + e.lo.x, St);
        const float qx = div_fma(e.hi.y + e.lo.y, Sd);
        if (!(us * qx < px)) {
            n = s;
            break;
        }
    }
    if (err) {
        if (lane == 0) {
            atomicOr(P.status, err);
            P.out_n[b] = -1;
        }
        put_task(P, b, lane, kModeNone, 0, 0.f, 0.f, 1.f, 0.f, 0);
        for (int32_t j = lane; j <= g; j += 32) P.out_tokens[t0 + j] = -1;
        commit_seq(P, b, -1, -1, -1, lane);
        enqueue_decided(P, b, lane);
        return;
    }
    const float un = __shfl_sync(0xFFFFFFFFu, u_draw, n);
    float rho = 1.f;
    if (n < g) {
        rho = div_fma(St, Sd);
        if (draw_uses_table<DT, VEC>(P, kModeResidual, Mt, Md)) rho *= exp2_fma((Mt - Md) * K);
    }
    put_task(P, b, lane, n < g ? kModeResidual : kModeBonus, n, Mt, n < g ? Md : 0.f, rho, un, n);
    enqueue_decided(P, b, lane);
}

// The check of a sequence's rows after its emitting slot n (P.prog), in the rule's order (target row
// s, then draft row s, for s = n + 1 .. g): polled until written (the streamers never wait), then the first
// row with a NaN / +inf chunk (SV_ERR_NONFINITE) or without a value above -inf (SV_ERR_EMPTY_ROW). Returns
// that error's bit, 0 when every row is clean, or the time-out bit.
__device__ __noinline__ uint32_t check_dead_rows(const Params& P, int32_t b, int32_t g, int32_t n, int lane) {
    const int nd = n < g ? 2 * (g - n) - 1 : 0;  // at most 61 rows
    if (nd <= 0) return 0u;
    const int nch = P.nchA;
    unsigned long long nan = 0ull, live = 0ull;
    const int total = nd * nch;
    for (int w0 = 0; w0 < total; w0 += 32) {
        const int w = w0 + lane;
        const bool in = w < total;
        const int i = in ? w / nch : 0, c = in ? w - i * nch : 0;
        const int32_t s = n + 1 + (i >> 1);
        const int32_t r = prog_q(P, b, s, i & 1);
        PartialWord q = in ? ld_word(P.partials + (size_t)r * nch + c) : 1ull;
        uint32_t spins = 0, nsl = 64;
        while (__any_sync(0xFFFFFFFFu, q == 0)) {
            if (++spins > P.spin) {
                if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                return 1u << SV_ERR_TIMEOUT;
            }
            __nanosleep(nsl);
            nsl = nsl < 256 ? 2 * nsl : 256;
            if (q == 0) q = ld_word(P.partials + (size_t)r * nch + c);
        }
        if (in) {
            const float m = __uint_as_float((uint32_t)q), sm = __uint_as_float((uint32_t)(q >> 32));
            if (sm != sm) nan |= 1ull << i;
            if (m > -INFINITY) live |= 1ull << i;
        }
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) {
        nan |= __shfl_xor_sync(0xFFFFFFFFu, nan, o);
        live |= __shfl_xor_sync(0xFFFFFFFFu, live, o);
    }
    const unsigned long long all = nd == 64 ? ~0ull : (1ull << nd) - 1ull;
    const unsigned long long bad = (nan | ~live) & all;
    if (!bad) return 0u;
    const int i = __ffsll((long long)bad) - 1;
    return (nan >> i) & 1ull ? 1u << SV_ERR_NONFINITE : 1u << SV_ERR_EMPTY_ROW;
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
    const float2 rq = mul2(f2(rho), eq.hi);
    return make_float2(gt_mask(ep.hi.x, rq.x), gt_mask(ep.hi.y, rq.y));
}

// Residual weight of a selected column, max(0, e_p - rho e_q) in float-float; 0 when not selected.
__device__ __forceinline__ ff resid_weight(float hp, float lp, float hq, float lq, float sel, ff rho) {
    if (sel == 0.f) return ff{0.f, 0.f};
    const ff w = ff_sub(ff_norm(hp, lp), ff_mul(rho, ff_norm(hq, lq)));
    return w.hi > 0.f ? w : ff{0.f, 0.f};
}

// Weight of one column in the find's element search: the precise p weight, or the residual weight of
// a selected column (float-float); 0 at or past k_hi.
template <int DT>
__device__ __forceinline__ ff column_weight(float lp, float lq, const TaskInfo& tk, const ExpConst& EC, bool resid,
                                            ff rho, const float* tab, bool removed) {
    const ff2 e = exp2_ff2(make_float2(lp, lq), make_float2(tk.m_p, tk.m_q), EC, tab);
    if (!resid) return removed ? ff{0.f, 0.f} : ff_norm(e.hi.x, e.lo.x);
    const bool sel = e.hi.x > tk.rho * e.hi.y;  // the selection rule of sel_mask
    return resid_weight(e.hi.x, e.lo.x, e.hi.y, e.lo.y, sel ? 1.f : 0.f, rho);
}
// The same in the value table's units, from the columns' raw bf16 codes (p in the low half of pq, q in
// the high half): the weights the sampler tasks summed for a draw that uses the table.
__device__ __forceinline__ ff column_weight_tab(uint32_t pq, const TaskInfo& tk, bool resid, ff rho, const char* vt,
                                                bool removed) {
    const ff2 e = tab_pair(pq, vt);
    if (!resid) return removed ? ff{0.f, 0.f} : ff_norm(e.hi.x, e.lo.x);
    const bool sel = e.hi.x > tk.rho * e.hi.y;  // the selection rule of sel_mask
    return resid_weight(e.hi.x, e.lo.x, e.hi.y, e.lo.y, sel ? 1.f : 0.f, rho);
}
// Column k's weight in the find, either way (TAB: the value table's, from the raw codes).
template <int DT, bool TAB>
__device__ __forceinline__ ff weight_at(const Params& P, size_t prow, size_t qrow, int32_t k, const TaskInfo& tk,
                                        const ExpConst& EC, bool resid, ff rho, const float* tab, const char* vt,
                                        bool removed) {
    if constexpr (TAB) {
        const uint32_t cp = __ldg((const unsigned short*)P.target + prow * (size_t)P.V + k);
        const uint32_t cq = resid ? __ldg((const unsigned short*)P.draft + qrow * (size_t)P.V + k) : 0u;
        return column_weight_tab(cp | cq << 16, tk, resid, rho, vt, removed);
    } else {
        const float lpk = logit_at<DT>(P.target, prow * (size_t)P.V + k);
        const float lqk = resid ? logit_at<DT>(P.draft, qrow * (size_t)P.V + k) : 0.f;
        return column_weight<DT>(lpk, lqk, tk, EC, resid, rho, tab, removed);
    }
}

// Inverse-CDF search over the columns [k_lo, k_hi) for the remaining target `rem`, kScanBlock columns
// per pass (16 consecutive columns per lane, float-float). Each lane keeps only its total; once the
// crossing lane is known, 16 lanes recompute its columns in parallel (their data are L1-resident) and
// a 16-lane prefix picks the column. Returns the first column whose running sum exceeds `rem`, or the
// last column of positive weight when the crossing is lost to rounding (or `tail_rule` asks for it).
template <int DT, bool VEC, bool TAB>
__device__ __noinline__ int32_t scan_elements(const Params& P, const TaskInfo& tk, size_t prow, size_t qrow, bool resid, ff rho,
                                 int32_t k_lo, int32_t k_hi, ff rem, bool tail_rule, int32_t rtok, int32_t nrm,
                                 const float* tab, const char* vt, int lane) {
    const ExpConst EC = exp_const(P);
    // a unit spans at most kSTask columns: NB passes; bf16 issues every pass's loads first
    constexpr int NB = kSTask / kScanBlock;
    constexpr bool kAhead = DT == SV_BF16;
    Cols16 cpa[kAhead ? NB : 1], cqa[kAhead ? NB : 1];
    if (kAhead) {
#pragma unroll
        for (int nb = 0; nb < (kAhead ? NB : 1); ++nb) {
            const int32_t k0 = k_lo + nb * kScanBlock + lane * kScanPerLane;
            cpa[nb] = load_cols16<DT, VEC>(P.target, prow, P.V, k0);
            if (resid) cqa[nb] = load_cols16<DT, VEC>(P.draft, qrow, P.V, k0);
        }
    }
    int32_t last_pos = -1;
#pragma unroll
    for (int nb = 0; nb < NB; ++nb) {
        const int32_t base = k_lo + nb * kScanBlock;
        if (base >= k_hi) break;
        const int32_t k0 = base + lane * kScanPerLane;
        Cols16 cp, cq;
        if (kAhead) {
            cp = cpa[kAhead ? nb : 0];
            cq = cqa[kAhead ? nb : 0];
        } else {
            cp = load_cols16<DT, VEC>(P.target, prow, P.V, k0);
            if (resid) cq = load_cols16<DT, VEC>(P.draft, qrow, P.V, k0);
        }
        ff tot{0.f, 0.f};
        int lastp = -1;
        const uint32_t rb = removed_bits(rtok, nrm, k0, kScanPerLane);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            ff w0, w1;
            if constexpr (TAB) {  // the pair word of the p row, and of the q row, by halves
                const uint32_t pw = cp.w[e], qw = resid ? cq.w[e] : 0u;
                w0 = column_weight_tab((pw & 0xFFFFu) | (qw << 16), tk, resid, rho, vt, (rb >> (2 * e)) & 1u);
                w1 = column_weight_tab((pw >> 16) | (qw & 0xFFFF0000u), tk, resid, rho, vt, (rb >> (2 * e + 1)) & 1u);
            } else {
                const float2 lpv = col2<DT>(cp, e), lqv = resid ? col2<DT>(cq, e) : f2(0.f);
                w0 = column_weight<DT>(lpv.x, lqv.x, tk, EC, resid, rho, tab, (rb >> (2 * e)) & 1u);
                w1 = column_weight<DT>(lpv.y, lqv.y, tk, EC, resid, rho, tab, (rb >> (2 * e + 1)) & 1u);
            }
            if (k0 + 2 * e < k_hi && w0.hi > 0.f) {
                tot = ff_add(tot, w0);
                lastp = k0 + 2 * e;
            }
            if (k0 + 2 * e + 1 < k_hi && w1.hi > 0.f) {
                tot = ff_add(tot, w1);
                lastp = k0 + 2 * e + 1;
            }
        }
        lastp = warp_max_i(lastp);
        if (lastp >= 0) last_pos = lastp;
        const ff incl = warp_inscan_ff(tot, lane);
        const ff btot = shfl_ff(incl, 31);
        if (!tail_rule && ff_gt(btot, rem)) {
            // the first lane whose inclusive prefix exceeds rem holds the crossing column
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, ff_gt(incl, rem));
            const int L = __ffs(hit) - 1;
            const ff pre = shfl_ff(exclusive_of(incl, lane), L);
            // lanes j < 16 take column kL + j of lane L
            const int32_t kL = base + L * kScanPerLane, kj = kL + (lane & 15);
            const uint32_t rj = removed_bits(rtok, nrm, kj, 1);
            ff w{0.f, 0.f};
            if (lane < kScanPerLane && kj < k_hi) {
                w = weight_at<DT, TAB>(P, prow, qrow, kj, tk, EC, resid, rho, tab, vt, rj != 0u);
                if (!(w.hi > 0.f)) w = ff{0.f, 0.f};
            }
            const ff c = ff_add(pre, warp_inscan_ff(w, lane));  // lanes >= 16 add zeros
            const uint32_t cross = __ballot_sync(0xFFFFFFFFu, lane < kScanPerLane && w.hi > 0.f && ff_gt(c, rem));
            if (cross) return kL + __ffs(cross) - 1;
            // the lane's sum crossed, its running sum fell short by rounding: its last positive column
            const uint32_t pos = __ballot_sync(0xFFFFFFFFu, lane < kScanPerLane && w.hi > 0.f);
            return pos ? kL + 31 - __clz(pos) : last_pos;
        }
        rem = ff_sub(rem, btot);
    }
    return last_pos;
}

// Element level of the find for the residual (or bonus) weights, inside sampler task `unit`: the
// crossing group from the groups' selected sums (polled until written), then the crossing column among
// that group's kGroupCols columns, 4 consecutive ones recomputed per lane. `rem` is the target left
// after the tasks before. Rounding that loses the crossing (or tail_rule) picks the last group, then
// column, of positive weight. Returns -1 when nothing in the task has positive weight, -2 on a time-out.
template <int DT, bool VEC, bool TAB>
__device__ __noinline__ int32_t group_search(const Params& P, int32_t b, int unit, const TaskInfo& tk, size_t prow, size_t qrow,
                                bool resid, ff rho, ff rem, bool tail_rule, int32_t rtok, const float* tab,
                                const char* vt, int lane) {
    static_assert(kGroupCols == 4 * 32, "four columns per lane");
    const Word* gw = P.groupw + (((size_t)b * P.nS + unit) * kGroups + (lane % kGroups)) * kGroupWords;
    Word wa = lane < kGroups ? ld_word(gw) : (Word)kWordMark, wb = lane < kGroups ? ld_word(gw + 1) : (Word)kWordMark;
    uint32_t spins = 0, ns = 32;
    while (__any_sync(0xFFFFFFFFu, wa == 0 || wb == 0)) {
        if (++spins > P.spin) {
            if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
            return -2;
        }
        __nanosleep(ns);
        ns = ns < 256 ? 2 * ns : 256;
        if (wa == 0) wa = ld_word(gw);
        if (wb == 0) wb = ld_word(gw + 1);
    }
    ff w = unpack_ff(wa);
    if (resid) w = ff_sub(w, ff_mul(rho, unpack_ff(wb)));
    if (!(w.hi > 0.f)) w = ff{0.f, 0.f};
    const ff incl = warp_inscan_ff(w, lane);
    const uint32_t gpos = __ballot_sync(0xFFFFFFFFu, w.hi > 0.f);
    if (!gpos) return -1;
    const uint32_t hit = tail_rule ? 0u : __ballot_sync(0xFFFFFFFFu, ff_gt(incl, rem));
    const int G = hit ? __ffs(hit) - 1 : 31 - __clz(gpos);
    const ff pre = shfl_ff(exclusive_of(incl, lane), G);
    // lane j: columns k0 + 4 j .. k0 + 4 j + 3 of the group
    const ExpConst EC = exp_const(P);
    const int32_t k0 = unit * kSTask + kGroupCols * G + 4 * lane;
    const uint32_t r4 = removed_bits(rtok, tk.nrm, k0, 4);
    ff cw[4];
    ff tot{0.f, 0.f};
    if constexpr (TAB) {  // rows 16-byte aligned, V a multiple of 8: the 4 columns are one 8-byte load per row
        uint2 pw = make_uint2(0u, 0u), qw = make_uint2(0u, 0u);
        if (k0 < P.V) {
            pw = __ldg((const uint2*)((const unsigned short*)P.target + prow * (size_t)P.V + k0));
            if (resid) qw = __ldg((const uint2*)((const unsigned short*)P.draft + qrow * (size_t)P.V + k0));
        }
        const uint32_t pws[2] = {pw.x, pw.y}, qws[2] = {qw.x, qw.y};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t p16 = e & 1 ? pws[e >> 1] >> 16 : pws[e >> 1] & 0xFFFFu;
            const uint32_t q16 = e & 1 ? qws[e >> 1] >> 16 : qws[e >> 1] & 0xFFFFu;
            cw[e] = ff{0.f, 0.f};
            if (k0 + e < P.V) {
                cw[e] = column_weight_tab(p16 | q16 << 16, tk, resid, rho, vt, (r4 >> e) & 1u);
                if (!(cw[e].hi > 0.f)) cw[e] = ff{0.f, 0.f};
            }
            tot = ff_add(tot, cw[e]);
        }
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int32_t k = k0 + e;
            cw[e] = ff{0.f, 0.f};
            if (k < P.V) {
                const float lpk = logit_at<DT>(P.target, prow * (size_t)P.V + k);
                const float lqk = resid ? logit_at<DT>(P.draft, qrow * (size_t)P.V + k) : 0.f;
                cw[e] = column_weight<DT>(lpk, lqk, tk, EC, resid, rho, tab, (r4 >> e) & 1u);
                if (!(cw[e].hi > 0.f)) cw[e] = ff{0.f, 0.f};
            }
            tot = ff_add(tot, cw[e]);
        }
    }
    const ff tin = warp_inscan_ff(tot, lane);
    const ff cincl = ff_add(pre, tin), cexcl = ff_add(pre, exclusive_of(tin, lane));
    const uint32_t lpos = __ballot_sync(0xFFFFFFFFu, tot.hi > 0.f);
    const uint32_t cross = hit ? __ballot_sync(0xFFFFFFFFu, ff_gt(cincl, rem)) : 0u;
    // the lane holding the crossing (or, failing that, the last lane of positive weight) picks the column
    const int J = cross ? __ffs(cross) - 1 : (lpos ? 31 - __clz(lpos) : -1);
    if (J < 0) return -1;
    int32_t col = -1;
    if (lane == J) {  // no collectives in here
        ff c = cexcl;
        int lastc = -1;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            if (cw[e].hi > 0.f) {
                c = ff_add(c, cw[e]);
                if (cross && col < 0 && ff_gt(c, rem)) col = k0 + e;
                lastc = k0 + e;
            }
        }
        if (col < 0) col = lastc;
    }
    return __shfl_sync(0xFFFFFFFFu, col, J);
}

// Find for sequence b (one warp): run by the warp that holds the sequence's last sampler task, after
// its own task. Exact normalisers from all task records (polled until written), the crossing task over
// the records' weights, then the crossing column inside that task.
template <int DT, bool VEC, bool TAB>
__device__ __noinline__ void find(const Params& P, int32_t b, const TaskInfo tk, size_t prow, size_t qrow,
                                  int32_t o0, const float* tab, const char* vt, int lane) {
    // the sequence's outputs are this warp's to write, unless a wait on the sequence gave up first
    if (claim_seq(P, b, 1u, lane) != 0u) return;
    // the accepted tokens (slot j on lane j < npos): the draft tokens, or a tree's accepted path (written
    // by the decision before the draw)
    int32_t acc_tok = -1, acc_node = -1;
    if (!P.parents) {
        if (lane < tk.npos) acc_tok = __ldg(P.tokens + o0 + lane);
    } else {
        const Word* pw = P.pathw + (size_t)b * kMaxRemoved + lane;
        Word v = lane < tk.npos ? ld_word(pw) : (Word)kWordMark << 32;
        uint32_t spins = 0, ns = 32;
        while (__any_sync(0xFFFFFFFFu, v == 0)) {
            if (++spins > P.spin) {
                if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                fail_outputs(P, b, lane);
                return;
            }
            __nanosleep(ns);
            ns = ns < 256 ? 2 * ns : 256;
            if (v == 0) v = ld_word(pw);
        }
        acc_node = (int32_t)((uint32_t)(v >> 32) & 0x7FFFFFFFu);
        acc_tok = (int32_t)(uint32_t)v;
    }
    const int nS = P.nS;
    const Word* rec = P.recw + (size_t)b * nS * kRecWords;
    // lane owns the run of tasks [s0, s1), read four tasks (16 words) at a time
    const int per = (nS + 31) / 32;
    const int s0 = min(nS, lane * per), s1 = min(nS, s0 + per);
    // Warp-collective (every lane calls it the same number of times): polls the words of tasks
    // i0 .. i0 + 3 until written (false on time-out), adds their sums to the lane's and returns each
    // task's selected sums.
    auto poll4 = [&](int i0, ff& lp, ff& lq, ff& la, ff& lb, ff (&va)[4], ff (&vb)[4]) -> bool {
        Word w[4][kRecWords];
#pragma unroll
        for (int k = 0; k < 4; ++k)
#pragma unroll
            for (int j = 0; j < kRecWords; ++j)
                w[k][j] = i0 + k < s1 ? ld_word(rec + (size_t)(i0 + k) * kRecWords + j) : (Word)kWordMark;
        uint32_t spins = 0, ns = 32;
        while (true) {
            bool missing = false;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int j = 0; j < kRecWords; ++j) missing |= w[k][j] == 0;
            if (!__any_sync(0xFFFFFFFFu, missing)) break;
            if (++spins > P.spin) {
                if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                return false;
            }
            __nanosleep(ns);
            ns = ns < 256 ? 2 * ns : 256;
#pragma unroll
            for (int k = 0; k < 4; ++k)
#pragma unroll
                for (int j = 0; j < kRecWords; ++j)
                    if (w[k][j] == 0) w[k][j] = ld_word(rec + (size_t)(i0 + k) * kRecWords + j);
        }
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            va[k] = unpack_ff(w[k][2]);
            vb[k] = unpack_ff(w[k][3]);
            lp = ff_add(lp, unpack_ff(w[k][0]));
            lq = ff_add(lq, unpack_ff(w[k][1]));
            la = ff_add(la, va[k]);
            lb = ff_add(lb, vb[k]);
        }
        return true;
    };
    // Per lane, no collective: task i's p total and selected sums, once every record is known written.
    auto read1 = [&](int i, ff& vp, ff& va, ff& vb) {
        const Word* r = rec + (size_t)i * kRecWords;
        vp = unpack_ff(ld_word(r));
        va = unpack_ff(ld_word(r + 2));
        vb = unpack_ff(ld_word(r + 3));
    };
    ff lp{0.f, 0.f}, lq{0.f, 0.f}, la{0.f, 0.f}, lb{0.f, 0.f};
    ff ka[4], kb[4];  // the lane's first four tasks, kept for the crossing search
    const int nchunk = (per + 3) / 4;  // the same on every lane
    if (!__all_sync(0xFFFFFFFFu, poll4(s0, lp, lq, la, lb, ka, kb))) {
        fail_outputs(P, b, lane);  // timed out (reported in the status word)
        return;
    }
    for (int q = 1; q < nchunk; ++q) {
        ff va[4], vb[4];
        if (!__all_sync(0xFFFFFFFFu, poll4(s0 + 4 * q, lp, lq, la, lb, va, vb))) {
            fail_outputs(P, b, lane);
            return;
        }
    }
    const ff sp = warp_sum_ff(lp);
    bool resid = tk.mode == kModeResidual;
    ff rho{0.f, 0.f};
    ff W = la;  // the lane's weight: p mass (bonus) or A - rho B (residual)
    if (resid) {
        rho = ff_div(sp, warp_sum_ff(lq));  // exact s_p / s_q
        W = ff_sub(la, ff_mul(rho, lb));
    }
    ff incl = warp_inscan_ff(W, lane);
    ff S = shfl_ff(incl, 31);
    bool by_p = false;
    if ((resid || tk.mode == kModeResidualPM || tk.mode == kModeResidualSet) && !(S.hi > 0.f)) {  // mass 0: p
        resid = false;
        by_p = true;
        W = lp;
        incl = warp_inscan_ff(W, lane);
        S = shfl_ff(incl, 31);
    }
    const ff target = ff_mul(ff{tk.u, 0.f}, S);
    // the first lane whose inclusive prefix exceeds the target searches its own run of tasks
    const uint32_t hit = __ballot_sync(0xFFFFFFFFu, ff_gt(incl, target));
    const ff pre = exclusive_of(incl, lane);
    auto unit_w = [&](const ff& vp, const ff& va, const ff& vb) {
        ff w = by_p ? vp : va;
        if (resid) w = ff_sub(w, ff_mul(rho, vb));
        return w;
    };
    int unit = -1;
    ff before{0.f, 0.f};
    bool tail_rule = false;
    if (hit) {
        const int L = __ffs(hit) - 1;
        if (lane == L) {  // no collectives in here
            ff c = pre;
            int lastu = -1;
            ff lastc{0.f, 0.f};
            for (int i = s0; i < s1 && unit < 0; ++i) {
                ff vp{0.f, 0.f}, va{0.f, 0.f}, vb{0.f, 0.f};
                if (i - s0 < 4 && !by_p) {
#pragma unroll
                    for (int k = 0; k < 4; ++k)
                        if (i - s0 == k) { va = ka[k]; vb = kb[k]; }
                } else {
                    read1(i, vp, va, vb);
                }
                const ff w = unit_w(vp, va, vb);
                if (w.hi > 0.f) {
                    const ff c2 = ff_add(c, w);
                    if (ff_gt(c2, target)) {
                        unit = i;
                        before = c;
                    }
                    lastu = i;
                    lastc = c;
                    c = c2;
                }
            }
            if (unit < 0) {  // the lane's sum crossed, its running sum fell short by rounding
                unit = lastu;
                before = lastc;
            }
        }
        unit = __shfl_sync(0xFFFFFFFFu, unit, L);
        before = shfl_ff(before, L);
    }
    if (unit < 0) {  // no crossing at all (rounding): the last task with positive weight
        int last = -1;
        for (int i = s0; i < s1; ++i) {  // per lane, no collectives
            ff vp, va, vb;
            read1(i, vp, va, vb);
            if (unit_w(vp, va, vb).hi > 0.f) last = i;
        }
        unit = warp_max_i(last);
        tail_rule = true;
    }
    int32_t token = -1;
    if (unit >= 0) {
        const ff rem = ff_sub(target, before);
        // the groups' sums cover the residual and bonus weights; the p fallback scans the task's columns
        int32_t rtok = -1;
        if (!by_p && !removed_tokens(P, b, tk, lane, rtok)) token = -2;
        if (!by_p && token != -2)
            token = group_search<DT, VEC, TAB>(P, b, unit, tk, prow, qrow, resid, rho, rem, tail_rule, rtok, tab, vt,
                                               lane);
        if (by_p || token == -1) {
            const int32_t k_lo = unit * kSTask, k_hi = min(P.V, k_lo + kSTask);
            token = scan_elements<DT, VEC, TAB>(P, tk, prow, qrow, resid, rho, k_lo, k_hi, rem, tail_rule, rtok,
                                                by_p ? 0 : tk.nrm, tab, vt, lane);
        }
    }
    if (token < 0) {  // a time-out (reported in the status word)
        fail_outputs(P, b, lane);
        return;
    }
    // every output of the sequence: the accepted tokens, the drawn one, -1 after it
    const int32_t g = __ldg(P.offs + b + 1) - o0, npos = tk.npos;
    if (P.prog) {  // slot order: the rows after the emitting slot pass their check first
        const uint32_t e = check_dead_rows(P, b, g, tk.n, lane);
        if (e) {
            if (lane == 0) atomicOr(P.status, e);
            fail_outputs(P, b, lane);
            return;
        }
    }
    if (lane <= g) P.out_tokens[o0 + b + lane] = lane < npos ? acc_tok : (lane == npos ? token : -1);
    if (P.out_path && lane < g) P.out_path[o0 + lane] = lane < npos ? acc_node : -1;
    if (lane == 0) {
        P.out_n[b] = npos;
        if (P.dbg.seq_mass) P.dbg.seq_mass[b] = ((double)S.hi + (double)S.lo) / ((double)sp.hi + (double)sp.lo);
    }
    commit_seq(P, b, npos, acc_tok, token, lane);
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

// The accumulation of one sampler task: sequence b, columns [i * kSTask, (i + 1) * kSTask). Lane L
// walks its 32 consecutive columns [32 L, 32 L + 32) in 4 steps of 8 (one 16-byte load per row; a
// bf16 task's loads are all issued before the first step), accumulating the p and q weights and their
// selected parts. It stores the selected sums of each group of kGroupLanes lanes, then the warp's sums
// as the task's record. TWOSUM: carry the rounding of l - m (see exp2_ff2). TAB: the weights are the
// value table's 2^(l K) (table units, bf16 only), Gp / Gq the grid constants of their rows' largest
// weights; otherwise the precise exponential's 2^((l - m) K) <= 1 (Gp = Gq = 12). rho_sel: the selection
// ratio in the weights' units.
template <int DT, bool VEC, bool TWOSUM, bool REMOVED, bool RESID, bool TAB>
__device__ __noinline__ void s_accumulate(const Params& P, int32_t b, int i, const TaskInfo& tk, size_t prow,
                                          size_t qrow, const float* tab, const char* vt, int lane, uint32_t lane_rm,
                                          float Gp, float Gq, float rho_sel) {
    // RESID: a residual draw (p and q rows); else p alone (bonus, point-mass and tree residuals). Each
    // kind is its own instantiation, so each hot path's code is only its own.
    constexpr bool resid = RESID;
    const float2 mp = f2(tk.m_p), mq = f2(tk.m_q);
    const int32_t cbase = i * kSTask;
    const ExpConst EC = exp_const(P);
    // REMOVED: a point-mass or tree residual whose removed columns include some of this task's (bit j of
    // lane_rm: the lane's column cbase + 32 lane + j); its selected sums leave them out. A separate
    // instantiation, so the ordinary tasks' code carries no trace of it.
    constexpr bool excl = REMOVED;
    // grid-split accumulators (see grid_hi): all p and q weights, and those of the selected columns
    float2 Ph = f2(0.f), Pl = f2(0.f), Qh = f2(0.f), Ql = f2(0.f);
    float2 Ah = f2(0.f), Al = f2(0.f), Bh = f2(0.f), Bl = f2(0.f);
    auto wp = [&](const Cols8& c, int h) {
        if constexpr (TAB) return tab_pair(c.w[h], vt);
        else return exp2_ff2<TWOSUM>(pair8<DT>(c, h), mp, EC, tab);
    };
    auto wq = [&](const Cols8& c, int h) {
        if constexpr (TAB) return tab_pair(c.w[h], vt);
        else return exp2_ff2<TWOSUM>(pair8<DT>(c, h), mq, EC, tab);
    };
    // one step: 8 consecutive columns k, k + 1, ... of the lane (4 pairs) of the p row, and of the q row
    // for a residual
    auto step = [&](const Cols8& cp, const Cols8& cq, int32_t k) {
        if (RESID) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const ff2 ep = wp(cp, h);
                const ff2 eq = wq(cq, h);
                const float2 mk = sel_mask(ep, eq, rho_sel);
                const float2 hp = grid_hi(ep.hi, Gp), hq = grid_hi(eq.hi, Gq);
                const float2 lp = add2(sub2(ep.hi, hp), ep.lo), lq = add2(sub2(eq.hi, hq), eq.lo);
                Ph = add2(Ph, hp);
                Pl = add2(Pl, lp);
                Qh = add2(Qh, hq);
                Ql = add2(Ql, lq);
                Ah = fma2(mk, hp, Ah);
                Al = fma2(mk, lp, Al);
                Bh = fma2(mk, hq, Bh);
                Bl = fma2(mk, lq, Bl);
            }
        } else if (REMOVED) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const ff2 ep = wp(cp, h);
                const int bit = k - (cbase + 32 * lane) + 2 * h;
                const float2 mk = make_float2((lane_rm >> bit) & 1u ? 0.f : 1.f, (lane_rm >> (bit + 1)) & 1u ? 0.f : 1.f);
                const float2 hp = grid_hi(ep.hi, Gp), lp = add2(sub2(ep.hi, hp), ep.lo);
                Ph = add2(Ph, hp);
                Pl = add2(Pl, lp);
                Ah = fma2(mk, hp, Ah);
                Al = fma2(mk, lp, Al);
            }
        } else {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
                const ff2 ep = wp(cp, h);
                const float2 hp = grid_hi(ep.hi, Gp);
                Ph = add2(Ph, hp);
                Pl = add2(Pl, add2(sub2(ep.hi, hp), ep.lo));
            }
        }
    };
    // a ring of D steps in flight: bf16 loads the whole task at once, fp32 two steps ahead. The step
    // loop stays rolled: under the statistics stream, instruction fetches are slow, and this loop's
    // code must stay small enough to remain cached.
    constexpr int kSteps = kSTask / 256;
    constexpr int D = DT == SV_BF16 ? kSteps : 2;
    Cols8 rp[D], rq[D];
#pragma unroll
    for (int d = 0; d < D; ++d) {
        rp[d] = load_cols8<DT, VEC>(P.target, prow, P.V, cbase + 32 * lane + 8 * d);
        if (resid) rq[d] = load_cols8<DT, VEC>(P.draft, qrow, P.V, cbase + 32 * lane + 8 * d);
    }
#pragma unroll 1
    for (int e = 0; e < kSteps; ++e) {
        const Cols8 cp = rp[0], cq = rq[0];
#pragma unroll
        for (int d = 0; d + 1 < D; ++d) {
            rp[d] = rp[d + 1];
            rq[d] = rq[d + 1];
        }
        if (e + D < kSteps) {
            const int32_t k1 = cbase + 32 * lane + 8 * (e + D);
            rp[D - 1] = load_cols8<DT, VEC>(P.target, prow, P.V, k1);
            if (resid) rq[D - 1] = load_cols8<DT, VEC>(P.draft, qrow, P.V, k1);
        }
        step(cp, cq, cbase + 32 * lane + 8 * e);
    }
    // the group words first (read by the find only, which polls them): sums over kGroupLanes lanes; the
    // record's selected sums continue the same butterfly from the group sums
    static_assert(kGroupLanes == 4, "two butterfly levels per group");
    Word* gw = P.groupw + (((size_t)b * P.nS + i) * kGroups + lane / kGroupLanes) * kGroupWords;
    ff mine;  // record word `lane` (lanes 0-3)
    if (resid) {
        ffp g = lane_ffp(Ah, Al, Bh, Bl);  // (selected p, selected q)
        g = ffp_add(g, shfl_xor_ffp(g, 1));
        g = ffp_add(g, shfl_xor_ffp(g, 2));
        if (lane % kGroupLanes == 0) {
            st_word(gw, pack_ff(ff{g.hi.x, g.lo.x}));
            st_word(gw + 1, pack_ff(ff{g.hi.y, g.lo.y}));
        }
        ffp t = lane_ffp(Ph, Pl, Qh, Ql);  // (all p, all q)
#pragma unroll
        for (int o = 16; o; o >>= 1) t = ffp_add(t, shfl_xor_ffp(t, o));
#pragma unroll
        for (int o = kGroupLanes; o < 32; o <<= 1) g = ffp_add(g, shfl_xor_ffp(g, o));
        const ffp r = lane & 2 ? g : t;
        mine = lane & 1 ? ff{r.hi.y, r.lo.y} : ff{r.hi.x, r.lo.x};
    } else {
        // excl: the group words hold the selected p sums; else the p sums (a bonus draw's selected sums)
        ff ga = excl ? lane_ff(Ah, Al) : lane_ff(Ph, Pl);
        ga = ff_add(ga, ff{__shfl_xor_sync(0xFFFFFFFFu, ga.hi, 1), __shfl_xor_sync(0xFFFFFFFFu, ga.lo, 1)});
        ga = ff_add(ga, ff{__shfl_xor_sync(0xFFFFFFFFu, ga.hi, 2), __shfl_xor_sync(0xFFFFFFFFu, ga.lo, 2)});
        if (lane % kGroupLanes == 0) {
            st_word(gw, pack_ff(ga));
            st_word(gw + 1, pack_ff(ff{0.f, 0.f}));
        }
        const ff sa = warp_sum_ff_from(ga, kGroupLanes);
        const ff sp = excl ? warp_sum_ff(lane_ff(Ph, Pl)) : sa;
        mine = (lane == 1 || lane == 3) ? ff{0.f, 0.f} : lane == 2 ? sa : sp;
    }
    if (lane < kRecWords) st_word(P.recw + ((size_t)b * P.nS + i) * kRecWords + lane, pack_ff(mine));
}

// Sampler task c: sequence b = c / nS, task i = c % nS. The warp reads the sequence's sampler work
// (polled), accumulates and stores the task; the warp holding the last task of a sequence then runs
// its find. vt: the value table (nullptr where the kernel has none).
template <int DT, bool VEC>
__device__ void s_task(const Params& P, uint32_t c, const float* tab, const char* vt, int lane) {
    // c / nS by a multiply-high with floor(2^64 / nS) + 1: exact for c, nS < 2^32 (no MUFU reciprocal)
    int32_t b = P.nS == 1 ? (int32_t)c : (int32_t)__umul64hi((unsigned long long)c, P.nS_recip);
    const int i = (int)(c - (uint32_t)b * (uint32_t)P.nS);
    if (P.prog) {  // slot order: c / nS is a position of the decision-order queue
        const uint32_t p = (uint32_t)b;
        uint32_t e = ld_u32(P.order + p);
        uint32_t spins = 0, ns = 32;
        while (__any_sync(0xFFFFFFFFu, e == 0u)) {
            if (++spins > P.spin) {  // give the position up (its decision fails its sequence) unless it came
                if (lane == 0) {
                    e = atomicCAS(P.order + p, 0u, kOrderLost);
                    if (e == 0u) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
                }
                e = __shfl_sync(0xFFFFFFFFu, e, 0);
                break;
            }
            __nanosleep(ns);
            ns = ns < 256 ? 2 * ns : 256;
            e = ld_u32(P.order + p);
        }
        if (e == 0u || e == kOrderLost) return;
        b = (int32_t)(e - 1u);
    }
    const int32_t o0 = __ldg(P.offs + b);
    TaskInfo tk;
    if (!get_task(P, b, lane, tk)) {
        give_up_seq(P, b, lane);
        return;
    }
    if (tk.mode == kModeNone) return;
    const size_t prow = (size_t)(o0 + b + tk.n), qrow = (size_t)(o0 + tk.n);
    uint32_t lane_rm = 0;  // the draw's removed columns among this lane's (point-mass and tree residuals)
    if (tk.nrm) {          // warp-uniform
        int32_t rtok = -1;
        if (!removed_tokens(P, b, tk, lane, rtok)) {
            give_up_seq(P, b, lane);
            return;
        }
        lane_rm = removed_bits(rtok, tk.nrm, i * kSTask + 32 * lane, 32);
    }
    const bool rm = __any_sync(0xFFFFFFFFu, lane_rm != 0u);
    const bool res = tk.mode == kModeResidual;
    if constexpr (DT == SV_BF16 && VEC) {
        if (vt && draw_uses_table<DT, VEC>(P, tk.mode, tk.m_p, tk.m_q)) {
            // value-table weights 2^(l K): below 2^(m K) in each row, which sets the grid constant
            const float Gp = grid_const(tk.m_p * P.K_hi), Gq = res ? grid_const(tk.m_q * P.K_hi) : 12.f;
            if (rm) s_accumulate<DT, VEC, false, true, false, true>(P, b, i, tk, prow, qrow, tab, vt, lane, lane_rm, Gp, Gq, tk.rho);
            else if (res) s_accumulate<DT, VEC, false, false, true, true>(P, b, i, tk, prow, qrow, tab, vt, lane, 0u, Gp, Gq, tk.rho);
            else s_accumulate<DT, VEC, false, false, false, true>(P, b, i, tk, prow, qrow, tab, vt, lane, 0u, Gp, Gq, tk.rho);
            if (i == P.nS - 1) find<DT, VEC, true>(P, b, tk, prow, qrow, o0, tab, vt, lane);
            return;
        }
    }
    // precise-exponential weights 2^((l - m) K) <= 1; rows whose maximum is near zero carry the rounding of
    // l - m (see exp2_ff2)
    const bool twosum = fabsf(tk.m_p) < kNeedTwoSum || (res && fabsf(tk.m_q) < kNeedTwoSum);
    if (rm) {
        if (twosum) s_accumulate<DT, VEC, true, true, false, false>(P, b, i, tk, prow, qrow, tab, vt, lane, lane_rm, 12.f, 12.f, tk.rho);
        else s_accumulate<DT, VEC, false, true, false, false>(P, b, i, tk, prow, qrow, tab, vt, lane, lane_rm, 12.f, 12.f, tk.rho);
    } else if (res) {
        if (twosum) s_accumulate<DT, VEC, true, false, true, false>(P, b, i, tk, prow, qrow, tab, vt, lane, 0u, 12.f, 12.f, tk.rho);
        else s_accumulate<DT, VEC, false, false, true, false>(P, b, i, tk, prow, qrow, tab, vt, lane, 0u, 12.f, 12.f, tk.rho);
    } else if (twosum) {
        s_accumulate<DT, VEC, true, false, false, false>(P, b, i, tk, prow, qrow, tab, vt, lane, 0u, 12.f, 12.f, tk.rho);
    } else {
        s_accumulate<DT, VEC, false, false, false, false>(P, b, i, tk, prow, qrow, tab, vt, lane, 0u, 12.f, 12.f, tk.rho);
    }
    if (i == P.nS - 1) find<DT, VEC, false>(P, b, tk, prow, qrow, o0, tab, vt, lane);
}

// ------------------------------------------------------------------------------------------------
// Statistics tasks
// ------------------------------------------------------------------------------------------------
struct ATask {
    int32_t r, ch;
    const char* rowp;
    int len;
};

// Source row of statistics row r. Greedy: the rows are the target rows themselves. Sampling: from the
// shared-memory row map when the batch has one (entry: draft flag in the sign bit, row index below),
// else through a sequence cursor that only moves forward (a warp visits its tasks in increasing
// order, so the owning sequence is found with a couple of cached offset reads instead of a search).
template <int DT, bool GREEDY>
__device__ __forceinline__ const char* stat_row_src(const Params& P, int32_t r, int32_t ch, int32_t& cur,
                                                    const int32_t* bases, const int32_t* rows) {
    const size_t esz = DT == SV_BF16 ? 2 : 4;
    size_t row = (size_t)r;
    bool draft = false;
    if (!GREEDY && !P.pm) {  // greedy and point-mass batches stream target rows only: row = r
        if (rows) {
            const int32_t v = rows[r];
            draft = v < 0;
            row = (size_t)(v & 0x7FFFFFFF);
        } else {
            while (cur + 1 < P.B && (bases ? bases[cur + 1] : stat_base<false>(P, cur + 1)) <= r) ++cur;
            const int32_t o0 = __ldg(P.offs + cur), g = __ldg(P.gammas + cur);
            const int32_t j = r - (2 * o0 + cur);
            draft = j > g;
            row = draft ? (size_t)(o0 + j - g - 1) : (size_t)(o0 + cur + j);
        }
    }
    return (const char*)(draft ? P.draft : P.target) + (row * (size_t)P.V + (size_t)ch * kAChunk) * esz;
}

// Source of slot-order row q (see prog_q): from the row map entry.
__device__ __forceinline__ const char* prog_row_src(const Params& P, int32_t q, int32_t ch, const int32_t* rows) {
    const uint32_t v = (uint32_t)rows[q];
    const size_t row = v & 0xFFFu;
    return (const char*)(v >> 31 ? P.draft : P.target) + (row * (size_t)P.V + (size_t)ch * kAChunk) * 2;
}

template <int DT, bool GREEDY>
__device__ __forceinline__ ATask a_task_at(const Params& P, uint32_t t, int32_t& cur, const int32_t* bases,
                                           const int32_t* rows) {
    ATask at;
    at.r = (int32_t)(t / (uint32_t)P.nchA);
    at.ch = (int32_t)(t % (uint32_t)P.nchA);
    at.rowp = stat_row_src<DT, GREEDY>(P, at.r, at.ch, cur, bases, rows);
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

// Decision of sequence b, run by its decider warp (or, cooperative, by the CTA's deciding warps); the
// deciding warps poll the partial words themselves.
template <int DT, bool VEC, bool GREEDY>
__device__ void lead_decide(const Params& P, int32_t b, const int32_t* bases, const float* tab, int lane, int wsub,
                            int nsub, CoopRows* co, int set) {
    int32_t o0, g;
    if (bases) {  // from the validated offsets cached in shared memory: no dependent global load
        const int32_t s0 = bases[b], s1 = bases[b + 1];
        o0 = GREEDY || P.pm ? s0 - b : (s0 - b) >> 1;
        g = GREEDY || P.pm ? s1 - s0 - 1 : (s1 - s0 - 1) >> 1;
    } else {
        o0 = __ldg(P.offs + b);
        g = __ldg(P.gammas + b);
    }
    decide<DT, VEC, GREEDY>(P, b, g, o0, lane, tab, wsub, nsub, co, set);
}

// A streamer warp on the bulk-copy path: its statistics tasks (statically strided over all streamers)
// arrive through a ring of kStages shared-memory stages filled by 1-D bulk copies, so up to
// kStages - 1 tasks stay in flight while one is reduced, without holding registers. The position (row or
// slot-order index, chunk) of the task being reduced and of the task that refills its stage advance
// incrementally; the refill's source is resolved before waiting on the stage, so its lookups overlap the
// wait and the reduction. In slot order (P.prog) the positions skip holes.
__device__ void stream_bulk(const Params& P, uint32_t nA, unsigned char* dsmem, const int32_t* bases,
                            const int32_t* rows, int warp, int lane) {
    uint64_t* bars = reinterpret_cast<uint64_t*>(dsmem + kStreamWarps * kStages * kStageBytes) + warp * kStages;
    unsigned char* bufs = dsmem + (size_t)warp * kStages * kStageBytes;
    const uint32_t SW = gridDim.x * kStreamWarps;
    const uint32_t sw = blockIdx.x * kStreamWarps + warp;
    const uint32_t nch = (uint32_t)P.nchA;
    const uint32_t dr = SW / nch, dc = SW % nch;
    const bool prog = P.prog;
    struct Pos {
        uint32_t t, q, c;  // task index, row (slot-order index in slot order), chunk
    };
    auto advance = [&](Pos& p) {
        p.t += SW;
        p.q += dr;
        p.c += dc;
        if (p.c >= nch) {
            p.c -= nch;
            ++p.q;
        }
    };
    // the statistics row of p (slot order: skipping holes)
    auto settle = [&](Pos& p) -> int32_t {
        if (!prog) return (int32_t)p.q;
        for (; p.t < nA; advance(p))
            if ((uint32_t)rows[p.q] != kProgHole) return (int32_t)p.q;
        return -1;
    };
    auto src_of = [&](int32_t r, uint32_t c, int32_t& cur) {
        return prog ? prog_row_src(P, r, (int32_t)c, rows) : stat_row_src<SV_BF16, false>(P, r, (int32_t)c, cur, bases, rows);
    };
    auto len_of = [&](uint32_t c) { return min(kAChunk, P.V - (int)c * kAChunk); };
    if (lane == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&bars[s], 1);
        fence_mbar_init();
    }
    __syncwarp();
    int32_t cur = 0;
    auto issue = [&](const char* src, uint32_t bytes, int s) {  // lane 0
        mbar_arrive_expect_tx(&bars[s], bytes);
        bulk_g2s(bufs + (size_t)s * kStageBytes, src, bytes, &bars[s]);
    };
    Pos rp{sw, sw / nch, sw % nch};  // task being reduced
    int32_t rr = settle(rp);
    Pos ip = rp;                     // next task to issue
    for (int s = 0; s < kStages; ++s) {
        const int32_t ir = settle(ip);
        if (ip.t < nA) {
            const char* src = src_of(ir, ip.c, cur);
            if (lane == 0) issue(src, (uint32_t)len_of(ip.c) * 2u, s);
            advance(ip);
        }
    }
    uint32_t parity = 0;  // bit s: parity of stage s's next completion
    int k = 0;
    for (; rp.t < nA; ++k) {
        const int s = k % kStages;
        const int32_t nr = settle(ip);
        const bool more = ip.t < nA;
        const char* nsrc = nullptr;
        uint32_t nbytes = 0;
        if (more) {
            nsrc = src_of(nr, ip.c, cur);
            nbytes = (uint32_t)len_of(ip.c) * 2u;
        }
        // one verdict for the whole warp: a time-out seen by some lanes only must not split it (a copy
        // always lands: this bound is the library's, never a caller's)
        const bool ok = __all_sync(0xFFFFFFFFu, mbar_wait(&bars[s], (parity >> s) & 1u, kSpinLimit));
        if (!ok) {
            // a copy that does not land: report, give every copy in flight (this stage's included) its
            // own bound to land before the shared memory is left, stop streaming
            if (lane == 0) atomicOr(P.status, 1u << SV_ERR_TIMEOUT);
            Pos q = rp;
            for (int i = 0; i < kStages; ++i) {
                settle(q);
                if (q.t >= nA) break;
                const int s2 = (k + i) % kStages;
                mbar_wait(&bars[s2], (parity >> s2) & 1u, kSpinLimit);
                advance(q);
            }
            return;
        }
        parity ^= 1u << s;
        ATask at;
        at.r = rr;
        at.ch = (int32_t)rp.c;
        at.len = len_of(rp.c);
        // the stage is refilled only once its task is reduced: with one copy per streamer in flight during
        // the reduction the stream keeps HBM busy without queueing the handoff loads of the decisions and
        // finds behind it (refilling right after the stage is read into registers measured slower)
        uint4 v[16];
        load_stage(bufs + (size_t)s * kStageBytes, at.len, lane, v);
        const SegStats st = stats_bf16(v, P.K_hi);
        __syncwarp();
        if (lane == 0 && more) {
            fence_proxy_async_smem();  // this stage's reads come before the copy that overwrites it
            issue(nsrc, nbytes, s);
        }
        if (more) advance(ip);
        a_finish<false>(P, at, st, lane);
        advance(rp);
        rr = settle(rp);
    }
}

// ------------------------------------------------------------------------------------------------
// The kernel
// ------------------------------------------------------------------------------------------------
template <int DT, bool VEC, bool GREEDY>
__global__ void __launch_bounds__(kThreads, 1) k_verify(const __grid_constant__ Params P) {
    constexpr bool kBulk = DT == SV_BF16 && VEC && !GREEDY;
    extern __shared__ __align__(128) unsigned char dsmem[];
    __shared__ float tab[2 * kExpTab];
    __shared__ int s_bad;
    __shared__ int32_t s_base[kBaseCache];
    __shared__ int32_t s_row[GREEDY ? 1 : kRowCache];
    __shared__ CoopRows s_coop;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (!GREEDY) fill_exp2_table(P, tab);
    if (tid == 0) {
        s_bad = __ldg(P.offs) != 0;
        s_coop.err[0] = s_coop.err[1] = 0u;
        s_coop.key[0] = s_coop.key[1] = ~0u;
    }
    __syncthreads();
    // every CTA checks the whole CSR structure before any row is read (and caches small batches' row
    // bases, b = 0..B, for the statistics tasks and the decisions)
    int bad = 0;
    const bool cache = P.B < kBaseCache;
    if (cache && tid == 0) {  // the end of the last sequence's rows
        const int32_t oB = __ldg(P.offs + P.B);
        s_base[P.B] = GREEDY || P.pm ? oB + P.B : 2 * oB + P.B;
    }
    for (int32_t b = tid; b < P.B; b += kThreads) {
        const int32_t o0 = __ldg(P.offs + b), o1 = __ldg(P.offs + b + 1), g = __ldg(P.gammas + b);
        const bool ok = g >= 0 && g <= P.max_gamma && o0 >= 0 && o1 - o0 == g;
        bad |= !ok;
        const int32_t sb = GREEDY || P.pm ? o0 + b : 2 * o0 + b;
        if (cache) s_base[b] = sb;
        if (kBulk && P.prog) {  // slot-order map (its size is checked by the host): every q of sequence b
            if (ok)
                for (int32_t sl = 0; sl <= P.max_gamma; ++sl) {
                    const uint32_t id = (uint32_t)b << 12 | (uint32_t)sl << 22;
                    s_row[prog_q(P, b, sl, false)] = (int32_t)(sl <= g ? id | (uint32_t)(o0 + b + sl) : kProgHole);
                    if (sl < P.max_gamma)
                        s_row[prog_q(P, b, sl, true)] =
                            (int32_t)(sl < g ? 0x80000000u | id | (uint32_t)(o0 + sl) : kProgHole);
                }
        } else if (!GREEDY && !P.pm && ok) {  // row map entries that fit (used only when every row fits)
            for (int32_t j = 0; j <= 2 * g && sb + j < kRowCache; ++j)
                s_row[sb + j] = j <= g ? o0 + b + j : (int32_t)(0x80000000u | (uint32_t)(o0 + j - g - 1));
        }
    }
    const int32_t* bases = cache ? s_base : nullptr;
    if (__syncthreads_or(bad) || s_bad) {
        if (blockIdx.x == 0) {
            for (int32_t b = tid; b < P.B; b += kThreads) {
                P.out_n[b] = -1;
                if (P.hist) P.next[b] = -1;
            }
            if (tid == 0) atomicOr(P.status, 1u << SV_ERR_BAD_OFFSETS);
        }
        return;
    }
    const int32_t oB = __ldg(P.offs + P.B);
    // the host bounds rows * nchA and B * nS below 2^31
    const uint32_t nA = (kBulk && P.prog ? prog_rows(P) : (uint32_t)(GREEDY || P.pm ? oB + P.B : 2 * oB + P.B)) *
                        (uint32_t)P.nchA;
    const uint32_t nStot = GREEDY ? 0u : (uint32_t)P.B * (uint32_t)P.nS;
    const int32_t* rows = (kBulk && P.prog) || (!GREEDY && !P.pm && 2 * oB + P.B <= kRowCache) ? s_row : nullptr;

    // Statistics. Bulk-copy path: the upper kStreamWarps warps of the CTA stream while the lower ones
    // build the sampler's value table, then decide and take sampler tasks. Other paths: every warp streams
    // its strided tasks from registers first.
    // The value table is built by the non-streaming warps, which wait for one another (named barrier 2)
    // and then only signal barrier 3; a streamer waits on barrier 3 once its stream is done, before its
    // first sampler task (by then the table is long finished).
    const bool use_tab = kBulk && P.use_tab;
    const char* vt = use_tab ? reinterpret_cast<const char*>(dsmem + kTabSmemOffset) : nullptr;
    constexpr int kBuilders = (kWarps - kStreamWarps) * 32;
    if (kBulk) {
        if (warp >= kWarps - kStreamWarps) {
            stream_bulk(P, nA, dsmem, bases, rows, warp - (kWarps - kStreamWarps), lane);
            if (use_tab) asm volatile("bar.sync 3, %0;" ::"r"(kThreads) : "memory");
        } else if (use_tab) {
            build_value_table(P, reinterpret_cast<float2*>(dsmem + kTabSmemOffset), tab, tid, kBuilders);
            asm volatile("bar.sync 2, %0;" ::"r"(kBuilders) : "memory");
            asm volatile("bar.arrive 3, %0;" ::"r"(kThreads) : "memory");
        }
    } else {
        const uint32_t W = gridDim.x * kWarps;
        int32_t cur = 0;
        for (uint32_t a = blockIdx.x * kWarps + warp; a < nA; a += W) {
            const ATask at = a_task_at<DT, GREEDY>(P, a, cur, bases, rows);
            const SegStats st = seg_stats<DT, VEC, GREEDY>(at.rowp, at.len, lane, P.K_hi);
            a_finish<GREEDY>(P, at, st, lane);
        }
    }
    // Work after the statistics:
    //   decisions, assigned statically: decider slot d (the non-streamer warps on the bulk-copy path,
    //     every warp otherwise) decides sequences d, d + ND, ... (each polls its sequence's partial
    //     words and, sampling, writes the sequence's sampler work);
    //   sampler tasks, claimed one at a time from a counter in sequence-major order by whichever warp
    //     is free (streamers join when their stream ends); the warp that claims a sequence's last task
    //     runs its find after the task.
    // Waits are bounded. A decision waits only on statistics tasks, which are done by warps that never
    // wait before finishing them. A sampler task waits on its decision, and a find on tasks of its own
    // sequence claimed before its own; a warp claims only when free, so every awaited word is produced
    // by a running warp that is not (transitively) waiting on the waiter.
    const bool streamer = kBulk && warp >= kWarps - kStreamWarps;
    const uint32_t ND = kBulk ? gridDim.x * (kWarps - kStreamWarps) : gridDim.x * kWarps;
    const uint32_t did = kBulk ? blockIdx.x * (kWarps - kStreamWarps) + warp : blockIdx.x * kWarps + warp;
    // Cooperative decisions when every CTA holds at most one: the non-streaming warps of CTA c share the
    // rows of sequence c (the decision's latency, not its throughput, is what the step waits for)
    const bool coop = kBulk && (uint32_t)P.B <= gridDim.x;
    if (kBulk && P.prog) {  // slot order: one warp decides a sequence, slot by slot
        const uint32_t d = coop ? (warp == 0 ? blockIdx.x : (uint32_t)P.B) : did;
        if (!streamer)
            for (uint32_t b = d; b < (uint32_t)P.B; b += coop ? (uint32_t)P.B : ND) {
                const int32_t s0 = bases[b], s1 = bases[b + 1];
                const int32_t o0 = P.pm ? s0 - (int32_t)b : (s0 - (int32_t)b) >> 1;
                const int32_t g = P.pm ? s1 - s0 - 1 : (s1 - s0 - 1) >> 1;
                decide_prog<DT, VEC>(P, (int32_t)b, g, o0, lane, tab);
            }
    } else if (coop) {
        if (!streamer && blockIdx.x < (uint32_t)P.B)
            lead_decide<DT, VEC, GREEDY>(P, (int32_t)blockIdx.x, bases, tab, lane, warp, kWarps - kStreamWarps, &s_coop, 0);
    } else if (!streamer) {
        for (uint32_t b = did; b < (uint32_t)P.B; b += ND) lead_decide<DT, VEC, GREEDY>(P, (int32_t)b, bases, tab, lane, 0, 1, &s_coop, 0);
    }
    if constexpr (!GREEDY) {
        while (true) {
            uint32_t t = 0;
            if (lane == 0) t = atomicAdd(&P.ctr->claim, 1u);
            t = __shfl_sync(0xFFFFFFFFu, t, 0);
            if (t >= nStot) break;
            s_task<DT, VEC>(P, t, tab, vt, lane);
        }
    }
}

// ------------------------------------------------------------------------------------------------
// Debug output beta_i = sum_x min(p_i(x), q_i(x)) (velog "6-1편. Speculative Decoding", §2-3: the
// probability that slot i's draft is accepted), recomputed from the logits after the step, one CTA per
// draft row: fp32 exponentials, fp64 sums. Point-mass drafts: beta_i = p_i(x_i). Not on the step's path.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ double block_sum(double v, double* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    double t = 0.0;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t += red[w];
    return t;
}
__device__ __forceinline__ float block_max(float v, double* red) {
    v = warp_max(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = (double)v;
    __syncthreads();
    float t = -INFINITY;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = fmaxf(t, (float)red[w]);
    return t;
}

template <int DT>
__global__ void __launch_bounds__(256) k_debug_beta(const __grid_constant__ Params P) {
    __shared__ double red[8];
    const int32_t r = (int32_t)blockIdx.x;  // draft slot
    if (*(volatile uint32_t*)P.status & (1u << SV_ERR_BAD_OFFSETS)) return;  // rows not owned reliably
    const int32_t R_d = __ldg(P.offs + P.B);
    if (r >= R_d) return;
    int32_t lo = 0, hi = P.B - 1;  // sequence b with offs[b] <= r < offs[b + 1]
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(P.offs + mid) <= r) lo = mid; else hi = mid - 1;
    }
    const int32_t b = lo, x = __ldg(P.tokens + r);
    if (x < 0 || x >= P.V) return;
    const size_t trow = (size_t)(r + b) * (size_t)P.V, drow = (size_t)r * (size_t)P.V;
    const float K = P.K_hi;
    float mt = -INFINITY, md = -INFINITY;
    for (int32_t k = threadIdx.x; k < P.V; k += blockDim.x) {
        mt = fmaxf(mt, logit_at<DT>(P.target, trow + k));
        if (!P.pm) md = fmaxf(md, logit_at<DT>(P.draft, drow + k));
    }
    mt = block_max(mt, red);
    if (!P.pm) md = block_max(md, red);
    double st = 0.0, sd = 0.0;
    for (int32_t k = threadIdx.x; k < P.V; k += blockDim.x) {
        st += (double)exp2f((logit_at<DT>(P.target, trow + k) - mt) * K);
        if (!P.pm) sd += (double)exp2f((logit_at<DT>(P.draft, drow + k) - md) * K);
    }
    st = block_sum(st, red);
    if (P.pm) {
        if (threadIdx.x == 0) P.dbg.beta[r] = (double)exp2f((logit_at<DT>(P.target, trow + x) - mt) * K) / st;
        return;
    }
    sd = block_sum(sd, red);
    double m = 0.0;
    for (int32_t k = threadIdx.x; k < P.V; k += blockDim.x) {
        const double pk = (double)exp2f((logit_at<DT>(P.target, trow + k) - mt) * K) / st;
        const double qk = (double)exp2f((logit_at<DT>(P.draft, drow + k) - md) * K) / sd;
        m += pk < qk ? pk : qk;
    }
    m = block_sum(m, red);
    if (threadIdx.x == 0) P.dbg.beta[r] = m;
}

// ------------------------------------------------------------------------------------------------
// Launch
// ------------------------------------------------------------------------------------------------
template <int DT, bool VEC, bool GREEDY>
static cudaError_t launch_typed(const Params& P, cudaStream_t st) {
    constexpr bool kBulk = DT == SV_BF16 && VEC && !GREEDY;
    constexpr int smem = kBulk ? kTabSmemOffset + kTabBytes : 0;  // stages, their barriers, the value table
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
    {  // small sampled batches (at most one statistics task per streaming warp of the persistent launch): one
       // CTA cluster per sequence (sv_debug.cluster: 1 never, 2 whenever the call allows it, greedy included;
       // a greedy step, a decision without a draw, is shorter as the persistent launch)
        int dev = 0, sms = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        int32_t C = 0;
        const int64_t rows = (int64_t)P.B * (greedy || P.pm ? P.max_gamma + 1 : 2 * P.max_gamma + 1);
        const bool small = P.dbg.cluster == 2u ||
                           (P.dbg.cluster == 0u && !greedy && rows * P.nchA <= (int64_t)sms * kStreamWarps);
        if (small && P.dbg.cluster != 1u && small_eligible(P, sms, &C)) return launch_small(P, dtype, C, st);
    }
    cudaError_t e = cudaMemsetAsync((char*)ws + L.zero_begin, 0, L.zero_end - L.zero_begin, st);
    if (e != cudaSuccess) return e;
    if (dtype == SV_BF16) {
        if (vec) e = greedy ? launch_typed<SV_BF16, true, true>(P, st) : launch_typed<SV_BF16, true, false>(P, st);
        else e = greedy ? launch_typed<SV_BF16, false, true>(P, st) : launch_typed<SV_BF16, false, false>(P, st);
    } else {
        if (vec) e = greedy ? launch_typed<SV_F32, true, true>(P, st) : launch_typed<SV_F32, true, false>(P, st);
        else e = greedy ? launch_typed<SV_F32, false, true>(P, st) : launch_typed<SV_F32, false, false>(P, st);
    }
    if (e != cudaSuccess || greedy || !P.dbg.beta || P.max_gamma == 0) return e;
    // debug output only: beta of every draft slot, after the step on the same stream
    const unsigned grid = (unsigned)((int64_t)P.B * P.max_gamma);
    if (dtype == SV_BF16) k_debug_beta<SV_BF16><<<grid, 256, 0, st>>>(P);
    else k_debug_beta<SV_F32><<<grid, 256, 0, st>>>(P);
    return cudaGetLastError();
}

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t nchA = ((size_t)V + kAChunk - 1) / kAChunk;
    const size_t nS = ((size_t)V + kSTask - 1) / kSTask;
    Layout L;
    // every region before the status word is cleared before every call, with one memset
    L.counters = 0;
    L.partials = up(L.counters + sizeof(Counters));
    L.taskw = up(L.partials + (size_t)B * (2 * (size_t)max_gamma + 1) * nchA * sizeof(PartialWord));
    L.recw = up(L.taskw + (size_t)B * kTaskWords * sizeof(Word));
    L.groupw = up(L.recw + (size_t)B * nS * kRecWords * sizeof(Word));
    L.remw = up(L.groupw + (size_t)B * nS * kGroups * kGroupWords * sizeof(Word));
    L.pathw = up(L.remw + (size_t)B * kMaxRemoved * sizeof(Word));
    L.seqstate = up(L.pathw + (size_t)B * kMaxRemoved * sizeof(Word));
    L.order = up(L.seqstate + (size_t)B * sizeof(uint32_t));
    L.status = up(L.order + (size_t)B * sizeof(uint32_t));
    L.zero_begin = 0;
    L.zero_end = L.status;
    L.total = up(L.status + sizeof(uint32_t));
    return L;
}

}  // namespace sv
