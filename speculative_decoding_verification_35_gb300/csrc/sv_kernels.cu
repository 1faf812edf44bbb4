// Kernels of the speculative-sampling verify step (sm_103a).
//
// The step, for each sequence of a CSR-packed batch (velog "6-1편. Speculative Decoding", §2 steps 3-4,
// §2-1, §2-2; greedy: "All About Transformer Inference", App. D steps 1-3):
//   k_stats        one pass over every logit the step needs: per (row, vocabulary chunk) the raw
//                  maximum, sum of exp((l - max) / T) in fp32 and (greedy) the first argmax.
//                  This pass moves almost all of the HBM traffic.
//   k_decide       one warp per sequence: merge the chunk partials of each row, evaluate
//                  u_i * q_i(x_i) < p_i(x_i) for every slot in fp64, find the first rejection with a
//                  warp ballot, write the accepted tokens and the draw each sequence needs.
//   k_sample_sums  the draw's weights in float-float precision (residual max(0, p - q) or p), summed
//                  per 512-token sub-chunk. The rows were streamed moments before (L2-resident).
//   k_sample_find  one warp per sequence: exact normalisers, inverse CDF over the sub-chunk sums,
//                  then over the 512 tokens of the crossing sub-chunk, in fp64.
// Precision: the accept test tolerates fp32 statistics (its decision moves with an error ~1e-7 of
// p/q); the inverse CDF over ~1e5 tokens does not, so the sampler recomputes its row(s) with a
// float-float exponential (relative error ~1e-9) and exact normalisers.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {

// ------------------------------------------------------------------------------------------------
// CSR structure checks. A sequence is read only when its own offsets are consistent with the
// batch total, so no row index can leave [0, R) whatever the offsets hold.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ bool batch_ok(const Params& P) {
    const int32_t oB = __ldg(P.offs + P.B);
    return __ldg(P.offs) == 0 && oB >= 0 && (long long)oB <= (long long)P.B * P.max_gamma;
}

__device__ __forceinline__ bool seq_ok(const Params& P, int32_t b, int32_t& g, int32_t& o0) {
    o0 = __ldg(P.offs + b);
    const int32_t o1 = __ldg(P.offs + b + 1), oB = __ldg(P.offs + P.B);
    g = __ldg(P.gammas + b);
    return o0 >= 0 && o0 <= o1 && o1 <= oB && o1 - o0 == g && g <= P.max_gamma;
}

// Statistics rows of a sequence: gamma + 1 target rows, then (sampling) gamma draft rows.
template <bool GREEDY>
__device__ __forceinline__ int32_t stat_rows(int32_t g) { return GREEDY ? g + 1 : 2 * g + 1; }

template <bool GREEDY>
__device__ __forceinline__ int32_t stat_base(const Params& P, int32_t b) {
    const int32_t o = __ldg(P.offs + b);
    return GREEDY ? o + b : 2 * o + b;
}

// Largest b with stat_base(b) <= r (terminates for any offsets).
template <bool GREEDY>
__device__ int32_t find_seq(const Params& P, int32_t r) {
    int32_t lo = 0, hi = P.B - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (stat_base<GREEDY>(P, mid) <= r) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// ------------------------------------------------------------------------------------------------
// k_validate: the whole CSR structure, before any row is read. One CTA; writes the batch flag every
// call (no stale state). Inconsistent offsets make row ownership ambiguous, so they fail the batch.
// ------------------------------------------------------------------------------------------------
__global__ void __launch_bounds__(kThreads) k_validate(const Params P) {
    __shared__ uint32_t s_bad;
    if (threadIdx.x == 0) s_bad = __ldg(P.offs) != 0;
    __syncthreads();
    uint32_t bad = 0;
    for (int32_t b = threadIdx.x; b < P.B; b += kThreads) {
        const int32_t o0 = __ldg(P.offs + b), o1 = __ldg(P.offs + b + 1), g = __ldg(P.gammas + b);
        bad |= !(g >= 0 && g <= P.max_gamma && o0 >= 0 && o1 - o0 == g);
    }
    if (bad) atomicOr(&s_bad, 1u);
    __syncthreads();
    if (threadIdx.x == 0) {
        *P.batch_bad = s_bad;
        if (s_bad) atomicOr(P.status, 1u << SV_ERR_BAD_OFFSETS);
    }
}

template <int DT>
__device__ __forceinline__ float logit_at(const void* base, size_t idx) {
    if (DT == SV_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)base + idx) << 16);
    return __ldg((const float*)base + idx);
}

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

// Table of 2^(j/64), j = 0..63, as float-float, built from the fp64 exp2 of the CUDA math library.
__device__ __forceinline__ void fill_exp2_table(float2* tab) {
    if (threadIdx.x < 64) {
        const double v = exp2((double)threadIdx.x * (1.0 / 64.0));
        const float hi = (float)v;
        tab[threadIdx.x] = make_float2(hi, (float)(v - (double)hi));
    }
}

// ------------------------------------------------------------------------------------------------
// k_stats: per (row, chunk) statistics. 32 elements per thread, 8192 per CTA item.
// ------------------------------------------------------------------------------------------------
template <int DT, bool VEC>
struct Loader {
    // elements per thread = 32; e(i) is the chunk offset of element i of thread t, increasing in i
    static constexpr int kPerLoad = VEC ? (DT == SV_BF16 ? 8 : 4) : 1;
    static constexpr int kLoads = 32 / kPerLoad;
    __device__ static __forceinline__ int offset(int i, int t) {
        return ((i / kPerLoad) * kThreads + t) * kPerLoad + (i % kPerLoad);
    }
    __device__ static __forceinline__ void load(const void* row, int len, int t, float (&x)[32]) {
        if (VEC && DT == SV_BF16) {
            const uint4* p = (const uint4*)row;
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                const int e0 = (q * kThreads + t) * 8;
                const uint4 v = e0 < len ? ldg_stream(p + q * kThreads + t)
                                         : make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u);
                x[q * 8 + 0] = bf16lo_to_f32(v.x); x[q * 8 + 1] = bf16hi_to_f32(v.x);
                x[q * 8 + 2] = bf16lo_to_f32(v.y); x[q * 8 + 3] = bf16hi_to_f32(v.y);
                x[q * 8 + 4] = bf16lo_to_f32(v.z); x[q * 8 + 5] = bf16hi_to_f32(v.z);
                x[q * 8 + 6] = bf16lo_to_f32(v.w); x[q * 8 + 7] = bf16hi_to_f32(v.w);
            }
        } else if (VEC) {
            const uint4* p = (const uint4*)row;
#pragma unroll
            for (int q = 0; q < kLoads; ++q) {
                const int e0 = (q * kThreads + t) * 4;
                const uint4 v = e0 < len ? ldg_stream(p + q * kThreads + t)
                                         : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
                x[q * 4 + 0] = __uint_as_float(v.x); x[q * 4 + 1] = __uint_as_float(v.y);
                x[q * 4 + 2] = __uint_as_float(v.z); x[q * 4 + 3] = __uint_as_float(v.w);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int e = i * kThreads + t;
                x[i] = e < len ? logit_at<DT>(row, (size_t)e) : -INFINITY;
            }
        }
    }
};

template <int DT, bool VEC, bool GREEDY>
__global__ void __launch_bounds__(kThreads) k_stats(const Params P) {
    __shared__ float s_redf[kThreads / 32];
    __shared__ int s_redi[kThreads / 32];
    __shared__ uint32_t s_redu[kThreads / 32];
    if (*P.batch_bad || !batch_ok(P)) return;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const int32_t oB = __ldg(P.offs + P.B);
    const int32_t total_rows = GREEDY ? oB + P.B : 2 * oB + P.B;
    const long long items = (long long)total_rows * P.nchunks;
    const size_t esz = DT == SV_BF16 ? 2 : 4;
    for (long long w = blockIdx.x; w < items; w += gridDim.x) {
        const int32_t r = (int32_t)(w / P.nchunks), c = (int32_t)(w % P.nchunks);
        const int32_t b = find_seq<GREEDY>(P, r);
        int32_t g, o0;
        if (!seq_ok(P, b, g, o0)) continue;
        const int32_t j = r - (GREEDY ? o0 + b : 2 * o0 + b);
        if (j < 0 || j >= stat_rows<GREEDY>(g)) continue;
        const size_t row = j <= g ? (size_t)(o0 + b + j) : (size_t)(o0 + j - g - 1);
        const char* base = (const char*)(j <= g ? P.target : P.draft);
        const int32_t k0 = c * kChunk;
        const int len = min(kChunk, P.V - k0);
        const char* rowp = base + (row * (size_t)P.V + (size_t)k0) * esz;

        float x[32];
        Loader<DT, VEC>::load(rowp, len, t, x);

        float m = -INFINITY;
        int arg = 0x7FFFFFFF;
        uint32_t bad = 0;
        if (GREEDY) {
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                bad |= (x[i] != x[i]);
                if (x[i] > m) { m = x[i]; arg = Loader<DT, VEC>::offset(i, t); }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) m = fmaxf(m, x[i]);
        }
        // block max (and first argmax)
        float wm = warp_max(m);
        if (GREEDY) {
            int a = (m == wm) ? arg : 0x7FFFFFFF;
#pragma unroll
            for (int o = 16; o; o >>= 1) a = min(a, __shfl_xor_sync(0xFFFFFFFFu, a, o));
            bad = warp_or(bad);
            if (lane == 0) { s_redf[warp] = wm; s_redi[warp] = a; s_redu[warp] = bad; }
        } else if (lane == 0) {
            s_redf[warp] = wm;
        }
        __syncthreads();
        float bm = s_redf[0];
#pragma unroll
        for (int i = 1; i < kThreads / 32; ++i) bm = fmaxf(bm, s_redf[i]);

        if (GREEDY) {
            if (t == 0) {
                int a = 0x7FFFFFFF;
                uint32_t bb = 0;
                for (int i = 0; i < kThreads / 32; ++i) {
                    if (s_redf[i] == bm) a = min(a, s_redi[i]);
                    bb |= s_redu[i];
                }
                uint32_t flags = (bb || bm == INFINITY) ? (1u << SV_ERR_NONFINITE) : 0u;
                P.partials[(size_t)r * P.nchunks + c] = Partial{bm, 0.f, a == 0x7FFFFFFF ? -1 : k0 + a, flags};
            }
        } else {
            float s = 0.f;
            if (bm != -INFINITY) {
                const float K = P.K_hi;
                const float mK = bm * K;
#pragma unroll
                for (int i = 0; i < 32; ++i) s += ex2_approx(__fmaf_rn(x[i], K, -mK));
            } else {
                // no finite maximum: only a NaN can still hide among the -inf entries
                bool nan = false;
#pragma unroll
                for (int i = 0; i < 32; ++i) nan |= x[i] != x[i];
                s = nan ? __int_as_float(0x7FC00000) : 0.f;
            }
            s = warp_sumf(s);
            __syncthreads();
            if (lane == 0) s_redf[warp] = s;
            __syncthreads();
            if (t == 0) {
                float tot = 0.f;
                for (int i = 0; i < kThreads / 32; ++i) tot += s_redf[i];
                // a NaN or +inf logit turns the sum into NaN (see the max pass above)
                const uint32_t flags = (tot != tot) ? (1u << SV_ERR_NONFINITE) : 0u;
                P.partials[(size_t)r * P.nchunks + c] = Partial{bm, tot, -1, flags};
            }
        }
        __syncthreads();
    }
}

// ------------------------------------------------------------------------------------------------
// k_decide: one warp per sequence.
// ------------------------------------------------------------------------------------------------
template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kThreads) k_decide(const Params P) {
    constexpr int kW = kThreads / 32;
    __shared__ float s_m[kW][2 * SV_MAX_GAMMA + 2];
    __shared__ double s_s[kW][2 * SV_MAX_GAMMA + 2];
    __shared__ int s_a[kW][SV_MAX_GAMMA + 1];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t b = blockIdx.x * kW + warp;
    if (b >= P.B) return;

    if (*P.batch_bad) {  // unusable offsets: every sequence fails, no token position is trusted
        if (lane == 0) {
            P.out_n[b] = -1;
            if (!GREEDY) P.tasks[b].mode = kModeNone;
        }
        return;
    }
    int32_t g = 0, o0 = 0;
    const bool bok = batch_ok(P);
    if (!(bok && seq_ok(P, b, g, o0))) {
        if (lane == 0) {
            atomicOr(P.status, 1u << SV_ERR_BAD_OFFSETS);
            P.out_n[b] = -1;
            if (!GREEDY) P.tasks[b].mode = kModeNone;
        }
        // tokens only where this sequence's slots are provably inside out_tokens
        const int32_t oB = __ldg(P.offs + P.B), a0 = __ldg(P.offs + b), a1 = __ldg(P.offs + b + 1);
        if (bok && a0 >= 0 && a0 <= a1 && a1 <= oB)
            for (int32_t j = lane; j <= a1 - a0; j += 32) P.out_tokens[a0 + b + j] = -1;
        return;
    }
    const int32_t t0 = o0 + b;
    // draft tokens
    int32_t x = 0;
    uint32_t err = 0;
    if (lane < g) {
        x = __ldg(P.tokens + o0 + lane);
        if (x < 0 || x >= P.V) err |= 1u << SV_ERR_BAD_TOKEN;
    }
    // merge chunk partials of each statistics row
    const int nrows = stat_rows<GREEDY>(g);
    const int32_t sbase = stat_base<GREEDY>(P, b);
    for (int jr = lane; jr < nrows; jr += 32) {
        const Partial* pp = P.partials + (size_t)(sbase + jr) * P.nchunks;
        float m = -INFINITY;
        int a = -1;
        uint32_t fl = 0;
        for (int c = 0; c < P.nchunks; ++c) {
            const Partial q = pp[c];
            fl |= q.flags;
            if (q.m > m) { m = q.m; a = q.arg; }
        }
        double s = 0.0;
        if (m == -INFINITY) {
            fl |= 1u << SV_ERR_EMPTY_ROW;
        } else if (!GREEDY) {
            for (int c = 0; c < P.nchunks; ++c) {
                const Partial q = pp[c];
                if (q.m != -INFINITY) s += (double)q.s * exp2(((double)q.m - (double)m) * P.K64);
            }
        }
        err |= fl;
        s_m[warp][jr] = m;
        s_s[warp][jr] = s;
        if (GREEDY) s_a[warp][jr] = a;
    }
    err = warp_or(err);
    __syncwarp();
    if (err) {
        if (lane == 0) {
            atomicOr(P.status, err);
            P.out_n[b] = -1;
            if (!GREEDY) P.tasks[b].mode = kModeNone;
        }
        for (int32_t j = lane; j <= g; j += 32) P.out_tokens[t0 + j] = -1;
        return;
    }

    if (GREEDY) {
        const int a = lane <= g ? s_a[warp][lane] : -1;
        if (lane <= g && P.dbg.row_argmax) P.dbg.row_argmax[t0 + lane] = a;
        const uint32_t mism = __ballot_sync(0xFFFFFFFFu, lane < g && x != a);
        const int n = mism ? __ffs(mism) - 1 : g;
        if (lane <= g) P.out_tokens[t0 + lane] = lane < n ? x : (lane == n ? a : -1);
        if (lane == 0) P.out_n[b] = n;
        return;
    }

    // sampling: accept test of every slot in fp64 (u * q(x) < p(x), p/q from exact logits)
    bool acc = true;
    if (lane < g) {
        const double lt = (double)logit_at<DT>(P.target, (size_t)(t0 + lane) * P.V + x);
        const double ld = (double)logit_at<DT>(P.draft, (size_t)(o0 + lane) * P.V + x);
        const double px = exp2((lt - (double)s_m[warp][lane]) * P.K64) / s_s[warp][lane];
        const double qx = exp2((ld - (double)s_m[warp][g + 1 + lane]) * P.K64) / s_s[warp][g + 1 + lane];
        const double u = philox_uniform(P.seed, P.step, (uint32_t)b, (uint32_t)lane, 0);
        acc = u * qx < px;
        if (P.dbg.p_x) P.dbg.p_x[o0 + lane] = px;
        if (P.dbg.q_x) P.dbg.q_x[o0 + lane] = qx;
    }
    if (P.dbg.row_lse) {
        const int32_t R_t = __ldg(P.offs + P.B) + P.B;
        for (int jr = lane; jr < nrows; jr += 32) {
            const double lse = (double)s_m[warp][jr] * P.invT64 + log(s_s[warp][jr]);
            const int32_t row = jr <= g ? t0 + jr : R_t + o0 + (jr - g - 1);
            P.dbg.row_lse[row] = lse;
        }
    }
    const uint32_t rej = __ballot_sync(0xFFFFFFFFu, lane < g && !acc);
    const int n = rej ? __ffs(rej) - 1 : g;
    if (lane <= g && lane != n) P.out_tokens[t0 + lane] = lane < n ? x : -1;
    if (lane == 0) {
        SeqTask tk;
        tk.mode = n < g ? kModeResidual : kModeBonus;
        tk.n = n;
        tk.prow = t0 + n;
        tk.qrow = n < g ? o0 + n : -1;
        tk.m_p = s_m[warp][n];
        tk.m_q = n < g ? s_m[warp][g + 1 + n] : 0.f;
        tk.rho = n < g ? (float)(s_s[warp][n] / s_s[warp][g + 1 + n]) : 1.f;
        tk.out_pos = t0 + n;
        tk.u = philox_uniform(P.seed, P.step, (uint32_t)b, (uint32_t)n, 1);
        P.tasks[b] = tk;
        P.out_n[b] = n;
    }
}

// ------------------------------------------------------------------------------------------------
// Sampler: weights of the draw in float-float.
// ------------------------------------------------------------------------------------------------
// Load the 16 logits k0 .. k0 + 15 of `row` (-inf past V).
template <int DT, bool VEC>
__device__ __forceinline__ void load16(const void* base, size_t row, int32_t V, int32_t k0, float (&x)[16]) {
    const size_t off = row * (size_t)V + (size_t)k0;
    if (VEC && k0 + 16 <= V) {
        if (DT == SV_BF16) {
            const uint4* p = (const uint4*)((const unsigned short*)base + off);
            const uint4 a = __ldg(p), c = __ldg(p + 1);
            const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) { x[2 * i] = bf16lo_to_f32(w[i]); x[2 * i + 1] = bf16hi_to_f32(w[i]); }
        } else {
            const float4* p = (const float4*)((const float*)base + off);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const float4 v = __ldg(p + i);
                x[4 * i] = v.x; x[4 * i + 1] = v.y; x[4 * i + 2] = v.z; x[4 * i + 3] = v.w;
            }
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) x[i] = k0 + i < V ? logit_at<DT>(base, off + i) : -INFINITY;
    }
}

// 2^((l - m) K) as float-float, the subtraction made exact first.
__device__ __forceinline__ ff weight_ff(float l, float m, float K_hi, float K_lo, const float2* tab) {
    float dh, dl;
    two_sum(l, -m, dh, dl);
    return exp2_ff(dh, dl, K_hi, K_lo, tab);
}

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) k_sample_sums(const Params P) {
    __shared__ float2 tab[64];
    fill_exp2_table(tab);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const long long items = (long long)P.B * P.nsub;
    for (long long w = (long long)blockIdx.x * (kThreads / 32) + warp; w < items;
         w += (long long)gridDim.x * (kThreads / 32)) {
        const int32_t b = (int32_t)(w / P.nsub), sc = (int32_t)(w % P.nsub);
        const SeqTask tk = P.tasks[b];
        if (tk.mode == kModeNone) continue;
        const bool resid = tk.mode == kModeResidual;
        const int32_t k0 = sc * kSub + lane * kSubPerLane;
        float lp[16], lq[16];
        load16<DT, VEC>(P.target, (size_t)tk.prow, P.V, k0, lp);
        if (resid) load16<DT, VEC>(P.draft, (size_t)tk.qrow, P.V, k0, lq);
        ffacc A, Bq, Pp, Qq;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const ff ep = weight_ff(lp[e], tk.m_p, P.K_hi, P.K_lo, tab);
            Pp.add(ep.hi, ep.lo);
            if (resid) {
                const ff eq = weight_ff(lq[e], tk.m_q, P.K_hi, P.K_lo, tab);
                Qq.add(eq.hi, eq.lo);
                if (ep.hi > tk.rho * eq.hi) {
                    A.add(ep.hi, ep.lo);
                    Bq.add(eq.hi, eq.lo);
                }
            }
        }
        const double sp = warp_sumd(Pp.value());
        double sa = sp, sb = 0.0, sq = 0.0;
        if (resid) {
            sa = warp_sumd(A.value());
            sb = warp_sumd(Bq.value());
            sq = warp_sumd(Qq.value());
        }
        if (lane == 0) P.subs[(size_t)b * P.nsub + sc] = SubSum{sa, sb, sp, sq};
    }
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

template <int DT, bool VEC>
__global__ void __launch_bounds__(kThreads) k_sample_find(const Params P) {
    __shared__ float2 tab[64];
    fill_exp2_table(tab);
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int32_t b = blockIdx.x * (kThreads / 32) + warp;
    if (b >= P.B) return;
    const SeqTask tk = P.tasks[b];
    if (tk.mode == kModeNone) return;
    const SubSum* ss = P.subs + (size_t)b * P.nsub;
    const int nsub = P.nsub;

    double sp = 0.0, sq = 0.0;
    for (int i = lane; i < nsub; i += 32) { sp += ss[i].p; sq += ss[i].q; }
    sp = warp_sumd(sp);
    sq = warp_sumd(sq);
    bool resid = tk.mode == kModeResidual;
    const double rho = resid ? sp / sq : 0.0;

    // sub-chunk weights: lane owns the contiguous range [s0, s1)
    const int per = (nsub + 31) / 32;
    const int s0 = min(nsub, lane * per), s1 = min(nsub, s0 + per);
    auto wsub = [&](int i, bool r) -> double { return r ? ss[i].a - rho * ss[i].b : ss[i].p; };
    double lsum = 0.0;
    for (int i = s0; i < s1; ++i) lsum += wsub(i, resid);
    double S = warp_sumd(lsum);
    if (resid && !(S > 0.0)) {  // residual mass 0 (only through rounding): draw from p
        resid = false;
        lsum = 0.0;
        for (int i = s0; i < s1; ++i) lsum += wsub(i, false);
        S = warp_sumd(lsum);
    }
    const double target = tk.u * S;

    // sub-chunk holding the crossing
    const double pre = warp_exscan(lsum, lane);
    int sc = -1;
    double before = 0.0;
    {
        int my_sc = -1;
        double my_before = 0.0;
        if (pre + lsum > target) {
            double c = pre;
            for (int i = s0; i < s1; ++i) {
                const double wi = wsub(i, resid);
                if (wi > 0.0 && c + wi > target) { my_sc = i; my_before = c; break; }
                c += wi;
            }
        }
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, my_sc >= 0);
        if (hit) {
            const int L = __ffs(hit) - 1;
            sc = __shfl_sync(0xFFFFFFFFu, my_sc, L);
            before = __shfl_sync(0xFFFFFFFFu, my_before, L);
        }
    }
    bool tail_rule = false;
    if (sc < 0) {  // rounding left no crossing: the last sub-chunk with positive weight
        int last = -1;
        for (int i = s0; i < s1; ++i)
            if (wsub(i, resid) > 0.0) last = i;
#pragma unroll
        for (int o = 16; o; o >>= 1) last = max(last, __shfl_xor_sync(0xFFFFFFFFu, last, o));
        sc = last;
        tail_rule = true;
    }

    int32_t token = -1;
    if (sc >= 0) {
        const int32_t k0 = sc * kSub + lane * kSubPerLane;
        float lp[16], lq[16];
        load16<DT, VEC>(P.target, (size_t)tk.prow, P.V, k0, lp);
        if (resid) load16<DT, VEC>(P.draft, (size_t)tk.qrow, P.V, k0, lq);
        double w[16];
        double tot = 0.0;
#pragma unroll
        for (int e = 0; e < 16; ++e) {
            const ff ep = weight_ff(lp[e], tk.m_p, P.K_hi, P.K_lo, tab);
            double we = (double)ep.hi + (double)ep.lo;
            if (resid) {
                const ff eq = weight_ff(lq[e], tk.m_q, P.K_hi, P.K_lo, tab);
                we = (ep.hi > tk.rho * eq.hi) ? fmax(0.0, we - rho * ((double)eq.hi + (double)eq.lo)) : 0.0;
            }
            w[e] = we;
            tot += we;
        }
        const double rem = target - before;
        const double lpre = warp_exscan(tot, lane);
        int my_k = -1;
        if (!tail_rule && lpre + tot > rem) {
            double c = lpre;
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                if (my_k < 0 && w[e] > 0.0 && c + w[e] > rem) my_k = k0 + e;
                c += w[e];
            }
        }
        const uint32_t hit = __ballot_sync(0xFFFFFFFFu, my_k >= 0);
        if (hit) {
            token = __shfl_sync(0xFFFFFFFFu, my_k, __ffs(hit) - 1);
        } else {  // no crossing inside (rounding): the last positive weight of the sub-chunk
            int last = -1;
#pragma unroll
            for (int e = 0; e < 16; ++e)
                if (w[e] > 0.0) last = k0 + e;
#pragma unroll
            for (int o = 16; o; o >>= 1) last = max(last, __shfl_xor_sync(0xFFFFFFFFu, last, o));
            token = last;
        }
    }
    if (lane == 0) {
        P.out_tokens[tk.out_pos] = token;
        if (P.dbg.seq_mass) P.dbg.seq_mass[b] = S / sp;
    }
}

// ------------------------------------------------------------------------------------------------
// Launch
// ------------------------------------------------------------------------------------------------
static int sm_count() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev >= 0 && dev < 64) {
        if (!cached[dev]) {
            int n = 0;
            cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
            cached[dev] = n > 0 ? n : 1;
        }
        return cached[dev];
    }
    return 1;
}

template <int DT, bool VEC>
static cudaError_t launch_typed(const Params& P, bool greedy, cudaStream_t st) {
    const int sms = sm_count();
    const long long max_rows = (long long)P.B * (greedy ? P.max_gamma + 1 : 2 * P.max_gamma + 1);
    const long long stat_items = max_rows * P.nchunks;
    const int g_stats = (int)std::max(1LL, std::min(stat_items, (long long)sms * 8));
    const int g_warp = (P.B + kThreads / 32 - 1) / (kThreads / 32);
    k_validate<<<1, kThreads, 0, st>>>(P);
    if (greedy) {
        k_stats<DT, VEC, true><<<g_stats, kThreads, 0, st>>>(P);
        k_decide<DT, true><<<g_warp, kThreads, 0, st>>>(P);
    } else {
        k_stats<DT, VEC, false><<<g_stats, kThreads, 0, st>>>(P);
        k_decide<DT, false><<<g_warp, kThreads, 0, st>>>(P);
        const long long sub_items = (long long)P.B * P.nsub;
        const int g_sub = (int)std::max(1LL, std::min((sub_items + 7) / 8, (long long)sms * 8));
        k_sample_sums<DT, VEC><<<g_sub, kThreads, 0, st>>>(P);
        k_sample_find<DT, VEC><<<g_warp, kThreads, 0, st>>>(P);
    }
    return cudaGetLastError();
}

cudaError_t launch_verify(const Params& P, int dtype, bool vec, bool greedy, cudaStream_t st) {
    if (P.B == 0) return cudaSuccess;
    if (dtype == SV_BF16) return vec ? launch_typed<SV_BF16, true>(P, greedy, st) : launch_typed<SV_BF16, false>(P, greedy, st);
    return vec ? launch_typed<SV_F32, true>(P, greedy, st) : launch_typed<SV_F32, false>(P, greedy, st);
}

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma) {
    auto up = [](size_t x) { return (x + 255) & ~(size_t)255; };
    const size_t nchunks = ((size_t)V + kChunk - 1) / kChunk;
    const size_t nsub = ((size_t)V + kSub - 1) / kSub;
    Layout L;
    L.partials = 0;
    L.tasks = up(L.partials + (size_t)B * (2 * (size_t)max_gamma + 1) * nchunks * sizeof(Partial));
    L.subs = up(L.tasks + (size_t)B * sizeof(SeqTask));
    L.status = up(L.subs + (size_t)B * nsub * sizeof(SubSum));
    L.batch_bad = L.status + 128;
    L.total = up(L.batch_bad + sizeof(uint32_t));
    return L;
}

}  // namespace sv
