// Vocabulary-sharded verify ("All About Transformer Inference", the model-parallel sections: the
// unembedding's output, the logits, sharded over the vocabulary across tensor-parallel ranks;
// "Accelerating Sonar through speculation", the tensor-parallel scheduling section). Each shard holds
// columns [v0, v0 + Vs) of every row. The step needs three exchanges, all between shards' small records:
//   1. per row and shard, the partial statistics of the shard's slice: raw max m_j, sum of
//      2^((l - m_j) K), the first argmax (global index) and the logit at the row's draft token when the
//      shard owns that column (ShardPartial, 16 B) -- exchanged by an all-gather;
//   2. every shard merges the gathered partials into the rows' statistics and makes the same decisions
//      (accept tests, first rejection; greedy: the whole output) and, for each sequence's draw, sums its
//      slice's weights exactly (float-float, relative to the merged row maxima) -- exchanged by an all-gather;
//   3. every shard finds the shard owning the draw's target u S from the gathered sums; that shard scans its
//      slice for the drawn column and writes the token, the others -1 -- combined by an element-wise max.
// The rule is the unsharded verify step's (velog "6-1편. Speculative Decoding", §2-1/§2-2), so the outputs
// equal the unsharded step's up to the rounding order of the sums.
#include <cfloat>
#include <cmath>

#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace sv {
namespace {

constexpr int kShThreads = 512;

template <int DT>
__device__ __forceinline__ float lg(const void* base, size_t idx) {
    if (DT == SV_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)base + idx) << 16);
    return __ldg((const float*)base + idx);
}

// CTA-wide max / sum helpers (kShThreads threads)
__device__ float cta_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int w = 0; w < kShThreads / 32; ++w) t = fmaxf(t, red[w]);
    return t;
}
__device__ float cta_sumf(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < kShThreads / 32; ++w) t += red[w];
    return t;
}
__device__ int cta_min_i(int v, int* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int t = 0x7FFFFFFF;
    for (int w = 0; w < kShThreads / 32; ++w) t = min(t, red[w]);
    return t;
}
// float-float sum over the CTA (every thread gets the total; summed in warp then warp-index order)
__device__ ff cta_sum_ff(ff v, ff* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = ff_add(v, ff{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)});
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    ff t{0.f, 0.f};
    for (int w = 0; w < kShThreads / 32; ++w) t = ff_add(t, red[w]);
    return t;
}

// The stats row r (targets first, then drafts) of sequence b, slot i; its draft token (-1 for a target row
// at slot gamma_b).
struct RowRef {
    int32_t b, slot, tok;
    bool draft;
};
__device__ RowRef row_ref(const ShardArgs& A, int32_t r) {
    RowRef R{0, 0, -1, false};
    const int32_t R_t = __ldg(A.offs + A.B) + A.B;
    R.draft = r >= R_t;
    const int32_t rr = R.draft ? r - R_t : r;
    // sequence b: offs[b] + (draft ? 0 : b) <= rr
    int32_t lo = 0, hi = A.B - 1;
    while (lo < hi) {
        const int32_t mid = (lo + hi + 1) >> 1;
        if (__ldg(A.offs + mid) + (R.draft ? 0 : mid) <= rr) lo = mid; else hi = mid - 1;
    }
    R.b = lo;
    R.slot = rr - __ldg(A.offs + lo) - (R.draft ? 0 : lo);
    const int32_t g = __ldg(A.offs + lo + 1) - __ldg(A.offs + lo), ti = __ldg(A.offs + lo) + R.slot;
    if (R.slot < g && A.tokens && ti >= 0 && ti < __ldg(A.offs + A.B)) R.tok = __ldg(A.tokens + ti);
    return R;
}

// 1. Partial statistics of every row's slice, one CTA per row.
template <int DT>
__global__ void __launch_bounds__(kShThreads) k_shard_stats(const __grid_constant__ ShardArgs A, ShardPartial* out) {
    __shared__ float redf[kShThreads / 32];
    __shared__ int redi[kShThreads / 32];
    const int32_t r = (int32_t)blockIdx.x;
    {  // every CTA checks the whole CSR structure before it reads a row (the decisions then fail the batch)
        int bad = threadIdx.x == 0 && __ldg(A.offs) != 0;
        for (int32_t b = threadIdx.x; b < A.B; b += kShThreads) {
            const int32_t o0 = __ldg(A.offs + b), g = __ldg(A.offs + b + 1) - o0;
            bad |= o0 < 0 || g < 0 || g > A.max_gamma || g != __ldg(A.gammas + b);
        }
        if (__syncthreads_or(bad)) {
            if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(A.status, 1u << SV_ERR_BAD_OFFSETS);
            return;
        }
    }
    const int32_t R_t = __ldg(A.offs + A.B) + A.B;
    const int32_t R_d = A.draft ? __ldg(A.offs + A.B) : 0;
    if (r >= R_t + R_d) return;
    const RowRef R = row_ref(A, r);
    const void* base = R.draft ? A.draft : A.target;
    const size_t row = (size_t)(R.draft ? r - R_t : r) * (size_t)A.Vs;
    float m = -INFINITY;
    int arg = 0x7FFFFFFF;
    uint32_t bad = 0;
    for (int32_t k = threadIdx.x; k < A.Vs; k += kShThreads) {
        const float l = lg<DT>(base, row + k);
        bad |= l != l || l == INFINITY;
        if (l > m) { m = l; arg = k; }
    }
    const float M = cta_max(m, redf);
    const int A0 = cta_min_i(m == M ? arg : 0x7FFFFFFF, redi);
    bad = __syncthreads_or(bad);
    float s = 0.f;
    if (!A.greedy && M != -INFINITY && !bad)
        for (int32_t k = threadIdx.x; k < A.Vs; k += kShThreads) s += exp2f((lg<DT>(base, row + k) - M) * A.K_hi);
    s = cta_sumf(s, redf);
    if (threadIdx.x == 0) {
        ShardPartial p;
        p.m = bad ? __int_as_float(0x7FC00000) : M;
        p.s = bad ? __int_as_float(0x7FC00000) : s;
        p.arg = M == -INFINITY || A0 == 0x7FFFFFFF ? -1 : A.v0 + A0;
        p.g = 0.f;
        if (R.tok >= A.v0 && R.tok < A.v0 + A.Vs) p.g = lg<DT>(base, row + (R.tok - A.v0));
        out[r] = p;
    }
}

// The merged statistics of row r from the S shards' partials (in shard order).
struct RowStat {
    float m, s;  // raw max, sum of 2^((l - m) K) (NaN: a NaN or +inf logit somewhere)
    int arg;     // first argmax over the whole row (-1: none)
};
__device__ RowStat merge_row(const ShardArgs& A, const ShardPartial* all, int32_t nrows, int32_t r) {
    RowStat R{-INFINITY, 0.f, -1};
    bool nan = false;
    for (int j = 0; j < A.S; ++j) {
        const ShardPartial p = all[(size_t)j * nrows + r];
        if (p.m != p.m) { nan = true; continue; }
        if (p.m > R.m) R.arg = p.arg;  // lower shards hold lower columns: the first max wins ties
        R.m = fmaxf(R.m, p.m);
    }
    if (nan) return RowStat{__int_as_float(0x7FC00000), __int_as_float(0x7FC00000), -1};
    if (R.m == -INFINITY || A.greedy) return R;
    for (int j = 0; j < A.S; ++j) {
        const ShardPartial p = all[(size_t)j * nrows + r];
        if (p.m != -INFINITY) R.s += p.s * exp2_fma((p.m - R.m) * A.K_hi);
    }
    return R;
}
__device__ __forceinline__ int owner_of(const ShardArgs& A, int32_t col) {
    int j = 0;
    while (j + 1 < A.S && col >= A.bounds[j + 1]) ++j;
    return j;
}

// 2a. Decisions, one warp per sequence (every shard computes the same ones). Writes n, the accepted tokens,
// -1 past the drawn slot, and the draw; greedy writes the whole output.
template <int DT>
__global__ void __launch_bounds__(256) k_shard_decide(const __grid_constant__ ShardArgs A, const ShardPartial* all,
                                                      ShardDraw* draws) {
    __shared__ float tab[2 * kExpTab];
    if (threadIdx.x < kExpTab) {
        tab[threadIdx.x] = A.exp2_tab[threadIdx.x].x;
        tab[kExpTab + threadIdx.x] = A.exp2_tab[threadIdx.x].y;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int32_t b = (int32_t)(blockIdx.x * 8 + (threadIdx.x >> 5));
    if (b >= A.B) return;
    if (*(volatile uint32_t*)A.status & (1u << SV_ERR_BAD_OFFSETS)) {  // rows not owned reliably: fail all
        if (lane == 0) {
            A.out_n[b] = -1;
            ShardDraw none{};
            none.mode = kModeNone;
            draws[b] = none;
        }
        return;
    }
    const int32_t o0 = __ldg(A.offs + b), g = __ldg(A.offs + b + 1) - o0, t0 = o0 + b;
    const int32_t R_t = __ldg(A.offs + A.B) + A.B, nrows = A.pm || A.greedy ? R_t : R_t + __ldg(A.offs + A.B);
    uint32_t err = 0;
    int32_t x = -1;
    if (lane < g) {
        x = __ldg(A.tokens + o0 + lane);
        if (x < 0 || x >= A.V) err |= 1u << SV_ERR_BAD_TOKEN;
    }
    // lane i: target row of slot i (i <= g) and draft row of slot i (i < g)
    RowStat T{-INFINITY, 0.f, -1}, D{0.f, 1.f, -1};
    if (lane <= g) T = merge_row(A, all, nrows, t0 + lane);
    if (lane < g && !A.pm && !A.greedy) D = merge_row(A, all, nrows, R_t + o0 + lane);
    if (lane <= g) {
        if (T.m != T.m || (lane < g && !A.pm && !A.greedy && D.m != D.m)) err |= 1u << SV_ERR_NONFINITE;
        else if (T.m == -INFINITY || (lane < g && !A.pm && !A.greedy && D.m == -INFINITY)) err |= 1u << SV_ERR_EMPTY_ROW;
    }
    err = __reduce_or_sync(0xFFFFFFFFu, err);
    ShardDraw dw{};
    if (err) {
        if (lane == 0) {
            atomicOr(A.status, err);
            A.out_n[b] = -1;
            dw.mode = kModeNone;
            draws[b] = dw;
        }
        for (int32_t j = lane; j <= g; j += 32) A.out_tokens[t0 + j] = -1;
        return;
    }
    if (A.greedy) {
        const uint32_t mism = __ballot_sync(0xFFFFFFFFu, lane < g && x != T.arg);
        const int n = mism ? __ffs(mism) - 1 : g;
        if (lane <= g) A.out_tokens[t0 + lane] = lane < n ? x : (lane == n ? T.arg : -1);
        if (lane == 0) {
            A.out_n[b] = n;
            dw.mode = kModeNone;
            draws[b] = dw;
        }
        return;
    }
    // p(x), q(x) from the owning shards' logits at x, over the merged normalisers
    bool acc = true;
    if (lane < g) {
        const int jo = owner_of(A, x);
        const float lt = all[(size_t)jo * nrows + t0 + lane].g;
        const float ld = A.pm ? 0.f : all[(size_t)jo * nrows + R_t + o0 + lane].g;
        const ExpConst EC{A.K_hi, A.K_lo, A.d_min};
        const ff2 e = exp2_ff2(make_float2(lt, ld), make_float2(T.m, A.pm ? 0.f : D.m), EC, tab);
        const float px = div_fma(e.hi.x + e.lo.x, T.s);
        const float qx = A.pm ? 1.f : div_fma(e.hi.y + e.lo.y, D.s);
        const float u = philox_uniform(A.seed, A.step, (uint32_t)b, (uint32_t)lane, 0);
        acc = u * qx < px;
    }
    const uint32_t rej = __ballot_sync(0xFFFFFFFFu, lane < g && !acc);
    const int n = rej ? __ffs(rej) - 1 : g;
    if (lane <= g && lane != n) A.out_tokens[t0 + lane] = lane < n ? x : -1;
    const float pm = __shfl_sync(0xFFFFFFFFu, T.m, n), ps = __shfl_sync(0xFFFFFFFFu, T.s, n);
    const float qm = __shfl_sync(0xFFFFFFFFu, D.m, n), qs = __shfl_sync(0xFFFFFFFFu, D.s, n);
    const int32_t xn = __shfl_sync(0xFFFFFFFFu, x, n < g ? n : 0);
    if (lane == 0) {
        A.out_n[b] = n;
        dw.mode = n < g ? (A.pm ? kModeResidualPM : kModeResidual) : kModeBonus;
        dw.n = n;
        dw.m_p = pm;
        dw.m_q = n < g && !A.pm ? qm : 0.f;
        dw.rho = n < g && !A.pm ? div_fma(ps, qs) : 1.f;
        dw.u = philox_uniform(A.seed, A.step, (uint32_t)b, (uint32_t)n, 1);
        dw.xcl = n < g && A.pm ? xn : -1;
        draws[b] = dw;
    }
}

// The weights of column k of a draw (relative to the merged row maxima), the residual's selection and the
// removed column of a point-mass draft: the same function for the sums and for the owner's scan.
template <int DT>
__device__ __forceinline__ void draw_weights(const ShardArgs& A, const ShardDraw& dw, size_t prow, size_t qrow, int32_t k,
                                             const ExpConst& EC, const float* tab, ff& ep, ff& eq, bool& sel) {
    const bool resid = dw.mode == kModeResidual;
    const float lp = lg<DT>(A.target, prow + k), lq = resid ? lg<DT>(A.draft, qrow + k) : 0.f;
    const ff2 e = exp2_ff2(make_float2(lp, lq), make_float2(dw.m_p, resid ? dw.m_q : 0.f), EC, tab);
    ep = ff_norm(e.hi.x, e.lo.x);
    eq = resid ? ff_norm(e.hi.y, e.lo.y) : ff{0.f, 0.f};
    sel = resid ? e.hi.x > dw.rho * e.hi.y : !(dw.mode == kModeResidualPM && A.v0 + k == dw.xcl);
}

// 2b. The draw's sums over this shard's slice, one CTA per sequence: all p weights, all q weights, and those
// of the selected columns (bonus: every column; point-mass residual: all but the draft token), float-float.
template <int DT>
__global__ void __launch_bounds__(kShThreads) k_shard_sums(const __grid_constant__ ShardArgs A, const ShardDraw* draws,
                                                           ff* sums) {
    __shared__ float tab[2 * kExpTab];
    __shared__ ff red[kShThreads / 32];
    if (threadIdx.x < kExpTab) {
        tab[threadIdx.x] = A.exp2_tab[threadIdx.x].x;
        tab[kExpTab + threadIdx.x] = A.exp2_tab[threadIdx.x].y;
    }
    __syncthreads();
    const int32_t b = (int32_t)blockIdx.x;
    const ShardDraw dw = draws[b];
    ff* out = sums + (size_t)b * 4;
    if (dw.mode == kModeNone) {
        if (threadIdx.x < 4) out[threadIdx.x] = ff{0.f, 0.f};
        return;
    }
    const int32_t o0 = __ldg(A.offs + b);
    const size_t prow = (size_t)(o0 + b + dw.n) * (size_t)A.Vs, qrow = (size_t)(o0 + dw.n) * (size_t)A.Vs;
    const ExpConst EC{A.K_hi, A.K_lo, A.d_min};
    ff P{0.f, 0.f}, Q{0.f, 0.f}, Sa{0.f, 0.f}, Sb{0.f, 0.f};
    for (int32_t k = threadIdx.x; k < A.Vs; k += kShThreads) {
        ff ep, eq;
        bool sel;
        draw_weights<DT>(A, dw, prow, qrow, k, EC, tab, ep, eq, sel);
        P = ff_add(P, ep);
        Q = ff_add(Q, eq);
        if (sel) {
            Sa = ff_add(Sa, ep);
            Sb = ff_add(Sb, eq);
        }
    }
    P = cta_sum_ff(P, red);
    Q = cta_sum_ff(Q, red);
    Sa = cta_sum_ff(Sa, red);
    Sb = cta_sum_ff(Sb, red);
    if (threadIdx.x == 0) {
        out[0] = P;
        out[1] = Q;
        out[2] = Sa;
        out[3] = Sb;
    }
}

// The draw's weight of column k given the exact normaliser ratio rho: the residual max(0, e_p - rho e_q) of
// a selected column, or the p weight (bonus, point-mass residual without its removed column, the p fallback).
__device__ __forceinline__ ff col_weight(const ShardDraw& dw, bool by_p, ff ep, ff eq, bool sel, ff rho) {
    if (by_p) return ep;
    if (!sel) return ff{0.f, 0.f};
    if (dw.mode != kModeResidual) return ep;
    const ff w = ff_sub(ep, ff_mul(rho, eq));
    return w.hi > 0.f ? w : ff{0.f, 0.f};
}

// 3. The owner of the draw's target and, on the owning shard, the drawn column: one CTA per sequence.
template <int DT>
__global__ void __launch_bounds__(kShThreads) k_shard_finish(const __grid_constant__ ShardArgs A, const ShardDraw* draws,
                                                             const ff* all_sums) {
    __shared__ float tab[2 * kExpTab];
    __shared__ ff red[kShThreads / 32];
    __shared__ int redi[kShThreads / 32];
    if (threadIdx.x < kExpTab) {
        tab[threadIdx.x] = A.exp2_tab[threadIdx.x].x;
        tab[kExpTab + threadIdx.x] = A.exp2_tab[threadIdx.x].y;
    }
    __syncthreads();
    const int32_t b = (int32_t)blockIdx.x;
    const ShardDraw dw = draws[b];
    if (dw.mode == kModeNone) return;  // greedy or failed: written by the decision
    const int32_t o0 = __ldg(A.offs + b), t0 = o0 + b;
    // every shard: the exact ratio and each shard's mass, summed in shard order
    ff sp{0.f, 0.f}, sq{0.f, 0.f};
    for (int j = 0; j < A.S; ++j) {
        sp = ff_add(sp, all_sums[((size_t)j * A.B + b) * 4]);
        sq = ff_add(sq, all_sums[((size_t)j * A.B + b) * 4 + 1]);
    }
    const bool resid = dw.mode == kModeResidual;
    const ff rho = resid ? ff_div(sp, sq) : ff{0.f, 0.f};
    auto mass = [&](int j, bool by_p) {
        const ff* s = all_sums + ((size_t)j * A.B + b) * 4;
        if (by_p) return s[0];
        ff w = s[2];
        if (resid) w = ff_sub(w, ff_mul(rho, s[3]));
        return w.hi > 0.f ? w : ff{0.f, 0.f};
    };
    ff S{0.f, 0.f};
    for (int j = 0; j < A.S; ++j) S = ff_add(S, mass(j, false));
    const bool by_p = !(S.hi > 0.f);  // a residual of mass 0: draw from p
    if (by_p) {
        S = ff{0.f, 0.f};
        for (int j = 0; j < A.S; ++j) S = ff_add(S, mass(j, true));
    }
    const ff target = ff_mul(ff{dw.u, 0.f}, S);
    int jo = -1, jlast = -1;
    ff before{0.f, 0.f}, c{0.f, 0.f}, before_last{0.f, 0.f};
    for (int j = 0; j < A.S; ++j) {
        const ff w = mass(j, by_p);
        if (!(w.hi > 0.f)) continue;
        const ff c2 = ff_add(c, w);
        if (jo < 0 && ff_gt(c2, target)) {
            jo = j;
            before = c;
        }
        jlast = j;
        before_last = c;
        c = c2;
    }
    const bool tail_rule = jo < 0;  // rounding lost the crossing: the last positive column overall
    if (tail_rule) {
        jo = jlast;
        before = before_last;
    }
    if (jo != A.shard) {
        if (threadIdx.x == 0) A.out_tokens[t0 + dw.n] = -1;  // another shard's column
        return;
    }
    // the owning shard: thread t scans the columns [t C, t C + C) of its slice
    const ff rem = ff_sub(target, before);
    const int32_t C = (A.Vs + kShThreads - 1) / kShThreads, k0 = threadIdx.x * C, k1 = min(A.Vs, k0 + C);
    const size_t prow = (size_t)(o0 + b + dw.n) * (size_t)A.Vs, qrow = (size_t)(o0 + dw.n) * (size_t)A.Vs;
    const ExpConst EC{A.K_hi, A.K_lo, A.d_min};
    ff tot{0.f, 0.f};
    int lastpos = -1;
    for (int32_t k = k0; k < k1; ++k) {
        ff ep, eq;
        bool sel;
        draw_weights<DT>(A, dw, prow, qrow, k, EC, tab, ep, eq, sel);
        const ff w = col_weight(dw, by_p, ep, eq, sel, rho);
        if (w.hi > 0.f) {
            tot = ff_add(tot, w);
            lastpos = k;
        }
    }
    // exclusive prefix of the threads' totals (warp scan, then the warps' totals in order)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    ff incl = tot;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff y{__shfl_up_sync(0xFFFFFFFFu, incl.hi, o), __shfl_up_sync(0xFFFFFFFFu, incl.lo, o)};
        if (lane >= o) incl = ff_add(y, incl);
    }
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    ff wbefore{0.f, 0.f};
    for (int w = 0; w < warp; ++w) wbefore = ff_add(wbefore, red[w]);
    const ff ex_lane{__shfl_up_sync(0xFFFFFFFFu, incl.hi, 1), __shfl_up_sync(0xFFFFFFFFu, incl.lo, 1)};
    const ff excl = ff_add(wbefore, lane ? ex_lane : ff{0.f, 0.f});
    const ff inc = ff_add(excl, tot);
    // the first thread whose inclusive prefix exceeds rem holds the crossing (lowest thread index)
    const bool holds = !tail_rule && tot.hi > 0.f && ff_gt(inc, rem) && !ff_gt(excl, rem);
    const int first = cta_min_i(holds ? (int)threadIdx.x : 0x7FFFFFFF, redi);
    const int lastp = -cta_min_i(-lastpos, redi);  // the slice's last column of positive weight
    if (first != 0x7FFFFFFF) {
        if ((int)threadIdx.x == first) {
            ff cc = excl;
            int32_t col = -1, lastc = -1;
            for (int32_t k = k0; k < k1 && col < 0; ++k) {
                ff ep, eq;
                bool sel;
                draw_weights<DT>(A, dw, prow, qrow, k, EC, tab, ep, eq, sel);
                const ff w = col_weight(dw, by_p, ep, eq, sel, rho);
                if (!(w.hi > 0.f)) continue;
                cc = ff_add(cc, w);
                lastc = k;
                if (ff_gt(cc, rem)) col = k;
            }
            if (col < 0) col = lastc;  // the thread's sum crossed, its running sum fell short by rounding
            A.out_tokens[t0 + dw.n] = A.v0 + col;
        }
    } else if (threadIdx.x == 0) {
        A.out_tokens[t0 + dw.n] = lastp >= 0 ? A.v0 + lastp : -1;
    }
}

}  // namespace

cudaError_t launch_shard(int stage, const ShardArgs& A, void* a, void* b, void* c) {
    cudaStream_t st = A.stream;
    const int32_t nrows = A.nrows;
    switch (stage) {
        case 0:
            if (nrows > 0) {
                if (A.dtype == SV_BF16) k_shard_stats<SV_BF16><<<nrows, kShThreads, 0, st>>>(A, (ShardPartial*)a);
                else k_shard_stats<SV_F32><<<nrows, kShThreads, 0, st>>>(A, (ShardPartial*)a);
            }
            break;
        case 1:
            if (A.dtype == SV_BF16) k_shard_decide<SV_BF16><<<(A.B + 7) / 8, 256, 0, st>>>(A, (const ShardPartial*)a, (ShardDraw*)b);
            else k_shard_decide<SV_F32><<<(A.B + 7) / 8, 256, 0, st>>>(A, (const ShardPartial*)a, (ShardDraw*)b);
            break;
        case 2:
            if (A.dtype == SV_BF16) k_shard_sums<SV_BF16><<<A.B, kShThreads, 0, st>>>(A, (const ShardDraw*)a, (ff*)b);
            else k_shard_sums<SV_F32><<<A.B, kShThreads, 0, st>>>(A, (const ShardDraw*)a, (ff*)b);
            break;
        default:
            if (A.dtype == SV_BF16) k_shard_finish<SV_BF16><<<A.B, kShThreads, 0, st>>>(A, (const ShardDraw*)a, (const ff*)b);
            else k_shard_finish<SV_F32><<<A.B, kShThreads, 0, st>>>(A, (const ShardDraw*)a, (const ff*)b);
    }
    return cudaGetLastError();
}

}  // namespace sv

// ------------------------------------------------------------------------------------------------
// C ABI (declared in include/specverify.h)
// ------------------------------------------------------------------------------------------------
namespace {
int shard_args(sv::ShardArgs& A, sv_dtype dtype, int32_t B, int32_t V, int32_t max_gamma, float temperature,
               void* stream) {
    using namespace sv;
    if (B < 0 || V < 1 || max_gamma < 0 || max_gamma > SV_MAX_GAMMA) return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    A = ShardArgs{};
    A.dtype = dtype;
    A.B = B;
    A.V = V;
    A.max_gamma = max_gamma;
    A.greedy = temperature == 0.f;
    const double K64 = A.greedy ? 0.0 : 1.4426950408889634074 / (double)temperature;
    A.K_hi = (float)K64;
    if (!A.greedy && !std::isfinite(A.K_hi)) return SV_ERR_INVALID_ARG;
    A.K_lo = (float)(K64 - (double)A.K_hi);
    A.d_min = A.greedy ? 0.f : (float)(-126.5 / (double)A.K_hi);
    for (int j = 0; j < 128; ++j) {
        const double v = std::exp2((double)j / 128.0);
        const float hi = (float)v;
        A.exp2_tab[j] = make_float2(hi, (float)(v - (double)hi));
    }
    A.stream = (cudaStream_t)stream;
    return SV_OK;
}
int shard_bounds(sv::ShardArgs& A, int32_t S, const int32_t* bounds, int32_t V) {
    if (S < 1 || S > sv::kMaxShards || !bounds || bounds[0] != 0 || bounds[S] != V) return SV_ERR_INVALID_ARG;
    for (int j = 0; j < S; ++j) {
        if (bounds[j + 1] <= bounds[j]) return SV_ERR_INVALID_ARG;
        A.bounds[j] = bounds[j];
    }
    A.bounds[S] = V;
    A.S = S;
    return SV_OK;
}
bool aligned4(const void* p) { return p && (uintptr_t)p % 4 == 0; }
}  // namespace

extern "C" {

int spec_shard_stats(const void* shard_target, const void* shard_draft, sv_dtype dtype, const int32_t* draft_tokens,
                     const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t v0, int32_t Vs,
                     int32_t max_gamma, float temperature, void* partials, uint32_t* device_status, void* cuda_stream) {
    sv::ShardArgs A;
    int rc = shard_args(A, dtype, B, V, max_gamma, temperature, cuda_stream);
    if (rc != SV_OK) return rc;
    if (v0 < 0 || Vs < 1 || (int64_t)v0 + Vs > V) return SV_ERR_INVALID_ARG;
    if (!shard_target || !aligned4(seq_offsets) || !aligned4(gammas) || !partials || (uintptr_t)partials % 16 ||
        !aligned4(device_status) || (max_gamma > 0 && !aligned4(draft_tokens)))
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    A.target = shard_target;
    A.draft = A.greedy ? nullptr : shard_draft;
    A.tokens = draft_tokens;
    A.offs = seq_offsets;
    A.gammas = gammas;
    A.v0 = v0;
    A.Vs = Vs;
    A.pm = !A.greedy && !shard_draft;
    A.status = device_status;
    const int64_t nrows = (int64_t)B * (max_gamma + 1) + (A.draft ? (int64_t)B * max_gamma : 0);
    if (nrows >= (1ll << 31)) return SV_ERR_INVALID_ARG;
    A.nrows = (int32_t)nrows;
    return sv::launch_shard(0, A, partials, nullptr, nullptr) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int spec_shard_decide(const void* all_partials, int32_t S, const int32_t* shard_bounds_host, const int32_t* draft_tokens,
                      const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t max_gamma,
                      float temperature, int32_t point_mass, uint64_t seed, uint64_t step, int32_t* out_tokens,
                      int32_t* out_num_accepted, void* draws, uint32_t* device_status, void* cuda_stream) {
    sv::ShardArgs A;
    int rc = shard_args(A, SV_BF16, B, V, max_gamma, temperature, cuda_stream);
    if (rc != SV_OK) return rc;
    if ((rc = shard_bounds(A, S, shard_bounds_host, V)) != SV_OK) return rc;
    if (!all_partials || (uintptr_t)all_partials % 16 || !aligned4(seq_offsets) || !aligned4(gammas) ||
        !aligned4(out_tokens) || !aligned4(out_num_accepted) || !draws || (uintptr_t)draws % 16 ||
        !aligned4(device_status) || (max_gamma > 0 && !aligned4(draft_tokens)))
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    A.tokens = draft_tokens;
    A.offs = seq_offsets;
    A.gammas = gammas;
    A.pm = !A.greedy && point_mass;
    A.seed = seed;
    A.step = step;
    A.out_tokens = out_tokens;
    A.out_n = out_num_accepted;
    A.status = device_status;
    return sv::launch_shard(1, A, const_cast<void*>(all_partials), draws, nullptr) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int spec_shard_sums(const void* shard_target, const void* shard_draft, sv_dtype dtype, int32_t v0, int32_t Vs,
                    const void* draws, const int32_t* seq_offsets, int32_t B, int32_t V, float temperature, void* sums,
                    void* cuda_stream) {
    sv::ShardArgs A;
    int rc = shard_args(A, dtype, B, V, 0, temperature, cuda_stream);
    if (rc != SV_OK) return rc;
    if (v0 < 0 || Vs < 1 || (int64_t)v0 + Vs > V || !shard_target || !draws || (uintptr_t)draws % 16 ||
        !aligned4(seq_offsets) || !sums || (uintptr_t)sums % 16)
        return SV_ERR_INVALID_ARG;
    if (B == 0 || A.greedy) return SV_OK;
    A.target = shard_target;
    A.draft = shard_draft;
    A.offs = seq_offsets;
    A.v0 = v0;
    A.Vs = Vs;
    return sv::launch_shard(2, A, const_cast<void*>(draws), sums, nullptr) == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}

int spec_shard_finish(int32_t shard, int32_t S, const int32_t* shard_bounds_host, const void* shard_target,
                      const void* shard_draft, sv_dtype dtype, const void* draws, const void* all_sums,
                      const int32_t* seq_offsets, int32_t B, int32_t V, float temperature, int32_t* out_tokens,
                      void* cuda_stream) {
    sv::ShardArgs A;
    int rc = shard_args(A, dtype, B, V, 0, temperature, cuda_stream);
    if (rc != SV_OK) return rc;
    if ((rc = shard_bounds(A, S, shard_bounds_host, V)) != SV_OK) return rc;
    if (shard < 0 || shard >= S || !shard_target || !draws || (uintptr_t)draws % 16 || !all_sums ||
        (uintptr_t)all_sums % 16 || !aligned4(seq_offsets) || !aligned4(out_tokens))
        return SV_ERR_INVALID_ARG;
    if (B == 0 || A.greedy) return SV_OK;
    A.shard = shard;
    A.v0 = A.bounds[shard];
    A.Vs = A.bounds[shard + 1] - A.bounds[shard];
    A.target = shard_target;
    A.draft = shard_draft;
    A.offs = seq_offsets;
    A.out_tokens = out_tokens;
    return sv::launch_shard(3, A, const_cast<void*>(draws), const_cast<void*>(all_sums), nullptr) == cudaSuccess
               ? SV_OK : SV_ERR_CUDA;
}

}  // extern "C"

static_assert(sizeof(sv::ShardPartial) == sizeof(sv_shard_partial), "the C ABI's partial record");
static_assert(sizeof(sv::ShardDraw) == sizeof(sv_shard_draw), "the C ABI's draw record");
