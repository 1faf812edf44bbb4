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
#include <algorithm>
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

// NaN-propagating maxima (a NaN operand gives NaN)
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}
__device__ __forceinline__ __nv_bfloat162 bits_bf162(uint32_t w) {
    __nv_bfloat162 r;
    memcpy(&r, &w, sizeof r);
    return r;
}

// CTA-wide max / sum helpers over NT threads (every thread gets the result)
template <int NT>
__device__ float cta_max(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = -INFINITY;
    for (int w = 0; w < NT / 32; ++w) t = fmaxf(t, red[w]);
    return t;
}
template <int NT>
__device__ float cta_sumf(float v, float* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xFFFFFFFFu, v, o);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float t = 0.f;
    for (int w = 0; w < NT / 32; ++w) t += red[w];
    return t;
}
template <int NT>
__device__ int cta_min_i(int v, int* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int t = 0x7FFFFFFF;
    for (int w = 0; w < NT / 32; ++w) t = min(t, red[w]);
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

// 1. Partial statistics of every row's slice, one CTA of kShStatThreads per row (all rows of a headline
// batch resident in one wave). Each thread keeps its running maximum, its first argmax and its sum of
// 2^((l - m) K) relative to that maximum, taking its columns in batches (rescaled when a batch raises it).
constexpr int kShStatThreads = 256;
template <int DT>
__global__ void __launch_bounds__(kShStatThreads, 5) k_shard_stats(const __grid_constant__ ShardArgs A, ShardPartial* out) {
    __shared__ float redf[kShStatThreads / 32];
    __shared__ int redi[kShStatThreads / 32];
    const int32_t r = (int32_t)blockIdx.x;
    {  // every CTA checks the whole CSR structure before it reads a row (the decisions then fail the batch)
        int bad = threadIdx.x == 0 && __ldg(A.offs) != 0;
        for (int32_t b = threadIdx.x; b < A.B; b += kShStatThreads) {
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
    float m = -INFINITY, s = 0.f;
    int arg = 0x7FFFFFFF;
    bool bad = false;
    const float K = A.K_hi;
    // n values x of columns col(i), increasing with i: the batch's maximum (fmax ignores NaN), the first
    // column attaining it only when it raises the running maximum, and NaN / +inf flagged by one compare
    auto take = [&](const float* x, int n, auto col) {
        float bm = -INFINITY;
        for (int i = 0; i < n; ++i) {
            bad |= !(x[i] <= FLT_MAX);
            bm = fmaxf(bm, x[i]);
        }
        if (bm > m) {
            int bi = 0;
            for (int i = n - 1; i >= 0; --i)
                if (x[i] == bm) bi = i;
            if (!A.greedy && m != -INFINITY) s *= ex2_approx((m - bm) * K);
            m = bm;
            arg = col(bi);
        }
        if (!A.greedy && m != -INFINITY) {
            const float nmK = -m * K;
            float s0 = 0.f, s1 = 0.f;
            for (int i = 0; i + 1 < n; i += 2) {
                s0 += ex2_approx(__fmaf_rn(x[i], K, nmK));
                s1 += ex2_approx(__fmaf_rn(x[i + 1], K, nmK));
            }
            if (n & 1) s0 += ex2_approx(__fmaf_rn(x[n - 1], K, nmK));
            s += s0 + s1;
        }
    };
    constexpr int PK = DT == SV_BF16 ? 8 : 4;  // values per 16-byte pack
    constexpr int NB = 4;                      // packs per batch: p, p + NT, p + 2 NT, p + 3 NT (coalesced)
    constexpr int NW = 4 * NB;                 // 32-bit words per batch
    const char* rp = (const char*)base + row * (DT == SV_BF16 ? 2 : 4);
    const bool vec = (uintptr_t)rp % 16 == 0 && A.Vs % PK == 0;
    if (vec) {
        // per batch: a NaN-propagating maximum over the raw words (bf16x2: two values an instruction; a NaN
        // or +inf anywhere shows in it), the first column attaining it only when it raises the running
        // maximum, then the sum with packed FMA / ADD and one MUFU ex2 per value
        const int32_t np = A.Vs / PK;
        const uint32_t ninf = DT == SV_BF16 ? 0xFF80FF80u : 0xFF800000u;  // -inf fills packs past the row
        const float2 K2 = f2(K);
        for (int32_t p = threadIdx.x; p < np; p += NB * kShStatThreads) {
            uint32_t w[NW];
#pragma unroll
            for (int u = 0; u < NB; ++u) {
                const uint4 v = p + u * kShStatThreads < np ? __ldg((const uint4*)rp + p + u * kShStatThreads)
                                                            : make_uint4(ninf, ninf, ninf, ninf);
                w[4 * u] = v.x; w[4 * u + 1] = v.y; w[4 * u + 2] = v.z; w[4 * u + 3] = v.w;
            }
            float bm;
            if (DT == SV_BF16) {
                __nv_bfloat162 mx = bits_bf162(w[0]);
#pragma unroll
                for (int i = 1; i < NW; ++i) mx = __hmax2_nan(mx, bits_bf162(w[i]));
                bm = fmax_nan(__low2float(mx), __high2float(mx));
            } else {
                bm = __uint_as_float(w[0]);
#pragma unroll
                for (int i = 1; i < NW; ++i) bm = fmax_nan(bm, __uint_as_float(w[i]));
            }
            bad |= !(bm <= FLT_MAX);  // NaN or +inf
            auto val = [&](int i) {
                return DT == SV_BF16 ? (i & 1 ? bf16hi_to_f32(w[i >> 1]) : bf16lo_to_f32(w[i >> 1]))
                                     : __uint_as_float(w[i]);
            };
            if (bm > m) {
                int bi = 0;
#pragma unroll
                for (int i = NB * PK - 1; i >= 0; --i)
                    if (val(i) == bm) bi = i;
                if (!A.greedy && m != -INFINITY) s *= ex2_approx((m - bm) * K);
                m = bm;
                arg = (p + (bi / PK) * kShStatThreads) * PK + bi % PK;
            }
            if (!A.greedy && m != -INFINITY) {
                const float2 nmK2 = f2(-m * K);
                float2 acc = f2(0.f);
#pragma unroll
                for (int i = 0; i < NB * PK; i += 2) {
                    const float2 t = fma2(make_float2(val(i), val(i + 1)), K2, nmK2);
                    acc = add2(acc, make_float2(ex2_approx(t.x), ex2_approx(t.y)));
                }
                s += acc.x + acc.y;
            }
        }
    } else {
        for (int32_t k = threadIdx.x; k < A.Vs; k += kShStatThreads) {
            const float x = lg<DT>(base, row + k);
            take(&x, 1, [&](int) { return k; });
        }
    }
    const float M = cta_max<kShStatThreads>(m, redf);
    const int A0 = cta_min_i<kShStatThreads>(m == M ? arg : 0x7FFFFFFF, redi);
    bad = __syncthreads_or(bad);
    s = cta_sumf<kShStatThreads>(!A.greedy && m != -INFINITY && M != -INFINITY ? s * ex2_approx((m - M) * K) : 0.f,
                                 redf);
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

// 2b. The draw's sums over this shard's slice, per 8192-column chunk: one CTA of kShSumThreads per (chunk,
// sequence), all p weights, all q weights, and those of the selected columns (bonus: every column;
// point-mass residual: all but the draft token). Thread t takes the column pairs t, t + 256, ... of the
// chunk (16 pairs): weights <= 1 (relative to the merged maxima) split on the 2^-20 grid, summed exactly
// (see grid_hi), then float-float across the CTA. Chunks past the slice hold zeros. bf16 rows on 16-byte
// boundaries are first copied into shared memory (cp.async), so that every load of the chunk is in flight
// at once; the rest read global memory directly.
constexpr int kShSumThreads = 256;
constexpr int kShRecSmem = 256;  // gathered sums records a finishing CTA stages in shared memory (8 KB)
static_assert(kShChunk == 2 * 16 * kShSumThreads, "16 column pairs per thread and chunk");

__device__ __forceinline__ void cp_async_wait_all() {
    cp_async_commit();
    cp_async_wait<0>();
}

// The accumulation over the thread's column pairs; LOAD(k) gives the logits of columns k, k + 1 of the p
// and q rows (q: -inf when unused).
template <bool TWOSUM, typename Load>
__device__ __forceinline__ void sums_pairs(const ShardArgs& A, const ShardDraw& dw, int32_t c0, int32_t c1,
                                           const float* tab, Load load, ff (&v)[4]) {
    const ExpConst EC{A.K_hi, A.K_lo, A.d_min};
    const bool resid = dw.mode == kModeResidual;
    float2 Ph = f2(0.f), Pl = f2(0.f), Qh = f2(0.f), Ql = f2(0.f), Ah = f2(0.f), Al = f2(0.f), Bh = f2(0.f), Bl = f2(0.f);
    constexpr int NP = kShChunk / (2 * kShSumThreads);
#pragma unroll 4
    for (int i = 0; i < NP; ++i) {
        const int32_t k = c0 + 2 * (int32_t)threadIdx.x + i * 2 * kShSumThreads;
        if (k >= c1) break;
        float2 lp, lq;
        load(k, lp, lq);
        const ff2 ep = exp2_ff2<TWOSUM>(lp, f2(dw.m_p), EC, tab);
        const ff2 eq = resid ? exp2_ff2<TWOSUM>(lq, f2(dw.m_q), EC, tab) : ff2{f2(0.f), f2(0.f)};
        float2 mk;
        if (resid) mk = make_float2(gt_mask(ep.hi.x, dw.rho * eq.hi.x), gt_mask(ep.hi.y, dw.rho * eq.hi.y));
        else mk = make_float2(A.v0 + k == dw.xcl ? 0.f : 1.f, A.v0 + k + 1 == dw.xcl ? 0.f : 1.f);
        const float2 hp = grid_hi(ep.hi), lpw = add2(sub2(ep.hi, hp), ep.lo);
        const float2 hq = grid_hi(eq.hi), lqw = add2(sub2(eq.hi, hq), eq.lo);
        Ph = add2(Ph, hp); Pl = add2(Pl, lpw); Qh = add2(Qh, hq); Ql = add2(Ql, lqw);
        Ah = fma2(mk, hp, Ah); Al = fma2(mk, lpw, Al); Bh = fma2(mk, hq, Bh); Bl = fma2(mk, lqw, Bl);
    }
    v[0] = ff_add(ff{Ph.x, Pl.x}, ff{Ph.y, Pl.y});
    v[1] = ff_add(ff{Qh.x, Ql.x}, ff{Qh.y, Ql.y});
    v[2] = ff_add(ff{Ah.x, Al.x}, ff{Ah.y, Al.y});
    v[3] = ff_add(ff{Bh.x, Bl.x}, ff{Bh.y, Bl.y});
}

template <int DT>
__global__ void __launch_bounds__(kShSumThreads, 3) k_shard_sums(const __grid_constant__ ShardArgs A,
                                                                 const ShardDraw* draws, ff* sums) {
    __shared__ float tab[2 * kExpTab];
    __shared__ ff red[4][kShSumThreads / 32];
    __shared__ __align__(16) uint32_t stage[2][kShChunk / 2];  // the chunk's p and q rows as bf16 pairs
    const int32_t b = (int32_t)(blockIdx.x / (uint32_t)A.nc), c = (int32_t)(blockIdx.x % (uint32_t)A.nc);
    const ShardDraw dw = draws[b];
    ff* out = sums + ((size_t)b * A.nc + c) * 4;
    const int32_t c0 = c * kShChunk, c1 = min(A.Vs, c0 + kShChunk);
    if (dw.mode == kModeNone || c0 >= c1) {
        if (threadIdx.x < 4) out[threadIdx.x] = ff{0.f, 0.f};
        return;
    }
    const int32_t o0 = __ldg(A.offs + b);
    const size_t prow = (size_t)(o0 + b + dw.n) * (size_t)A.Vs, qrow = (size_t)(o0 + dw.n) * (size_t)A.Vs;
    const bool resid = dw.mode == kModeResidual;
    const bool staged = DT == SV_BF16 && A.Vs % 8 == 0 && (uintptr_t)A.target % 16 == 0 &&
                        (!resid || (uintptr_t)A.draft % 16 == 0);
    if (staged) {  // 16-byte packs of both rows (the chunk's width is a multiple of 8 columns)
        const int32_t npk = (c1 - c0) / 8;
        const char* gp = (const char*)A.target + (prow + c0) * 2;
        const char* gq = (const char*)A.draft + (qrow + c0) * 2;
        for (int32_t i = threadIdx.x; i < npk; i += kShSumThreads) {
            cp_async16(&stage[0][4 * i], gp + 16 * (size_t)i);
            if (resid) cp_async16(&stage[1][4 * i], gq + 16 * (size_t)i);
        }
    }
    if (threadIdx.x < kExpTab) {
        tab[threadIdx.x] = A.exp2_tab[threadIdx.x].x;
        tab[kExpTab + threadIdx.x] = A.exp2_tab[threadIdx.x].y;
    }
    if (staged) cp_async_wait_all();
    __syncthreads();
    ff v[4];
    auto run = [&](auto load) {
        // bf16 rows whose maxima are not near zero need no rounding correction of l - m (see exp2_ff2)
        if (DT == SV_BF16 && fabsf(dw.m_p) >= kNeedTwoSum && (!resid || fabsf(dw.m_q) >= kNeedTwoSum))
            sums_pairs<false>(A, dw, c0, c1, tab, load, v);
        else
            sums_pairs<true>(A, dw, c0, c1, tab, load, v);
    };
    if (staged) {
        run([&](int32_t k, float2& lp, float2& lq) {
            const uint32_t wp = stage[0][(k - c0) >> 1];
            lp = make_float2(bf16lo_to_f32(wp), bf16hi_to_f32(wp));
            if (resid) {
                const uint32_t wq = stage[1][(k - c0) >> 1];
                lq = make_float2(bf16lo_to_f32(wq), bf16hi_to_f32(wq));
            } else {
                lq = f2(-INFINITY);
            }
        });
    } else {
        run([&](int32_t k, float2& lp, float2& lq) {
            const bool two = k + 1 < c1;
            lp = make_float2(lg<DT>(A.target, prow + k), two ? lg<DT>(A.target, prow + k + 1) : -INFINITY);
            lq = resid ? make_float2(lg<DT>(A.draft, qrow + k), two ? lg<DT>(A.draft, qrow + k + 1) : -INFINITY)
                       : f2(-INFINITY);
        });
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int o = 16; o; o >>= 1)
            v[i] = ff_add(v[i], ff{__shfl_xor_sync(0xFFFFFFFFu, v[i].hi, o), __shfl_xor_sync(0xFFFFFFFFu, v[i].lo, o)});
        if ((threadIdx.x & 31) == 0) red[i][threadIdx.x >> 5] = v[i];
    }
    __syncthreads();
    if (threadIdx.x < 4) {
        ff t{0.f, 0.f};
        for (int w = 0; w < kShSumThreads / 32; ++w) t = ff_add(t, red[threadIdx.x][w]);  // in warp order
        out[threadIdx.x] = t;
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

// Warp-wide float-float helpers (all 32 lanes take part).
__device__ __forceinline__ ff shfl_ff(ff v, int src) {
    return ff{__shfl_sync(0xFFFFFFFFu, v.hi, src), __shfl_sync(0xFFFFFFFFu, v.lo, src)};
}
// the sum over the warp, the same on every lane (each butterfly stage adds the same pair on both lanes)
__device__ __forceinline__ ff warp_sum_ff(ff v) {
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = ff_add(v, ff{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)});
    return v;
}
// inclusive prefix over lanes 0..lane
__device__ __forceinline__ ff warp_scan_ff(ff v, int lane) {
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff y{__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
        if (lane >= o) v = ff_add(y, v);
    }
    return v;
}

// 3. The (shard, chunk) that holds the draw's target and, on the owning shard, the drawn column: one CTA per
// sequence. Warp 0 of every shard finds the owner from the gathered chunk sums (records in shard, then chunk
// order: ratio, masses, total, prefix; the same arithmetic on every shard). The owner scans that chunk:
// thread t takes 16 contiguous columns, exact sums of their selected weights (A - rho B for a residual), a
// CTA-wide prefix, then the crossing thread's warp weighs its 16 columns one a lane and scans them.
template <int DT>
__global__ void __launch_bounds__(kShThreads) k_shard_finish(const __grid_constant__ ShardArgs A, const ShardDraw* draws,
                                                             const ff* all_sums) {
    __shared__ float tab[2 * kExpTab];
    __shared__ ff red[kShThreads / 32];
    __shared__ int redi[kShThreads / 32];
    __shared__ ff s_rec[kShRecSmem][4];
    __shared__ ff s_rho, s_rem;
    __shared__ int s_owner, s_byp, s_tail, s_col;
    if (threadIdx.x < kExpTab) {
        tab[threadIdx.x] = A.exp2_tab[threadIdx.x].x;
        tab[kExpTab + threadIdx.x] = A.exp2_tab[threadIdx.x].y;
    }
    const int32_t b = (int32_t)blockIdx.x;
    const ShardDraw dw = draws[b];
    if (dw.mode == kModeNone) return;  // greedy or failed: written by the decision
    const int32_t o0 = __ldg(A.offs + b), t0 = o0 + b;
    const bool resid = dw.mode == kModeResidual;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // the sequence's gathered records, staged in shared memory when they fit
    const int32_t nrec = A.S * A.nc;
    const bool staged = nrec <= kShRecSmem;
    if (staged)
        for (int32_t i = threadIdx.x; i < nrec * 4; i += kShThreads) {
            const int32_t j = i / (A.nc * 4), r = i % (A.nc * 4);
            s_rec[i / 4][i % 4] = all_sums[((size_t)j * A.B + b) * A.nc * 4 + r];
        }
    if (threadIdx.x == 0) s_col = -1;
    __syncthreads();
    if (warp == 0) {
        auto rec = [&](int32_t r) {
            return staged ? &s_rec[r][0] : all_sums + (((size_t)(r / A.nc) * A.B + b) * A.nc + r % A.nc) * 4;
        };
        ff sp{0.f, 0.f}, sq{0.f, 0.f};
        for (int32_t r = lane; r < nrec; r += 32) {
            sp = ff_add(sp, rec(r)[0]);
            sq = ff_add(sq, rec(r)[1]);
        }
        sp = warp_sum_ff(sp);
        sq = warp_sum_ff(sq);
        const ff rho = resid ? ff_div(sp, sq) : ff{0.f, 0.f};
        auto mass = [&](int32_t r, bool by_p) {
            if (r >= nrec) return ff{0.f, 0.f};
            const ff* x = rec(r);
            if (by_p) return x[0];
            ff w = x[2];
            if (resid) w = ff_sub(w, ff_mul(rho, x[3]));
            return w.hi > 0.f ? w : ff{0.f, 0.f};
        };
        ff S{0.f, 0.f};
        for (int32_t r = lane; r < nrec; r += 32) S = ff_add(S, mass(r, false));
        S = warp_sum_ff(S);
        const bool by_p = !(S.hi > 0.f);  // a residual of mass 0: draw from p
        if (by_p) {
            S = ff{0.f, 0.f};
            for (int32_t r = lane; r < nrec; r += 32) S = ff_add(S, mass(r, true));
            S = warp_sum_ff(S);
        }
        const ff target = ff_mul(ff{dw.u, 0.f}, S);
        // the first record of positive mass whose inclusive prefix exceeds the target; else (rounding) the
        // last record of positive mass
        int32_t owner = -1, lastr = -1;
        ff before{0.f, 0.f}, before_last{0.f, 0.f}, carry{0.f, 0.f};
        for (int32_t g = 0; g < nrec; g += 32) {
            const ff w = mass(g + lane, by_p);
            const ff inc = ff_add(carry, warp_scan_ff(w, lane));
            const ff up = shfl_ff(inc, lane ? lane - 1 : 0);
            const ff exc = lane ? up : carry;
            const bool pos = w.hi > 0.f;
            const uint32_t cross = __ballot_sync(0xFFFFFFFFu, pos && ff_gt(inc, target));
            if (cross) {
                const int f = __ffs(cross) - 1;
                owner = g + f;
                before = shfl_ff(exc, f);
                break;
            }
            const uint32_t pb = __ballot_sync(0xFFFFFFFFu, pos);
            if (pb) {
                const int l = 31 - __clz(pb);
                lastr = g + l;
                before_last = shfl_ff(exc, l);
            }
            carry = shfl_ff(inc, 31);
        }
        if (lane == 0) {
            s_tail = owner < 0;
            if (owner < 0) {
                owner = lastr;
                before = before_last;
            }
            s_owner = owner;
            s_byp = by_p;
            s_rho = rho;
            s_rem = ff_sub(target, before);
        }
    }
    __syncthreads();
    const int32_t owner = s_owner;
    const bool by_p = s_byp, tail_rule = s_tail;
    if (owner < 0 || owner / A.nc != A.shard) {
        if (threadIdx.x == 0) A.out_tokens[t0 + dw.n] = -1;  // another shard's column
        return;
    }
    const ff rho = s_rho, rem = s_rem;
    const int32_t kc0 = (owner % A.nc) * kShChunk, kc1 = min(A.Vs, kc0 + kShChunk);
    constexpr int C = kShChunk / kShThreads;  // 16 columns per thread
    const int32_t k0 = kc0 + (int32_t)threadIdx.x * C, k1 = min(kc1, k0 + C);
    const size_t prow = (size_t)(o0 + b + dw.n) * (size_t)A.Vs, qrow = (size_t)(o0 + dw.n) * (size_t)A.Vs;
    const ExpConst EC{A.K_hi, A.K_lo, A.d_min};
    // the thread's total: exact sums of its selected p (and q) weights, A - rho B for a residual
    float2 Ah = f2(0.f), Al = f2(0.f), Bh = f2(0.f), Bl = f2(0.f);
    float2 LP[C / 2], LQ[C / 2];  // the thread's columns, loaded before use
#pragma unroll
    for (int i = 0; i < C / 2; ++i) {
        const int32_t k = k0 + 2 * i;
        LP[i] = make_float2(k < k1 ? lg<DT>(A.target, prow + k) : -INFINITY,
                            k + 1 < k1 ? lg<DT>(A.target, prow + k + 1) : -INFINITY);
        LQ[i] = make_float2(resid && k < k1 ? lg<DT>(A.draft, qrow + k) : -INFINITY,
                            resid && k + 1 < k1 ? lg<DT>(A.draft, qrow + k + 1) : -INFINITY);
    }
#pragma unroll
    for (int i = 0; i < C / 2; ++i) {
        const int32_t k = k0 + 2 * i;
        if (k >= k1) break;
        const float2 lp = LP[i], lq = LQ[i];
        const ff2 ep = exp2_ff2(lp, f2(dw.m_p), EC, tab);
        const ff2 eq = resid ? exp2_ff2(lq, f2(dw.m_q), EC, tab) : ff2{f2(0.f), f2(0.f)};
        float2 mk;
        if (by_p) mk = f2(1.f);
        else if (resid) mk = make_float2(gt_mask(ep.hi.x, dw.rho * eq.hi.x), gt_mask(ep.hi.y, dw.rho * eq.hi.y));
        else mk = make_float2(A.v0 + k == dw.xcl ? 0.f : 1.f, A.v0 + k + 1 == dw.xcl ? 0.f : 1.f);
        const float2 hp = grid_hi(ep.hi), lpw = add2(sub2(ep.hi, hp), ep.lo);
        const float2 hq = grid_hi(eq.hi), lqw = add2(sub2(eq.hi, hq), eq.lo);
        Ah = fma2(mk, hp, Ah); Al = fma2(mk, lpw, Al);
        Bh = fma2(mk, hq, Bh); Bl = fma2(mk, lqw, Bl);
    }
    ff tot = ff_add(ff{Ah.x, Al.x}, ff{Ah.y, Al.y});
    if (resid && !by_p) tot = ff_sub(tot, ff_mul(rho, ff_add(ff{Bh.x, Bl.x}, ff{Bh.y, Bl.y})));
    if (!(tot.hi > 0.f)) tot = ff{0.f, 0.f};
    // exclusive prefix of the threads' totals (warp scan, then the warps' totals in order)
    const ff incl = warp_scan_ff(tot, lane);
    if (lane == 31) red[warp] = incl;
    __syncthreads();
    ff wbefore{0.f, 0.f};
    for (int w = 0; w < warp; ++w) wbefore = ff_add(wbefore, red[w]);
    const ff ex_lane = shfl_ff(incl, lane ? lane - 1 : 0);
    const ff excl = ff_add(wbefore, lane ? ex_lane : ff{0.f, 0.f});
    const ff inc = ff_add(excl, tot);
    // the first thread whose inclusive prefix exceeds rem holds the crossing (lowest thread index)
    const bool holds = !tail_rule && tot.hi > 0.f && ff_gt(inc, rem) && !ff_gt(excl, rem);
    const int first = cta_min_i<kShThreads>(holds ? (int)threadIdx.x : 0x7FFFFFFF, redi);
    if (first != 0x7FFFFFFF && warp == first / 32) {
        // the crossing thread's columns, one a lane: weights, their prefix from the thread's exclusive
        // prefix, the first positive column past rem (else, rounding, its last positive column)
        const int32_t f0 = kc0 + first * C, f1 = min(kc1, f0 + C);
        const ff base = shfl_ff(excl, first & 31);
        ff w{0.f, 0.f};
        if (lane < C && f0 + lane < f1) {
            ff ep, eq;
            bool sel;
            draw_weights<DT>(A, dw, prow, qrow, f0 + lane, EC, tab, ep, eq, sel);
            w = col_weight(dw, by_p, ep, eq, sel, rho);
        }
        const ff cc = ff_add(base, warp_scan_ff(w, lane));
        const bool pos = w.hi > 0.f;
        const uint32_t cross = __ballot_sync(0xFFFFFFFFu, pos && ff_gt(cc, rem));
        const uint32_t pb = __ballot_sync(0xFFFFFFFFu, pos);
        if (lane == 0 && pb) s_col = f0 + (cross ? __ffs(cross) - 1 : 31 - __clz(pb));
    }
    __syncthreads();
    int32_t col = s_col;
    if (col < 0) {  // no crossing (the tail rule, or rounding): the chunk's last column of positive weight
        int lastpos = -1;
        for (int32_t k = k0; k < k1; ++k) {
            ff ep, eq;
            bool sel;
            draw_weights<DT>(A, dw, prow, qrow, k, EC, tab, ep, eq, sel);
            if (col_weight(dw, by_p, ep, eq, sel, rho).hi > 0.f) lastpos = k;
        }
        col = -cta_min_i<kShThreads>(-lastpos, redi);
    }
    if (threadIdx.x == 0) A.out_tokens[t0 + dw.n] = col >= 0 ? A.v0 + col : -1;
}

}  // namespace

cudaError_t launch_shard(int stage, const ShardArgs& A, void* a, void* b, void* c) {
    cudaStream_t st = A.stream;
    const int32_t nrows = A.nrows;
    switch (stage) {
        case 0:
            if (nrows > 0) {
                if (A.dtype == SV_BF16) k_shard_stats<SV_BF16><<<nrows, kShStatThreads, 0, st>>>(A, (ShardPartial*)a);
                else k_shard_stats<SV_F32><<<nrows, kShStatThreads, 0, st>>>(A, (ShardPartial*)a);
            }
            break;
        case 1:
            if (A.dtype == SV_BF16) k_shard_decide<SV_BF16><<<(A.B + 7) / 8, 256, 0, st>>>(A, (const ShardPartial*)a, (ShardDraw*)b);
            else k_shard_decide<SV_F32><<<(A.B + 7) / 8, 256, 0, st>>>(A, (const ShardPartial*)a, (ShardDraw*)b);
            break;
        case 2:
            if (A.dtype == SV_BF16) k_shard_sums<SV_BF16><<<A.nc * A.B, kShSumThreads, 0, st>>>(A, (const ShardDraw*)a, (ff*)b);
            else k_shard_sums<SV_F32><<<A.nc * A.B, kShSumThreads, 0, st>>>(A, (const ShardDraw*)a, (ff*)b);
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
    int32_t w = 0;
    for (int j = 0; j < S; ++j) w = std::max(w, bounds[j + 1] - bounds[j]);
    A.nc = (w + sv::kShChunk - 1) / sv::kShChunk;
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

int32_t spec_shard_chunks(int32_t S, const int32_t* shard_bounds_host) {
    sv::ShardArgs A{};
    if (S < 1 || S > sv::kMaxShards || !shard_bounds_host) return 0;
    return shard_bounds(A, S, shard_bounds_host, shard_bounds_host[S]) == SV_OK ? A.nc : 0;
}

int spec_shard_sums(int32_t shard, int32_t S, const int32_t* shard_bounds_host, const void* shard_target,
                    const void* shard_draft, sv_dtype dtype, const void* draws, const int32_t* seq_offsets, int32_t B,
                    int32_t V, float temperature, void* sums, void* cuda_stream) {
    sv::ShardArgs A;
    int rc = shard_args(A, dtype, B, V, 0, temperature, cuda_stream);
    if (rc != SV_OK) return rc;
    if ((rc = shard_bounds(A, S, shard_bounds_host, V)) != SV_OK) return rc;
    if (shard < 0 || shard >= S || !shard_target || !draws || (uintptr_t)draws % 16 || !aligned4(seq_offsets) ||
        !sums || (uintptr_t)sums % 16)
        return SV_ERR_INVALID_ARG;
    if (B == 0 || A.greedy) return SV_OK;
    if ((int64_t)A.nc * B >= (1ll << 31)) return SV_ERR_INVALID_ARG;  // one CTA per (sequence, chunk)
    A.shard = shard;
    A.v0 = A.bounds[shard];
    A.Vs = A.bounds[shard + 1] - A.bounds[shard];
    A.target = shard_target;
    A.draft = shard_draft;
    A.offs = seq_offsets;
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
static_assert(sv::kShChunk == SV_SHARD_CHUNK, "the C ABI's sums chunk");
