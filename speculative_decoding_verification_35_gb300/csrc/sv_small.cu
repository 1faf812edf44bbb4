// Small-batch verify: one thread-block cluster per sequence, its CTAs holding contiguous vocabulary slices
// of the sequence's rows. The step is the vocabulary-sharded protocol ("All About Transformer Inference",
// the model-parallel sections; the rule of velog "6-1편. Speculative Decoding", §2-1/§2-2), with the
// shards as the CTAs of a cluster and the exchanges in distributed shared memory behind cluster barriers:
//   1. each CTA: every row's partial statistics over its slice (raw max, sum of 2^((l - m) K), first
//      argmax, the logit at the row's draft token when the slice holds it);
//   2. CTA 0: the merged statistics, the accept tests, the first rejection (greedy: the whole output) and
//      the draw (mode, slot, row maxima, selection ratio, uniform);
//   3. each CTA: the draw's exact sums over its slice (float-float on the 2^-20 grid, see grid_hi);
//   4. every CTA finds the slice holding the draw's target u S (the same arithmetic on each); that CTA
//      scans its slice for the drawn column and writes it.
// For a sampled batch whose persistent launch would give each statistics warp at most one task, a step is
// then a chain of four phases on shared memory instead of handoff words polled across the GPU (a greedy
// step, one decision without a draw, stays shorter as the persistent launch unless forced here). Every
// wait is a cluster barrier among CTAs that the hardware schedules together; nothing is polled.
#include <algorithm>
#include <cfloat>
#include <cmath>

#include <cooperative_groups.h>
#include <cuda_bf16.h>

#include "sv_device.cuh"
#include "sv_internal.h"

namespace cg = cooperative_groups;

namespace sv {
namespace {

constexpr int kSmThreads = 512;
constexpr int kSmWarps = kSmThreads / 32;
constexpr int kSmRows = 2 * SV_MAX_GAMMA + 1;
constexpr int kSmBatch = 8;    // 16-byte loads a lane issues together in phase 1
constexpr int kSmParts = 128;  // piece records of a CTA (rows x pieces; one piece a row always fits)

struct SmRec {  // one row's partial statistics over a CTA's slice
    float m, s;     // raw max, sum of 2^((l - m) K) (NaN: a NaN or +inf logit in the slice)
    int32_t arg;    // first argmax in the slice, as a global column (-1: none)
    float g;        // the logit at the row's draft token if the slice holds that column, else 0
};
struct SmDraw {  // the sequence's draw, written by CTA 0
    int32_t mode, n;
    float m_p, m_q, rho, u;
    int32_t xcl, pad;
};

template <int DT>
__device__ __forceinline__ float lgs(const void* base, size_t idx) {
    if (DT == SV_BF16) return __uint_as_float((uint32_t)__ldg((const unsigned short*)base + idx) << 16);
    return __ldg((const float*)base + idx);
}

__device__ __forceinline__ ff shfl_ff(ff v, int src) {
    return ff{__shfl_sync(0xFFFFFFFFu, v.hi, src), __shfl_sync(0xFFFFFFFFu, v.lo, src)};
}
__device__ __forceinline__ ff warp_scan_ff(ff v, int lane) {  // inclusive prefix over lanes 0..lane
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const ff y{__shfl_up_sync(0xFFFFFFFFu, v.hi, o), __shfl_up_sync(0xFFFFFFFFu, v.lo, o)};
        if (lane >= o) v = ff_add(y, v);
    }
    return v;
}
__device__ __forceinline__ ff warp_sum_ff(ff v) {  // the same on every lane
#pragma unroll
    for (int o = 16; o; o >>= 1)
        v = ff_add(v, ff{__shfl_xor_sync(0xFFFFFFFFu, v.hi, o), __shfl_xor_sync(0xFFFFFFFFu, v.lo, o)});
    return v;
}
__device__ int cta_min_i(int v, int* red) {
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xFFFFFFFFu, v, o));
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    int t = 0x7FFFFFFF;
    for (int w = 0; w < kSmWarps; ++w) t = min(t, red[w]);
    return t;
}

// the draw's weights of column k (relative to the merged row maxima) and the residual's selection
template <int DT>
__device__ __forceinline__ void draw_weights(const Params& P, const SmDraw& dw, size_t prow, size_t qrow, int32_t k,
                                             const ExpConst& EC, const float* tab, ff& ep, ff& eq, bool& sel) {
    const bool resid = dw.mode == kModeResidual;
    const float lp = lgs<DT>(P.target, prow + k), lq = resid ? lgs<DT>(P.draft, qrow + k) : 0.f;
    const ff2 e = exp2_ff2(make_float2(lp, lq), make_float2(dw.m_p, resid ? dw.m_q : 0.f), EC, tab);
    ep = ff_norm(e.hi.x, e.lo.x);
    eq = resid ? ff_norm(e.hi.y, e.lo.y) : ff{0.f, 0.f};
    sel = resid ? e.hi.x > dw.rho * e.hi.y : !(dw.mode == kModeResidualPM && k == dw.xcl);
}
// the draw's weight of a column given the exact normaliser ratio rho (by_p: the p fallback)
__device__ __forceinline__ ff col_weight(const SmDraw& dw, bool by_p, ff ep, ff eq, bool sel, ff rho) {
    if (by_p) return ep;
    if (!sel) return ff{0.f, 0.f};
    if (dw.mode != kModeResidual) return ep;
    const ff w = ff_sub(ep, ff_mul(rho, eq));
    return w.hi > 0.f ? w : ff{0.f, 0.f};
}

template <int DT>
__global__ void __launch_bounds__(kSmThreads, 1) k_small(const __grid_constant__ Params P, int32_t C) {
    cg::cluster_group cl = cg::this_cluster();
    // every CTA of the cluster must have started before another one stores into its shared memory: arrive
    // now, wait just before the first remote store
    auto started = cl.barrier_arrive();
    const int32_t j = (int32_t)cl.block_rank();
    const int32_t b = (int32_t)(blockIdx.x / (uint32_t)C);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    __shared__ SmRec part[kSmParts];  // rows x pieces
    __shared__ SmRec allrec[8][kSmRows];  // CTA 0: every slice's row records, stored by their CTAs
    __shared__ SmDraw draw;               // stored into every CTA by CTA 0
    __shared__ ff allsum[8][4];           // every slice's draw sums, stored into every CTA by their CTAs
    __shared__ float tab[2 * kExpTab];
    __shared__ ff red[4][kSmWarps];
    __shared__ ff redt[kSmWarps];
    __shared__ int redi[kSmWarps];
    __shared__ ff s_rho, s_rem;
    __shared__ int s_owner, s_byp, s_tail, s_col;
    __shared__ int32_t s_tok[32];   // CTA 0: the draft tokens of slots 0 .. g - 1
    __shared__ float s_u[2][32];    // CTA 0: the accept and draw uniforms of every slot
    if (tid < kExpTab) {
        tab[tid] = P.exp2_tab[tid].x;
        tab[kExpTab + tid] = P.exp2_tab[tid].y;
    }
    // the CSR structure, checked by every CTA before any row is read (a bad structure fails every sequence)
    {
        int bad = tid == 0 && __ldg(P.offs) != 0;
        for (int32_t s = tid; s < P.B; s += kSmThreads) {
            const int32_t o0 = __ldg(P.offs + s), g = __ldg(P.offs + s + 1) - o0;
            bad |= o0 < 0 || g < 0 || g > P.max_gamma || g != __ldg(P.gammas + s);
        }
        if (__syncthreads_or(bad)) {
            if (j == 0 && tid == 0) {
                P.out_n[b] = -1;
                if (P.hist) P.next[b] = -1;
                atomicOr(P.status, 1u << SV_ERR_BAD_OFFSETS);
            }
            return;  // every CTA of the cluster returns here, before any exchange
        }
    }
    const bool greedy = P.K_hi == 0.f;
    const int32_t o0 = __ldg(P.offs + b), g = __ldg(P.offs + b + 1) - o0, t0 = o0 + b;
    const bool has_d = !greedy && !P.pm;
    const int32_t nrows = g + 1 + (has_d ? g : 0);
    const int32_t V = P.V;
    const int32_t v0 = (int32_t)((int64_t)V * j / C), v1 = (int32_t)((int64_t)V * (j + 1) / C);
    const float K = P.K_hi;
    const ExpConst EC{P.K_hi, P.K_lo, P.d_min};
    if (j == 0 && warp == kSmWarps - 1) {  // the decision's inputs that need no statistics, under phase 1
        s_tok[lane] = lane < g ? __ldg(P.tokens + o0 + lane) : -1;
        if (!greedy) {
            const uint32_t seq = P.seq_base + (uint32_t)b;
            s_u[0][lane] = philox_uniform(P.seed, P.step, seq, (uint32_t)lane, 0);
            s_u[1][lane] = philox_uniform(P.seed, P.step, seq, (uint32_t)lane, 1);
        }
    }

    // 1. partial statistics of every row over the slice. The slice of a row is cut into np pieces so that
    // every warp has an item (row r, piece p); a warp reads its piece with 16-byte loads (scalar elements
    // before the first aligned address and after the last whole vector); a tie in the maximum goes to the
    // lower column, whatever order a lane takes its columns in.
    const int32_t Ls = v1 - v0;
    const int32_t np = max(1, min(kSmWarps / nrows, Ls / 256));  // pieces a row: at most one item a warp
    auto piece_lo = [&](int32_t p) {  // interior boundaries on 64-column multiples (aligned vectors)
        if (p == 0 || p == np) return p == 0 ? v0 : v1;
        return max(v0, (v0 + (int32_t)((int64_t)Ls * p / np)) & ~63);
    };
    auto row_of = [&](int32_t r, const void*& base, int32_t& slot) {
        const bool dr = r > g;
        slot = dr ? r - g - 1 : r;
        base = dr ? P.draft : P.target;
        return (size_t)(dr ? o0 + slot : t0 + slot) * (size_t)V;
    };
    for (int32_t it = warp; it < nrows * np; it += kSmWarps) {
        const int32_t r = it / np, p = it - r * np;
        const void* base;
        int32_t slot;
        const size_t row = row_of(r, base, slot);
        const int32_t a = piece_lo(p), e = piece_lo(p + 1);
        constexpr int ES = DT == SV_BF16 ? 2 : 4, VE = 16 / ES;
        const uintptr_t addr = (uintptr_t)base + (row + (size_t)a) * ES;
        int32_t head = e - a, nvec = 0;  // an address that is not element-aligned: all scalar
        if (addr % ES == 0) {
            head = min(e - a, (int32_t)(((16 - addr % 16) % 16) / ES));
            nvec = (e - a - head) / VE;
        }
        const int32_t body = a + head, tail = body + nvec * VE;
        float m = -INFINITY, s = 0.f;
        int arg = 0x7FFFFFFF;
        bool bad = false;
        auto take = [&](const auto& x, int32_t k0) {  // the values x[i] at columns k0 + i
            constexpr int n = (int)(sizeof(x) / sizeof(float));
            float vm = x[0];
            int vi = 0;
            bad |= !(x[0] <= FLT_MAX);
#pragma unroll
            for (int i = 1; i < n; ++i) {
                bad |= !(x[i] <= FLT_MAX);
                if (x[i] > vm) { vm = x[i]; vi = i; }
            }
            if (vm > m) {
                if (!greedy && m != -INFINITY) s *= ex2_approx((m - vm) * K);
                m = vm;
                arg = k0 + vi;
            } else if (vm == m && k0 + vi < arg) {  // columns are not taken in order: the first maximum
                arg = k0 + vi;
            }
            if (!greedy && m != -INFINITY) {
#pragma unroll
                for (int i = 0; i < n; ++i) s += ex2_approx((x[i] - m) * K);
            }
        };
        // the scalar columns before and after the vectors (fewer than a vector each, unless the address is
        // not element-aligned), loaded before the vectors so that their latency overlaps
        const bool edge = body - a <= 32 && e - tail <= 32;
        float xh = 0.f, xt = 0.f;
        if (edge) {
            if (lane < body - a) xh = lgs<DT>(base, row + a + lane);
            if (lane < e - tail) xt = lgs<DT>(base, row + tail + lane);
        }
        const uint4* vp = (const uint4*)((const char*)base + (row + (size_t)body) * ES);
        for (int32_t v0b = 0; v0b < nvec; v0b += 32 * kSmBatch) {
            uint4 u[kSmBatch];
#pragma unroll
            for (int i = 0; i < kSmBatch; ++i) {
                const int32_t v = v0b + lane + 32 * i;
                if (v < nvec) u[i] = __ldg(vp + v);
            }
#pragma unroll
            for (int i = 0; i < kSmBatch; ++i) {
                const int32_t v = v0b + lane + 32 * i;
                if (v < nvec) {
                    float x[VE];
                    const uint32_t w[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        if (DT == SV_BF16) {
                            x[2 * q] = __uint_as_float(w[q] << 16);
                            x[2 * q + 1] = __uint_as_float(w[q] & 0xFFFF0000u);
                        } else {
                            x[q] = __uint_as_float(w[q]);
                        }
                    }
                    take(x, body + v * VE);
                }
            }
        }
        if (edge) {
            if (lane < body - a) {
                const float x[1] = {xh};
                take(x, a + lane);
            }
            if (lane < e - tail) {
                const float x[1] = {xt};
                take(x, tail + lane);
            }
        } else {
            for (int32_t k = a + lane; k < body; k += 32) {
                const float x[1] = {lgs<DT>(base, row + k)};
                take(x, k);
            }
            for (int32_t k = tail + lane; k < e; k += 32) {
                const float x[1] = {lgs<DT>(base, row + k)};
                take(x, k);
            }
        }
        float M = m;
#pragma unroll
        for (int o = 16; o; o >>= 1) M = fmaxf(M, __shfl_xor_sync(0xFFFFFFFFu, M, o));
        int A = m == M ? arg : 0x7FFFFFFF;
        float S = !greedy && m != -INFINITY && M != -INFINITY ? s * ex2_approx((m - M) * K) : 0.f;
#pragma unroll
        for (int o = 16; o; o >>= 1) {
            A = min(A, __shfl_xor_sync(0xFFFFFFFFu, A, o));
            S += __shfl_xor_sync(0xFFFFFFFFu, S, o);
        }
        const bool bd = __any_sync(0xFFFFFFFFu, bad);
        if (lane == 0) {
            SmRec q;
            q.m = bd ? __int_as_float(0x7FC00000) : M;
            q.s = bd ? __int_as_float(0x7FC00000) : S;
            q.arg = M == -INFINITY || A == 0x7FFFFFFF ? -1 : A;
            q.g = 0.f;
            if (slot < g) {
                const int32_t x = __ldg(P.tokens + o0 + slot);
                if (x >= a && x < e) q.g = lgs<DT>(base, row + x);
            }
            part[it] = q;
        }
    }
    __syncthreads();
    cl.barrier_wait(std::move(started));
    // the row's record over the slice: its pieces merged in column order, stored into CTA 0
    if (tid < nrows) {
        const void* base;
        int32_t slot;
        row_of(tid, base, slot);
        const int32_t x = slot < g ? __ldg(P.tokens + o0 + slot) : -1;
        float M = -INFINITY, S = 0.f, gx = 0.f;
        int arg = -1;
        bool nan = false;
        for (int32_t p = 0; p < np; ++p) {
            const SmRec q = part[tid * np + p];
            if (q.m != q.m) nan = true;
            else if (q.m > M) { M = q.m; arg = q.arg; }
            if (x >= piece_lo(p) && x < piece_lo(p + 1)) gx = q.g;
        }
        if (!nan && !greedy && M != -INFINITY) {
            for (int32_t p = 0; p < np; ++p) {
                const SmRec q = part[tid * np + p];
                if (q.m != -INFINITY) S += q.s * exp2_fma((q.m - M) * K);
            }
        }
        SmRec q;
        q.m = nan ? __int_as_float(0x7FC00000) : M;
        q.s = nan ? __int_as_float(0x7FC00000) : S;
        q.arg = nan ? -1 : arg;
        q.g = gx;
        *cl.map_shared_rank(&allrec[j][tid], 0u) = q;
    }
    cl.sync();

    // 2. the decision, by warp 0 of CTA 0 (lane i: slot i)
    if (j == 0 && warp == 0) {
        // merged statistics of row r from the C slices (in slice order)
        auto merged = [&](int32_t r, float& M, float& S, int& arg) {
            M = -INFINITY;
            S = 0.f;
            arg = -1;
            bool nan = false;
            for (int32_t i = 0; i < C; ++i) {
                const SmRec q = allrec[i][r];
                if (q.m != q.m) { nan = true; continue; }
                if (q.m > M) arg = q.arg;  // lower slices hold lower columns: the first max wins ties
                M = fmaxf(M, q.m);
            }
            if (nan) { M = S = __int_as_float(0x7FC00000); arg = -1; return; }
            if (M == -INFINITY || greedy) return;
            for (int32_t i = 0; i < C; ++i) {
                const SmRec q = allrec[i][r];
                if (q.m != -INFINITY) S += q.s * exp2_fma((q.m - M) * K);
            }
        };
        auto gval = [&](int32_t r, int32_t x) {  // the logit at column x of row r, from the slice holding it
            int32_t i = (int32_t)(((int64_t)x * C) / V);
            while (i + 1 < C && x >= (int32_t)((int64_t)V * (i + 1) / C)) ++i;
            while (i > 0 && x < (int32_t)((int64_t)V * i / C)) --i;
            return allrec[i][r].g;
        };
        int32_t x = -1;
        uint32_t tcode = 0;
        if (lane < g) {
            x = s_tok[lane];
            if (x < 0 || x >= V) tcode = SV_ERR_BAD_TOKEN;
        }
        float Tm = -INFINITY, Ts = 0.f, Dm = 0.f, Ds = 1.f;
        int Ta = -1, Da = -1;
        if (lane <= g) merged(lane, Tm, Ts, Ta);
        if (lane < g && has_d) merged(g + 1 + lane, Dm, Ds, Da);
        // the first failure in the rule's order: a bad draft token, then target row i before draft row i
        uint32_t code = 0;
        {
            const uint32_t tb = __ballot_sync(0xFFFFFFFFu, tcode != 0u);
            if (tb) {
                code = SV_ERR_BAD_TOKEN;
            } else {
                uint32_t key = ~0u;
                if (lane <= g) {
                    const uint32_t ct = Tm != Tm ? SV_ERR_NONFINITE : (Tm == -INFINITY ? SV_ERR_EMPTY_ROW : 0u);
                    if (ct) key = min(key, (2u * (uint32_t)lane) << 4 | ct);
                }
                if (lane < g && has_d) {
                    const uint32_t cd = Dm != Dm ? SV_ERR_NONFINITE : (Dm == -INFINITY ? SV_ERR_EMPTY_ROW : 0u);
                    if (cd) key = min(key, (2u * (uint32_t)lane + 1u) << 4 | cd);
                }
                key = __reduce_min_sync(0xFFFFFFFFu, key);
                if (key != ~0u) code = key & 15u;
            }
        }
        SmDraw dw{};
        dw.mode = kModeNone;
        dw.xcl = -1;
        int32_t n = -1, acc = -1, drawn = -1;
        if (code) {
            if (lane == 0) {
                atomicOr(P.status, 1u << code);
                P.out_n[b] = -1;
            }
            for (int32_t s = lane; s <= g; s += 32) P.out_tokens[t0 + s] = -1;
        } else if (greedy) {
            const uint32_t mism = __ballot_sync(0xFFFFFFFFu, lane < g && x != Ta);
            n = mism ? __ffs(mism) - 1 : g;
            if (lane <= g) P.out_tokens[t0 + lane] = lane < n ? x : (lane == n ? Ta : -1);
            if (lane == 0) P.out_n[b] = n;
            acc = x;
            drawn = __shfl_sync(0xFFFFFFFFu, Ta, n);
        } else {
            bool ok = true;
            if (lane < g) {
                const float lt = gval(lane, x), ld = P.pm ? 0.f : gval(g + 1 + lane, x);
                const ff2 e = exp2_ff2(make_float2(lt, ld), make_float2(Tm, P.pm ? 0.f : Dm), EC, tab);
                const float px = div_fma(e.hi.x + e.lo.x, Ts);
                const float qx = P.pm ? 1.f : div_fma(e.hi.y + e.lo.y, Ds);
                ok = s_u[0][lane] * qx < px;
            }
            const uint32_t rej = __ballot_sync(0xFFFFFFFFu, lane < g && !ok);
            n = rej ? __ffs(rej) - 1 : g;
            if (lane <= g && lane != n) P.out_tokens[t0 + lane] = lane < n ? x : -1;
            if (lane == 0) P.out_n[b] = n;
            dw.mode = n < g ? (P.pm ? kModeResidualPM : kModeResidual) : kModeBonus;
            dw.n = n;
            dw.m_p = __shfl_sync(0xFFFFFFFFu, Tm, n);
            const float ps = __shfl_sync(0xFFFFFFFFu, Ts, n);
            const float qm = __shfl_sync(0xFFFFFFFFu, Dm, n), qs = __shfl_sync(0xFFFFFFFFu, Ds, n);
            dw.m_q = n < g && !P.pm ? qm : 0.f;
            dw.rho = n < g && !P.pm ? div_fma(ps, qs) : 1.f;
            dw.u = s_u[1][n];
            dw.xcl = n < g && P.pm ? __shfl_sync(0xFFFFFFFFu, x, n) : -1;
        }
        if (lane < C) *cl.map_shared_rank(&draw, (unsigned)lane) = dw;
        // the fused update of a greedy or failed sequence (a sampled one's is written with its token)
        if (P.hist && (code || greedy)) {
            const int32_t L = n >= 0 ? P.lens[b] : 0;
            if (n < 0 || L < 0 || (int64_t)L + n + 1 > P.cap) {
                if (lane == 0) {
                    P.next[b] = -1;
                    if (n >= 0) atomicOr(P.status, 1u << SV_ERR_CAPACITY);
                }
            } else {
                int32_t* h = P.hist + (size_t)b * (size_t)P.cap + (size_t)L;
                if (lane < n) h[lane] = acc;
                if (lane == n) h[n] = drawn;
                if (lane == 0) {
                    P.lens[b] = L + n + 1;
                    P.next[b] = drawn;
                }
            }
        }
    }
    cl.sync();

    // 3. the draw's exact sums over the slice: all p weights, all q weights, those of the selected columns
    const SmDraw dw = draw;
    const bool sampled = dw.mode != kModeNone;
    const bool resid = dw.mode == kModeResidual;
    const size_t prow = (size_t)(t0 + dw.n) * (size_t)V, qrow = (size_t)(o0 + dw.n) * (size_t)V;
    if (sampled) {
        // thread t: column pairs v0 + 2 t + 1024 i; exact grid sums folded into float-float every 16 pairs
        ff acc4[4] = {ff{0.f, 0.f}, ff{0.f, 0.f}, ff{0.f, 0.f}, ff{0.f, 0.f}};
        float2 Ph = f2(0.f), Pl = f2(0.f), Qh = f2(0.f), Ql = f2(0.f), Ah = f2(0.f), Al = f2(0.f), Bh = f2(0.f),
               Bl = f2(0.f);
        int cnt = 0;
        auto fold = [&]() {
            acc4[0] = ff_add(acc4[0], ff_add(ff{Ph.x, Pl.x}, ff{Ph.y, Pl.y}));
            acc4[1] = ff_add(acc4[1], ff_add(ff{Qh.x, Ql.x}, ff{Qh.y, Ql.y}));
            acc4[2] = ff_add(acc4[2], ff_add(ff{Ah.x, Al.x}, ff{Ah.y, Al.y}));
            acc4[3] = ff_add(acc4[3], ff_add(ff{Bh.x, Bl.x}, ff{Bh.y, Bl.y}));
            Ph = Pl = Qh = Ql = Ah = Al = Bh = Bl = f2(0.f);
        };
        for (int32_t k = v0 + 2 * tid; k < v1; k += 2 * kSmThreads) {
            const bool two = k + 1 < v1;
            const float2 lp = make_float2(lgs<DT>(P.target, prow + k), two ? lgs<DT>(P.target, prow + k + 1) : -INFINITY);
            const float2 lq = resid ? make_float2(lgs<DT>(P.draft, qrow + k), two ? lgs<DT>(P.draft, qrow + k + 1)
                                                                                  : -INFINITY)
                                    : f2(-INFINITY);
            const ff2 ep = exp2_ff2(lp, f2(dw.m_p), EC, tab);
            const ff2 eq = resid ? exp2_ff2(lq, f2(dw.m_q), EC, tab) : ff2{f2(0.f), f2(0.f)};
            float2 mk;
            if (resid) mk = make_float2(gt_mask(ep.hi.x, dw.rho * eq.hi.x), gt_mask(ep.hi.y, dw.rho * eq.hi.y));
            else mk = make_float2(k == dw.xcl ? 0.f : 1.f, k + 1 == dw.xcl ? 0.f : 1.f);
            const float2 hp = grid_hi(ep.hi), lpw = add2(sub2(ep.hi, hp), ep.lo);
            const float2 hq = grid_hi(eq.hi), lqw = add2(sub2(eq.hi, hq), eq.lo);
            Ph = add2(Ph, hp); Pl = add2(Pl, lpw); Qh = add2(Qh, hq); Ql = add2(Ql, lqw);
            Ah = fma2(mk, hp, Ah); Al = fma2(mk, lpw, Al); Bh = fma2(mk, hq, Bh); Bl = fma2(mk, lqw, Bl);
            if (++cnt == 16) {
                fold();
                cnt = 0;
            }
        }
        fold();
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            acc4[i] = warp_sum_ff(acc4[i]);
            if (lane == 0) red[i][warp] = acc4[i];
        }
        __syncthreads();
        if (tid < 4) {
            ff t{0.f, 0.f};
            for (int w = 0; w < kSmWarps; ++w) t = ff_add(t, red[tid][w]);  // in warp order
            for (int32_t i = 0; i < C; ++i) *cl.map_shared_rank(&allsum[j][tid], (unsigned)i) = t;
        }
    }
    cl.sync();

    // 4. the slice holding the target, then its drawn column. Warp 0 of every CTA reads the C records in
    // slice order (the same arithmetic everywhere); the owning CTA scans its slice.
    if (sampled) {
        if (warp == 0) {
            auto recw = [&](int32_t i, int f) { return &allsum[i][f]; };
            ff sp{0.f, 0.f}, sq{0.f, 0.f};
            for (int32_t i = lane; i < C; i += 32) {
                sp = ff_add(sp, *recw(i, 0));
                sq = ff_add(sq, *recw(i, 1));
            }
            sp = warp_sum_ff(sp);
            sq = warp_sum_ff(sq);
            const ff rho = resid ? ff_div(sp, sq) : ff{0.f, 0.f};
            auto mass = [&](int32_t i, bool by_p) {
                if (i >= C) return ff{0.f, 0.f};
                if (by_p) return *recw(i, 0);
                ff w = *recw(i, 2);
                if (resid) w = ff_sub(w, ff_mul(rho, *recw(i, 3)));
                return w.hi > 0.f ? w : ff{0.f, 0.f};
            };
            // both candidate masses are summed by every lane (no warp collective sits under a branch)
            const ff w0 = mass(lane, false), w1 = mass(lane, true);
            const ff S0 = warp_sum_ff(w0), S1 = warp_sum_ff(w1);
            const bool by_p = __shfl_sync(0xFFFFFFFFu, (int)!(S0.hi > 0.f), 0) != 0;  // a residual of mass 0: from p
            const ff w = by_p ? w1 : w0;
            const ff S = by_p ? S1 : S0;
            const ff target = ff_mul(ff{dw.u, 0.f}, S);
            const ff inc = warp_scan_ff(w, lane);
            const ff up = shfl_ff(inc, lane ? lane - 1 : 0);  // every lane takes part in the shuffle
            const ff exc = lane ? up : ff{0.f, 0.f};
            const bool pos = w.hi > 0.f;
            const uint32_t cross = __ballot_sync(0xFFFFFFFFu, pos && ff_gt(inc, target));
            const uint32_t pb = __ballot_sync(0xFFFFFFFFu, pos);
            int owner = -1;
            ff before{0.f, 0.f};
            int tail = 0;
            if (cross) {
                owner = __ffs(cross) - 1;
                before = shfl_ff(exc, owner);
            } else if (pb) {  // rounding lost the crossing: the last slice of positive mass
                owner = 31 - __clz(pb);
                before = shfl_ff(exc, owner);
                tail = 1;
            }
            if (lane == 0) {
                s_owner = owner;
                s_byp = by_p;
                s_tail = tail;
                s_rho = rho;
                s_rem = ff_sub(target, before);
                s_col = -1;
            }
        }
        __syncthreads();
        if (s_owner < 0 && j == 0 && tid == 0) P.out_tokens[t0 + dw.n] = -1;  // nothing of positive weight
        if (s_owner == j) {
            const ff rho = s_rho, rem = s_rem;
            const bool by_p = s_byp, tail_rule = s_tail;
            // thread t: columns [c0, c1) of the slice, contiguous
            const int32_t per = (v1 - v0 + kSmThreads - 1) / kSmThreads;
            const int32_t c0 = min(v1, v0 + tid * per), c1 = min(v1, c0 + per);
            float2 Ah = f2(0.f), Al = f2(0.f), Bh = f2(0.f), Bl = f2(0.f);
            for (int32_t k = c0; k < c1; k += 2) {
                const bool two = k + 1 < c1;
                const float2 lp = make_float2(lgs<DT>(P.target, prow + k), two ? lgs<DT>(P.target, prow + k + 1) : -INFINITY);
                const float2 lq = resid ? make_float2(lgs<DT>(P.draft, qrow + k), two ? lgs<DT>(P.draft, qrow + k + 1)
                                                                                      : -INFINITY)
                                        : f2(-INFINITY);
                const ff2 ep = exp2_ff2(lp, f2(dw.m_p), EC, tab);
                const ff2 eq = resid ? exp2_ff2(lq, f2(dw.m_q), EC, tab) : ff2{f2(0.f), f2(0.f)};
                float2 mk;
                if (by_p) mk = f2(1.f);
                else if (resid) mk = make_float2(gt_mask(ep.hi.x, dw.rho * eq.hi.x), gt_mask(ep.hi.y, dw.rho * eq.hi.y));
                else mk = make_float2(k == dw.xcl ? 0.f : 1.f, k + 1 == dw.xcl ? 0.f : 1.f);
                const float2 hp = grid_hi(ep.hi), lpw = add2(sub2(ep.hi, hp), ep.lo);
                const float2 hq = grid_hi(eq.hi), lqw = add2(sub2(eq.hi, hq), eq.lo);
                Ah = fma2(mk, hp, Ah); Al = fma2(mk, lpw, Al);
                Bh = fma2(mk, hq, Bh); Bl = fma2(mk, lqw, Bl);
            }
            ff tot = ff_add(ff{Ah.x, Al.x}, ff{Ah.y, Al.y});
            if (resid && !by_p) tot = ff_sub(tot, ff_mul(rho, ff_add(ff{Bh.x, Bl.x}, ff{Bh.y, Bl.y})));
            if (!(tot.hi > 0.f)) tot = ff{0.f, 0.f};
            const ff incl = warp_scan_ff(tot, lane);
            if (lane == 31) redt[warp] = incl;
            __syncthreads();
            ff wbefore{0.f, 0.f};
            for (int w = 0; w < warp; ++w) wbefore = ff_add(wbefore, redt[w]);
            const ff ex_lane = shfl_ff(incl, lane ? lane - 1 : 0);
            const ff excl = ff_add(wbefore, lane ? ex_lane : ff{0.f, 0.f});
            const ff inc = ff_add(excl, tot);
            const bool holds = !tail_rule && tot.hi > 0.f && ff_gt(inc, rem) && !ff_gt(excl, rem);
            const int first = cta_min_i(holds ? tid : 0x7FFFFFFF, redi);
            if (first != 0x7FFFFFFF && warp == first / 32) {
                // the crossing thread's columns, one a lane (at most 32: the slice has at most 16384)
                const int32_t f0 = min(v1, v0 + first * per), f1 = min(v1, f0 + per);
                const ff base = shfl_ff(excl, first & 31);
                ff w{0.f, 0.f};
                if (f0 + lane < f1) {
                    ff ep, eq;
                    bool sel;
                    draw_weights<DT>(P, dw, prow, qrow, f0 + lane, EC, tab, ep, eq, sel);
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
            if (col < 0) {  // no crossing (the tail rule, or rounding): the slice's last column of positive weight
                int lastpos = -1;
                for (int32_t k = c0; k < c1; ++k) {
                    ff ep, eq;
                    bool sel;
                    draw_weights<DT>(P, dw, prow, qrow, k, EC, tab, ep, eq, sel);
                    if (col_weight(dw, by_p, ep, eq, sel, rho).hi > 0.f) lastpos = k;
                }
                col = -cta_min_i(-lastpos, redi);
            }
            if (warp == 0) {
                const int32_t drawn = col;  // a column of positive weight exists in the owning slice
                if (lane == 0) P.out_tokens[t0 + dw.n] = drawn;
                if (P.hist) {  // the fused update: the accepted drafts and the drawn token
                    const int32_t n = dw.n;
                    const int32_t L = P.lens[b];
                    if (L < 0 || (int64_t)L + n + 1 > P.cap) {
                        if (lane == 0) {
                            P.next[b] = -1;
                            atomicOr(P.status, 1u << SV_ERR_CAPACITY);
                        }
                    } else {
                        int32_t* h = P.hist + (size_t)b * (size_t)P.cap + (size_t)L;
                        if (lane < n) h[lane] = __ldg(P.tokens + o0 + lane);
                        if (lane == n) h[n] = drawn;
                        if (lane == 0) {
                            P.lens[b] = L + n + 1;
                            P.next[b] = drawn;
                        }
                    }
                }
            }
        }
    }
    // no remote access follows the last cluster barrier: a CTA may leave as soon as it is done
}

}  // namespace

bool small_eligible(const Params& P, int sms, int32_t* clusters) {
    if (P.parents || P.dbg.row_lse || P.dbg.row_argmax || P.dbg.p_x || P.dbg.q_x || P.dbg.seq_mass || P.dbg.beta)
        return false;
    if (P.B < 1 || P.max_gamma > SV_MAX_GAMMA) return false;
    // slices of at most 16384 columns (a crossing thread's columns fit one warp), at most 8 CTAs a cluster
    const int32_t C = std::min<int32_t>(8, std::max<int32_t>(1, (P.V + 4095) / 4096));
    if ((int64_t)P.V > (int64_t)C * 16384) return false;
    if ((int64_t)P.B * C > sms) return false;
    *clusters = C;
    return true;
}

cudaError_t launch_small(const Params& P, int dtype, int32_t C, cudaStream_t st) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(P.B * C));
    cfg.blockDim = dim3(kSmThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == SV_BF16) return cudaLaunchKernelEx(&cfg, k_small<SV_BF16>, P, C);
    return cudaLaunchKernelEx(&cfg, k_small<SV_F32>, P, C);
}

}  // namespace sv
