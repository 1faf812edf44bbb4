// Internal interface between the C ABI (sv_api.cu) and the verify kernel (sv_kernels.cu).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/specverify.h"

namespace sv {

constexpr int kThreads = 512;               // threads per CTA (one CTA per SM: its shared memory holds the
                                            // bulk-copy stages and the sampler's value table)
constexpr int kWarps = kThreads / 32;       // independent warp workers per CTA
constexpr int kAChunk = 4096;               // vocabulary columns of one statistics task (one warp, one row)
constexpr int kSTask = 1024;                // vocabulary columns of one sampler task (one warp): the unit
                                            // of the inverse-CDF search's first level
constexpr int kScanBlock = 512;             // columns the find's element scan covers per pass
constexpr int kScanPerLane = kScanBlock / 32;  // 16 consecutive columns per lane
constexpr int kStreamWarps = 8;             // statistics streamers per CTA on the bulk-copy path
constexpr int kStages = 2;                  // bulk-copy stages per streamer (128 KB in flight per SM:
                                            // enough for the HBM rate, short enough that other requests
                                            // and instruction fetches are not queued far behind)
constexpr int kStageBytes = kAChunk * 2;    // one bf16 statistics task
constexpr int kTmaSmemBytes = kStreamWarps * kStages * (kStageBytes + 8);

// The sampler's value table (bf16 logits): 2^(l K) as float-float for every bf16 magnitude in
// [2^-26, 64) of either sign, indexed by the bf16 code itself: entry (s << 12) | i holds sign s and
// magnitude code 0x3280 + i (0x3280 = 2^-26, 0x427F = 63.75). Entry i = 0 stands for every magnitude
// below 2^-26 and holds 2^0 (l = 0); the last negative entry (l = -63.75) holds 0 and stands for every
// logit at or below it, -inf included. A draw uses the table only when its rows' maxima make those two
// stand-ins negligible (tab_ok); its weights are then 2^(l K) instead of 2^((l - m) K), a per-row scale
// that cancels in every ratio the inverse CDF uses.
constexpr uint32_t kTabCodeLo = 0x3280u;    // bf16 code of 2^-26
constexpr uint32_t kTabCodeHi = 0x427Fu;    // bf16 code of 63.75
constexpr int kTabHalf = 4096;              // entries per sign
constexpr int kTabBytes = 2 * kTabHalf * 8; // 64 KB
constexpr int kTabSmemOffset = (kTmaSmemBytes + 15) & ~15;  // after the stages and their barriers
constexpr int kProgMinTasks = 4096;  // statistics tasks (bound) from which a sampled call streams in slot order
constexpr int kTabMinTasks = 2048;  // sampler tasks (sequences x 1024-column tasks) from which a call builds
                                    // the table: below, its build (~4 us at the launch's start) would sit on
                                    // the step's critical path instead of under the stream
constexpr int kBaseCache = 1024;            // batches up to this size keep their row bases in shared memory
constexpr int kRowCache = 2048;             // sampling batches with up to this many statistics rows keep a
                                            // row map (target or draft, row index) in shared memory

// kModeResidualPM: the residual of a point-mass draft (no draft rows): p with the draft column removed.
// kModeResidualSet: a token-tree node whose candidates were all rejected: p with their tokens removed.
enum : int32_t { kModeNone = 0, kModeResidual = 1, kModeBonus = 2, kModeResidualPM = 3, kModeResidualSet = 4 };
constexpr int kMaxRemoved = 32;  // removed-token words per sequence (a node has at most 31 children)
constexpr uint32_t kSpinLimit = 1u << 21;  // polls before a wait gives up (about 1 s with back-off)

// Data handed between warps of one launch is written as 64-bit words, each exactly once per call with
// one relaxed store, into a region zeroed before the call, and each non-zero once written. A reader
// polls the words themselves (bounded back-off): no fence, flag or counter orders them.
typedef unsigned long long Word;

// Partial statistics of one (row, chunk):
//   sampling: low = bits(raw max m), high = bits(sum of 2^((l - m) K)) (m = +0 implies sum >= 1;
//             sum = 0 implies m = -inf; a NaN or +inf logit makes the sum NaN);
//   greedy:   low = bits(m), high = (first argmax + 1) | (1 << 31 if a NaN was seen).
typedef Word PartialWord;

// A sequence's sampler work, written by its decision as kTaskWords words:
//   w0 = (0x80000000 | mode << 8 | n) << 32 | bits(m_p)   mode kMode*, n the emitting slot
//   w1 = bits(rho) << 32 | bits(m_q)                      rho = approximate s_p / s_q (> 0);
//                                                         kModeResidualPM: (x + 1) << 32, x the
//                                                         draft token (the column the draw removes);
//                                                         kModeResidualSet: k << 32, k removed tokens
//                                                         in the sequence's removed-token words
//   w2 = (0x80000000 | npos) << 32 | bits(u)              u the draw's uniform, npos the output slot
//                                                         of the drawn token (n, except in a tree)
// m_p, m_q are the raw-logit maxima of the draw's target and draft rows.
constexpr int kTaskWords = 4;
constexpr uint32_t kWordMark = 0x80000000u;

// A sampler task's record, kRecWords words: word k = bits(lo) << 32 | (bits(hi) | 0x80000000) of a
// non-negative float-float sum over the task's columns of the weights 2^((l - m) K):
//   k = 0: all p weights, 1: all q weights, 2: p weights of the selected columns, 3: q weights of the
//   selected columns (a bonus draw stores its p total as 0 and 2, zeros as 1 and 3; the residual of a
//   point-mass draft stores its p total as 0, the total without the removed column as 2, zeros as 1
//   and 3).
constexpr int kRecWords = 4;
// Per group of kGroupLanes lanes of a sampler task (lane L covers the task's columns [32 L, 32 L + 32),
// so group G covers [128 G, 128 G + 128)): two words, the group's selected p weights and selected q
// weights (a bonus draw: its p weights and 0), packed like the record words. The find locates the
// crossing group from them.
constexpr int kGroupLanes = 4;
constexpr int kGroups = 32 / kGroupLanes;            // 8 per task
constexpr int kGroupCols = kSTask / kGroups;         // 128 columns
constexpr int kGroupWords = 2;

// Counters of one call (zeroed before the kernel by the launch sequence).
constexpr uint32_t kOrderLost = 0xFFFFFFFFu;
struct Counters {
    uint32_t claim;    // sampler tasks claimed: in sequence-major order, or (slot order) in decision order
    uint32_t decided;  // slot order: decisions published (positions in the decision-order queue)
    uint32_t pad[30];
};

struct Params {
    const void* target;
    const void* draft;
    const int32_t* tokens;
    const int32_t* offs;
    const int32_t* gammas;
    int32_t B, V, max_gamma;
    int32_t pm;        // point-mass drafts: sampling without draft rows (q_i = 1 at x_i)
    int32_t nchA;      // statistics chunks per row
    int32_t nS;        // sampler tasks per sequence
    unsigned long long nS_recip;  // floor(2^64 / nS) + 1 (nS >= 2): c / nS = high 64 bits of c * nS_recip
    float K_hi, K_lo;  // log2(e) / T as float-float
    float d_min;       // clamp of l - m in the precise exponential (about -126.5 / K)
    int32_t use_tab;         // the CTAs build the value table (batches with enough sampler work, bf16 rows)
    float tab_mlo, tab_mhi;  // a draw uses the value table when its rows' raw maxima lie in [tab_mlo, tab_mhi]
    int32_t prog;      // slot order: statistics streamed slot by slot, each decision made at its first
                       // rejection, the rows after it checked by the sequence's find (bf16 bulk-copy path,
                       // linear sampled drafts, no per-row debug output, row bases and map in shared memory)
    uint32_t spin;     // polls before a wait on another warp's word gives up (kSpinLimit unless a caller
                       // testing the time-out path asks for fewer)
    double invT64;     // 1 / T (debug output of the row log-normalisers only)
    uint64_t seed, step;
    uint32_t seq_base;  // global index of sequence 0: sequence b's uniforms are keyed by seq_base + b
    int32_t* out_tokens;
    int32_t* out_n;
    uint32_t* status;
    sv_debug dbg;
    // workspace
    PartialWord* partials;  // [B * (2 max_gamma + 1) * nchA]
    Word* taskw;            // [B * kTaskWords]
    Word* recw;             // [B * nS * kRecWords]
    Word* groupw;           // [B * nS * kGroups * kGroupWords]
    Word* remw;             // [B * kMaxRemoved] removed tokens of a tree draw: 0x80000000 << 32 | token
    Word* pathw;            // [B * kMaxRemoved] accepted path of a sampled tree: (0x80000000 | node) << 32 | token
    uint32_t* seqstate;     // [B] who writes a sampled sequence's outputs: 0 open, 1 its find, 2 failed (a wait
                            // on the sequence gave up); claimed by compare-and-swap
    uint32_t* order;        // [B] slot order: the decision-order queue, entry p = b + 1 of the p-th decided
                            // sequence (0: not yet; kOrderLost: a claimer gave up waiting for it)
    const int32_t* parents; // token trees: parent node of each non-root node (nullptr: linear drafts)
    int32_t* out_path;      // token trees: the accepted nodes (nullable)
    Counters* ctr;
    // fused post-verify update (spec_verify_fused); hist == nullptr: none
    int32_t* hist;
    int32_t cap;
    int32_t* lens;
    int32_t* next;
    float2 exp2_tab[128];  // 2^(j/128), j = 0..127, as (hi, lo) floats, built on the host
};

// Vocabulary-sharded verify (sv_shard.cu): one shard's view of the step.
struct ShardPartial {  // per row and shard, 16 bytes (sv_shard_partial in the C ABI)
    float m;           // raw max of the slice (NaN: a NaN or +inf logit in the slice)
    float s;           // sum over the slice of 2^((l - m) K) (sampling)
    int32_t arg;       // first argmax of the slice as a global column (-1: none)
    float g;           // the logit at the row's draft token when this shard holds that column, else 0
};
struct ShardDraw {     // per sequence, 32 bytes (sv_shard_draw in the C ABI)
    int32_t mode, n;   // kMode*, the emitting slot
    float m_p, m_q;    // merged raw maxima of the draw's target and draft rows
    float rho;         // selection ratio s_p / s_q (approximate)
    float u;           // the draw's uniform
    int32_t xcl;       // point-mass residual: the removed column (global), else -1
    int32_t pad;
};
constexpr int kMaxShards = 8;
constexpr int kShChunk = 8192;     // columns per sums record (SV_SHARD_CHUNK)
struct ShardArgs {
    const void* target;   // this shard's slice of the target rows, [R_t, Vs]
    const void* draft;    // this shard's slice of the draft rows, [R_d, Vs] (nullptr: greedy or point-mass)
    int32_t dtype;
    const int32_t* tokens;
    const int32_t* offs;
    const int32_t* gammas;
    int32_t B, V, Vs, v0, max_gamma;
    int32_t S, shard;               // shard count and this shard's index
    int32_t bounds[kMaxShards + 1]; // first column of each shard, V last
    int32_t greedy, pm;
    float K_hi, K_lo, d_min;
    uint64_t seed, step;
    int32_t* out_tokens;
    int32_t* out_n;
    uint32_t* status;
    int32_t nrows;                  // grid of the statistics kernel (an upper bound of the rows)
    int32_t nc;                     // sums records per sequence and shard: chunks of the widest shard
    cudaStream_t stream;
    float2 exp2_tab[128];
};
// Small batches: one CTA cluster per sequence (sv_small.cu). small_eligible: the call can take that path
// (sets the cluster size); launch_small: the launch.
bool small_eligible(const Params& P, int sms, int32_t* clusters);
cudaError_t launch_small(const Params& P, int dtype, int32_t clusters, cudaStream_t st);

// stage 0: statistics (a = partials of this shard); 1: decisions (a = all partials, b = draws);
// 2: sums (a = draws, b = this shard's per-chunk sums); 3: finish (a = draws, b = all shards' sums)
cudaError_t launch_shard(int stage, const ShardArgs& A, void* a, void* b, void* c);

struct Layout {
    size_t counters, partials, taskw, recw, groupw, remw, pathw, seqstate, order, status;
    size_t zero_begin, zero_end;  // byte range the launch sequence clears
    size_t total;
};

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma);

// Enqueue the whole verify step on `stream`: one memset of the zeroed regions and one cooperative
// launch.
// dtype: SV_F32 / SV_BF16; vec: rows 16-byte aligned and V * elem_size a multiple of 16.
cudaError_t launch_verify(const Params& P, const Layout& L, void* workspace, int dtype, bool vec, bool greedy,
                          cudaStream_t stream);

}  // namespace sv
