// Internal interface between the C ABI (sv_api.cu) and the verify kernel (sv_kernels.cu).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/specverify.h"

namespace sv {

constexpr int kThreads = 256;               // threads per CTA
constexpr int kWarps = kThreads / 32;       // independent warp workers per CTA
constexpr int kAChunk = 4096;               // vocabulary columns of one statistics task (one warp, one row)
constexpr int kSub = 512;                   // sampler sub-chunk: the finest unit of the inverse-CDF search
constexpr int kSubPerLane = kSub / 32;      // 16 consecutive columns per lane
constexpr int kSTask = 1024;                // vocabulary columns of one sampler task (one warp)
constexpr int kSubPerTask = kSTask / kSub;  // 2
constexpr int kStreamWarps = 4;             // statistics streamers per CTA on the bulk-copy path
constexpr int kStages = 3;                  // bulk-copy stages per streamer
constexpr int kStageBytes = kAChunk * 2;    // one bf16 statistics task
constexpr int kTmaSmemBytes = kStreamWarps * kStages * (kStageBytes + 8);
constexpr int kFlagStride = 32;             // ready flags one per 128-byte line (words)
constexpr int kBaseCache = 1024;            // batches up to this size keep their row bases in shared memory

enum : int32_t { kModeNone = 0, kModeResidual = 1, kModeBonus = 2 };

// Partial statistics of one (row, chunk), one 64-bit word written with a single store. The region is
// zeroed before every call and a written word is never 0, so readers poll the word itself:
//   sampling: low = bits(raw max m), high = bits(sum of 2^((l - m) K)) (m = +0 implies sum >= 1;
//             sum = 0 implies m = -inf; a NaN or +inf logit makes the sum NaN);
//   greedy:   low = bits(m), high = (first argmax + 1) | (1 << 31 if a NaN was seen).
typedef unsigned long long PartialWord;

// What the sampler draws for one sequence, written by the decision step. 48 bytes, 16-byte
// aligned: readers fetch it with 16-byte loads.
struct alignas(16) SeqTask {
    int32_t mode;    // kMode*
    int32_t n;       // emitting slot
    int32_t prow;    // target row of the draw
    int32_t qrow;    // draft row of the draw (residual), -1 otherwise
    float m_p, m_q;  // raw-logit row maxima
    float rho;       // approximate s_p / s_q: selects the tokens with p > q
    int32_t out_pos; // index into out_tokens of the emitting slot
    double u;        // uniform of the draw
    int32_t pad[2];
};

// Counters of one call (zeroed before the kernel by the launch sequence).
struct Counters {
    uint32_t claim;  // sampler tasks claimed, in sequence order
    uint32_t pad[31];
};

struct Params {
    const void* target;
    const void* draft;
    const int32_t* tokens;
    const int32_t* offs;
    const int32_t* gammas;
    int32_t B, V, max_gamma;
    int32_t nchA;      // statistics chunks per row
    int32_t nsub;      // sampler sub-chunks per row
    int32_t nS;        // sampler tasks per sequence
    float K_hi, K_lo;  // log2(e) / T as float-float
    double K64;        // log2(e) / T
    double invT64;     // 1 / T
    uint64_t seed, step;
    int32_t* out_tokens;
    int32_t* out_n;
    uint32_t* status;
    sv_debug dbg;
    // workspace
    PartialWord* partials;  // [B * (2 max_gamma + 1) * nchA]
    SeqTask* tasks;     // [B]
    double2* subs;      // [B * nsub]: (sum_sel 2^{(l_p-m_p)K}, sum_sel 2^{(l_q-m_q)K}) per sub-chunk
    double2* stot;      // [B * nS]: (sum_all p-weight, sum_all q-weight) per sampler task
    Counters* ctr;
    uint32_t* s_done;   // [B] sampler tasks finished per sequence
    uint32_t* seq_ready;  // [B * kFlagStride] set (release) once a sequence's sampler task record is written
};

struct Layout {
    size_t counters, s_done, seq_ready, partials, tasks, subs, stot, status;
    size_t zero_begin, zero_end;  // byte range the launch sequence clears
    size_t total;
};

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma);

// Enqueue the whole verify step on `stream`: one memset of the counters and one cooperative launch.
// dtype: SV_F32 / SV_BF16; vec: rows 16-byte aligned and V * elem_size a multiple of 16.
cudaError_t launch_verify(const Params& P, const Layout& L, void* workspace, int dtype, bool vec, bool greedy,
                          cudaStream_t stream);

}  // namespace sv
