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
constexpr int kSTask = 2048;                // vocabulary columns of one sampler task (one warp)
constexpr int kSubPerTask = kSTask / kSub;  // 4

enum : int32_t { kModeNone = 0, kModeResidual = 1, kModeBonus = 2 };

// Partial statistics of one (row, chunk): raw-logit max, sum of 2^((l - m) K) in fp32, first
// argmax (greedy) and error flags (bit codes of sv_status).
struct Partial {
    float m;
    float s;
    int32_t arg;
    uint32_t flags;
};

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
    Partial* partials;  // [B * (2 max_gamma + 1) * nchA]
    SeqTask* tasks;     // [B]
    double2* subs;      // [B * nsub]: (sum_sel 2^{(l_p-m_p)K}, sum_sel 2^{(l_q-m_q)K}) per sub-chunk
    double2* stot;      // [B * nS]: (sum_all p-weight, sum_all q-weight) per sampler task
    Counters* ctr;
    uint32_t* a_done;   // [B] statistics tasks finished per sequence
    uint32_t* s_done;   // [B] sampler tasks finished per sequence
    uint32_t* seq_ready;  // [B] set (release) once a sequence's sampler task record is written
};

struct Layout {
    size_t partials, tasks, subs, stot, counters, a_done, s_done, seq_ready, status;
    size_t zero_begin, zero_end;  // byte range the launch sequence clears
    size_t total;
};

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma);

// Enqueue the whole verify step on `stream`: one memset of the counters and one cooperative launch.
// dtype: SV_F32 / SV_BF16; vec: rows 16-byte aligned and V * elem_size a multiple of 16.
cudaError_t launch_verify(const Params& P, const Layout& L, void* workspace, int dtype, bool vec, bool greedy,
                          cudaStream_t stream);

}  // namespace sv
