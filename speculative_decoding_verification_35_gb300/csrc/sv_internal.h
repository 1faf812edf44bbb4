// Internal interface between the C ABI (sv_api.cu) and the kernels (sv_kernels.cu).
#pragma once
#include <cstddef>
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/specverify.h"

namespace sv {

constexpr int kThreads = 256;       // threads per CTA of every kernel
constexpr int kChunk = 8192;        // vocabulary elements per statistics work item
constexpr int kSub = 512;           // vocabulary elements per sampler sub-chunk (one warp)
constexpr int kSubPerLane = kSub / 32;

enum : int32_t { kModeNone = 0, kModeResidual = 1, kModeBonus = 2 };

// Partial statistics of one (row, chunk): raw-logit max, sum of 2^((l - m) * K) in fp32,
// argmax (greedy) and error flags (bit code of sv_status).
struct Partial {
    float m;
    float s;
    int32_t arg;
    uint32_t flags;
};

// What the sampler has to draw for one sequence, written by the decision kernel.
struct SeqTask {
    int32_t mode;   // kMode*
    int32_t n;      // emitting slot
    int32_t prow;   // target row of the draw
    int32_t qrow;   // draft row of the draw (residual), -1 otherwise
    float m_p, m_q; // raw-logit row maxima
    float rho;      // approximate s_p / s_q: selects the tokens with p > q
    int32_t out_pos;// index into out_tokens of the emitting slot
    double u;       // uniform of the draw
};

// Precise sums of one sampler sub-chunk, all relative to the row maxima:
// a = sum_sel 2^{(l_p - m_p) K}, b = sum_sel 2^{(l_q - m_q) K}, p / q = the same over all tokens.
struct SubSum {
    double a, b, p, q;
};

struct Params {
    const void* target;
    const void* draft;
    const int32_t* tokens;
    const int32_t* offs;
    const int32_t* gammas;
    int32_t B, V, max_gamma;
    int32_t nchunks, nsub;
    float K_hi, K_lo;  // log2(e) / T as float-float
    double K64;        // log2(e) / T
    double invT64;     // 1 / T
    uint64_t seed, step;
    int32_t* out_tokens;
    int32_t* out_n;
    uint32_t* status;
    sv_debug dbg;
    Partial* partials;
    SeqTask* tasks;
    SubSum* subs;
    uint32_t* batch_bad;  // written by k_validate each call: nonzero when the CSR offsets are unusable
};

struct Layout {
    size_t partials, tasks, subs, status, batch_bad, total;
};

Layout workspace_layout(int32_t B, int32_t V, int32_t max_gamma);

// Enqueue the whole verify step on `stream`. dtype: SV_F32 / SV_BF16; vec: rows are 16-byte
// aligned and V * elem_size is a multiple of 16; greedy: temperature == 0.
cudaError_t launch_verify(const Params& P, int dtype, bool vec, bool greedy, cudaStream_t stream);

}  // namespace sv
