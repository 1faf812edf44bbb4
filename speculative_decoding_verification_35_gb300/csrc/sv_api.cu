// C ABI of libspecverify (declared in include/specverify.h): host-side validation, workspace layout
// and the launch of the verify step on the caller's stream.
#include <algorithm>
#include <cmath>
#include <cstdint>
#include <vector>

#include "sv_internal.h"

using namespace sv;

extern "C" {

size_t spec_verify_workspace_size(int32_t B, int32_t V, int32_t max_gamma) {
    if (B < 0 || V < 1 || max_gamma < 0 || max_gamma > SV_MAX_GAMMA) return 0;
    return workspace_layout(B, V, max_gamma).total;
}

int spec_verify_status_from_bits(uint32_t bits) {
    static const int order[] = {SV_ERR_BAD_OFFSETS, SV_ERR_BAD_TOKEN, SV_ERR_NONFINITE, SV_ERR_EMPTY_ROW,
                                SV_ERR_TIMEOUT, SV_ERR_CAPACITY};
    for (int c : order)
        if (bits & (1u << c)) return c;
    for (int c = 1; c < 32; ++c)
        if (bits & (1u << c)) return c;
    return SV_OK;
}

const char* spec_verify_status_string(int status) {
    switch (status) {
        case SV_OK: return "SV_OK";
        case SV_ERR_INVALID_ARG: return "SV_ERR_INVALID_ARG: bad scalar, NULL or misaligned pointer, or unsupported size";
        case SV_ERR_CUDA: return "SV_ERR_CUDA: a CUDA call or kernel launch failed";
        case SV_ERR_BAD_TOKEN: return "SV_ERR_BAD_TOKEN: a draft token lies outside [0, V)";
        case SV_ERR_BAD_OFFSETS: return "SV_ERR_BAD_OFFSETS: seq_offsets / gammas inconsistent or gamma above max_gamma";
        case SV_ERR_NONFINITE: return "SV_ERR_NONFINITE: NaN or +inf logit";
        case SV_ERR_EMPTY_ROW: return "SV_ERR_EMPTY_ROW: a row whose logits are all -inf";
        case SV_ERR_TIMEOUT: return "SV_ERR_TIMEOUT: a bounded device wait gave up";
        case SV_ERR_WORKSPACE: return "SV_ERR_WORKSPACE: workspace missing, too small or not 256-byte aligned";
        case SV_ERR_CAPACITY: return "SV_ERR_CAPACITY: a sequence's token history would overflow its capacity";
        default: return "unknown status";
    }
}

}  // extern "C"

namespace {
struct CommitBufs {
    int32_t* history;
    int32_t capacity;
    int32_t* lengths;
    int32_t* next_tokens;
};

int verify_impl(const void* target_logits, const void* draft_logits, sv_dtype dtype, const int32_t* draft_tokens,
                const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t max_gamma,
                float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                uint32_t* device_status, void* workspace, size_t workspace_bytes, const sv_debug* debug,
                const CommitBufs* commit, const int32_t* parents, int32_t* out_path, void* cuda_stream,
                bool validate_only = false, uint32_t seq_base = 0) {
    if (B < 0 || V < 1 || max_gamma < 0 || max_gamma > SV_MAX_GAMMA) return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (!(temperature >= 0.f) || !std::isfinite(temperature)) return SV_ERR_INVALID_ARG;
    const bool greedy = temperature == 0.f;
    const double K64 = greedy ? 0.0 : 1.4426950408889634074 / (double)temperature;
    const float K_hi = (float)K64;
    if (!greedy && !std::isfinite(K_hi)) return SV_ERR_INVALID_ARG;
    if (!target_logits || !seq_offsets || !gammas || !out_tokens || !out_num_accepted) return SV_ERR_INVALID_ARG;
    if (max_gamma > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;  // no draft logits: point-mass drafts
    const size_t esz = dtype == SV_BF16 ? 2 : 4;
    if ((uintptr_t)target_logits % esz || (draft_logits && (uintptr_t)draft_logits % esz)) return SV_ERR_INVALID_ARG;
    if ((uintptr_t)seq_offsets % 4 || (uintptr_t)gammas % 4 || (uintptr_t)out_tokens % 4 ||
        (uintptr_t)out_num_accepted % 4 || (draft_tokens && (uintptr_t)draft_tokens % 4))
        return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    // task indices are 32-bit on the device: statistics tasks and tickets stay below 2^31
    const uint64_t nchA = ((uint64_t)V + kAChunk - 1) / kAChunk, nS = ((uint64_t)V + kSTask - 1) / kSTask;
    if ((uint64_t)B * (2 * (uint64_t)max_gamma + 1) * nchA >= (1ull << 31) || (uint64_t)B * (nS + 1) >= (1ull << 31))
        return SV_ERR_INVALID_ARG;
    const Layout L = workspace_layout(B, V, max_gamma);
    if (!workspace || workspace_bytes < L.total || (uintptr_t)workspace % 256) return SV_ERR_WORKSPACE;
    if (validate_only) return SV_OK;

    const bool uses_draft = !greedy && max_gamma > 0 && draft_logits;
    const bool vec = (uintptr_t)target_logits % 16 == 0 && (!uses_draft || (uintptr_t)draft_logits % 16 == 0) &&
                     ((size_t)V * esz) % 16 == 0;
    char* ws = (char*)workspace;
    Params P{};
    P.target = target_logits;
    P.draft = draft_logits;
    P.tokens = draft_tokens;
    P.offs = seq_offsets;
    P.gammas = gammas;
    P.B = B;
    P.V = V;
    P.max_gamma = max_gamma;
    P.pm = !greedy && !draft_logits;
    P.nchA = (V + kAChunk - 1) / kAChunk;
    P.nS = (V + kSTask - 1) / kSTask;
    P.nS_recip = P.nS >= 2 ? ~0ull / (unsigned long long)P.nS + 1ull : 0ull;
    P.K_hi = K_hi;
    P.K_lo = (float)(K64 - (double)K_hi);
    P.d_min = greedy ? 0.f : (float)(-126.5 / (double)K_hi);
    // The sampler's value table serves a draw whose rows' maxima m make its two stand-ins negligible and
    // keep its sums finite: m <= 63.75 (no logit above the table), m >= -63.75 + 60 / K (every logit at
    // or below -63.75, taken as weight 0, lies 2^60 below the row's largest weight) and m K <= 96 (sums of
    // up to 2^31 weights of at most 2^96 stay finite).
    P.use_tab = !greedy && (int64_t)B * P.nS >= kTabMinTasks;
    P.tab_mlo = greedy ? 1.f : (float)(-63.75 + 60.0 / (double)K_hi);
    P.tab_mhi = greedy ? 0.f : (float)std::min(63.75, 96.0 / (double)K_hi);
    {
        // Slot order pays where drafts have their own rows (their acceptance varies) and the statistics
        // stream is long enough for early decisions to overlap it. Measured per step: B = 64, gamma = 5,
        // V = 128256 (22528 statistics tasks): 54.3 against 55.2 us; B = 8, V = 32000 (576 tasks, streamed
        // in ~3 us): 24.6 against 23.1 us, so small batches keep sequence order (kProgMinTasks); point-mass
        // batches, whose planted drafts are mostly accepted, also measured faster in sequence order (37.6
        // against 39.2 us at the headline size).
        const bool row_dbg = debug && (debug->row_lse || debug->row_argmax || debug->p_x || debug->q_x || debug->beta);
        const int64_t rows = (int64_t)B * (2 * (int64_t)max_gamma + 1);
        const uint32_t order = debug ? debug->order : 0u;
        P.prog = !greedy && !P.pm && dtype == SV_BF16 && vec && !parents && !row_dbg && B < kBaseCache &&
                 rows <= kRowCache && order != 1u && (order == 2u || rows * P.nchA >= kProgMinTasks);
    }
    P.invT64 = greedy ? 0.0 : 1.0 / (double)temperature;
    P.seed = seed;
    P.step = step;
    P.seq_base = seq_base;
    P.out_tokens = out_tokens;
    P.out_n = out_num_accepted;
    P.status = device_status ? device_status : (uint32_t*)(ws + L.status);
    if (debug) P.dbg = *debug;
    P.spin = debug && debug->spin_limit ? debug->spin_limit : kSpinLimit;
    for (int j = 0; j < 128; ++j) {  // Tang's table: 2^(j/128) as a float pair (hi, lo)
        const double v = std::exp2((double)j / 128.0);
        const float hi = (float)v;
        P.exp2_tab[j] = make_float2(hi, (float)(v - (double)hi));
    }
    P.partials = (PartialWord*)(ws + L.partials);
    P.taskw = (Word*)(ws + L.taskw);
    P.recw = (Word*)(ws + L.recw);
    P.groupw = (Word*)(ws + L.groupw);
    P.remw = (Word*)(ws + L.remw);
    P.pathw = (Word*)(ws + L.pathw);
    P.seqstate = (uint32_t*)(ws + L.seqstate);
    P.order = (uint32_t*)(ws + L.order);
    P.ctr = (Counters*)(ws + L.counters);
    P.parents = parents;
    P.out_path = out_path;
    if (commit) {
        P.hist = commit->history;
        P.cap = commit->capacity;
        P.lens = commit->lengths;
        P.next = commit->next_tokens;
    }
    const cudaError_t e = launch_verify(P, L, workspace, (int)dtype, vec, greedy, (cudaStream_t)cuda_stream);
    return e == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
}  // namespace

extern "C" {

int spec_verify_ex(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                   const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                   int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed,
                   uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                   uint32_t* device_status, void* workspace, size_t workspace_bytes,
                   const sv_debug* debug, void* cuda_stream) {
    return verify_impl(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                       temperature, seed, step, out_tokens, out_num_accepted, device_status, workspace,
                       workspace_bytes, debug, nullptr, nullptr, nullptr, cuda_stream);
}

int spec_verify_range(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                      int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed,
                      uint64_t step, uint32_t seq_base, int32_t* out_tokens, int32_t* out_num_accepted,
                      uint32_t* device_status, void* workspace, size_t workspace_bytes,
                      const sv_debug* debug, void* cuda_stream) {
    return verify_impl(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                       temperature, seed, step, out_tokens, out_num_accepted, device_status, workspace,
                       workspace_bytes, debug, nullptr, nullptr, nullptr, cuda_stream, false, seq_base);
}

int spec_verify_fused(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                      const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas,
                      int32_t B, int32_t V, int32_t max_gamma, float temperature, uint64_t seed, uint64_t step,
                      int32_t* out_tokens, int32_t* out_num_accepted, uint32_t* device_status, void* workspace,
                      size_t workspace_bytes, int32_t* history, int32_t capacity, int32_t* lengths,
                      int32_t* next_tokens, void* cuda_stream) {
    if (capacity < 1) return SV_ERR_INVALID_ARG;
    if (B > 0) {
        const void* ptrs[] = {history, lengths, next_tokens};
        for (const void* p : ptrs)
            if (!p || (uintptr_t)p % 4) return SV_ERR_INVALID_ARG;
        if (max_gamma > 0 && !draft_tokens) return SV_ERR_INVALID_ARG;  // the appended drafts
    }
    const CommitBufs c{history, capacity, lengths, next_tokens};
    return verify_impl(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                       temperature, seed, step, out_tokens, out_num_accepted, device_status, workspace,
                       workspace_bytes, nullptr, &c, nullptr, nullptr, cuda_stream);
}

int spec_verify_tree(const void* target_logits, sv_dtype dtype, const int32_t* draft_tokens, const int32_t* parents,
                     const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, int32_t max_gamma,
                     float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted,
                     int32_t* out_path, uint32_t* device_status, void* workspace, size_t workspace_bytes,
                     void* cuda_stream) {
    if (max_gamma > 0 && (!parents || (uintptr_t)parents % 4)) return SV_ERR_INVALID_ARG;
    if (out_path && (uintptr_t)out_path % 4) return SV_ERR_INVALID_ARG;
    // max_gamma 0: every tree is a root alone, which the linear path handles identically (a draw from p)
    return verify_impl(target_logits, nullptr, dtype, draft_tokens, seq_offsets, gammas, B, V, max_gamma,
                       temperature, seed, step, out_tokens, out_num_accepted, device_status, workspace,
                       workspace_bytes, nullptr, nullptr, max_gamma > 0 ? parents : nullptr, out_path, cuda_stream);
}

int spec_verify_host(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                     const int32_t* draft_tokens, const int32_t* seq_offsets, const int32_t* gammas, int32_t B,
                     int32_t V, int32_t max_gamma, float temperature, uint64_t seed, uint64_t step,
                     int32_t* out_tokens, int32_t* out_num_accepted, const sv_device_buffers* dev,
                     uint32_t* device_status, void* workspace, size_t workspace_bytes, void* cuda_stream) {
    if (!dev || B < 0 || V < 1 || max_gamma < 0 || max_gamma > SV_MAX_GAMMA || (B > 0 && !seq_offsets))
        return SV_ERR_INVALID_ARG;
    if (dtype != SV_F32 && dtype != SV_BF16) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    // the draft rows, from the host copy of the offsets (the device re-checks the whole structure)
    const int64_t R_d = seq_offsets[B];
    if (R_d < 0 || R_d > (int64_t)B * max_gamma) return SV_ERR_INVALID_ARG;
    const int64_t R_t = R_d + B;
    const bool with_draft = draft_logits != nullptr;
    const bool with_tokens = draft_tokens != nullptr;
    if (!target_logits || !gammas || !out_tokens || !out_num_accepted || (with_draft && !dev->draft_logits) ||
        (with_tokens && !dev->draft_tokens))
        return SV_ERR_INVALID_ARG;
    // every argument check of the step, on the staging buffers, before anything is enqueued
    const int rc = verify_impl(dev->target_logits, with_draft ? dev->draft_logits : nullptr, dtype,
                               with_tokens ? dev->draft_tokens : nullptr, dev->seq_offsets, dev->gammas, B, V,
                               max_gamma, temperature, seed, step, dev->out_tokens, dev->out_num_accepted,
                               device_status, workspace, workspace_bytes, nullptr, nullptr, nullptr, nullptr,
                               cuda_stream, true);
    if (rc != SV_OK) return rc;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    const size_t esz = dtype == SV_BF16 ? 2 : 4;
    auto h2d = [&](void* d, const void* h, size_t bytes) {
        return bytes == 0 || cudaMemcpyAsync(d, h, bytes, cudaMemcpyHostToDevice, st) == cudaSuccess;
    };
    if (!h2d(dev->target_logits, target_logits, (size_t)R_t * (size_t)V * esz) ||
        (with_draft && !h2d(dev->draft_logits, draft_logits, (size_t)R_d * (size_t)V * esz)) ||
        (with_tokens && !h2d(dev->draft_tokens, draft_tokens, (size_t)R_d * sizeof(int32_t))) ||
        !h2d(dev->seq_offsets, seq_offsets, (size_t)(B + 1) * sizeof(int32_t)) ||
        !h2d(dev->gammas, gammas, (size_t)B * sizeof(int32_t)))
        return SV_ERR_CUDA;
    const int r2 = verify_impl(dev->target_logits, with_draft ? dev->draft_logits : nullptr, dtype,
                               with_tokens ? dev->draft_tokens : nullptr, dev->seq_offsets, dev->gammas, B, V,
                               max_gamma, temperature, seed, step, dev->out_tokens, dev->out_num_accepted,
                               device_status, workspace, workspace_bytes, nullptr, nullptr, nullptr, nullptr,
                               cuda_stream);
    if (r2 != SV_OK) return r2;
    if (cudaMemcpyAsync(out_tokens, dev->out_tokens, (size_t)R_t * sizeof(int32_t), cudaMemcpyDeviceToHost, st) !=
            cudaSuccess ||
        cudaMemcpyAsync(out_num_accepted, dev->out_num_accepted, (size_t)B * sizeof(int32_t), cudaMemcpyDeviceToHost,
                        st) != cudaSuccess)
        return SV_ERR_CUDA;
    return SV_OK;
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                const int32_t* seq_offsets, const int32_t* gammas, int32_t B, int32_t V, float temperature,
                uint64_t seed, uint64_t step, int32_t* out_tokens, int32_t* out_num_accepted) {
    if (B < 0 || !gammas) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    std::vector<int32_t> g((size_t)B);
    if (cudaMemcpy(g.data(), gammas, sizeof(int32_t) * (size_t)B, cudaMemcpyDeviceToHost) != cudaSuccess)
        return SV_ERR_CUDA;
    int32_t max_gamma = 0;
    for (int32_t v : g) {
        if (v < 0 || v > SV_MAX_GAMMA) return SV_ERR_INVALID_ARG;
        max_gamma = std::max(max_gamma, v);
    }
    const size_t need = spec_verify_workspace_size(B, V, max_gamma);
    if (!need) return SV_ERR_INVALID_ARG;
    void* ws = nullptr;
    uint32_t* st = nullptr;
    if (cudaMalloc(&ws, need) != cudaSuccess) return SV_ERR_CUDA;
    if (cudaMalloc((void**)&st, sizeof(uint32_t)) != cudaSuccess) {
        cudaFree(ws);
        return SV_ERR_CUDA;
    }
    int rc = SV_OK;
    uint32_t bits = 0;
    if (cudaMemsetAsync(st, 0, sizeof(uint32_t), 0) != cudaSuccess) rc = SV_ERR_CUDA;
    if (rc == SV_OK)
        rc = spec_verify_ex(target_logits, draft_logits, SV_BF16, draft_tokens, seq_offsets, gammas, B, V,
                            max_gamma, temperature, seed, step, out_tokens, out_num_accepted, st, ws, need,
                            nullptr, nullptr);
    if (rc == SV_OK && (cudaStreamSynchronize(0) != cudaSuccess ||
                        cudaMemcpy(&bits, st, sizeof(uint32_t), cudaMemcpyDeviceToHost) != cudaSuccess))
        rc = SV_ERR_CUDA;
    cudaFree(st);
    cudaFree(ws);
    if (rc != SV_OK) return rc;
    return spec_verify_status_from_bits(bits);
}

}  // extern "C"
