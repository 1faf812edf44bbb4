// N-gram drafter (spec_draft_ngram, declared in include/specverify.h): proposes drafts from each
// sequence's own token history, with no draft model (velog "6-1편. Speculative Decoding", §"drafter
// types", N-gram: the tokens that followed an earlier occurrence of the most recent n tokens are reused
// as the guess). Two launches on the caller's stream: a search (one CTA per sequence, the history row
// staged in shared memory), then one CTA that prefix-sums the draft lengths into CSR offsets and packs
// the drafted tokens.
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/specverify.h"

namespace sv {

constexpr int kNgThreads = 256;
constexpr int kNgMaxCap = 32768;  // history tokens staged per CTA (up to 128 KB of shared memory)

// Sequence b (CTA b): for n = n_max .. n_min, the last n tokens h[L-n .. L-1] are looked for at every
// earlier start s < L - n (the occurrence ends before the last token); the largest matching s wins, and
// the draft is h[s+n .. s+n+gamma-1] with gamma = min(gamma_max, L - (s + n)). No match: gamma 0.
__global__ void __launch_bounds__(kNgThreads) k_ngram_search(const int32_t* __restrict__ history, int32_t capacity,
                                                             const int32_t* __restrict__ lengths, int32_t n_min,
                                                             int32_t n_max, int32_t gamma_max,
                                                             int32_t* __restrict__ gammas,
                                                             int32_t* __restrict__ match_pos, uint32_t* status) {
    extern __shared__ int32_t h[];
    __shared__ int s_best;
    const int32_t b = blockIdx.x;
    int32_t L = lengths[b];
    if (L < 0 || L > capacity) {  // an inconsistent length: no draft, flagged
        if (threadIdx.x == 0) {
            gammas[b] = 0;
            match_pos[b] = L < 0 ? 0 : capacity;
            if (status) atomicOr(status, 1u << SV_ERR_INVALID_ARG);
        }
        return;
    }
    const int32_t* row = history + (size_t)b * (size_t)capacity;
    for (int32_t k = threadIdx.x; k < L; k += kNgThreads) h[k] = row[k];
    __syncthreads();
    int32_t gamma = 0, pos = L;
    for (int32_t n = n_max; n >= n_min && gamma == 0 && gamma_max > 0; --n) {
        if (L < n + 1) continue;
        // candidates s = L - n - 1 down to 0, kNgThreads at a time; the first block with a match holds
        // the largest s
        for (int32_t top = L - n - 1; top >= 0; top -= kNgThreads) {
            if (threadIdx.x == 0) s_best = -1;
            __syncthreads();
            const int32_t s = top - (int32_t)threadIdx.x;
            if (s >= 0) {
                bool eq = true;
                for (int32_t j = 0; j < n && eq; ++j) eq = h[s + j] == h[L - n + j];
                if (eq) atomicMax(&s_best, s);
            }
            __syncthreads();
            const int best = s_best;
            __syncthreads();
            if (best >= 0) {
                pos = best + n;
                gamma = min(gamma_max, L - pos);
                break;
            }
        }
    }
    if (threadIdx.x == 0) {
        gammas[b] = gamma;
        match_pos[b] = pos;
    }
}

// One CTA: seq_offsets = prefix sums of gammas (block scan over chunks of kNgThreads sequences), then
// draft_tokens[seq_offsets[b] + j] = history[b * capacity + match_pos[b] + j], j < gammas[b].
__global__ void __launch_bounds__(kNgThreads) k_ngram_pack(const int32_t* __restrict__ history, int32_t capacity,
                                                           int32_t B, const int32_t* __restrict__ gammas,
                                                           const int32_t* __restrict__ match_pos,
                                                           int32_t* __restrict__ seq_offsets,
                                                           int32_t* __restrict__ draft_tokens) {
    __shared__ int32_t scan[kNgThreads];
    __shared__ int32_t carry;
    if (threadIdx.x == 0) {
        carry = 0;
        seq_offsets[0] = 0;
    }
    __syncthreads();
    for (int32_t b0 = 0; b0 < B; b0 += kNgThreads) {
        const int32_t b = b0 + (int32_t)threadIdx.x;
        const int32_t g = b < B ? gammas[b] : 0;
        scan[threadIdx.x] = g;
        __syncthreads();
        for (int o = 1; o < kNgThreads; o <<= 1) {  // inclusive Hillis-Steele scan
            const int32_t v = threadIdx.x >= (unsigned)o ? scan[threadIdx.x - o] : 0;
            __syncthreads();
            scan[threadIdx.x] += v;
            __syncthreads();
        }
        const int32_t end = carry + scan[threadIdx.x], start = end - g;
        if (b < B) {
            seq_offsets[b + 1] = end;
            const int32_t* src = history + (size_t)b * (size_t)capacity + match_pos[b];
            for (int32_t j = 0; j < g; ++j) draft_tokens[start + j] = src[j];
        }
        __syncthreads();
        if (threadIdx.x == kNgThreads - 1) carry = end;
        __syncthreads();
    }
}

}  // namespace sv

extern "C" int spec_draft_ngram(const int32_t* history, int32_t capacity, const int32_t* lengths, int32_t B,
                                int32_t n_min, int32_t n_max, int32_t gamma_max, int32_t* draft_tokens,
                                int32_t* gammas, int32_t* seq_offsets, int32_t* match_pos, uint32_t* device_status,
                                void* cuda_stream) {
    if (B < 0 || capacity < 1 || capacity > sv::kNgMaxCap || n_min < 1 || n_max < n_min || gamma_max < 0 ||
        gamma_max > SV_MAX_GAMMA)
        return SV_ERR_INVALID_ARG;
    if (!seq_offsets || (uintptr_t)seq_offsets % 4) return SV_ERR_INVALID_ARG;
    if (B > 0) {
        const void* ptrs[] = {history, lengths, draft_tokens, gammas, match_pos};
        for (const void* p : ptrs)
            if (!p || (uintptr_t)p % 4) return SV_ERR_INVALID_ARG;
    }
    if (device_status && (uintptr_t)device_status % 4) return SV_ERR_INVALID_ARG;
    const cudaStream_t st = (cudaStream_t)cuda_stream;
    const size_t smem = (size_t)capacity * sizeof(int32_t);
    if (smem > 40 * 1024 &&  // near or above the default 48 KB limit (with the static bytes): opt in
        cudaFuncSetAttribute(sv::k_ngram_search, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
        return SV_ERR_CUDA;
    if (B > 0)
        sv::k_ngram_search<<<B, sv::kNgThreads, smem, st>>>(
            history, capacity, lengths, n_min, n_max, gamma_max, gammas, match_pos, device_status);
    sv::k_ngram_pack<<<1, sv::kNgThreads, 0, st>>>(history, capacity, B, gammas, match_pos, seq_offsets, draft_tokens);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
