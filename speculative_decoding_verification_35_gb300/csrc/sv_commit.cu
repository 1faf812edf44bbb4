// Post-verify update (spec_verify_commit, declared in include/specverify.h): appends each sequence's
// emitted tokens to its device-side history and sets its next input token, on the stream of the verify
// call, with no host synchronisation ("Accelerating Sonar through speculation", §"MTP scheduling").
#include <cstdint>

#include <cuda_runtime.h>

#include "../../include/specverify.h"

namespace sv {

// One warp per sequence (grid-strided); lane j copies slot j (n + 1 <= 32 slots, as gamma <= 31).
__global__ void __launch_bounds__(256) k_commit(const int32_t* __restrict__ out_tokens,
                                                const int32_t* __restrict__ out_n,
                                                const int32_t* __restrict__ offs, int32_t B,
                                                int32_t* __restrict__ history, int32_t capacity,
                                                int32_t* __restrict__ lengths, int32_t* __restrict__ next_tokens,
                                                uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const int32_t warps = (int32_t)(gridDim.x * (blockDim.x >> 5));
    for (int32_t b = (int32_t)(blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)); b < B; b += warps) {
        const int32_t n = out_n[b];
        const int32_t o0 = offs[b], g = offs[b + 1] - o0;
        const int32_t L = lengths[b];
        uint32_t err = 0;
        // n above the sequence's gap, or above the largest gamma a verify call writes (lanes 0..31 copy
        // the slots), means the outputs are not a verify call's: nothing is appended
        if (n >= 0 && (n > g || n > SV_MAX_GAMMA || o0 < 0)) err = 1u << SV_ERR_BAD_OFFSETS;
        else if (n >= 0 && (L < 0 || (int64_t)L + n + 1 > capacity)) err = 1u << SV_ERR_CAPACITY;
        if (n < 0 || err) {
            if (lane == 0) {
                next_tokens[b] = -1;
                if (err && status) atomicOr(status, err);
            }
            continue;
        }
        const int32_t t0 = o0 + b;
        if (lane <= n) history[(size_t)b * (size_t)capacity + (size_t)(L + lane)] = out_tokens[t0 + lane];
        if (lane == 0) {
            lengths[b] = L + n + 1;
            next_tokens[b] = out_tokens[t0 + n];
        }
    }
}

}  // namespace sv

extern "C" int spec_verify_commit(const int32_t* out_tokens, const int32_t* out_num_accepted,
                                  const int32_t* seq_offsets, int32_t B, int32_t* history, int32_t capacity,
                                  int32_t* lengths, int32_t* next_tokens, uint32_t* device_status,
                                  void* cuda_stream) {
    if (B < 0 || capacity < 1) return SV_ERR_INVALID_ARG;
    if (B == 0) return SV_OK;
    const void* ptrs[] = {out_tokens, out_num_accepted, seq_offsets, history, lengths, next_tokens};
    for (const void* p : ptrs)
        if (!p || (uintptr_t)p % 4) return SV_ERR_INVALID_ARG;
    if (device_status && (uintptr_t)device_status % 4) return SV_ERR_INVALID_ARG;
    const int warps_per_cta = 8;
    int32_t grid = (B + warps_per_cta - 1) / warps_per_cta;
    if (grid > 4096) grid = 4096;
    sv::k_commit<<<grid, 32 * warps_per_cta, 0, (cudaStream_t)cuda_stream>>>(
        out_tokens, out_num_accepted, seq_offsets, B, history, capacity, lengths, next_tokens, device_status);
    return cudaGetLastError() == cudaSuccess ? SV_OK : SV_ERR_CUDA;
}
