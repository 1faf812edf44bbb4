// spec_verify_noalloc: the verify step for callers that cannot allocate device memory.
//
// Some callers may not call cudaMalloc at all: code that runs inside a CUDA stream capture it does
// not own, allocator-less runtimes, or hooks invoked where a hidden device allocation (and the
// synchronisation it can imply) is not allowed. For them this entry point runs the same kernel as
// spec_verify_ex, with its scratch taken from one fixed array compiled into the library instead of a
// caller-provided workspace. It allocates nothing and frees nothing.
#include <atomic>
#include <cstdint>

#include "sv_internal.h"

namespace {

// Fixed scratch: 8 MiB, enough for every batch with spec_verify_workspace_size(B, V, max_gamma) up to
// that size. Every GPU that loads the library keeps this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of the array, per device. The host-side name `g_noalloc_scratch` is only a
// stand-in; the address a kernel may use comes from cudaGetSymbolAddress with that device current.
constexpr int kMaxDevices = 64;
std::atomic<void*> g_scratch_addr[kMaxDevices];

}  // namespace

extern "C" int spec_verify_noalloc(const void* target_logits, const void* draft_logits, sv_dtype dtype,
                                   const int32_t* draft_tokens, const int32_t* seq_offsets,
                                   const int32_t* gammas, int32_t B, int32_t V, int32_t max_gamma,
                                   float temperature, uint64_t seed, uint64_t step, int32_t* out_tokens,
                                   int32_t* out_num_accepted, uint32_t* device_status,
                                   const sv_debug* debug, void* cuda_stream) {
    if (B < 0 || V < 1 || max_gamma < 0 || max_gamma > SV_MAX_GAMMA) return SV_ERR_INVALID_ARG;
    const size_t need = spec_verify_workspace_size(B, V, max_gamma);
    if (need > kNoAllocScratchBytes) return SV_ERR_WORKSPACE;  // batch too large for the fixed scratch
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SV_ERR_CUDA;
    void* scratch = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (!scratch) {
        // first call on this device: look up the array's device address once
        if (cudaGetSymbolAddress(&scratch, g_noalloc_scratch) != cudaSuccess || !scratch) return SV_ERR_CUDA;
        g_scratch_addr[dev].store(scratch, std::memory_order_release);
    }
    return spec_verify_ex(target_logits, draft_logits, dtype, draft_tokens, seq_offsets, gammas, B, V,
                          max_gamma, temperature, seed, step, out_tokens, out_num_accepted, device_status,
                          scratch, kNoAllocScratchBytes, debug, cuda_stream);
}
