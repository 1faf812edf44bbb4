// Test helper (GPU): evaluates the library's device Philox4x32-10 and curand's
// curand_Philox4x32_10(counter, key) on the same inputs, so a test can compare them word for word.
#include <cstdint>
#include <cuda_runtime.h>
#include <curand_kernel.h>

#include "../../speculative_decoding_verification_35_gb300/csrc/sv_device.cuh"

__global__ void k_philox_both(int n, const uint4* ctr, const uint2* key, uint4* ours, uint4* ref) {
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= n) return;
    ours[i] = sv::philox4x32_10(ctr[i], key[i]);
    ref[i] = curand_Philox4x32_10(ctr[i], key[i]);
}

extern "C" int philox_check(int n, const uint32_t* ctr, const uint32_t* key, uint32_t* ours, uint32_t* ref) {
    uint4 *dc = nullptr, *d_o = nullptr, *d_r = nullptr;
    uint2* dk = nullptr;
    const size_t n4 = sizeof(uint4) * (size_t)n, n2 = sizeof(uint2) * (size_t)n;
    if (cudaMalloc(&dc, n4) || cudaMalloc(&dk, n2) || cudaMalloc(&d_o, n4) || cudaMalloc(&d_r, n4)) return 1;
    cudaMemcpy(dc, ctr, n4, cudaMemcpyHostToDevice);
    cudaMemcpy(dk, key, n2, cudaMemcpyHostToDevice);
    k_philox_both<<<(n + 255) / 256, 256>>>(n, dc, dk, d_o, d_r);
    int rc = cudaDeviceSynchronize() != cudaSuccess;
    cudaMemcpy(ours, d_o, n4, cudaMemcpyDeviceToHost);
    cudaMemcpy(ref, d_r, n4, cudaMemcpyDeviceToHost);
    cudaFree(dc); cudaFree(dk); cudaFree(d_o); cudaFree(d_r);
    return rc;
}
