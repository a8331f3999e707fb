/*
 * Device fill routines for the seeded synthetic-input generator
 * (ds4g_synth.h): bit-identical to synth_host.c for the same arguments.
 * Used by the tests and the benchmark to fill caller-owned device buffers.
 */
#include <cuda_runtime.h>
#include <stdint.h>
#include "ds4g_synth.h"

enum { FMT_F32 = 0, FMT_BF16 = 1, FMT_F16 = 2, FMT_TOKENS = 3 };

__global__ void synth_fill_kernel(void *dst, int fmt, size_t n, uint64_t key, float scale,
                                  float offset, uint64_t index0, uint32_t vocab)
{
    size_t stride = (size_t)gridDim.x * blockDim.x;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        uint64_t idx = index0 + (uint64_t)i;
        switch (fmt) {
        case FMT_F32:
            ((float *)dst)[i] = offset + syn_value(key, idx, scale);
            break;
        case FMT_BF16:
            ((uint16_t *)dst)[i] = syn_to_bf16(syn_value(key, idx, scale));
            break;
        case FMT_F16:
            ((uint16_t *)dst)[i] = syn_to_f16(syn_value(key, idx, scale));
            break;
        default:
            ((int32_t *)dst)[i] = syn_token(key, idx, vocab);
            break;
        }
    }
}

/* Returns 0 on success, or the CUDA error code of the launch. */
extern "C" int synth_fill_dev(void *dst, int fmt, size_t n, uint64_t seed, uint64_t tensor_id,
                              float scale, float offset, uint64_t index0, uint32_t vocab,
                              void *stream)
{
    if (n == 0) return 0;
    if (fmt < FMT_F32 || fmt > FMT_TOKENS || dst == nullptr) return (int)cudaErrorInvalidValue;
    int blocks = (int)((n + 255) / 256);
    if (blocks > 152 * 32) blocks = 152 * 32;
    synth_fill_kernel<<<blocks, 256, 0, (cudaStream_t)stream>>>(
        dst, fmt, n, syn_key(seed, tensor_id), scale, offset, index0, vocab);
    return (int)cudaGetLastError();
}
