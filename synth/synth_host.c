/*
 * Host fill routines for the seeded synthetic-input generator (ds4g_synth.h).
 * Element i of a fill is element (index0 + i) of the tensor stream, so any
 * slice of a tensor can be regenerated without the rest.
 */
#include <stddef.h>
#include <stdint.h>
#include "ds4g_synth.h"

void synth_fill_f32(float *dst, size_t n, uint64_t seed, uint64_t tensor_id,
                    float scale, float offset, uint64_t index0)
{
    uint64_t key = syn_key(seed, tensor_id);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; i++)
        dst[i] = offset + syn_value(key, index0 + (uint64_t)i, scale);
}

void synth_fill_bf16(uint16_t *dst, size_t n, uint64_t seed, uint64_t tensor_id,
                     float scale, uint64_t index0)
{
    uint64_t key = syn_key(seed, tensor_id);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; i++)
        dst[i] = syn_to_bf16(syn_value(key, index0 + (uint64_t)i, scale));
}

void synth_fill_f16(uint16_t *dst, size_t n, uint64_t seed, uint64_t tensor_id,
                    float scale, uint64_t index0)
{
    uint64_t key = syn_key(seed, tensor_id);
    #pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < (int64_t)n; i++)
        dst[i] = syn_to_f16(syn_value(key, index0 + (uint64_t)i, scale));
}

void synth_fill_tokens(int32_t *dst, size_t n, uint64_t seed, uint64_t tensor_id,
                       uint32_t vocab, uint64_t index0)
{
    uint64_t key = syn_key(seed, tensor_id);
    for (size_t i = 0; i < n; i++)
        dst[i] = syn_token(key, index0 + (uint64_t)i, vocab);
}

/* Conversion helpers exposed for the generator's own tests. */
uint16_t synth_f32_to_bf16(float f) { return syn_to_bf16(f); }
uint16_t synth_f32_to_f16(float f) { return syn_to_f16(f); }
int32_t synth_ih4(uint64_t seed, uint64_t tensor_id, uint64_t index)
{
    return syn_ih4(syn_hash(syn_key(seed, tensor_id), index));
}
