/*
 * ds4g_synth.h -- seeded, counter-based generator for synthetic inputs.
 *
 * This header is the only code shared by the oracle (oracle/) and the CUDA
 * library's tests and benchmark: it produces weights, KV-cache contents, token
 * ids and logits from (seed, tensor id, element index), identically on the
 * host (C) and on the device (CUDA).  It contains none of the layer's
 * arithmetic: no norm, no projection, no attention, no sampling.
 *
 * Definition of one element (all integer arithmetic except one multiply):
 *   key   = mix64(seed * G + tensor_id * G2 + 1)
 *   h     = mix64(key + (index + 1) * G)
 *   s     = sum of the four 16-bit lanes of h            (exact integer)
 *   z     = s - 131070                                    (Irwin-Hall(4), centred)
 *   value = (float)z * scale                              (one IEEE multiply)
 * where mix64 is the SplitMix64 output function (Steele, Lea & Flood,
 * "Fast splittable pseudorandom number generators", OOPSLA 2014), G is the
 * 64-bit golden-ratio increment it uses and scale = sigma * sqrt(3) / 65536
 * rounded to float once on the host, so that value has standard deviation
 * sigma (a sum of four uniforms on [0, 65535] has variance 65536^2 / 3).
 * Values are bounded by +-3.46 sigma.  BF16 and F16 tensors are the float
 * value rounded to nearest-even in the storage format.
 */
#ifndef DS4G_SYNTH_H
#define DS4G_SYNTH_H

#include <stdint.h>
#include <string.h>

#if defined(__CUDACC__)
#define SYN_FN static __host__ __device__ __forceinline__
#else
#define SYN_FN static inline
#endif

#define SYN_GOLDEN 0x9E3779B97F4A7C15ull
#define SYN_GOLDEN2 0xD1B54A32D192ED03ull

/* Tensor kinds; a tensor id is (layer << 32) | (kind << 24) | expert. */
enum {
    SYN_ATTN_NORM = 1, SYN_WQ_A = 2, SYN_WQ_B = 3, SYN_WKV_A = 4, SYN_WK_B = 5,
    SYN_WV_B = 6, SYN_WO = 7, SYN_FFN_NORM = 8, SYN_W_ROUTER = 9, SYN_W_GATE = 10,
    SYN_W_UP = 11, SYN_W_DOWN = 12, SYN_WS_GATE = 13, SYN_WS_UP = 14, SYN_WS_DOWN = 15,
    SYN_TOK_EMBD = 16, SYN_LM_HEAD = 17, SYN_KV_K = 18, SYN_KV_V = 19, SYN_TOKENS = 20,
    SYN_LOGITS = 21, SYN_MISC = 22
};
#define SYN_GLOBAL_LAYER 0xFFFFu

SYN_FN uint64_t syn_tensor_id(uint32_t layer, uint32_t kind, uint32_t expert)
{
    return ((uint64_t)layer << 32) | ((uint64_t)kind << 24) | (uint64_t)(expert & 0xFFFFFFu);
}

SYN_FN uint64_t syn_mix64(uint64_t z)
{
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

SYN_FN uint64_t syn_key(uint64_t seed, uint64_t tensor_id)
{
    return syn_mix64(seed * SYN_GOLDEN + tensor_id * SYN_GOLDEN2 + 1ull);
}

SYN_FN uint64_t syn_hash(uint64_t key, uint64_t index)
{
    return syn_mix64(key + (index + 1ull) * SYN_GOLDEN);
}

/* Centred Irwin-Hall(4) integer in [-131070, 131070]. */
SYN_FN int32_t syn_ih4(uint64_t h)
{
    uint32_t s = (uint32_t)(h & 0xFFFFu) + (uint32_t)((h >> 16) & 0xFFFFu) +
                 (uint32_t)((h >> 32) & 0xFFFFu) + (uint32_t)(h >> 48);
    return (int32_t)s - 131070;
}

SYN_FN float syn_value(uint64_t key, uint64_t index, float scale)
{
    return (float)syn_ih4(syn_hash(key, index)) * scale;
}

SYN_FN uint32_t syn_f32_bits(float f)
{
#if defined(__CUDA_ARCH__)
    return __float_as_uint(f);
#else
    uint32_t u;
    memcpy(&u, &f, 4);
    return u;
#endif
}

/* float -> bfloat16 bits, round to nearest even (values here are finite). */
SYN_FN uint16_t syn_to_bf16(float f)
{
    uint32_t u = syn_f32_bits(f);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* float -> IEEE binary16 bits, round to nearest even; handles the subnormal
 * range and saturates to infinity beyond the largest finite half. */
SYN_FN uint16_t syn_to_f16(float f)
{
    uint32_t u = syn_f32_bits(f);
    uint32_t sign = (u >> 16) & 0x8000u;
    uint32_t a = u & 0x7FFFFFFFu;
    if (a >= 0x477FF000u) return (uint16_t)(sign | 0x7C00u);  /* rounds to >= 65520: inf */
    if (a < 0x38800000u) {                                     /* below 2^-14: subnormal half */
        if (a < 0x33000000u) return (uint16_t)sign;            /* below 2^-25: rounds to 0 */
        uint32_t e = a >> 23;
        uint32_t m = (a & 0x7FFFFFu) | 0x800000u;
        /* half subnormal unit is 2^-24; value = m * 2^(e-150); units = m * 2^(e-126) */
        uint32_t shift = 126u - e;                             /* in [14, 24] */
        uint32_t q = m >> shift;
        uint32_t rem = m & ((1u << shift) - 1u);
        uint32_t halfway = 1u << (shift - 1u);
        if (rem > halfway || (rem == halfway && (q & 1u))) q += 1u;
        return (uint16_t)(sign | q);
    }
    /* normal: rebias exponent 127 -> 15 and round the 13 dropped mantissa bits */
    uint32_t r = a - 0x38000000u;
    uint32_t lsb = (r >> 13) & 1u;
    r += 0xFFFu + lsb;
    return (uint16_t)(sign | (r >> 13));
}

/* Token id uniform in [0, vocab) (modulo bias below 1e-14 for vocab < 2^18). */
SYN_FN int32_t syn_token(uint64_t key, uint64_t index, uint32_t vocab)
{
    return (int32_t)(syn_hash(key, index) % (uint64_t)vocab);
}

#endif /* DS4G_SYNTH_H */
