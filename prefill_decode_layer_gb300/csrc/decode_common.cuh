// Device helpers shared by the decode kernels (per-stage and persistent forms).
#pragma once

#include "common.cuh"

namespace ds4g {

__device__ __forceinline__ int gwarp() { return (threadIdx.x >> 5) * gridDim.x + blockIdx.x; }
__device__ __forceinline__ int gwarps() { return (blockDim.x >> 5) * gridDim.x; }

// Copy n f32 (n % 4 == 0) from global to shared memory, four 16-byte loads in flight
// per thread, and return this thread's partial sum of squares.  CG: read through L2
// only (data written by other CTAs of the same running grid).
template <bool CG = false>
__device__ __forceinline__ float load_f32_sumsq(const float *src, float *dst, int n)
{
    float ss = 0.f;
    for (int base = threadIdx.x * 4; base < n; base += blockDim.x * 16) {
        float4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = base + j * blockDim.x * 4;
            const float4 *p = reinterpret_cast<const float4 *>(src + i);
            v[j] = i < n ? (CG ? __ldcg(p) : *p) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = base + j * blockDim.x * 4;
            if (i < n) {
                *reinterpret_cast<float4 *>(dst + i) = v[j];
                ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
            }
        }
    }
    return ss;
}

// Same for an f16 embedding row (n % 8 == 0), widened to f32.
__device__ __forceinline__ float load_f16_sumsq(const uint16_t *src, float *dst, int n)
{
    float ss = 0.f;
    for (int base = threadIdx.x * 8; base < n; base += blockDim.x * 32) {
        uint4 v[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = base + j * blockDim.x * 8;
            v[j] = i < n ? *reinterpret_cast<const uint4 *>(src + i) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int i = base + j * blockDim.x * 8;
            if (i < n) {
                const __half *h = reinterpret_cast<const __half *>(&v[j]);
#pragma unroll
                for (int t = 0; t < 8; ++t) {
                    const float f = __half2float(h[t]);
                    dst[i + t] = f;
                    ss = fmaf(f, f, ss);
                }
            }
        }
    }
    return ss;
}

// xs = xs * rsqrt(ss / H + eps) * g, after a block-wide sum of the partial sums.
__device__ __forceinline__ void finish_norm(float ss, const float *g, int H, float eps, float *xs,
                                            float *red)
{
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)H + eps);
    for (int i = threadIdx.x * 4; i < H; i += blockDim.x * 4) {
        float4 v = *reinterpret_cast<float4 *>(xs + i);
        const float4 gg = *reinterpret_cast<const float4 *>(g + i);
        v.x = v.x * inv * gg.x; v.y = v.y * inv * gg.y; v.z = v.z * inv * gg.z; v.w = v.w * inv * gg.w;
        *reinterpret_cast<float4 *>(xs + i) = v;
    }
    __syncthreads();
}

template <bool CG = false>
__device__ __forceinline__ void copy_f32(const float *src, float *dst, int n)
{
    (void)load_f32_sumsq<CG>(src, dst, n);
}

}  // namespace ds4g
