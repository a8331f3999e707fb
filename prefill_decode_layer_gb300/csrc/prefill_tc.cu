// Layer-major prefill on the tensor cores (page "ds4.c 学习笔记 -- 端到端推理流程",
// 阶段三 prefill_layer_major_cpu: every layer runs over the whole chunk before the
// next, so each layer's weights are read once per chunk).
//
// Same steps, order and fixed reductions as the SIMT form in prefill.cu, with every
// weight contraction a tcgen05 GEMM (tc_gemm.cuh).  Activations entering a GEMM are
// BF16 (the router's input a BF16 hi/lo pair; every activation a pair in the hi/lo
// mode); the residual and the router scores stay FP32, the routed experts' per-slot
// rows are BF16 (FP32 in the hi/lo mode).  The buffers are those of the SIMT form:
// an FP32-sized buffer holds exactly one hi and one lo BF16 array.  The shared
// expert's GEMMs run on the session's side stream.  Weight tensor maps are built
// once per model, activation maps once per session.
#include <type_traits>

#include "kernels.h"
#include "prefill_problems.cuh"
#include "prefill_tc.h"
#include "tc_gemm.cuh"

namespace ds4g {

// ------------------------------------------------------------------ small kernels

// RMSNorm of each residual row into hi/lo BF16 (lo == nullptr: hi only): one CTA per
// token row, each thread keeping up to four float4s in registers between the two
// passes (H <= 16 x blockDim.x).
__global__ void __launch_bounds__(1024) k_rmsnorm_hilo(const float *X, const float *g, bf16 *hi, bf16 *lo,
                                                       int H, float eps)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    __shared__ float red[32];
    const int t = blockIdx.x, nv = H / 4;
    const float4 *x = reinterpret_cast<const float4 *>(X + (size_t)t * H);
    float4 v[4];
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        v[u] = i < nv ? x[i] : make_float4(0.f, 0.f, 0.f, 0.f);
        ss = fmaf(v[u].x, v[u].x, fmaf(v[u].y, v[u].y, fmaf(v[u].z, v[u].z, fmaf(v[u].w, v[u].w, ss))));
    }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)H + eps);
#pragma unroll
    for (int u = 0; u < 4; ++u) {
        const int i = threadIdx.x + u * blockDim.x;
        if (i >= nv) continue;
        const float4 gv = reinterpret_cast<const float4 *>(g)[i];
        __align__(8) bf16 h[4], l[4];
        split_hilo(v[u].x * inv * gv.x, h[0], l[0]);
        split_hilo(v[u].y * inv * gv.y, h[1], l[1]);
        split_hilo(v[u].z * inv * gv.z, h[2], l[2]);
        split_hilo(v[u].w * inv * gv.w, h[3], l[3]);
        *reinterpret_cast<uint2 *>(hi + (size_t)t * H + 4 * i) = *reinterpret_cast<const uint2 *>(h);
        if (lo) *reinterpret_cast<uint2 *>(lo + (size_t)t * H + 4 * i) = *reinterpret_cast<const uint2 *>(l);
    }
}
// H / 16 threads (each keeps four float4s): a token row of 4096 takes 256 threads,
// so that eight CTAs fit on an SM (0.08 ms per 8 x 4096 prefill against 1024).
static int rmsnorm_threads(int H) { return (H / 16 + 31) / 32 * 32; }

// ------------------------------------------------------------------ attention on the tensor cores
//
// Windowed causal MQA for a chunk with warp-level BF16 MMAs (m16n8k16, FP32
// accumulation).  All heads of a token share one K/V window, so a warp takes 16
// heads of one token as the 16 rows of its tiles: S = Q K^T over the window's keys,
// a row softmax in registers, O = P V.  Q and P enter the MMAs as hi/lo BF16 pairs
// (two MMAs each), K and V are BF16 already.  A CTA serves 16 consecutive tokens:
// the union of their windows (at most W + 15 keys) is staged once in shared memory
// (rows padded by 16 bytes so that ldmatrix rows fall in distinct banks, plus 16
// zero rows for the padding of the last 16-key step).  Head dimension 128, window
// <= 128.

static constexpr int kAttnTB = 16;                     // tokens per CTA
static constexpr int kAttnHD = 128;                    // head dimension of this kernel
static constexpr int kAttnMaxW = 128;                  // largest window
static constexpr int kAttnPitch = kAttnHD + 8;         // bf16 per staged K/V row
static constexpr int kAttnMaxT = kAttnMaxW / 8 + 2;    // 8-key tiles a window can touch (even)

__device__ __forceinline__ uint32_t pack_bf16(float a, float b)   // a in the low half
{
    const uint32_t lo = __bfloat16_as_ushort(__float2bfloat16_rn(a));
    const uint32_t hi = __bfloat16_as_ushort(__float2bfloat16_rn(b));
    return lo | (hi << 16);
}
__device__ __forceinline__ void split_pack(float a, float b, uint32_t &hi, uint32_t &lo)
{
    const bf16 ha = __float2bfloat16_rn(a), hb = __float2bfloat16_rn(b);
    hi = (uint32_t)__bfloat16_as_ushort(ha) | ((uint32_t)__bfloat16_as_ushort(hb) << 16);
    lo = pack_bf16(a - __bfloat162float(ha), b - __bfloat162float(hb));
}
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
        "{%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t (&r)[4], const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(smem_u32(p)));
}

size_t attn_mma_smem(const Dims &d)
{
    const int rows = d.W + kAttnTB - 1 + 15 + 16;   // window union, alignment, padding
    return 2 * (size_t)rows * kAttnPitch * 2;
}

__global__ void __launch_bounds__(256) k_attn_prefill_mma(const float *Q, bf16 *o_hi, bf16 *o_lo,
                                                          const bf16 *kc, const bf16 *vc, int p0, int n,
                                                          Dims d)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    extern __shared__ __align__(16) unsigned char sm_attn[];
    const int W = d.W, NH = d.NH, QD = d.QD;
    const int t0 = blockIdx.x * kAttnTB;
    const int tend = min(t0 + kAttnTB, n);
    // Staged keys [kbase, kend), kbase a multiple of 16.  Tiles start at absolute key
    // positions that are multiples of 16, so a token's sums run in the same order
    // however the prompt was cut into chunks (batch-invariant results); a window's
    // last 16-key step may run up to 15 rows past the keys: 16 zero rows follow.
    const int kbase = (max(0, p0 + t0 - W + 1) / 16) * 16, kend = p0 + tend;
    const int nrows = kend - kbase + 16;
    bf16 *Ks = reinterpret_cast<bf16 *>(sm_attn);
    bf16 *Vs = Ks + (size_t)nrows * kAttnPitch;
    for (int i = threadIdx.x; i < nrows * (kAttnHD / 8); i += blockDim.x) {
        const int r = i / (kAttnHD / 8), c = (i % (kAttnHD / 8)) * 8;
        uint4 kv = make_uint4(0, 0, 0, 0), vv = make_uint4(0, 0, 0, 0);
        if (kbase + r < kend) {
            kv = *reinterpret_cast<const uint4 *>(kc + (size_t)(kbase + r) * kAttnHD + c);
            vv = *reinterpret_cast<const uint4 *>(vc + (size_t)(kbase + r) * kAttnHD + c);
        }
        *reinterpret_cast<uint4 *>(Ks + (size_t)r * kAttnPitch + c) = kv;
        *reinterpret_cast<uint4 *>(Vs + (size_t)r * kAttnPitch + c) = vv;
    }
    __syncthreads();
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c2 = (lane & 3) * 2;
    const int ngroups = (NH + 15) / 16;
    const float scale = rsqrtf((float)kAttnHD);
    for (int item = warp; item < (tend - t0) * ngroups; item += 8) {
        const int t = t0 + item / ngroups, h0 = (item % ngroups) * 16;
        const int pos = p0 + t, klo = max(0, pos - W + 1);
        const int ra = h0 + g, rb = h0 + g + 8;   // the two query rows (heads) of this thread
        // S = Q K^T over 8-key tiles [s0, s0 + 8 * nt) of the staged rows
        const int s0 = (klo / 16) * 16 - kbase;
        const int nt = ((pos - kbase + 1 - s0 + 15) / 16) * 2;   // even
        float S[kAttnMaxT][4];
#pragma unroll
        for (int j = 0; j < kAttnMaxT; ++j) S[j][0] = S[j][1] = S[j][2] = S[j][3] = 0.f;
        const float *qa = Q + (size_t)t * QD + (size_t)ra * kAttnHD;
        const float *qb = Q + (size_t)t * QD + (size_t)rb * kAttnHD;
#pragma unroll 1
        for (int k0 = 0; k0 < kAttnHD; k0 += 16) {
            uint32_t ah[4], al[4];
            {
                float2 x0 = make_float2(0.f, 0.f), x1 = x0, x2 = x0, x3 = x0;
                if (ra < NH) {
                    x0 = *reinterpret_cast<const float2 *>(qa + k0 + c2);
                    x2 = *reinterpret_cast<const float2 *>(qa + k0 + 8 + c2);
                }
                if (rb < NH) {
                    x1 = *reinterpret_cast<const float2 *>(qb + k0 + c2);
                    x3 = *reinterpret_cast<const float2 *>(qb + k0 + 8 + c2);
                }
                split_pack(x0.x * scale, x0.y * scale, ah[0], al[0]);
                split_pack(x1.x * scale, x1.y * scale, ah[1], al[1]);
                split_pack(x2.x * scale, x2.y * scale, ah[2], al[2]);
                split_pack(x3.x * scale, x3.y * scale, ah[3], al[3]);
            }
#pragma unroll
            for (int j = 0; j < kAttnMaxT; j += 2) {
                if (j < nt) {
                    // keys s0 + 8j .. +15, dims k0 .. k0+15: matrices (keys 0-7, dims 0-7),
                    // (keys 0-7, dims 8-15), (keys 8-15, dims 0-7), (keys 8-15, dims 8-15)
                    uint32_t b[4];
                    const int kr = s0 + 8 * j + (lane & 7) + ((lane >> 4) << 3);
                    const int kcol = k0 + ((lane >> 3) & 1) * 8;
                    ldsm_x4(b, Ks + (size_t)kr * kAttnPitch + kcol);
                    mma_16816(S[j], ah, b[0], b[1]);
                    mma_16816(S[j], al, b[0], b[1]);
                    mma_16816(S[j + 1], ah, b[2], b[3]);
                    mma_16816(S[j + 1], al, b[2], b[3]);
                }
            }
        }
        // mask to the window, then row max / exp / sum (rows ra: S[.][0..1], rb: S[.][2..3])
        float ma = -INFINITY, mb = -INFINITY;
#pragma unroll
        for (int j = 0; j < kAttnMaxT; ++j) {
            const int kabs = kbase + s0 + 8 * j + c2;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const bool ok = j < nt && kabs + u >= klo && kabs + u <= pos;
                if (!ok) {
                    S[j][u] = -INFINITY;
                    S[j][2 + u] = -INFINITY;
                }
                ma = fmaxf(ma, S[j][u]);
                mb = fmaxf(mb, S[j][2 + u]);
            }
        }
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 1));
        ma = fmaxf(ma, __shfl_xor_sync(0xffffffffu, ma, 2));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 1));
        mb = fmaxf(mb, __shfl_xor_sync(0xffffffffu, mb, 2));
        float suma = 0.f, sumb = 0.f;
#pragma unroll
        for (int j = 0; j < kAttnMaxT; ++j) {
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                S[j][u] = S[j][u] == -INFINITY ? 0.f : __expf(S[j][u] - ma);
                S[j][2 + u] = S[j][2 + u] == -INFINITY ? 0.f : __expf(S[j][2 + u] - mb);
                suma += S[j][u];
                sumb += S[j][2 + u];
            }
        }
        suma += __shfl_xor_sync(0xffffffffu, suma, 1);
        suma += __shfl_xor_sync(0xffffffffu, suma, 2);
        sumb += __shfl_xor_sync(0xffffffffu, sumb, 1);
        sumb += __shfl_xor_sync(0xffffffffu, sumb, 2);
        // O = P V, 16 keys per step; P's C-fragment layout is the A-fragment layout
        float O[kAttnHD / 8][4];
#pragma unroll
        for (int q = 0; q < kAttnHD / 8; ++q) O[q][0] = O[q][1] = O[q][2] = O[q][3] = 0.f;
#pragma unroll
        for (int j = 0; j < kAttnMaxT; j += 2) {
            if (j < nt) {
                uint32_t ph[4], pl[4];
                split_pack(S[j][0], S[j][1], ph[0], pl[0]);
                split_pack(S[j][2], S[j][3], ph[1], pl[1]);
                split_pack(S[j + 1][0], S[j + 1][1], ph[2], pl[2]);
                split_pack(S[j + 1][2], S[j + 1][3], ph[3], pl[3]);
#pragma unroll
                for (int q = 0; q < kAttnHD / 8; q += 2) {
                    // keys s0 + 8j .. +15 x dims 8q .. 8q+15, transposed: matrices (keys 0-7,
                    // dims 0-7), (keys 8-15, dims 0-7), (keys 0-7, dims 8-15), (keys 8-15, dims 8-15)
                    uint32_t b[4];
                    const int vr = s0 + 8 * j + (lane & 7) + (((lane >> 3) & 1) << 3);
                    const int vcol = 8 * q + ((lane >> 4) << 3);
                    ldsm_x4_t(b, Vs + (size_t)vr * kAttnPitch + vcol);
                    mma_16816(O[q], ph, b[0], b[1]);
                    mma_16816(O[q], pl, b[0], b[1]);
                    mma_16816(O[q + 1], ph, b[2], b[3]);
                    mma_16816(O[q + 1], pl, b[2], b[3]);
                }
            }
        }
        const float ia = 1.f / suma, ib = 1.f / sumb;
#pragma unroll
        for (int q = 0; q < kAttnHD / 8; ++q) {
            const int dcol = 8 * q + c2;
            uint32_t h, l;
            if (ra < NH) {
                split_pack(O[q][0] * ia, O[q][1] * ia, h, l);
                const size_t oi = (size_t)t * QD + (size_t)ra * kAttnHD + dcol;
                *reinterpret_cast<uint32_t *>(o_hi + oi) = h;
                *reinterpret_cast<uint32_t *>(o_lo + oi) = l;
            }
            if (rb < NH) {
                split_pack(O[q][2] * ib, O[q][3] * ib, h, l);
                const size_t oi = (size_t)t * QD + (size_t)rb * kAttnHD + dcol;
                *reinterpret_cast<uint32_t *>(o_hi + oi) = h;
                *reinterpret_cast<uint32_t *>(o_lo + oi) = l;
            }
        }
    }
}

bool attn_mma_eligible(const Dims &d) { return d.HD == kAttnHD && d.W <= kAttnMaxW && d.kvdt == DS4G_BF16; }

cudaError_t attn_mma_setup(const Dims &d, int max_smem)
{
    if (!attn_mma_eligible(d)) return cudaSuccess;
    if (attn_mma_smem(d) > (size_t)max_smem) return cudaErrorInvalidValue;
    return allow_max_dyn_smem((const void *)k_attn_prefill_mma, max_smem);
}

// ------------------------------------------------------------------ epilogues
// Functors of the tensor-core GEMM.  Direct form (kDirect): the thread of the
// epilogue that owns token m passes 32 adjacent features f0 .. f0 + 31 of it at a
// time; load32 fetches what their store needs from global memory (issued ahead by
// the GEMM), store32 writes.  Staged form: the same for 4 features at a time
// (load4, store4), with the GEMM's instructions covering 4 tokens x 32 features.

// 32 values as BF16 hi (and lo, unless null) halves: 4 16-byte stores each
__device__ __forceinline__ void store_hilo32(bf16 *hi, bf16 *lo, const float (&v)[32])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t wh[4], wl[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) split2_hilo(v[8 * q + 2 * j], v[8 * q + 2 * j + 1], wh[j], wl[j]);
        reinterpret_cast<uint4 *>(hi)[q] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
        if (lo) reinterpret_cast<uint4 *>(lo)[q] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
    }
}
// 32 values as FP32 (8 16-byte stores) or BF16, rounded to nearest even (4)
__device__ __forceinline__ void store32(float *p, const float (&v)[32])
{
#pragma unroll
    for (int q = 0; q < 8; ++q)
        reinterpret_cast<float4 *>(p)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}
__device__ __forceinline__ void store32(bf16 *p, const float (&v)[32])
{
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        uint32_t w[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
            w[j] = pack_bf16x2(__float2bfloat16_rn(v[8 * q + 2 * j]), __float2bfloat16_rn(v[8 * q + 2 * j + 1]));
        reinterpret_cast<uint4 *>(p)[q] = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// (cos, sin) of the 16 RoPE pairs of features f0 .. f0 + 31 of a head (f0 % 32 == 0)
struct Rope16 {
    float4 cs[8];   // pairs 2k and 2k + 1 in cs[k]
};
__device__ __forceinline__ Rope16 rope16(const float2 *rope, int pos, int HD, int f0)
{
    Rope16 r;
    const float4 *p = reinterpret_cast<const float4 *>(rope + (size_t)pos * (HD / 2) + (f0 % HD) / 2);
#pragma unroll
    for (int k = 0; k < 8; ++k) r.cs[k] = p[k];
    return r;
}
// v rotated pair by pair: (v[2i], v[2i+1]) by the angle of pair i
__device__ __forceinline__ void rotate32(const float (&v)[32], const Rope16 &r, float (&o)[32])
{
#pragma unroll
    for (int k = 0; k < 8; ++k) {
        const float4 c = r.cs[k];
        o[4 * k] = v[4 * k] * c.x - v[4 * k + 1] * c.y;
        o[4 * k + 1] = v[4 * k] * c.y + v[4 * k + 1] * c.x;
        o[4 * k + 2] = v[4 * k + 2] * c.z - v[4 * k + 3] * c.w;
        o[4 * k + 3] = v[4 * k + 2] * c.w + v[4 * k + 3] * c.z;
    }
}

struct EpiHiLo {   // out[m][n..n+3] as hi/lo BF16 (the next GEMM's input; lo may be null)
    bf16 *hi, *lo;
    int ld;
    static constexpr bool kDirect = false;
    using Aux = tc::NoAux;
    __device__ Aux load4(int, int, int) const { return {}; }
    __device__ void store4(int m, int n, const float (&v)[4], const Aux &, int) const
    {
        uint32_t h0, l0, h1, l1;
        split2_hilo(v[0], v[1], h0, l0);
        split2_hilo(v[2], v[3], h1, l1);
        *reinterpret_cast<uint2 *>(hi + (size_t)m * ld + n) = make_uint2(h0, h1);
        if (lo) *reinterpret_cast<uint2 *>(lo + (size_t)m * ld + n) = make_uint2(l0, l1);
    }
};

struct EpiQRope {   // Q[m][f0..f0+31] = RoPE(q) in FP32 (the attention's input)
    float *Q;
    const float2 *rope;
    int QD, HD, p0;
    static constexpr bool kDirect = true;
    using Aux = Rope16;
    __device__ Aux load32(int m, int f0, int) const { return rope16(rope, p0 + m, HD, f0); }
    __device__ void store32(int m, int f0, const float (&v)[32], const Aux &cs, int) const
    {
        float r[32];
        rotate32(v, cs, r);
        ds4g::store32(Q + (size_t)m * QD + f0, r);
    }
};

struct EpiQRopeHiLo {   // RoPE(q) as hi/lo BF16 [token][head][dim] rows (the tcgen05 attention's input; lo may be null)
    bf16 *hi, *lo;
    const float2 *rope;
    int QD, HD, p0;
    static constexpr bool kDirect = true;
    using Aux = Rope16;
    __device__ Aux load32(int m, int f0, int) const { return rope16(rope, p0 + m, HD, f0); }
    __device__ void store32(int m, int f0, const float (&v)[32], const Aux &cs, int) const
    {
        float r[32];
        rotate32(v, cs, r);
        const size_t o = (size_t)m * QD + f0;
        store_hilo32(hi + o, lo ? lo + o : nullptr, r);
    }
};

__device__ __forceinline__ float4 rope_pairs(const float2 *rope, int pos, int HD, int n)
{   // (cos, sin) of the RoPE pairs (n % HD)/2 and the next one
    return *reinterpret_cast<const float4 *>(rope + (size_t)pos * (HD / 2) + (n % HD) / 2);
}

template <typename TKV>
struct EpiKVRope {   // features [0, HD): K with RoPE, [HD, 2HD): V; appended at p0 + m
    TKV *kc, *vc;
    const float2 *rope;
    int HD, p0;
    static constexpr bool kDirect = false;
    using Aux = float4;
    __device__ Aux load4(int m, int n, int) const
    {
        return n < HD ? rope_pairs(rope, p0 + m, HD, n) : make_float4(1.f, 0.f, 1.f, 0.f);
    }
    __device__ void store4(int m, int n, const float (&v)[4], const Aux &cs, int) const
    {
        const size_t row = (size_t)(p0 + m) * HD;
        if (n < HD) {
            kc[row + n] = from_f32<TKV>(v[0] * cs.x - v[1] * cs.y);
            kc[row + n + 1] = from_f32<TKV>(v[0] * cs.y + v[1] * cs.x);
            kc[row + n + 2] = from_f32<TKV>(v[2] * cs.z - v[3] * cs.w);
            kc[row + n + 3] = from_f32<TKV>(v[2] * cs.w + v[3] * cs.z);
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) vc[row + n - HD + j] = from_f32<TKV>(v[j]);
        }
    }
};

struct EpiAddX {   // residual: X[m][n..n+3] += v
    float *X;
    int H;
    static constexpr bool kDirect = false;
    using Aux = float4;
    __device__ Aux load4(int m, int n, int) const { return *reinterpret_cast<const float4 *>(X + (size_t)m * H + n); }
    __device__ void store4(int m, int n, const float (&v)[4], const Aux &x, int) const
    {
        *reinterpret_cast<float4 *>(X + (size_t)m * H + n) =
            make_float4(x.x + v[0], x.y + v[1], x.z + v[2], x.w + v[3]);
    }
};

struct EpiScores {   // router scores of reduction part s: S[s][m][n..n+3] in FP32
    float *S;
    int E;
    size_t part;   // elements between the parts' score arrays
    static constexpr bool kDirect = false;
    using Aux = tc::NoAux;
    __device__ Aux load4(int, int, int) const { return {}; }
    __device__ void store4(int m, int n, const float (&v)[4], const Aux &, int s) const
    {
        *reinterpret_cast<float4 *>(S + s * part + (size_t)m * E + n) = make_float4(v[0], v[1], v[2], v[3]);
    }
};

// Per-slot routed rows: 4 consecutive values as FP32 or BF16 (RNE); acc_row16 adds w
// times the values of 16 bytes of a row (4 FP32 or 8 BF16, widened exactly) to r.
__device__ __forceinline__ void store_row4(float *p, const float (&v)[4])
{
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
}
__device__ __forceinline__ void store_row4(bf16 *p, const float (&v)[4])
{
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16x2(__float2bfloat16_rn(v[0]), __float2bfloat16_rn(v[1])),
                                               pack_bf16x2(__float2bfloat16_rn(v[2]), __float2bfloat16_rn(v[3])));
}
__device__ __forceinline__ void acc_row16(float w, const uint4 &q, float (&r)[4], float)
{
    r[0] = fmaf(w, __uint_as_float(q.x), r[0]);
    r[1] = fmaf(w, __uint_as_float(q.y), r[1]);
    r[2] = fmaf(w, __uint_as_float(q.z), r[2]);
    r[3] = fmaf(w, __uint_as_float(q.w), r[3]);
}
__device__ __forceinline__ void acc_row16(float w, const uint4 &q, float (&r)[8], bf16)
{
    const uint32_t a[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        r[2 * j] = fmaf(w, __uint_as_float(a[j] << 16), r[2 * j]);
        r[2 * j + 1] = fmaf(w, __uint_as_float(a[j] & 0xffff0000u), r[2 * j + 1]);
    }
}
template <typename TY>
struct EpiRoutedRows {   // routed expert output of grouped row m into its (token, slot) row (FP32 or BF16)
    TY *YS;
    const int *rows;
    int H;
    int nrows;     // (token, slot) rows of the launch: a row index outside is never written
    int *status;
    static constexpr bool kDirect = false;
    using Aux = int;
    __device__ Aux load4(int m, int, int) const { return rows[m]; }
    __device__ void store4(int, int n, const float (&v)[4], const Aux &r, int) const
    {
        if ((unsigned)r >= (unsigned)nrows) {
            atomicCAS(status, 0, DS4G_EINVAL);
            return;
        }
        store_row4(YS + (size_t)r * H + n, v);
    }
};

struct EpiSwiGLU {   // h[m][i0 .. i0+31] = silu(gate) * up as hi/lo BF16 (lo may be null), 16-byte stores
    bf16 *hi, *lo;
    int ld;
    __device__ void store_row(int m, int i0, const float (&h)[32], int) const
    {
        const size_t o = (size_t)m * ld + i0;
        store_hilo32(hi + o, lo ? lo + o : nullptr, h);
    }
};

// x[t] += sum over slots s (in order) of w[t][s] * YS[t*K + s]: the selected experts'
// outputs (FP32, or BF16 rows widened exactly), after the shared expert's down
// projection was added by its GEMM.  A thread takes 16 bytes of each slot's row a
// step (4 FP32 or 8 BF16 values), the slots' loads in flight together.  With gnext:
// also the next layer's attention RMSNorm of the new row, as BF16 hi/lo into hi, lo
// (what k_rmsnorm_hilo would write next; lo may be null); each thread reads back the
// residual values it has just written.
template <typename TY>
__global__ void __launch_bounds__(256) k_moe_combine(float *X, const TY *YS, const float *wts, int H, int K,
                                                     const float *gnext, float eps, bf16 *nhi, bf16 *nlo)
{
    pdl_wait();      // inputs of the previous kernel (programmatic launch)
    pdl_trigger();
    constexpr int VEC = 16 / (int)sizeof(TY);   // values per thread and step
    const int t = blockIdx.x, step = blockDim.x * VEC;
    float w[8];
#pragma unroll
    for (int s = 0; s < 8; ++s) w[s] = s < K ? wts[(size_t)t * K + s] : 0.f;
    float *xrow = X + (size_t)t * H;
    for (int i = threadIdx.x * VEC; i < H; i += step) {
        uint4 y[8];
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (s < K) y[s] = *reinterpret_cast<const uint4 *>(YS + ((size_t)t * K + s) * H + i);
        float r[VEC];
#pragma unroll
        for (int k = 0; k < VEC; ++k) r[k] = 0.f;
#pragma unroll
        for (int s = 0; s < 8; ++s)
            if (s < K) acc_row16(w[s], y[s], r, TY{});
        float4 *x = reinterpret_cast<float4 *>(xrow + i);
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const float4 xv = x[q];
            x[q] = make_float4(xv.x + r[4 * q], xv.y + r[4 * q + 1], xv.z + r[4 * q + 2], xv.w + r[4 * q + 3]);
        }
    }
    if (!gnext) return;
    __shared__ float red[32];
    float ss = 0.f;
    for (int i = threadIdx.x * VEC; i < H; i += step)
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const float4 v = reinterpret_cast<const float4 *>(xrow + i)[q];
            ss = fmaf(v.x, v.x, fmaf(v.y, v.y, fmaf(v.z, v.z, fmaf(v.w, v.w, ss))));
        }
    ss = block_sum(ss, red);
    const float inv = rsqrtf(ss / (float)H + eps);
    for (int i = threadIdx.x * VEC; i < H; i += step)
#pragma unroll
        for (int q = 0; q < VEC / 4; ++q) {
            const int j = i + 4 * q;
            const float4 v = *reinterpret_cast<const float4 *>(xrow + j);
            const float4 gv = *reinterpret_cast<const float4 *>(gnext + j);
            __align__(8) bf16 h[4], l[4];
            split_hilo(v.x * inv * gv.x, h[0], l[0]);
            split_hilo(v.y * inv * gv.y, h[1], l[1]);
            split_hilo(v.z * inv * gv.z, h[2], l[2]);
            split_hilo(v.w * inv * gv.w, h[3], l[3]);
            *reinterpret_cast<uint2 *>(nhi + (size_t)t * H + j) = *reinterpret_cast<const uint2 *>(h);
            if (nlo) *reinterpret_cast<uint2 *>(nlo + (size_t)t * H + j) = *reinterpret_cast<const uint2 *>(l);
        }
}

// ------------------------------------------------------------------ maps and eligibility

bool tc_prefill_eligible(const Dims &d)
{
    return d.wdt == DS4G_BF16 && d.H % 128 == 0 && d.H <= 16384 && d.RQ % 128 == 0 && d.RKV % 128 == 0 &&
           d.QD % 128 == 0 && d.HD % 128 == 0 && d.E % 128 == 0 && d.I % 128 == 0;
}

cudaError_t tc_layer_maps(const Dims &d, const LayerPtrs &w, TcLayerMaps &m)
{
    using tc::make_map_bf16;
    const int H = d.H, I = d.I, E = d.E;
    cudaError_t e;
    if ((e = make_map_bf16(&m.wqa, w.wq_a, d.RQ, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wkva, w.wkv_a, d.RKV, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wqb, w.wq_b, d.QD, d.RQ, d.RQ, 128))) return e;
    if ((e = make_map_bf16(&m.wkb, w.wk_b, d.HD, d.RKV, d.RKV, 128))) return e;
    if ((e = make_map_bf16(&m.wvb, w.wv_b, d.HD, d.RKV, d.RKV, 128))) return e;
    if ((e = make_map_bf16(&m.wo, w.wo, H, d.QD, d.QD, 128))) return e;
    if ((e = make_map_bf16(&m.wr, w.w_router, E, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wsg, w.ws_gate, I, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wsu, w.ws_up, I, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wsd, w.ws_down, H, I, I, 128))) return e;
    if ((e = make_map_bf16(&m.wg, w.w_gate, E * I, H, H, 128))) return e;
    if ((e = make_map_bf16(&m.wu, w.w_up, E * I, H, H, 128))) return e;
    return make_map_bf16(&m.wd, w.w_down, E * H, I, I, 128);
}

TcActPtrs tc_act_ptrs(const Dims &d, const PrefillBufs &pb)
{
    const size_t P = pb.P, PK = (size_t)pb.P * d.K, RC = d.RQ + d.RKV;
    TcActPtrs a;
    a.xn_hi = (bf16 *)pb.XN;
    a.xn_lo = a.xn_hi + P * d.H;
    a.c_hi = (bf16 *)pb.C;
    a.c_lo = a.c_hi + P * RC;
    a.o_hi = (bf16 *)pb.O;
    a.o_lo = a.o_hi + P * d.QD;
    a.hg_hi = (bf16 *)pb.HG;
    a.hg_lo = a.hg_hi + PK * d.I;
    a.hs_hi = (bf16 *)pb.HS;
    a.hs_lo = a.hs_hi + P * d.I;
    return a;
}

cudaError_t tc_act_maps(const Dims &d, const PrefillBufs &pb, TcActMaps &m)
{
    using tc::make_map_bf16;
    const TcActPtrs a = tc_act_ptrs(d, pb);
    const int P = pb.P, PK = pb.P * d.K, RC = d.RQ + d.RKV;
    cudaError_t e;
    if ((e = make_map_bf16(&m.xn_hi, a.xn_hi, P, d.H, d.H, tc::BT))) return e;
    if ((e = make_map_bf16(&m.xn_lo, a.xn_lo, P, d.H, d.H, tc::BT))) return e;
    if ((e = make_map_bf16(&m.c_hi, a.c_hi, P, RC, RC, tc::BT))) return e;
    if ((e = make_map_bf16(&m.c_lo, a.c_lo, P, RC, RC, tc::BT))) return e;
    if ((e = make_map_bf16(&m.o_hi, a.o_hi, P, d.QD, d.QD, tc::BT))) return e;
    if ((e = make_map_bf16(&m.o_lo, a.o_lo, P, d.QD, d.QD, tc::BT))) return e;
    if ((e = make_map_bf16(&m.hg_hi, a.hg_hi, PK, d.I, d.I, tc::BT))) return e;
    if ((e = make_map_bf16(&m.hg_lo, a.hg_lo, PK, d.I, d.I, tc::BT))) return e;
    if ((e = make_map_bf16(&m.hs_hi, a.hs_hi, P, d.I, d.I, tc::BT))) return e;
    if ((e = make_map_bf16(&m.hs_lo, a.hs_lo, P, d.I, d.I, tc::BT))) return e;
    if (!attn_tc_eligible(d)) return cudaSuccess;
    const bf16 *q_hi = (const bf16 *)pb.Q;   // the query buffer as hi then lo BF16 halves
    if ((e = attn_tc_row_map(d, P, q_hi, m.q_hi))) return e;
    if ((e = attn_tc_row_map(d, P, q_hi + (size_t)P * d.QD, m.q_lo))) return e;
    if ((e = attn_tc_row_map(d, P, a.o_hi, m.oa_hi))) return e;   // the attention output's [token][head] rows
    return attn_tc_row_map(d, P, a.o_lo, m.oa_lo);
}

// ------------------------------------------------------------------ one chunk

template <typename TKV, bool HL>
static cudaError_t chunk_tc_t(const Dims &d, const LayerPtrs *layers, const TcLayerMaps *lm,
                              const TcActMaps &am, const TcKVMaps *kvm, void *const *kcs, void *const *vcs,
                              const float2 *rope,
                              const uint16_t *tok_embd, const PrefillBufs &pb, int p0, int n,
                              cudaStream_t st, int nsm)
{
    cudaError_t e;
    const int H = d.H, K = d.K, nent = n * K, I = d.I;
    const TcActPtrs ap = tc_act_ptrs(d, pb);
    const int ny = (n + tc::BT - 1) / tc::BT;
    const int max_tiles = nent / tc::BT + d.E + 1;
    // timing mode: an event after every launch, tagged with its kind
    auto mark = [&](int kind) {
        PrefillBufs::Timing *tm = pb.tm;
        if (!tm || tm->n >= PrefillBufs::Timing::kMax) return;
        cudaEventRecord(tm->ev[tm->n], st);
        tm->kind[tm->n++] = kind;
    };
    mark(-1);
    if ((e = launch_pdl(k_embed_rows, dim3(n), dim3(256), 0, st, tok_embd, (const int *)pb.tok, pb.X, H))) return e;
        mark(DS4G_K_P_EMBED);
    bool normed = false;   // xn holds the next layer's attention RMSNorm already
    for (int l = 0; l <= d.L; ++l) {
        for (int i = 0; i < pb.n_rec; ++i)
            if ((e = cudaMemcpyAsync(pb.rec_dst[i] + (size_t)l * H, pb.X + (size_t)pb.rec_row[i] * H,
                                     (size_t)H * 4, cudaMemcpyDeviceToDevice, st)))
                return e;
        if (l == d.L) break;
        const LayerPtrs &w = layers[l];
        const TcLayerMaps &m = lm[l];
        TKV *kc = (TKV *)kcs[l], *vc = (TKV *)vcs[l];
        tc::Args a{};
        a.status = pb.status;
        a.m_tok = n;
        // ---- attention half (its RMSNorm came with the previous layer's combine)
        if (!normed &&
            (e = launch_pdl(k_rmsnorm_hilo, dim3(n), dim3(rmsnorm_threads(H)), 0, st, (const float *)pb.X,
                            (const float *)w.attn_norm, ap.xn_hi, HL ? ap.xn_lo : nullptr, H, d.eps)))
            return e;
        if (!normed) mark(DS4G_K_P_NORM);
        a.n_out = d.RQ + d.RKV, a.k = H, a.piece_rows = d.RQ, a.x_col0 = 0;
        if ((e = tc::launch<false, HL>(m.wqa, m.wkva, am.xn_hi, am.xn_lo, a, EpiHiLo{ap.c_hi, HL ? ap.c_lo : nullptr, d.RQ + d.RKV},
                                   ny, nsm, st)))
            return e;
        mark(DS4G_K_P_QKV_A);
        a.n_out = d.QD, a.k = d.RQ, a.piece_rows = 0, a.x_col0 = 0;
        const bool attn_tc = kvm != nullptr;   // tcgen05 attention: queries as hi/lo BF16
        if (attn_tc) {
            bf16 *q_hi = (bf16 *)pb.Q, *q_lo = q_hi + (size_t)pb.P * d.QD;
            if ((e = tc::launch<false, HL>(m.wqb, m.wqb, am.c_hi, am.c_lo, a,
                                       EpiQRopeHiLo{q_hi, HL ? q_lo : nullptr, rope, d.QD, d.HD, p0}, ny, nsm, st)))
                return e;
            mark(DS4G_K_P_Q_B);
        } else if ((e = tc::launch<false, HL>(m.wqb, m.wqb, am.c_hi, am.c_lo, a,
                                          EpiQRope{(float *)pb.Q, rope, d.QD, d.HD, p0}, ny, nsm, st))) {
            return e;
        }
        if (!attn_tc) mark(DS4G_K_P_Q_B);
        a.n_out = 2 * d.HD, a.k = d.RKV, a.piece_rows = d.HD, a.x_col0 = d.RQ;
        if ((e = tc::launch<false, HL>(m.wkb, m.wvb, am.c_hi, am.c_lo, a, EpiKVRope<TKV>{kc, vc, rope, d.HD, p0}, ny,
                                   nsm, st)))
            return e;
        mark(DS4G_K_P_KV_B);
        if (attn_tc) {
            if ((e = attn_prefill_tc(d, am.q_hi, am.q_lo, kvm[l], am.oa_hi, am.oa_lo, p0, n, pb.status, st,
                                     nsm, HL)))
                return e;
        } else if constexpr (std::is_same<TKV, bf16>::value) {
            if (attn_mma_eligible(d)) {
                k_attn_prefill_mma<<<(n + kAttnTB - 1) / kAttnTB, 256, attn_mma_smem(d), st>>>(
                    (const float *)pb.Q, ap.o_hi, ap.o_lo, kc, vc, p0, n, d);
                ++launch_count();
                if ((e = cudaGetLastError())) return e;
            } else if ((e = attn_prefill_hilo<TKV>(d, (const float *)pb.Q, ap.o_hi, ap.o_lo, kc, vc, p0, n, st))) {
                return e;
            }
        } else if ((e = attn_prefill_hilo<TKV>(d, (const float *)pb.Q, ap.o_hi, ap.o_lo, kc, vc, p0, n, st))) {
            return e;
        }
        mark(DS4G_K_P_ATTN);
        a.n_out = H, a.k = d.QD, a.piece_rows = 0, a.x_col0 = 0;
        if ((e = tc::launch<false, HL>(m.wo, m.wo, am.o_hi, am.o_lo, a, EpiAddX{pb.X, H}, ny, nsm, st)))
            return e;
        mark(DS4G_K_P_WO);
        // ---- MoE half
        if ((e = launch_pdl(k_rmsnorm_hilo, dim3(n), dim3(rmsnorm_threads(H)), 0, st, (const float *)pb.X,
                            (const float *)w.ffn_norm, ap.xn_hi, ap.xn_lo, H, d.eps)))
            return e;
        mark(DS4G_K_P_NORM);
        // The shared expert's gate/up and down read only the FFN RMSNorm and write the
        // residual before the combine: on the side stream they overlap the router, the
        // top-k, the grouping and the routed GEMMs (not in timing mode).
        const bool fork = pb.side && !pb.tm;
        cudaStream_t sst = fork ? pb.side : st;
        if (fork) {
            if ((e = cudaEventRecord(pb.ev_fork, st))) return e;
            if ((e = cudaStreamWaitEvent(pb.side, pb.ev_fork, 0))) return e;
        }
        auto shared_gu = [&]() -> cudaError_t {
            tc::Args sa = a;
            sa.ksplit = 0, sa.n_out = I, sa.k = H;
            return tc::launch<true, HL>(m.wsg, m.wsu, am.xn_hi, am.xn_lo, sa,
                                        EpiSwiGLU{ap.hs_hi, HL ? ap.hs_lo : nullptr, I}, ny, nsm, sst);
        };
        auto shared_down = [&]() -> cudaError_t {
            tc::Args sa = a;
            sa.ksplit = 0, sa.n_out = H, sa.k = I;
            return tc::launch<false, HL>(m.wsd, m.wsd, am.hs_hi, am.hs_lo, sa, EpiAddX{pb.X, H}, ny, nsm, sst);
        };
        if (fork) {
            if ((e = shared_gu())) return e;
            if ((e = shared_down())) return e;
            if ((e = cudaEventRecord(pb.ev_join, pb.side))) return e;
        }
        // The router's reduction in fixed parts (twice the tiles on the SMs; the parts'
        // scores are summed in order by the top-k), whatever the chunk.
        const int parts = router_parts(d.E);
        a.n_out = d.E, a.k = H, a.ksplit = parts;
        const size_t part = (size_t)pb.P * d.E;
        if ((e = tc::launch<false, true>(m.wr, m.wr, am.xn_hi, am.xn_lo, a, EpiScores{pb.S, d.E, part}, ny, nsm,
                                         st)))
            return e;
        mark(DS4G_K_P_ROUTER);
        a.ksplit = 0;
        if ((e = launch_pdl(k_router_topk, dim3((n * 32 + 255) / 256), dim3(256), 0, st, (const float *)pb.S,
                            parts, part, pb.ids, pb.wts, n, d.E, K, pb.status)))
            return e;
        mark(DS4G_K_P_TOPK);
        if ((e = group_by_expert(pb, nent, d.E, tc::BT, st))) return e;
        mark(DS4G_K_P_GROUP);
        // routed gate/up + SwiGLU (grouped; the GEMM gathers each group's token rows of
        // the normalised input itself), then the shared expert's
        tc::Args g{};
        g.status = pb.status;
        g.m_tok = n;
        g.n_out = I, g.k = H, g.tiles = pb.tiles, g.off = pb.off;
        g.grow = pb.rows, g.gdiv = K, g.gx_hi = ap.xn_hi, g.gx_lo = ap.xn_lo, g.gld = H;
        if ((e = tc::launch<true, HL>(m.wg, m.wu, am.xn_hi, am.xn_lo, g, EpiSwiGLU{ap.hg_hi, HL ? ap.hg_lo : nullptr, I}, max_tiles,
                                  nsm, st)))
            return e;
        mark(DS4G_K_P_GATE_UP);
        g.grow = nullptr;
        if (!fork) {
            if ((e = shared_gu())) return e;
            mark(DS4G_K_P_SHARED_GU);
        }
        // routed down (grouped) into per-(token, slot) rows; the shared expert's down
        // projection into the residual; then the weighted routed rows, slot order
        // The routed rows are FP32 with hi/lo activations, else BF16: each expert's
        // output is rounded once before the fixed-order weighted sum, and the down GEMM
        // writes and the combine reads half the bytes.
        using TY = std::conditional_t<HL, float, bf16>;
        TY *ys = reinterpret_cast<TY *>(pb.YS);
        g.n_out = H, g.k = I;
        if ((e = tc::launch<false, HL>(m.wd, m.wd, am.hg_hi, am.hg_lo, g, EpiRoutedRows<TY>{ys, pb.rows, H, nent, pb.status},
                                   max_tiles, nsm, st)))
            return e;
        mark(DS4G_K_P_DOWN);
        if (!fork) {
            if ((e = shared_down())) return e;
            mark(DS4G_K_P_SHARED_DOWN);
        } else if ((e = cudaStreamWaitEvent(st, pb.ev_join, 0))) {
            return e;
        }
        const float *gn = l + 1 < d.L ? layers[l + 1].attn_norm : nullptr;
        if ((e = launch_pdl(k_moe_combine<TY>, dim3(n), dim3(256), 0, st, pb.X, (const TY *)ys,
                            (const float *)pb.wts, H, K, gn, d.eps, ap.xn_hi, HL ? ap.xn_lo : nullptr)))
            return e;
        mark(DS4G_K_P_COMBINE);
        normed = gn != nullptr;
    }
    return cudaGetLastError();
}

cudaError_t prefill_chunk_tc(const Dims &d, const LayerPtrs *layers, const TcLayerMaps *lm,
                             const TcActMaps &am, const TcKVMaps *kvm, void *const *kc, void *const *vc,
                             const float2 *rope, const uint16_t *tok_embd, const PrefillBufs &pb, int p0, int n,
                             cudaStream_t st, int nsm, bool hilo)
{
    if (d.kvdt != DS4G_BF16)
        return hilo ? chunk_tc_t<float, true>(d, layers, lm, am, nullptr, kc, vc, rope, tok_embd, pb, p0, n, st, nsm)
                    : chunk_tc_t<float, false>(d, layers, lm, am, nullptr, kc, vc, rope, tok_embd, pb, p0, n, st,
                                               nsm);
    return hilo ? chunk_tc_t<bf16, true>(d, layers, lm, am, kvm, kc, vc, rope, tok_embd, pb, p0, n, st, nsm)
                : chunk_tc_t<bf16, false>(d, layers, lm, am, kvm, kc, vc, rope, tok_embd, pb, p0, n, st, nsm);
}

}  // namespace ds4g
