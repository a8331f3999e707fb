// Shared device helpers and host-side structures of the ds4g library.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ds4g.h"

namespace ds4g {

using bf16 = __nv_bfloat16;

// Model dimensions, copied into every kernel's arguments.
struct Dims {
    int L, H, NH, HD, RQ, RKV, W, E, K, I, V, QD;  // QD = NH * HD
    float eps;
    int wdt, kvdt;
};

// One layer's weight pointers (device).
struct LayerPtrs {
    const float *attn_norm;
    const void *wq_a, *wq_b, *wkv_a, *wk_b, *wv_b, *wo;
    const float *ffn_norm;
    const void *w_router, *w_gate, *w_up, *w_down, *ws_gate, *ws_up, *ws_down;
};

// Decode-step activations (device, inside the session buffer).
struct DecodeBufs {
    float *x;        // [H]   residual: layer input, then layer output
    float *xm;       // [H]   residual after the attention half
    float *xn2;      // [H]   normalised residual entering the MoE
    float *c;        // [RQ+RKV] Q and KV latents
    float *q;        // [QD]  queries after RoPE
    float *o;        // [QD]  attention output
    float *scores;   // [E]   router scores
    int *ids;        // [L*K] selected experts per layer
    float *wts;      // [L*K] their weights
    float *h;        // [(K+1)*I] SwiGLU hidden
    float *logits;   // [V]
    float *hidden;   // [H]   final hidden state
    unsigned *counters;  // [8] grid-completion tickets (reset by their last user)
    int *status;         // session status word (DS4G_* error raised on the device)
    float *layer_x;      // optional [L+1][H]: the residual entering each layer (row 0 the
                         // embedding), then the final hidden state; null: not recorded
    float *x_out;        // optional [H]: the final hidden state written here as well (the
                         // device view of a pinned host buffer); persistent kernel only
};

// Arguments of every decode kernel: one layer at one position.
struct StepArgs {
    Dims d;
    LayerPtrs w;
    void *kc, *vc;          // this layer's K and V caches [n_ctx][HD]
    const float2 *rope;     // [n_ctx][HD/2] (cos, sin)
    DecodeBufs b;
    const uint16_t *tok_embd;
    const void *lm_head;
    int layer, pos, token;  // token >= 0 only for the first layer's first kernel
};

// Arguments of the persistent decode kernel: every layer of one token.
struct PersistArgs {
    Dims d;
    const LayerPtrs *layers;   // device [L]
    void *const *kc;           // device [L]
    void *const *vc;           // device [L]
    const float2 *rope;
    DecodeBufs b;
    const uint16_t *tok_embd;
    const void *lm_head;
    int pos, token, logits;
    unsigned *bar;             // [0] grid-barrier arrivals, [1] K/V rows published (both only grow)
    unsigned bar_base;         // its value when this launch starts
    unsigned kv_base;          // value of the K/V-row counter (bar[1]) when this launch starts
    unsigned *qflag;           // [NH] query halves published, per head (split queries; only grow)
    unsigned q_base;           // value of every qflag entry when this launch starts
    int split_q;               // each head's queries are computed by two CTAs (2 NH + 2 <= grid)
    int *status;               // DS4G_ETIMEOUT if a barrier wait gave up
    unsigned long long *trace; // optional [events][gridDim] stage start times (ns)
    int trace_events;
    unsigned *done_flag;       // optional: device view of a pinned host word; the last CTA to
    unsigned done_seq;         // finish writes done_seq there (system-scope release) once every
                               // output of the launch is written
};

// ------------------------------------------------------------------ device helpers

// Programmatic dependent launch: wait for the preceding grid's results, and
// allow the next grid to be scheduled.  Both are no-ops without the attribute.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger()
{
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

__device__ __forceinline__ uint64_t policy_evict_first()
{
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

// 16-byte read-only streaming load that does not allocate in L1 and marks the
// line first-to-evict in L2 (weights are read once per step).
__device__ __forceinline__ uint4 ld_stream(const void *ptr, uint64_t pol)
{
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(ptr), "l"(pol));
    return r;
}

// Asynchronous bulk prefetch of [p, p + bytes) into L2 (16-byte aligned, bytes % 16 == 0).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes)
{
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

// 16-byte asynchronous global -> shared copy (no register staging) and its wait.
__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const unsigned s = (unsigned)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// Top-k of the scores s[0..E) (E <= 1024) by one warp: values sel[k] and ids[k],
// largest first, equal scores to the lower id.  A NaN ranks as -inf, so the K ids
// are always distinct valid experts; returns false if a selected score was not
// finite (the caller raises DS4G_ENONFINITE).
//  - E <= 256: lane l holds experts l, l+32, ... (at most eight), sorted once by a
//    19-comparator network; each of the K rounds is then one warp arg-max over the
//    lanes' heads, and the winning lane shifts its list.
//  - larger E: each round rescans the lane's untaken experts.
__device__ __forceinline__ bool topk_better(float va, int ia, float vb, int ib)
{
    return va > vb || (va == vb && ia < ib);
}
// One comparator of the sorting network: the better of entries I and J ends at I.
// (Template indices keep both arrays in registers; indices read from a table
// put them in local memory.)
template <int I, int J> __device__ __forceinline__ void topk_cswap(float (&v)[8], int (&id)[8])
{
    const bool sw = topk_better(v[J], id[J], v[I], id[I]);
    const float vi = v[I], vj = v[J];
    const int ii = id[I], ij = id[J];
    v[I] = sw ? vj : vi;
    v[J] = sw ? vi : vj;
    id[I] = sw ? ij : ii;
    id[J] = sw ? ii : ij;
}
__device__ __forceinline__ bool warp_topk(const float *s, int E, int K, float *sel, int *ids, int lane)
{
    bool finite = true;
    if (E <= 256) {
        float v[8];
        int id[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int e = lane + 32 * u;
            const float x = e < E ? s[e] : -INFINITY;
            v[u] = x != x ? -INFINITY : x;
            id[u] = e < E ? e : 0x7fffffff;   // padding: loses every tie to a real expert
        }
        topk_cswap<0, 2>(v, id); topk_cswap<1, 3>(v, id); topk_cswap<4, 6>(v, id);
        topk_cswap<5, 7>(v, id); topk_cswap<0, 4>(v, id); topk_cswap<1, 5>(v, id);
        topk_cswap<2, 6>(v, id); topk_cswap<3, 7>(v, id); topk_cswap<0, 1>(v, id);
        topk_cswap<2, 3>(v, id); topk_cswap<4, 5>(v, id); topk_cswap<6, 7>(v, id);
        topk_cswap<2, 4>(v, id); topk_cswap<3, 5>(v, id); topk_cswap<1, 4>(v, id);
        topk_cswap<3, 6>(v, id); topk_cswap<1, 2>(v, id); topk_cswap<3, 4>(v, id);
        topk_cswap<5, 6>(v, id);
#pragma unroll
        for (int k = 0; k < 8; ++k) {   // K <= 8
            if (k >= K) break;
            float bv = v[0];
            int bi = id[0];
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) {
                const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
                const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
                if (topk_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
            }
            sel[k] = bv;
            ids[k] = bi;
            finite = finite && isfinite(bv);
            if (id[0] == bi) {   // this lane's head was taken
#pragma unroll
                for (int u = 0; u < 7; ++u) { v[u] = v[u + 1]; id[u] = id[u + 1]; }
                v[7] = -INFINITY;
                id[7] = 0x7fffffff;
            }
        }
        return finite;
    }
    unsigned taken = 0u;  // bit j: expert lane + 32 j is already chosen
#pragma unroll
    for (int k = 0; k < 8; ++k) {   // K <= 8; fixed bounds keep sel/ids in registers
        if (k >= K) break;
        float bv = -INFINITY;
        int bi = E;  // above every id: any untaken expert beats it
        for (int e = lane, j = 0; e < E; e += 32, ++j) {
            if ((taken >> j) & 1u) continue;
            float v = s[e];
            if (v != v) v = -INFINITY;
            if (topk_better(v, e, bv, bi)) { bv = v; bi = e; }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
            if (topk_better(ov, oi, bv, bi)) { bv = ov; bi = oi; }
        }
        sel[k] = bv;
        ids[k] = bi;
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        finite = finite && isfinite(bv);
    }
    return finite;
}

// Order-preserving 32-bit key of a score: for non-NaN floats a, b (with -0 taken
// as +0), a > b exactly when key(a) > key(b), and a == b when the keys are equal.
__device__ __forceinline__ unsigned topk_key(float v)
{
    const unsigned u = __float_as_uint(v == 0.f ? 0.f : v);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float topk_unkey(unsigned k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}
template <int I, int J> __device__ __forceinline__ void topk_cswap_key(unsigned (&k)[8], int (&id)[8])
{
    const bool sw = k[J] > k[I] || (k[J] == k[I] && id[J] < id[I]);
    const unsigned ki = k[I], kj = k[J];
    const int ii = id[I], ij = id[J];
    k[I] = sw ? kj : ki;
    k[J] = sw ? ki : kj;
    id[I] = sw ? ij : ii;
    id[J] = sw ? ii : ij;
}
// The same selection as warp_topk for E <= 256, from registers: lane l passes the
// scores of experts l, l+32, ... in x[0..8).  Each of the K rounds is two warp
// reductions (redux.sync): the largest head key, then the lowest id among the
// lanes holding it; the warp-wide shuffle butterfly of warp_topk takes five
// dependent exchange steps per round instead.
__device__ __forceinline__ bool warp_topk_r256(const float (&x)[8], int E, int K, float *sel, int *ids,
                                               int lane)
{
    unsigned k8[8];
    int id[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
        const int e = lane + 32 * u;
        const float v = e < E ? x[u] : -INFINITY;
        k8[u] = topk_key(v != v ? -INFINITY : v);
        id[u] = e < E ? e : 0x7fffffff;   // padding: loses every tie to a real expert
    }
    topk_cswap_key<0, 2>(k8, id); topk_cswap_key<1, 3>(k8, id); topk_cswap_key<4, 6>(k8, id);
    topk_cswap_key<5, 7>(k8, id); topk_cswap_key<0, 4>(k8, id); topk_cswap_key<1, 5>(k8, id);
    topk_cswap_key<2, 6>(k8, id); topk_cswap_key<3, 7>(k8, id); topk_cswap_key<0, 1>(k8, id);
    topk_cswap_key<2, 3>(k8, id); topk_cswap_key<4, 5>(k8, id); topk_cswap_key<6, 7>(k8, id);
    topk_cswap_key<2, 4>(k8, id); topk_cswap_key<3, 5>(k8, id); topk_cswap_key<1, 4>(k8, id);
    topk_cswap_key<3, 6>(k8, id); topk_cswap_key<1, 2>(k8, id); topk_cswap_key<3, 4>(k8, id);
    topk_cswap_key<5, 6>(k8, id);
    bool finite = true;
#pragma unroll
    for (int k = 0; k < 8; ++k) {   // K <= 8
        if (k >= K) break;
        const unsigned m = __reduce_max_sync(0xffffffffu, k8[0]);
        const unsigned bi = __reduce_min_sync(0xffffffffu, k8[0] == m ? (unsigned)id[0] : 0x7fffffffu);
        const float bv = topk_unkey(m);
        sel[k] = bv;
        ids[k] = (int)bi;
        finite = finite && isfinite(bv);
        if (k8[0] == m && (unsigned)id[0] == bi) {   // this lane's head was taken
#pragma unroll
            for (int u = 0; u < 7; ++u) { k8[u] = k8[u + 1]; id[u] = id[u + 1]; }
            k8[7] = topk_key(-INFINITY);
            id[7] = 0x7fffffff;
        }
    }
    return finite;
}

// SwiGLU of one gate/up pair: silu(g) * u.
__device__ __forceinline__ float silu_mul(float g, float u) { return g / (1.f + expf(-g)) * u; }

// An FP32 value as a BF16 pair: hi = bf16(v), lo = bf16(v - hi); hi + lo carries
// about 16 significant bits of v.
__device__ __forceinline__ void split_hilo(float v, bf16 &h, bf16 &l)
{
    h = __float2bfloat16_rn(v);
    l = __float2bfloat16_rn(v - __bfloat162float(h));
}
// Two BF16 values in one 32-bit word, a in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(bf16 a, bf16 b)
{
    return (uint32_t)__bfloat16_as_ushort(a) | ((uint32_t)__bfloat16_as_ushort(b) << 16);
}

// split_hilo of two values, each half packed as a BF16 pair (a in the low half).
__device__ __forceinline__ void split2_hilo(float a, float b, uint32_t &hi, uint32_t &lo)
{
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    const __nv_bfloat162 l = __floats2bfloat162_rn(a - __low2float(h), b - __high2float(h));
    hi = *reinterpret_cast<const uint32_t *>(&h);
    lo = *reinterpret_cast<const uint32_t *>(&l);
}

template <typename T> struct VecOf;
template <> struct VecOf<bf16> { static constexpr int n = 8; };
template <> struct VecOf<float> { static constexpr int n = 4; };

// acc += dot(16 bytes of weights, x[0..n)) with x 16-byte aligned in shared memory.
template <typename TW> __device__ __forceinline__ float dotv(const uint4 &w, const float *x,
                                                            float acc);
template <> __device__ __forceinline__ float dotv<bf16>(const uint4 &w, const float *x, float acc)
{
    const float4 a = *reinterpret_cast<const float4 *>(x);
    const float4 b = *reinterpret_cast<const float4 *>(x + 4);
    acc = fmaf(__uint_as_float(w.x << 16), a.x, acc);
    acc = fmaf(__uint_as_float(w.x & 0xffff0000u), a.y, acc);
    acc = fmaf(__uint_as_float(w.y << 16), a.z, acc);
    acc = fmaf(__uint_as_float(w.y & 0xffff0000u), a.w, acc);
    acc = fmaf(__uint_as_float(w.z << 16), b.x, acc);
    acc = fmaf(__uint_as_float(w.z & 0xffff0000u), b.y, acc);
    acc = fmaf(__uint_as_float(w.w << 16), b.z, acc);
    acc = fmaf(__uint_as_float(w.w & 0xffff0000u), b.w, acc);
    return acc;
}
template <> __device__ __forceinline__ float dotv<float>(const uint4 &w, const float *x, float acc)
{
    const float4 a = *reinterpret_cast<const float4 *>(x);
    acc = fmaf(__uint_as_float(w.x), a.x, acc);
    acc = fmaf(__uint_as_float(w.y), a.y, acc);
    acc = fmaf(__uint_as_float(w.z), a.z, acc);
    acc = fmaf(__uint_as_float(w.w), a.w, acc);
    return acc;
}

// Per-lane partial dot products of R weight rows (global) with one vector xs
// (shared memory), over nvec 16-byte vectors.  Lane l takes vectors l, l+32, ...;
// U vectors per row are in flight at once.  Reduce with warp_sum afterwards.
template <typename TW, int R, int U>
__device__ __forceinline__ void gemv_rows(const TW *const (&rows)[R], const float *xs, int nvec,
                                          float (&acc)[R], int lane, uint64_t pol)
{
    constexpr int VEC = VecOf<TW>::n;
    for (int v0 = lane; v0 < nvec; v0 += 32 * U) {
        uint4 w[R][U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
#pragma unroll
            for (int r = 0; r < R; ++r)
                w[r][u] = (v < nvec) ? ld_stream(rows[r] + (size_t)v * VEC, pol)
                                     : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int v = v0 + 32 * u;
            if (v < nvec) {
#pragma unroll
                for (int r = 0; r < R; ++r) acc[r] = dotv<TW>(w[r][u], xs + v * VEC, acc[r]);
            }
        }
    }
}

// Block-wide sum (fixed order: per-warp shuffle tree, then warp 0 over warps).
__device__ __forceinline__ float block_sum(float v, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_sum(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    float t = 0.f;
    if (warp == 0) {
        t = lane < nw ? red[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    t = red[0];
    return t;
}

__device__ __forceinline__ float block_max(float v, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    v = warp_max(v);
    __syncthreads();
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        float t = lane < nw ? red[lane] : -INFINITY;
        t = warp_max(t);
        if (lane == 0) red[0] = t;
    }
    __syncthreads();
    return red[0];
}

template <typename T> __device__ __forceinline__ float to_f32(T v);
template <> __device__ __forceinline__ float to_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ float to_f32<bf16>(bf16 v) { return __bfloat162float(v); }

template <typename T> __device__ __forceinline__ T from_f32(float v);
template <> __device__ __forceinline__ float from_f32<float>(float v) { return v; }
template <> __device__ __forceinline__ bf16 from_f32<bf16>(float v) { return __float2bfloat16_rn(v); }

// ------------------------------------------------------------------ host helpers

// Kernels launched by the calling thread (a session has one owner thread).
inline uint64_t &launch_count()
{
    static thread_local uint64_t n = 0;
    return n;
}

// Allow a kernel the largest dynamic shared memory the device offers beside its
// static shared memory.
static inline cudaError_t allow_max_dyn_smem(const void *f, int optin)
{
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, f);
    if (e) return e;
    return cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                optin - (int)fa.sharedSizeBytes);
}

// Launch with programmatic stream serialisation so the kernel may be scheduled
// while its predecessor drains (the kernel itself waits with pdl_wait()).
template <typename... KArgs, typename... Args>
static inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block,
                                     size_t smem, cudaStream_t st, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    ++launch_count();
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace ds4g
