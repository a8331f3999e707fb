// Persistent decode step: every layer of one token (page "ds4.c 学习笔记 --
// 端到端推理流程", 阶段四 4.2, run once per layer) and optionally the lm_head (4.3)
// in ONE cooperative launch of one CTA per SM.
//
// Batch-1 decode streams 275 MB of weights per layer and does almost no math
// with them, so the whole design is about keeping HBM busy:
//  - Warp 11 of every CTA is a producer: one thread walks the CTA's share of every
//    stage's weight rows, in stage order, and copies them with TMA bulk copies
//    (cp.async.bulk, 16 KB per item) into a ring of shared-memory slots guarded by
//    full/empty mbarriers.  Weights do not depend on the token, so the producer
//    runs ahead across stage boundaries, grid barriers and the small stages
//    (attention, router); only the routed experts wait for this layer's top-k.
//  - Warps 0-10 consume.  Item i lands in slot i mod 11 and is taken by warp
//    i mod 11, so every warp owns one slot and waits only for that slot's next
//    phase (an mbarrier parity wait cannot tell phase k from phase k+2).  The warp
//    dots the item's rows with the stage's activation vector (also in shared
//    memory) with several loads and accumulators in flight, frees the slot, and
//    only then runs the stage's epilogue, so epilogue latency never holds a slot.
//  - Stages are separated by grid-wide barriers among the consumer threads
//    (named barrier 1 inside the CTA, then an arrival counter + generation word).
//    Activations written by other CTAs in this launch are read through L2.
//  - Each CTA owns a contiguous, balanced share of each stage's rows, so copies
//    are large and contiguous.
//  - Every wait (mbarrier or grid barrier) gives up after a bounded time, raises
//    the session's status word and lets the CTA return: nothing can hang.
//  - Reductions have a fixed order; the expert down-projections keep per-expert
//    partial sums and combine them in slot order, so results do not depend on
//    timing.
#include <algorithm>

#include "common.cuh"
#include "kernels.h"
#include "sm100.cuh"

namespace ds4g {

static constexpr int kNSlot = 11;                   // ring slots
static constexpr int kNC = kNSlot;                  // consumer warps, one per slot
static constexpr int kCT = kNC * 32;                // consumer threads
static constexpr int kPThreads = kCT + 32;          // + the producer warp
static constexpr int kDoneTicket = 1;              // DecodeBufs::counters slot of the completion ticket
static constexpr int kSlot = 16384;                 // bytes per ring slot
static constexpr int kMaxR = 32;                    // rows per item at most

// ------------------------------------------------------------------ helpers

// Barrier among the consumer warps only (the producer never joins).
__device__ __forceinline__ void csync() { asm volatile("bar.sync 1, %0;" ::"r"(kCT) : "memory"); }

// Optional device self-checks (built with -DDS4G_DEVICE_CHECKS): a violated
// condition is recorded in the status word as 1000 + site and the access skipped.
#ifdef DS4G_DEVICE_CHECKS
#define DS4G_CHECK(cond, site, status)                      \
    (!(cond) ? (atomicCAS((status), 0, 1000 + (site)), false) : true)
#else
#define DS4G_CHECK(cond, site, status) true
#endif

// ------------------------------------------------------------------ shared state

struct Shared {
    uint64_t full[kNSlot];
    uint64_t empty[kNSlot];
    uint64_t scores_ready;    // one arrival per layer: router scores complete (consumers)
    uint64_t ids_ready;       // one arrival per layer: top-k known (producer warp)
    LayerPtrs lw[2];          // consumers' copy of layer l's pointers in lw[l & 1]
    int ids[8];
    float w[9];
    int abort_flag;
    float red[32];
};

// Tracing: thread 0 stamps the start of stage `ev` of this launch.
__device__ __forceinline__ void stamp(const PersistArgs &a, int ev)
{
    if (a.trace && threadIdx.x == 0 && ev < a.trace_events)
        a.trace[(size_t)ev * gridDim.x + blockIdx.x] = global_ns();
}

// Grid barrier among consumer threads of all CTAs; false if it gave up.  The
// arrival counter only grows: barrier k of the launch is complete once it reaches
// bar_base + k * gridDim.x (bar_base: arrivals of earlier launches, from the host).
// Thread 0 adds its arrival with release semantics (covering the CTA's writes,
// ordered by the named barrier before it) and polls with acquire loads.
__device__ __forceinline__ bool grid_sync(const PersistArgs &a, unsigned &target, Shared &S)
{
    csync();
    if (threadIdx.x == 0) {
        target += gridDim.x;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(a.bar) : "memory");
        const long long t0 = clock64();
        while ((int)(ld_acquire_gpu(a.bar) - target) < 0) {
            if (clock64() - t0 > kWaitCycles) {
                atomicExch(a.status, DS4G_ETIMEOUT);
                S.abort_flag = 1;
                break;
            }
        }
    }
    csync();
    return *(volatile int *)&S.abort_flag == 0;
}

// L2 prefetch of a byte range (16-byte aligned start and size), in bulk requests.
__device__ __forceinline__ void prefetch_range(const void *p, size_t bytes)
{
    const char *c = static_cast<const char *>(p);
    while (bytes > 0) {
        const uint32_t n = (uint32_t)(bytes < ((size_t)1 << 20) ? bytes : ((size_t)1 << 20));
        prefetch_l2(c, n);
        c += n;
        bytes -= n;
    }
}

// ------------------------------------------------------------------ work items
// A stage's weight rows come in pieces (matrices); each piece is cut into chunks
// of whole rows of at most kSlot bytes (and kMaxR rows, an even number).  A CTA
// owns a contiguous, balanced range of the stage's chunks.  Producer and
// consumers enumerate the same sequence.

struct Piece {
    const void *base;
    int rows, K;       // rows of K elements
    int rpc;           // rows per chunk
};

__device__ __forceinline__ int chunks_of(const Piece &p) { return (p.rows + p.rpc - 1) / p.rpc; }

template <typename TW> __device__ __forceinline__ Piece piece(const void *b, int rows, int K)
{
    Piece p;
    p.base = b;
    p.rows = rows;
    p.K = K;
    p.rpc = min(kMaxR, max(1, kSlot / (K * (int)sizeof(TW))));
    if (p.rpc > 1) p.rpc &= ~1;   // even, so RoPE pairs never straddle chunks
    return p;
}

// Stages 2-3 of a layer are one stage.  CTA h < NH computes the queries of head h
// (its HD rows of W_qb) and attends for that head; CTA NH computes the new K row
// (W_kb) and CTA NH+1 the new V row (W_vb), and they publish them through the kv
// counter.  With split queries (2 NH + 2 CTAs or more), CTA h computes only the
// first HD/2 query rows of head h and CTA NH+2+h the second half, which it writes
// to global memory and publishes through the head's query flag; the work of a
// head CTA before its attention halves.  Other CTAs have no work in it.
// kind: 0 head, 1 K, 2 V, 3 second query half, -1 none.
__device__ __forceinline__ int qkv_kind(int nh, int split)
{
    const int c = blockIdx.x;
    if (c < nh) return 0;
    if (c == nh) return 1;
    if (c == nh + 1) return 2;
    return split && c < 2 * nh + 2 ? 3 : -1;
}
// The head a kind-0 or kind-3 CTA serves, and the first query row it computes.
__device__ __forceinline__ int qkv_head(int nh, int kind)
{
    return kind == 3 ? (int)blockIdx.x - nh - 2 : (int)blockIdx.x;
}
__device__ __forceinline__ int qkv_row0(const Dims &d, int kind) { return kind == 3 ? d.HD / 2 : 0; }
template <typename TW>
__device__ __forceinline__ Piece qkv_piece(const LayerPtrs &w, const Dims &d, int kind, int split)
{
    if (kind == 0 || kind == 3) {
        const int h = qkv_head(d.NH, kind), rows = split ? d.HD / 2 : d.HD;
        return piece<TW>(static_cast<const TW *>(w.wq_b) + ((size_t)h * d.HD + qkv_row0(d, kind)) * d.RQ, rows,
                         d.RQ);
    }
    return piece<TW>(kind == 1 ? w.wk_b : w.wv_b, d.HD, d.RKV);
}

__device__ __forceinline__ void cta_range(int n, int &lo, int &hi)
{
    lo = (int)((long long)n * blockIdx.x / gridDim.x);
    hi = (int)((long long)n * (blockIdx.x + 1) / gridDim.x);
}

struct Chunk {
    int piece, row0, nrows;
};

template <int NP>
__device__ __forceinline__ Chunk locate(const Piece (&P)[NP], int j)
{
    Chunk c{0, 0, 0};
#pragma unroll
    for (int p = 0; p < NP; ++p) {
        const int n = chunks_of(P[p]);
        if (j < n) {
            c.piece = p;
            c.row0 = j * P[p].rpc;
            c.nrows = min(P[p].rpc, P[p].rows - c.row0);
            return c;
        }
        j -= n;
    }
    return c;
}

template <int NP> __device__ __forceinline__ int total_chunks(const Piece (&P)[NP])
{
    int n = 0;
#pragma unroll
    for (int p = 0; p < NP; ++p) n += chunks_of(P[p]);
    return n;
}

// ------------------------------------------------------------------ consumer math

// Activation vectors in shared memory are stored in a lane-friendly order.  With
// 16-byte weight vectors of VEC elements, lane t of a warp reads weight vector
// v = 32*blk + t and needs the VEC activations x[v*VEC ..].  For BF16 weights
// (VEC = 8) those are two float4s; stored plainly they sit 32 bytes apart and a
// warp's float4 load hits every bank pair twice.  So within each block of 32
// vectors the first halves of all vectors come first, then the second halves:
// each float4 load of a warp is one contiguous 512-byte run (no bank conflict).
// A partial last block of m vectors keeps the same shape with m in place of 32.
// For FP32 weights (VEC = 4) the plain order is already conflict-free.
// `xperm4` maps the float4 index f of a segment of nvec vectors to its slot.
template <typename TW> __device__ __forceinline__ int xperm4(int f, int nvec);
template <> __device__ __forceinline__ int xperm4<float>(int f, int) { return f; }
template <> __device__ __forceinline__ int xperm4<bf16>(int f, int nvec)
{
    const int v = f >> 1, h = f & 1, blk = v >> 5, t = v & 31;
    const int m = min(32, nvec - (blk << 5));
    return (blk << 6) + h * m + t;
}

// The activations lane-vector v needs, loaded from the permuted layout.
template <typename TW> struct XFrag;
template <> struct XFrag<bf16> {
    float4 a, b;
    __device__ __forceinline__ void zero() { a = b = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void load(const float4 *x4, int v, int nvec)
    {
        const int blk = v >> 5, t = v & 31, m = min(32, nvec - (blk << 5));
        a = x4[(blk << 6) + t];
        b = x4[(blk << 6) + m + t];
    }
    // Two-wide FP32 FMAs: the even and the odd weights of the vector accumulate in
    // the two halves of acc (a BF16 pair widens to two floats with one shift and one
    // mask).
    __device__ __forceinline__ float2 dot(const uint4 &w, float2 acc) const
    {
        acc = __ffma2_rn(make_float2(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u)),
                         make_float2(a.x, a.y), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u)),
                         make_float2(a.z, a.w), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(w.z << 16), __uint_as_float(w.z & 0xffff0000u)),
                         make_float2(b.x, b.y), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(w.w << 16), __uint_as_float(w.w & 0xffff0000u)),
                         make_float2(b.z, b.w), acc);
        return acc;
    }
};
template <> struct XFrag<float> {
    float4 a;
    __device__ __forceinline__ void zero() { a = make_float4(0.f, 0.f, 0.f, 0.f); }
    __device__ __forceinline__ void load(const float4 *x4, int v, int) { a = x4[v]; }
    __device__ __forceinline__ float2 dot(const uint4 &w, float2 acc) const
    {
        acc = __ffma2_rn(make_float2(__uint_as_float(w.x), __uint_as_float(w.y)), make_float2(a.x, a.y), acc);
        acc = __ffma2_rn(make_float2(__uint_as_float(w.z), __uint_as_float(w.w)), make_float2(a.z, a.w), acc);
        return acc;
    }
};
__device__ __forceinline__ float hsum(float2 v) { return v.x + v.y; }

// Vectors per lane kept in registers by the short-row path (32 floats of x).
template <typename TW> struct ShortRow { static constexpr int NU = 32 / VecOf<TW>::n; };

// Dot products of `nr` rows (stride K, shared memory) with the permuted vector x,
// by one warp; the warp-reduced result of row r goes to res[r] (lane 0).  Lane t
// takes 16-byte vectors t, t+32, ...
//  - Short rows (K/VEC <= 32*NU): the lane's x fragments are loaded once into
//    registers and reused for every row, two rows at a time.  (A transposed
//    butterfly that reduces eight rows at once is faster in isolation but made the
//    whole decode step slower.)
//  - Long rows: two rows share each x fragment load; four weight vectors per row
//    are in flight and two accumulators alternate.
// Not inlined: every stage runs the same copy, which stays in the instruction cache.
template <typename TW>
__device__ __noinline__ void warp_dots(const TW *rows, int nr, int K, const float *x, float *res,
                                       int lane)
{
    constexpr int VEC = VecOf<TW>::n;
    constexpr int NU = ShortRow<TW>::NU;
    const int nvec = K / VEC;
    const float4 *x4 = reinterpret_cast<const float4 *>(x);
    const uint4 *w4 = reinterpret_cast<const uint4 *>(rows);   // row r starts at r * nvec
    if (nvec <= 32 * NU) {
        XFrag<TW> xf[NU];
#pragma unroll
        for (int u = 0; u < NU; ++u) {
            xf[u].zero();   // lanes past the end multiply zero weights by zeros
            if (lane + 32 * u < nvec) xf[u].load(x4, lane + 32 * u, nvec);
        }
        int r = 0;
        for (; r + 1 < nr; r += 2) {
            const uint4 *r0 = w4 + (size_t)r * nvec, *r1 = r0 + nvec;
            uint4 q0[NU], q1[NU];
#pragma unroll
            for (int u = 0; u < NU; ++u) {
                const int v = lane + 32 * u;
                q0[u] = v < nvec ? r0[v] : make_uint4(0, 0, 0, 0);
                q1[u] = v < nvec ? r1[v] : make_uint4(0, 0, 0, 0);
            }
            float2 a0 = {0.f, 0.f}, a1 = {0.f, 0.f}, b0 = {0.f, 0.f}, b1 = {0.f, 0.f};
#pragma unroll
            for (int u = 0; u < NU; u += 2) {
                a0 = xf[u].dot(q0[u], a0);
                a1 = xf[u].dot(q1[u], a1);
                if (u + 1 < NU) {
                    b0 = xf[u + 1].dot(q0[u + 1], b0);
                    b1 = xf[u + 1].dot(q1[u + 1], b1);
                }
            }
            const float s0 = warp_sum(hsum(a0) + hsum(b0));
            const float s1 = warp_sum(hsum(a1) + hsum(b1));
            if (lane == 0) {
                res[r] = s0;
                res[r + 1] = s1;
            }
        }
        if (r < nr) {
            const uint4 *r0 = w4 + (size_t)r * nvec;
            float2 a0 = {0.f, 0.f}, b0 = {0.f, 0.f};
#pragma unroll
            for (int u = 0; u < NU; u += 2) {
                const int v = lane + 32 * u;
                if (v < nvec) a0 = xf[u].dot(r0[v], a0);
                if (u + 1 < NU && v + 32 < nvec) b0 = xf[u + 1].dot(r0[v + 32], b0);
            }
            const float s0 = warp_sum(hsum(a0) + hsum(b0));
            if (lane == 0) res[r] = s0;
        }
        return;
    }
    int r = 0;
    for (; r + 1 < nr; r += 2) {
        const uint4 *r0 = w4 + (size_t)r * nvec, *r1 = r0 + nvec;
        float2 a0 = {0.f, 0.f}, a1 = {0.f, 0.f}, b0 = {0.f, 0.f}, b1 = {0.f, 0.f};
        int v = lane;
        for (; v + 96 < nvec; v += 128) {
            uint4 q0[4], q1[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                q0[u] = r0[v + 32 * u];
                q1[u] = r1[v + 32 * u];
            }
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
                XFrag<TW> xa, xb;
                xa.load(x4, v + 32 * u, nvec);
                xb.load(x4, v + 32 * (u + 1), nvec);
                a0 = xa.dot(q0[u], a0);
                a1 = xa.dot(q1[u], a1);
                b0 = xb.dot(q0[u + 1], b0);
                b1 = xb.dot(q1[u + 1], b1);
            }
        }
        for (; v < nvec; v += 32) {
            XFrag<TW> xa;
            xa.load(x4, v, nvec);
            a0 = xa.dot(r0[v], a0);
            a1 = xa.dot(r1[v], a1);
        }
        const float s0 = warp_sum(hsum(a0) + hsum(b0));
        const float s1 = warp_sum(hsum(a1) + hsum(b1));
        if (lane == 0) {
            res[r] = s0;
            res[r + 1] = s1;
        }
    }
    if (r < nr) {
        const uint4 *r0 = w4 + (size_t)r * nvec;
        float2 a0 = {0.f, 0.f}, b0 = {0.f, 0.f};
        int v = lane;
        for (; v + 96 < nvec; v += 128) {
            uint4 q0[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) q0[u] = r0[v + 32 * u];
#pragma unroll
            for (int u = 0; u < 4; u += 2) {
                XFrag<TW> xa, xb;
                xa.load(x4, v + 32 * u, nvec);
                xb.load(x4, v + 32 * (u + 1), nvec);
                a0 = xa.dot(q0[u], a0);
                b0 = xb.dot(q0[u + 1], b0);
            }
        }
        for (; v < nvec; v += 32) {
            XFrag<TW> xa;
            xa.load(x4, v, nvec);
            a0 = xa.dot(r0[v], a0);
        }
        const float s0 = warp_sum(hsum(a0) + hsum(b0));
        if (lane == 0) res[r] = s0;
    }
}

// 16 bytes of K/V storage widened to floats.
template <typename T> __device__ __forceinline__ void unpack(const uint4 &u, float *f);
template <> __device__ __forceinline__ void unpack<bf16>(const uint4 &u, float *f)
{
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int t = 0; t < 4; ++t) {
        f[2 * t] = __uint_as_float(w[t] << 16);
        f[2 * t + 1] = __uint_as_float(w[t] & 0xffff0000u);
    }
}
template <> __device__ __forceinline__ void unpack<float>(const uint4 &u, float *f)
{
    f[0] = __uint_as_float(u.x);
    f[1] = __uint_as_float(u.y);
    f[2] = __uint_as_float(u.z);
    f[3] = __uint_as_float(u.w);
}

// Consumer-thread helpers (threads 0 .. kCT-1).
__device__ __forceinline__ float csum(float v, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_sum(v);
    csync();
    if (lane == 0) red[warp] = v;
    csync();
    float t = 0.f;
    if (warp == 0) {
        t = lane < kNC ? red[lane] : 0.f;
        t = warp_sum(t);
        if (lane == 0) red[0] = t;
    }
    csync();
    t = red[0];
    return t;
}
__device__ __forceinline__ float cmax(float v, float *red)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    v = warp_max(v);
    csync();
    if (lane == 0) red[warp] = v;
    csync();
    if (warp == 0) {
        float t = lane < kNC ? red[lane] : -INFINITY;
        t = warp_max(t);
        if (lane == 0) red[0] = t;
    }
    csync();
    return red[0];
}
// Activation vector (written by other CTAs in this launch, so read through L2)
// into shared memory in the permuted order of segments of `seg` elements; up to
// eight 16-byte loads in flight per thread.  Returns this thread's partial sum of
// squares.
template <typename TW>
__device__ __noinline__ float cload(const float *src, float *dst, int n, int seg)
{
    constexpr int B = 8;
    const int nv = seg / VecOf<TW>::n, s4 = seg / 4;
    float ss = 0.f;
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    const float4 *g4 = reinterpret_cast<const float4 *>(src);
    for (int base = threadIdx.x; base < n / 4; base += kCT * B) {
        float4 v[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int f = base + j * kCT;
            v[j] = f < n / 4 ? __ldcg(g4 + f) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int f = base + j * kCT;
            if (f < n / 4) {
                const int s = f / s4, fl = f - s * s4;
                d4[s * s4 + xperm4<TW>(fl, nv)] = v[j];
                ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
            }
        }
    }
    return ss;
}
// RMSNorm input with its gain folded in: dst = x * g (permuted, one segment of n),
// where x is an activation vector written by other CTAs (read through L2) and g the
// norm gain; x and g are loaded together.  Returns this thread's partial sum of
// squares of x: the caller forms 1/rms and applies it to the dot products, since
// W (x * g / rms) = (W (x * g)) / rms.
template <typename TW>
__device__ __noinline__ float cload_g(const float *src, const float *g, float *dst, int n)
{
    constexpr int B = 6;
    const int nv = n / VecOf<TW>::n;
    float ss = 0.f;
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    const float4 *s4 = reinterpret_cast<const float4 *>(src);
    const float4 *g4 = reinterpret_cast<const float4 *>(g);
    for (int base = threadIdx.x; base < n / 4; base += kCT * B) {
        float4 v[B], gv[B];
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int f = base + j * kCT;
            v[j] = f < n / 4 ? __ldcg(s4 + f) : make_float4(0, 0, 0, 0);
            gv[j] = f < n / 4 ? __ldg(g4 + f) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < B; ++j) {
            const int f = base + j * kCT;
            if (f < n / 4) {
                d4[xperm4<TW>(f, nv)] = make_float4(v[j].x * gv[j].x, v[j].y * gv[j].y, v[j].z * gv[j].z,
                                                    v[j].w * gv[j].w);
                ss = fmaf(v[j].x, v[j].x, fmaf(v[j].y, v[j].y, fmaf(v[j].z, v[j].z, fmaf(v[j].w, v[j].w, ss))));
            }
        }
    }
    return ss;
}
// The same for the f16 embedding row (read-only); the plain row also goes to
// `plain` (the residual stream) when it is non-null.
template <typename TW>
__device__ __noinline__ float cload_f16_g(const uint16_t *src, const float *g, float *dst, int n,
                                          float *plain)
{
    const int nv = n / VecOf<TW>::n;
    float ss = 0.f;
    float4 *d4 = reinterpret_cast<float4 *>(dst);
    for (int base = threadIdx.x * 8; base < n; base += kCT * 24) {
        uint4 v[3];
        float4 g0[3], g1[3];
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int i = base + j * kCT * 8;
            const bool in = i < n;
            v[j] = in ? __ldg(reinterpret_cast<const uint4 *>(src + i)) : make_uint4(0, 0, 0, 0);
            g0[j] = in ? __ldg(reinterpret_cast<const float4 *>(g + i)) : make_float4(0, 0, 0, 0);
            g1[j] = in ? __ldg(reinterpret_cast<const float4 *>(g + i + 4)) : make_float4(0, 0, 0, 0);
        }
#pragma unroll
        for (int j = 0; j < 3; ++j) {
            const int i = base + j * kCT * 8;
            if (i < n) {
                const __half2 *h = reinterpret_cast<const __half2 *>(&v[j]);
                const float2 p0 = __half22float2(h[0]), p1 = __half22float2(h[1]);
                const float2 p2 = __half22float2(h[2]), p3 = __half22float2(h[3]);
                const float4 lo = make_float4(p0.x, p0.y, p1.x, p1.y);
                const float4 hi = make_float4(p2.x, p2.y, p3.x, p3.y);
                d4[xperm4<TW>(i / 4, nv)] =
                    make_float4(lo.x * g0[j].x, lo.y * g0[j].y, lo.z * g0[j].z, lo.w * g0[j].w);
                d4[xperm4<TW>(i / 4 + 1, nv)] =
                    make_float4(hi.x * g1[j].x, hi.y * g1[j].y, hi.z * g1[j].z, hi.w * g1[j].w);
                if (plain) {
                    *reinterpret_cast<float4 *>(plain + i) = lo;
                    *reinterpret_cast<float4 *>(plain + i + 4) = hi;
                }
                ss = fmaf(lo.x, lo.x, fmaf(lo.y, lo.y, fmaf(lo.z, lo.z, fmaf(lo.w, lo.w, ss))));
                ss = fmaf(hi.x, hi.x, fmaf(hi.y, hi.y, fmaf(hi.z, hi.z, fmaf(hi.w, hi.w, ss))));
            }
        }
    }
    return ss;
}

// Sliding-window MQA for head h: the query (after RoPE, times 1/sqrt(HD)) is in
// att[0, HD); the K/V rows of the window (positions lo_w .. pos) are read straight
// from L2 (the current row was written by another CTA of this launch).  Scores:
// `tpk` adjacent threads share a key, each holding up to eight 16-byte vectors of it
// in flight.  Output: thread t accumulates vector t % nkv of V over the keys
// j = g, g + G, ... (g = t / nkv), and the G partial sums are added in group order.
template <typename TKV, class KvWait>
__device__ __forceinline__ bool attention_head(const PersistArgs &a, int h, const TKV *kw, const TKV *vw, int n,
                                               float *att, float *red, KvWait &&kv_wait)
{
    const Dims &d = a.d;
    constexpr int KVEC = VecOf<TKV>::n;
    const int HD = d.HD, nkv = HD / KVEC;
    int tpk = 1;
    while (tpk * 8 < nkv) tpk <<= 1;
    const int kpp = kCT / tpk, G = kCT / nkv;
    const float *qs = att;           // [HD]
    float *ps = att + HD;            // [W]
    float *op = ps + d.W;            // [G][HD]
    const int t = threadIdx.x, sub = t % tpk, c = t % nkv, g = t / nkv;
    // A window that fits one pass (every key has its threads, every thread at most
    // eight V rows) issues all of its K and V loads at once.  The rows before the
    // current position are final: they are requested before waiting for the current
    // K and V rows (published by other CTAs of this launch through the kv counter).
    const bool one_pass = n <= kpp && n <= 8 * G;
    uint4 kq[8], vq[8];
    if (one_pass) {
        const int j = t / tpk;
        const uint4 *kr = reinterpret_cast<const uint4 *>(kw + (size_t)j * HD);
#pragma unroll
        for (int u = 0; u < 8; ++u) {
            const int v = sub + tpk * u;
            kq[u] = j < n - 1 && v < nkv ? __ldcg(kr + v) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int jv = g + k * G;
            vq[k] = g < G && jv < n - 1 ? __ldcg(reinterpret_cast<const uint4 *>(vw + (size_t)jv * HD) + c)
                                        : make_uint4(0, 0, 0, 0);
        }
    }
    if (!kv_wait()) return false;
    if (one_pass) {   // the current position's rows
        const int j = t / tpk;
        if (j == n - 1) {
            const uint4 *kr = reinterpret_cast<const uint4 *>(kw + (size_t)j * HD);
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = sub + tpk * u;
                if (v < nkv) kq[u] = __ldcg(kr + v);
            }
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int jv = g + k * G;
            if (g < G && jv == n - 1)
                vq[k] = __ldcg(reinterpret_cast<const uint4 *>(vw + (size_t)jv * HD) + c);
        }
    }
    float m = -INFINITY;
    for (int j0 = 0; j0 < n; j0 += kpp) {
        const int j = j0 + t / tpk;
        float s = 0.f;
        if (j < n) {
            if (!one_pass) {
                const uint4 *kr = reinterpret_cast<const uint4 *>(kw + (size_t)j * HD);
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int v = sub + tpk * u;
                    kq[u] = v < nkv ? __ldcg(kr + v) : make_uint4(0, 0, 0, 0);
                }
            }
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int v = sub + tpk * u;
                if (v < nkv) s = dotv<TKV>(kq[u], qs + v * KVEC, s);
            }
        }
        for (int o = 1; o < tpk; o <<= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
        if (j < n) {
            if (sub == 0) ps[j] = s;
            m = fmaxf(m, s);
        }
    }
    m = cmax(m, red);
    float sum = 0.f;
    for (int j = t; j < n; j += kCT) {
        const float e = __expf(ps[j] - m);
        ps[j] = e;
        sum += e;
    }
    sum = csum(sum, red);
    const float inv = 1.f / sum;
    if (g < G) {
        float acc[KVEC];
#pragma unroll
        for (int e = 0; e < KVEC; ++e) acc[e] = 0.f;
        if (one_pass) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int jv = g + k * G;
                if (jv < n) {
                    float vv[KVEC];
                    unpack<TKV>(vq[k], vv);
                    const float pj = ps[jv];
#pragma unroll
                    for (int e = 0; e < KVEC; ++e) acc[e] = fmaf(pj, vv[e], acc[e]);
                }
            }
        } else {
            for (int j = g; j < n; j += G) {
                float vv[KVEC];
                unpack<TKV>(__ldcg(reinterpret_cast<const uint4 *>(vw + (size_t)j * HD) + c), vv);
                const float pj = ps[j];
#pragma unroll
                for (int e = 0; e < KVEC; ++e) acc[e] = fmaf(pj, vv[e], acc[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < KVEC; ++e) op[g * HD + c * KVEC + e] = acc[e];
    }
    csync();
    for (int i = t; i < HD; i += kCT) {
        float acc = 0.f;
        for (int gg = 0; gg < G; ++gg) acc += op[gg * HD + i];
        a.b.o[(size_t)h * HD + i] = acc * inv;
    }
    csync();
    return true;
}

// ------------------------------------------------------------------ the kernel
// Shared-memory layout (dynamic part): ring [kNSlot][kSlot] bytes, then per-warp
// row results [kNC][kMaxR], the activation vector xs [vmax], the producer's score
// copy [E] and the stage-7 partial results; stage 3 reuses xs as scratch.
// The two roles are written as separate functions (inlined into the kernel, which
// reads its arguments straight from the parameter bank).

// Producer warp (warp kNC): lane 0 issues every copy; the whole warp computes each
// layer's top-k.
template <typename TW>
__device__ __forceinline__ void producer_warp(const PersistArgs &a, Shared &S, unsigned char *sm_raw)
{
    const Dims &d = a.d;
    const int I = d.I, H = d.H, K = d.K;
    const int RB = min(kMaxR, max(1, kSlot / (I * (int)sizeof(TW))));  // rows per down chunk
    const int vmax = max(max(H, d.QD), max(d.RQ + d.RKV, (K + 1) * I));
    unsigned char *ring = sm_raw;                                          // [kNSlot][kSlot]
    float *res_all = reinterpret_cast<float *>(ring + kNSlot * kSlot);     // [kNC][kMaxR]
    float *xs = res_all + kNC * kMaxR;                                     // [vmax]
    float *sc = xs + vmax;                                                 // [E] producer's
    const int lane = threadIdx.x & 31;
    // ======================= producer warp =======================
    // Lane 0 issues every copy; the whole warp computes each layer's top-k.
    const uint64_t pol = policy_evict_first();
    volatile int *ab = &S.abort_flag;
    unsigned it = 0;
    // one item = up to two contiguous copies into the next ring slot
    auto issue = [&](const void *s0, uint32_t b0, const void *s1, uint32_t b1, int site,
                     const void *lo0, size_t ext0) -> bool {
        const int slot = it % kNSlot;
        const unsigned use = it / kNSlot;
        if (!mbar_wait(&S.empty[slot], (use & 1u) ^ 1u, ab)) return false;
        unsigned char *dst = ring + (size_t)slot * kSlot;
        const bool ok =
            DS4G_CHECK(((uintptr_t)s0 & 15u) == 0 && (b0 & 15u) == 0 && b0 > 0, site, a.status) &&
            DS4G_CHECK(b0 + b1 <= (uint32_t)kSlot, site + 1, a.status) &&
            DS4G_CHECK((const char *)s0 >= (const char *)lo0 &&
                           (const char *)s0 + b0 <= (const char *)lo0 + ext0, site + 2, a.status) &&
            DS4G_CHECK(b1 == 0 || (((uintptr_t)s1 & 15u) == 0 && (b1 & 15u) == 0), site + 3,
                       a.status) &&
            DS4G_CHECK((smem_u32(dst) & 15u) == 0, site + 4, a.status);
        if (ok) {
            mbar_expect_tx(&S.full[slot], b0 + b1);
            bulk_g2s(dst, s0, b0, &S.full[slot], pol);
            if (b1) bulk_g2s(dst + b0, s1, b1, &S.full[slot], pol);
        } else {
            mbar_arrive(&S.full[slot]);   // complete the phase without data
        }
        ++it;
        return true;
    };
    // Before leaving, wait (bounded) until the copies of the last items landed, so
    // no bulk copy is in flight when the CTA exits, even after an abort.
    auto drain = [&]() {
        const unsigned n = it < (unsigned)kNSlot ? it : (unsigned)kNSlot;
        for (unsigned k = 1; k <= n; ++k) {
            const unsigned idx = it - k;
            volatile int never = 0;
            mbar_wait(&S.full[idx % kNSlot], (idx / kNSlot) & 1u, &never);
        }
    };
    auto stream = [&](const auto &P) -> bool {
        int lo, hi;
        cta_range(total_chunks(P), lo, hi);
        for (int j = lo; j < hi; ++j) {
            const Chunk c = locate(P, j);
            const Piece &p = P[c.piece];
            const TW *src = static_cast<const TW *>(p.base) + (size_t)c.row0 * p.K;
            if (!issue(src, (uint32_t)(c.nrows * p.K * sizeof(TW)), nullptr, 0, 10 + 10 * c.piece,
                       p.base, (size_t)p.rows * p.K * sizeof(TW)))
                return false;
        }
        return true;
    };
    // every chunk of one piece (a work list owned by this CTA alone)
    auto stream_all = [&](const Piece &pc) -> bool {
        for (int j = 0; j < chunks_of(pc); ++j) {
            const int row0 = j * pc.rpc, nr = min(pc.rpc, pc.rows - row0);
            const TW *src = static_cast<const TW *>(pc.base) + (size_t)row0 * pc.K;
            if (!issue(src, (uint32_t)(nr * pc.K * sizeof(TW)), nullptr, 0, 20, pc.base,
                       (size_t)pc.rows * pc.K * sizeof(TW)))
                return false;
        }
        return true;
    };
    // gate and up rows i of the shared expert (e < 0) or of expert e
    struct Experts {   // one layer's expert matrices (s: shared expert)
        const void *gate, *up, *down, *s_gate, *s_up, *s_down;
    };
    auto issue_gu = [&](const Experts &x, int e, int i) -> bool {
        const size_t off = ((e < 0 ? (size_t)0 : (size_t)e * I) + i) * H;
        const void *gbase = e < 0 ? x.s_gate : x.gate;
        const TW *g = static_cast<const TW *>(gbase) + off;
        const TW *u = static_cast<const TW *>(e < 0 ? x.s_up : x.up) + off;
        const size_t gext = (e < 0 ? (size_t)I : (size_t)d.E * I) * H * sizeof(TW);
        return issue(g, H * sizeof(TW), u, H * sizeof(TW), 70, gbase, gext);
    };
    if (lane == 0 && blockIdx.x == 0) prefetch_l2(a.tok_embd + (size_t)a.token * H, H * 2);
    bool ok = true;
    for (int l = 0; l < d.L && ok; ++l) {
        const LayerPtrs &w = a.layers[l];   // read from global memory as needed
        // the expert pointers stay in registers: the routed copies follow the top-k
        const Experts xp = {w.w_gate, w.w_up, w.w_down, w.ws_gate, w.ws_up, w.ws_down};
        int slo, shi, rlo, rhi;
        cta_range(I, slo, shi);        // this CTA's shared-expert rows
        cta_range(K * I, rlo, rhi);    // and routed rows (s-th selected expert: s*I + i)
        if (lane == 0) {
            if (blockIdx.x == 0) {
                prefetch_l2(w.attn_norm, H * 4);
                prefetch_l2(w.ffn_norm, H * 4);
            }
            const Piece P1[2] = {piece<TW>(w.wq_a, d.RQ, H), piece<TW>(w.wkv_a, d.RKV, H)};
            const int kind = qkv_kind(d.NH, a.split_q);
            const Piece P4[1] = {piece<TW>(w.wo, H, d.QD)};
            const Piece P5[1] = {piece<TW>(w.w_router, d.E, H)};
            ok = stream(P1) && (kind < 0 || stream_all(qkv_piece<TW>(w, d, kind, a.split_q))) && stream(P4) &&
                 stream(P5);
            for (int i = slo; ok && i < shi; ++i) ok = issue_gu(xp, -1, i);
        }
        // top-k once every CTA has written its router scores for this layer
        bool go = __shfl_sync(0xffffffffu, ok, 0) && mbar_wait(&S.scores_ready, (unsigned)l & 1u, ab);
        if (!__all_sync(0xffffffffu, go)) { ok = false; break; }
        float sel[8] = {};
        int ids[8] = {};
        bool finite;
        if (d.E <= 256) {   // lane l: experts l, l + 32, ... straight from the loads
            float v[8];
#pragma unroll
            for (int u = 0; u < 8; ++u) {
                const int e = lane + 32 * u;
                v[u] = e < d.E ? __ldcg(a.b.scores + e) : 0.f;
            }
            finite = warp_topk_r256(v, d.E, K, sel, ids, lane);
        } else {
            for (int e0 = 0; e0 < d.E; e0 += 256) {   // eight loads in flight per lane
                float v[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = e0 + lane + 32 * u;
                    v[u] = e < d.E ? __ldcg(a.b.scores + e) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int e = e0 + lane + 32 * u;
                    if (e < d.E) sc[e] = v[u];
                }
            }
            __syncwarp();
            finite = warp_topk(sc, d.E, K, sel, ids, lane);
        }
        // Gate weights, softmax over the selected scores: lane k < K takes the k-th
        // selected expert; every lane sums the K terms in selection order.
        {
            float mys = sel[0];
            int myid = ids[0];
#pragma unroll
            for (int k = 1; k < 8; ++k)
                if (lane == k) {
                    mys = sel[k];
                    myid = ids[k];
                }
            const float wv = expf(mys - sel[0]);
            float sum = 0.f;
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const float wk = __shfl_sync(0xffffffffu, wv, k);
                if (k < K) sum += wk;
            }
            if (lane < K) {
                // an id always indexes a real expert: copy addresses are built from it
                const bool valid = (unsigned)myid < (unsigned)d.E;
                if (!valid) atomicCAS(a.status, 0, DS4G_ENONFINITE);
                S.ids[lane] = valid ? myid : 0;
                S.w[lane] = wv / sum;
                if (blockIdx.x == 0) {
                    a.b.ids[l * K + lane] = myid;
                    a.b.wts[l * K + lane] = wv / sum;
                }
            }
            __syncwarp();
        }
        if (lane == 0) {
            if (!finite) atomicCAS(a.status, 0, DS4G_ENONFINITE);
            S.w[K] = 1.f;
            mbar_arrive(&S.ids_ready);   // consumers start stage 6; the combine reads S.w
            int dlo, dhi;   // this CTA's output rows of the down projections, in chunks of RB
            cta_range(H, dlo, dhi);
            for (int j = rlo; ok && j < rhi; ++j) ok = issue_gu(xp, S.ids[j / I], j % I);
            for (int r0 = dlo; ok && r0 < dhi; r0 += RB) {
                const int nr = min(RB, dhi - r0);
                for (int t = 0; ok && t <= K; ++t) {
                    const TW *base = t == 0 ? static_cast<const TW *>(xp.s_down)
                                            : static_cast<const TW *>(xp.down) +
                                                  (size_t)S.ids[t - 1] * H * I;
                    const void *dbase = t == 0 ? xp.s_down : xp.down;
                    const size_t dext = (t == 0 ? (size_t)H : (size_t)d.E * H) * I * sizeof(TW);
                    ok = issue(base + (size_t)r0 * I, (uint32_t)(nr * I * sizeof(TW)), nullptr, 0, 80,
                               dbase, dext);
                }
            }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (lane == 0) {
        if (ok && a.logits) {
            const Piece PL[1] = {piece<TW>(a.lm_head, d.V, H)};
            stream(PL);
        }
        drain();
    }
}

// Consumer warps 0 .. kNC-1.
template <typename TW, typename TKV>
__device__ __forceinline__ void consumer_warps(const PersistArgs &a, Shared &S, unsigned char *sm_raw)
{
    const Dims &d = a.d;
    const int I = d.I, H = d.H, K = d.K;
    const int RB = min(kMaxR, max(1, kSlot / (I * (int)sizeof(TW))));  // rows per down chunk
    const int vmax = max(max(H, d.QD), max(d.RQ + d.RKV, (K + 1) * I));
    unsigned char *ring = sm_raw;                                          // [kNSlot][kSlot]
    float *res_all = reinterpret_cast<float *>(ring + kNSlot * kSlot);     // [kNC][kMaxR]
    float *xs = res_all + kNC * kMaxR;                                     // [vmax]
    float *sc = xs + vmax;                                                 // [E] producer's
    float *ybuf = sc + d.E;   // [(row chunks per CTA) * (K + 1) * RB] stage-7 results
    float *att = xs + d.RQ + d.RKV;   // stages 2-3: q, scores, partial outputs (after the latents)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // ========================= consumers =========================
    unsigned target = a.bar_base;   // grid-barrier arrivals expected so far
    unsigned it = 0;  // same item counter as the producer
    volatile int *ab = &S.abort_flag;
    float *res = res_all + warp * kMaxR;   // this warp's row results

    // Item idx (this warp's: idx % kNC == warp): wait, compute(slot) -> res, free
    // the slot, then epilogue() reading res.
    auto consume = [&](unsigned idx, auto &&compute, auto &&epilogue) -> bool {
        const int slot = idx % kNSlot;
        if (!mbar_wait(&S.full[slot], (idx / kNSlot) & 1u, ab)) {
            S.abort_flag = 1;
            atomicExch(a.status, DS4G_ETIMEOUT);
            return false;
        }
        compute(ring + (size_t)slot * kSlot);
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.empty[slot]);
        epilogue();
        __syncwarp();
        return true;
    };
    // A plain stage: this CTA's chunks; epi(piece, row0, nrows) reads res.
    auto run_stage = [&](const auto &P, const float *x, auto &&epi) -> bool {
        int lo, hi;
        cta_range(total_chunks(P), lo, hi);
        const unsigned base = it;
        it = base + (unsigned)(hi - lo);
        for (int j = lo; j < hi; ++j) {
            const unsigned idx = base + (unsigned)(j - lo);
            if ((int)(idx % kNC) != warp) continue;
            const Chunk c = locate(P, j);
            const Piece &p = P[c.piece];
            if (!consume(idx,
                         [&](const unsigned char *sl) {
                             warp_dots<TW>(reinterpret_cast<const TW *>(sl), c.nrows, p.K, x, res, lane);
                         },
                         [&]() { epi(c.piece, c.row0, c.nrows); }))
                return false;
        }
        return true;
    };

    constexpr int kLP = sizeof(LayerPtrs) / sizeof(void *);
    if (threadIdx.x < kLP)
        reinterpret_cast<const void **>(&S.lw[0])[threadIdx.x] =
            reinterpret_cast<const void *const *>(&a.layers[0])[threadIdx.x];
    csync();
    for (int l = 0; l < d.L; ++l) {
        const LayerPtrs &w = S.lw[l & 1];   // loaded a stage ahead (see stage 7)
        TKV *kc = static_cast<TKV *>(a.kc[l]);
        TKV *vc = static_cast<TKV *>(a.vc[l]);
        const int lo_w = max(0, a.pos - d.W + 1);

        // ---- stage 1: RMSNorm + [W_qa; W_kva]
        stamp(a, l * 7 + 0);
        {
            // the window's earlier K/V rows are final: start bringing them to L2 now
            if (threadIdx.x == 0 && (int)blockIdx.x < d.NH && a.pos > lo_w) {
                const size_t bytes = (size_t)(a.pos - lo_w) * d.HD * sizeof(TKV);
                prefetch_l2(kc + (size_t)lo_w * d.HD, (uint32_t)bytes);
                prefetch_l2(vc + (size_t)lo_w * d.HD, (uint32_t)bytes);
            }
            // the plain embedding row: the residual (CTA 0) and, when recorded, the
            // input of layer 0 (the last CTA)
            float *plain = blockIdx.x == 0 ? a.b.x : blockIdx.x == gridDim.x - 1 ? a.b.layer_x : nullptr;
            float ss = l == 0 ? cload_f16_g<TW>(a.tok_embd + (size_t)a.token * H, w.attn_norm, xs, H, plain)
                              : cload_g<TW>(a.b.x, w.attn_norm, xs, H);
            const float inv = rsqrtf(csum(ss, S.red) / (float)H + d.eps);
            const Piece P[2] = {piece<TW>(w.wq_a, d.RQ, H), piece<TW>(w.wkv_a, d.RKV, H)};
            if (!run_stage(P, xs, [&](int p, int row0, int nr) {
                    const int o = (p == 0 ? 0 : d.RQ) + row0;
                    for (int r = lane; r < nr; r += 32) a.b.c[o + r] = res[r] * inv;
                }))
                return;
        }
        if (!grid_sync(a, target, S)) return;

        // ---- stages 2-3: queries of one head + attention (head CTAs); K or V row (two CTAs)
        stamp(a, l * 7 + 1);
        {
            const int kind = qkv_kind(d.NH, a.split_q);
            const bool qk = kind == 0 || kind == 3;   // query rows
            const int qh = qkv_head(d.NH, kind), qrow0 = qkv_row0(d, kind);
            const float scale_q = rsqrtf((float)d.HD);
            float *qs = att;   // [HD] this head's queries after RoPE, times 1/sqrt(HD)
            if (kind >= 0) {
                if (qk) cload<TW>(a.b.c, xs, d.RQ, d.RQ);
                else cload<TW>(a.b.c + d.RQ, xs + d.RQ, d.RKV, d.RKV);
                csync();
                const Piece P = qkv_piece<TW>(w, d, kind, a.split_q);
                const float *x = qk ? xs : xs + d.RQ;
                const float2 *rope = a.rope + (size_t)a.pos * (d.HD / 2);
                const float scale = rsqrtf((float)d.HD);
                const int nch = chunks_of(P);
                const unsigned base = it;
                it = base + (unsigned)nch;
                for (int j = 0; j < nch; ++j) {
                    const unsigned idx = base + (unsigned)j;
                    if ((int)(idx % kNC) != warp) continue;
                    const int row0 = j * P.rpc, nr = min(P.rpc, P.rows - row0);
                    if (!consume(idx,
                                 [&](const unsigned char *sl) {
                                     warp_dots<TW>(reinterpret_cast<const TW *>(sl), nr, P.K, x, res, lane);
                                 },
                                 [&]() {
                                     for (int q = lane; q < nr / 2; q += 32) {   // row pairs
                                         const int row = qrow0 + row0 + 2 * q;  // within the head
                                         float e = res[2 * q], o = res[2 * q + 1];
                                         if (kind != 2) {
                                             const float2 cs = rope[row / 2];
                                             const float re = e * cs.x - o * cs.y, ro = e * cs.y + o * cs.x;
                                             e = re;
                                             o = ro;
                                         }
                                         if (qk) {
                                             if (kind == 0) {
                                                 qs[row] = e * scale;
                                                 qs[row + 1] = o * scale;
                                             }
                                             // for inspection, and the second half's way to its head CTA
                                             a.b.q[(size_t)qh * d.HD + row] = e;
                                             a.b.q[(size_t)qh * d.HD + row + 1] = o;
                                         } else {
                                             TKV *dst = (kind == 1 ? kc : vc) + (size_t)a.pos * d.HD;
                                             dst[row] = from_f32<TKV>(e);
                                             dst[row + 1] = from_f32<TKV>(o);
                                         }
                                     }
                                 }))
                        return;
                }
                csync();
                // publish the new K or V row, or the query half: the release (as in grid_sync)
                // covers the CTA's writes, ordered before it by the named barrier above; a full
                // fence here would also wait for the producer's copies in flight
                if (kind > 0 && threadIdx.x == 0) {
                    unsigned *ctr = kind == 3 ? a.qflag + qh : a.bar + 1;
                    asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
                }
            }
            stamp(a, l * 7 + 2);
            if (threadIdx.x == 0) {
                // HBM has little to do while the heads run: bring this CTA's W_o rows that
                // the ring does not hold yet (those after its first kNSlot) into L2.  (A
                // bulk prefetch of whole stages early in the layer was slower: it queued
                // ahead of the stages' own latency-critical loads.)
                const Piece P[1] = {piece<TW>(w.wo, H, d.QD)};
                int lo, hi;
                cta_range(total_chunks(P), lo, hi);
                if (hi - lo > kNSlot) {
                    const Chunk c0 = locate(P, lo + kNSlot), c1 = locate(P, hi - 1);
                    prefetch_range(static_cast<const TW *>(w.wo) + (size_t)c0.row0 * d.QD,
                                   (size_t)(c1.row0 + c1.nrows - c0.row0) * d.QD * sizeof(TW));
                }
            }
            if (kind == 0) {
                // waits for this position's K and V rows (two arrivals per layer) and, with
                // split queries, for the second half of this head's queries
                auto kv_wait = [&]() -> bool {
                    if (threadIdx.x == 0) {
                        const unsigned want = a.kv_base + 2u * (unsigned)(l + 1);
                        const long long t0 = clock64();
                        while ((int)(ld_acquire_gpu(a.bar + 1) - want) < 0) {
                            if (clock64() - t0 > kWaitCycles) {
                                atomicExch(a.status, DS4G_ETIMEOUT);
                                S.abort_flag = 1;
                                break;
                            }
                        }
                        const unsigned qwant = a.q_base + (unsigned)(l + 1);
                        while (a.split_q && *ab == 0 && (int)(ld_acquire_gpu(a.qflag + qh) - qwant) < 0) {
                            if (clock64() - t0 > kWaitCycles) {
                                atomicExch(a.status, DS4G_ETIMEOUT);
                                S.abort_flag = 1;
                                break;
                            }
                        }
                    }
                    csync();
                    if (*ab) return false;
                    if (a.split_q) {
                        for (int i = threadIdx.x; i < d.HD / 2; i += kCT)
                            qs[d.HD / 2 + i] = __ldcg(a.b.q + (size_t)qh * d.HD + d.HD / 2 + i) * scale_q;
                        csync();
                    }
                    return true;
                };
                if (!attention_head<TKV>(a, blockIdx.x, kc + (size_t)lo_w * d.HD, vc + (size_t)lo_w * d.HD,
                                         a.pos - lo_w + 1, att, S.red, kv_wait))
                    return;
            }
        }
        if (!grid_sync(a, target, S)) return;

        // ---- stage 4: xm = x + W_o o
        stamp(a, l * 7 + 3);
        {
            cload<TW>(a.b.o, xs, d.QD, d.QD);
            csync();
            const Piece P[1] = {piece<TW>(w.wo, H, d.QD)};
            if (!run_stage(P, xs, [&](int, int row0, int nr) {
                    for (int r = lane; r < nr; r += 32)
                        a.b.xm[row0 + r] = __ldcg(a.b.x + row0 + r) + res[r];
                }))
                return;
        }
        if (!grid_sync(a, target, S)) return;

        // ---- stage 5: RMSNorm + router scores (xs keeps x * g; inv2 = 1/rms)
        stamp(a, l * 7 + 4);
        if (threadIdx.x == 0) {   // likewise during the router: the shared expert's rows of
                                  // stages 6 and 7 (the routed rows wait for the top-k)
            int slo, shi;
            cta_range(I, slo, shi);
            if (shi > slo) {
                prefetch_range(static_cast<const TW *>(w.ws_gate) + (size_t)slo * H, (size_t)(shi - slo) * H * sizeof(TW));
                prefetch_range(static_cast<const TW *>(w.ws_up) + (size_t)slo * H, (size_t)(shi - slo) * H * sizeof(TW));
            }
            int dlo, dhi;
            cta_range(H, dlo, dhi);
            if (dhi > dlo)
                prefetch_range(static_cast<const TW *>(w.ws_down) + (size_t)dlo * I, (size_t)(dhi - dlo) * I * sizeof(TW));
        }
        float inv2;
        {
            float ss = cload_g<TW>(a.b.xm, w.ffn_norm, xs, H);
            inv2 = rsqrtf(csum(ss, S.red) / (float)H + d.eps);
            if (blockIdx.x == 0) {   // the normalised vector, for inspection
                const float4 *x4 = reinterpret_cast<const float4 *>(xs);
                for (int f = threadIdx.x; f < H / 4; f += kCT) {
                    const float4 v = x4[xperm4<TW>(f, H / VecOf<TW>::n)];
                    reinterpret_cast<float4 *>(a.b.xn2)[f] =
                        make_float4(v.x * inv2, v.y * inv2, v.z * inv2, v.w * inv2);
                }
            }
            const Piece P[1] = {piece<TW>(w.w_router, d.E, H)};
            if (!run_stage(P, xs, [&](int, int row0, int nr) {
                    for (int r = lane; r < nr; r += 32) a.b.scores[row0 + r] = res[r] * inv2;
                }))
                return;
        }
        if (!grid_sync(a, target, S)) return;
        if (threadIdx.x == 0) mbar_arrive(&S.scores_ready);   // the producer warp runs top-k

        // ---- stage 6: shared + routed gate/up + SwiGLU (shared rows first)
        stamp(a, l * 7 + 5);
        // Hold the shared rows until the producer warp has the top-k: it then runs
        // alone on the SM, and the shared rows are computed while the first routed
        // rows are on their way.
        if (threadIdx.x == 0 && !mbar_wait(&S.ids_ready, (unsigned)l & 1u, ab)) {
            S.abort_flag = 1;
            atomicExch(a.status, DS4G_ETIMEOUT);
        }
        csync();
        if (*ab) return;
        {
            int slo, shi, rlo, rhi;
            cta_range(I, slo, shi);
            cta_range(K * I, rlo, rhi);
            const int nsh = shi - slo, nitems = nsh + (rhi - rlo);
            const unsigned base = it;
            it = base + (unsigned)nitems;
            for (int jj = 0; jj < nitems; ++jj) {
                const unsigned idx = base + (unsigned)jj;
                if ((int)(idx % kNC) != warp) continue;
                const int j = jj < nsh ? slo + jj : rlo + (jj - nsh);
                const int slot = jj < nsh ? K : j / I;   // h rows: selected 0..K-1, shared K
                const int i = jj < nsh ? j : j % I;
                if (!consume(idx,
                             [&](const unsigned char *sl) {
                                 warp_dots<TW>(reinterpret_cast<const TW *>(sl), 2, H, xs, res, lane);
                             },
                             [&]() {
                                 if (lane == 0) {
                                     const float gv = res[0] * inv2, uv = res[1] * inv2;
                                     a.b.h[(size_t)slot * I + i] = gv / (1.f + expf(-gv)) * uv;
                                 }
                             }))
                    return;
            }
        }
        if (!grid_sync(a, target, S)) return;

        // ---- stage 7: down-projections, per-expert results, combine + residual
        stamp(a, l * 7 + 6);
        if (l + 1 < d.L && threadIdx.x < kLP)   // next layer's pointers (visible after the
            reinterpret_cast<const void **>(&S.lw[(l + 1) & 1])[threadIdx.x] =   // barriers below)
                reinterpret_cast<const void *const *>(&a.layers[l + 1])[threadIdx.x];
        {
            float *hs = xs;  // [(K+1) * I]
            cload<TW>(a.b.h, hs, (K + 1) * I, I);
            csync();
            // this CTA's output rows [dlo, dhi) (balanced to one row), in chunks of RB rows
            int dlo, dhi;
            cta_range(H, dlo, dhi);
            const int nch = (dhi - dlo + RB - 1) / RB;
            const unsigned base = it;
            const int nitems = nch * (K + 1);
            it = base + (unsigned)nitems;
            for (int j = 0; j < nitems; ++j) {
                const unsigned idx = base + (unsigned)j;
                if ((int)(idx % kNC) != warp) continue;
                const int b = j / (K + 1), t = j % (K + 1);
                const int r0 = dlo + b * RB, nr = min(RB, dhi - r0);
                const int slot = t == 0 ? K : t - 1;
                if (!consume(idx,
                             [&](const unsigned char *sl) {
                                 warp_dots<TW>(reinterpret_cast<const TW *>(sl), nr, I,
                                               hs + (size_t)slot * I, res, lane);
                             },
                             [&]() {
                                 float *yy = ybuf + ((size_t)b * (K + 1) + t) * RB;
                                 for (int r = lane; r < nr; r += 32) yy[r] = res[r];
                             }))
                    return;
            }
            csync();
            // combine in fixed order: shared expert first, then the selected experts
            for (int rr = threadIdx.x; rr < dhi - dlo; rr += kCT) {
                const int b = rr / RB, r = rr % RB, row = dlo + rr;
                float tot = 0.f;
                for (int t = 0; t <= K; ++t) {
                    const int slot = t == 0 ? K : t - 1;
                    tot = fmaf(S.w[slot], ybuf[((size_t)b * (K + 1) + t) * RB + r], tot);
                }
                const float xo = __ldcg(a.b.xm + row) + tot;
                a.b.x[row] = xo;
                if (a.b.layer_x) a.b.layer_x[(size_t)(l + 1) * H + row] = xo;
                if (a.b.x_out && l + 1 == d.L) a.b.x_out[row] = xo;
            }
        }
        if (l + 1 < d.L || a.logits)
            if (!grid_sync(a, target, S)) return;
    }

    // ---- lm_head: logits = W_lm x
    stamp(a, d.L * 7);
    if (a.logits) {
        cload<TW>(a.b.x, xs, H, H);
        csync();
        const Piece P[1] = {piece<TW>(a.lm_head, d.V, H)};
        if (!run_stage(P, xs, [&](int, int row0, int nr) {
                for (int r = lane; r < nr; r += 32) a.b.logits[row0 + r] = res[r];
            }))
            return;
    }
    csync();
    stamp(a, d.L * 7 + 1);
    if (a.done_flag && threadIdx.x == 0) {
        // every consumer thread's outputs of this launch precede the csync above; the
        // last CTA through the ticket tells the waiting host thread
        __threadfence_system();
        const unsigned t = atomicAdd(&a.b.counters[kDoneTicket], 1u);
        if (t == gridDim.x - 1) {
            a.b.counters[kDoneTicket] = 0u;   // ready for the next launch
            __threadfence_system();
            st_release_sys(a.done_flag, a.done_seq);
        }
    }
}

template <typename TW, typename TKV>
__global__ void __launch_bounds__(kPThreads, 1) k_decode_persistent(const __grid_constant__ PersistArgs a)
{
    extern __shared__ __align__(128) unsigned char sm_raw[];
    __shared__ Shared S;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNSlot; ++i) {
            mbar_init(&S.full[i], 1);
            mbar_init(&S.empty[i], 1);
        }
        mbar_init(&S.scores_ready, 1);
        mbar_init(&S.ids_ready, 1);
        S.abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();   // the only whole-CTA barrier: roles split below
    if ((threadIdx.x >> 5) == kNC)
        producer_warp<TW>(a, S, sm_raw);
    else
        consumer_warps<TW, TKV>(a, S, sm_raw);
}

// ------------------------------------------------------------------ host side

static int rows_per_down_chunk(const Dims &d)
{
    const int wsz = d.wdt == DS4G_BF16 ? 2 : 4;
    return std::min(kMaxR, std::max(1, kSlot / (d.I * wsz)));
}

size_t persistent_smem(const Dims &d)
{
    const size_t kvs = d.kvdt == DS4G_BF16 ? 2 : 4;
    const int vmax = std::max(std::max(d.H, d.QD), std::max(d.RQ + d.RKV, (d.K + 1) * d.I));
    const int RB = rows_per_down_chunk(d);
    const int nrb = (d.H + RB - 1) / RB;
    int nsm = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev);
    const int ymax = ((nrb + std::max(nsm, 1) - 1) / std::max(nsm, 1) + 1) * (d.K + 1) * RB;
    const size_t region =
        std::max((size_t)(vmax + d.E + ymax), (size_t)(d.RQ + d.RKV + d.HD + d.W + kCT * 8)) * 4;
    (void)kvs;
    return (size_t)kNSlot * kSlot + (size_t)kNC * kMaxR * 4 + region;
}

template <typename TW, typename TKV> static const void *kernel_of()
{
    return (const void *)k_decode_persistent<TW, TKV>;
}

static const void *persistent_kernel(const Dims &d)
{
    if (d.wdt == DS4G_BF16)
        return d.kvdt == DS4G_BF16 ? kernel_of<bf16, bf16>() : kernel_of<bf16, float>();
    return d.kvdt == DS4G_BF16 ? kernel_of<float, bf16>() : kernel_of<float, float>();
}

// Whether the persistent kernel applies: cooperative launch with one CTA per SM,
// every chunk fits a ring slot and holds whole RoPE pairs.
cudaError_t persistent_setup(const Dims &d, int max_smem, int nsm, bool *ok)
{
    *ok = false;
    const void *f = persistent_kernel(d);
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, f);
    if (e) return e;
    if (persistent_smem(d) + fa.sharedSizeBytes > (size_t)max_smem) return cudaSuccess;
    if ((e = allow_max_dyn_smem(f, max_smem))) return e;
    int dev = 0, coop = 0, per_sm = 0;
    if ((e = cudaGetDevice(&dev))) return e;
    if ((e = cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev))) return e;
    if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, f, kPThreads,
                                                             persistent_smem(d))))
        return e;
    const int wsz = d.wdt == DS4G_BF16 ? 2 : 4;
    // every chunk fits a ring slot; RoPE pieces (K = RQ, RKV) hold at least one row pair
    const bool rows_fit = (size_t)std::max(d.H, d.QD) * wsz <= kSlot && (size_t)d.I * wsz <= kSlot &&
                          2 * (size_t)d.H * wsz <= kSlot &&
                          2 * (size_t)std::max(d.RQ, d.RKV) * wsz <= kSlot;
    // one CTA per head plus the K and V writers must exist
    *ok = coop && per_sm >= 1 && nsm > 0 && rows_fit && d.NH + 2 <= nsm;
    return cudaSuccess;
}

cudaError_t decode_persistent(const PersistArgs &a, cudaStream_t st, int nsm)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(nsm);
    cfg.blockDim = dim3(kPThreads);
    cfg.dynamicSmemBytes = persistent_smem(a.d);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    void *args[] = {const_cast<PersistArgs *>(&a)};
    ++launch_count();
    return cudaLaunchKernelExC(&cfg, persistent_kernel(a.d), args);
}

}  // namespace ds4g
