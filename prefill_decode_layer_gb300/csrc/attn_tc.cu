// Windowed causal multi-query attention of the layer-major prefill on the 5th-
// generation tensor cores (tcgen05, TMEM accumulators, TMA operand tiles).
//
// Page "ds4.c 学习笔记 -- 端到端推理流程", 阶段三 prefill_layer_major_cpu: a layer's
// attention over the whole chunk, each token attending to the keys of its sliding
// window (its own position and the W - 1 before it) through one shared K/V head.
//
// A CTA block is 128 query rows: the NH heads of 128 / NH consecutive tokens (row
// r = token_in_block * NH + head, so the rows of a block are rows blk*128 .. of the
// [token][head] query array).  All of them read the same keys: the union of their
// windows, staged once.  Per block:
//   S = (Qhi + Qlo) K^T      M 128 rows x N keys (<= KR) x K 128 dims, hi and lo
//                            query tiles into one FP32 accumulator in TMEM;
//   softmax                  one thread per row reads its S row from TMEM, masks it
//                            to the token's window, and writes P = exp(scale (S -
//                            max)) as BF16 hi/lo rows into shared memory (the row
//                            sum stays FP32 in a register);
//   O = (Phi + Plo) V        M 128 x N 128 dims x K keys, V read MN-major (its rows
//                            are keys) straight from the TMA tile;
//   out                      O / sum as BF16 hi/lo rows (the W_o GEMM's input).
// Keys are staged from an absolute position that is a multiple of 16 and every
// reduction runs over absolute 16-key steps (keys outside a row's window add exact
// zeros), so a token's result does not depend on how the prompt was cut into
// chunks or blocks.
//
// Roles (160 threads, one CTA per SM, persistent over blocks):
//   warps 0-3        softmax and output of rows 32w .. 32w + 31 (their TMEM lanes);
//   warp 4 lane 0    TMA and MMA issue.  The next block's Q and K tiles load while
//                    this block's softmax runs, its V tile while this block's
//                    output is written; two TMEM buffers (S, then O in the same
//                    columns) let the next block's S run during this block's output.
// Every wait is bounded; a CTA that gives up raises DS4G_ETIMEOUT, drains its copies
// and MMAs, frees its TMEM and returns.
#include <cuda.h>

#include "prefill_tc.h"
#include "sm100.cuh"
#include "tc_gemm.cuh"

namespace ds4g {

static constexpr int kTaHD = 128;         // head dimension
static constexpr int kTaRows = 128;       // query rows per block (MMA M)
static constexpr int kTaMaxW = 128;       // largest window
static constexpr int kTaThreads = 160;
static constexpr uint32_t kTaQBox = kTaRows * 64 * 2;   // one 64-dim box of 128 query rows (16 KB)

// Staged key rows for NH heads: the union of 128 / NH windows, from a 16-aligned
// start, rounded up to 16.
static int ta_key_rows(int W, int NH) { return ((W + kTaRows / NH - 1 + 15) + 15) / 16 * 16; }

// Shared-memory layout of one CTA (offsets from the 1024-aligned base).
struct TaLayout {
    uint32_t qhi, qlo, k, v, phi, plo, bars, total;
    __host__ __device__ explicit TaLayout(int KR)
    {
        const uint32_t kv = (uint32_t)KR * 128 * 2;   // two 64-dim boxes of KR rows
        const uint32_t p = (uint32_t)KR * kTaRows * 2;   // P rows (BF16), one of hi / lo
        qhi = 0;
        qlo = 2 * kTaQBox;
        k = 4 * kTaQBox;
        v = k + kv;
        phi = v + kv;
        plo = phi + p;
        bars = plo + p;
        total = bars + 256;
    }
};

bool attn_tc_eligible(const Dims &d)
{
    const bool nh_ok = d.NH == 16 || d.NH == 32 || d.NH == 64 || d.NH == 128;
    return d.kvdt == DS4G_BF16 && d.HD == kTaHD && nh_ok && d.W >= 1 && d.W <= kTaMaxW;
}

size_t attn_tc_smem(const Dims &d) { return 1024 + TaLayout(ta_key_rows(d.W, d.NH)).total; }

__global__ void __launch_bounds__(kTaThreads, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap qhi, const __grid_constant__ CUtensorMap qlo,
                      const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      bf16 *o_hi, bf16 *o_lo, int p0, int n, int NH, int W, int KR, int *status)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const TaLayout L(KR);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L.bars);
    uint64_t *bar_qk = bar, *bar_v = bar + 1, *bar_s = bar + 2, *bar_p = bar + 3, *bar_o = bar + 4;
    uint64_t *bar_oe = bar + 5;   // [2]: TMEM buffer drained by the output threads
    uint64_t *done = bar + 7;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 8);
    int *abort_flag = reinterpret_cast<int *>(tslot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int TB = kTaRows / NH;   // tokens per block
    const int nblk = (n + TB - 1) / TB;
    const uint32_t sbase = smem_u32(sm);
    const uint32_t kvbox = (uint32_t)KR * 128;   // bytes of one 64-dim K or V box
    // keys staged for block blk: [kbase, kbase + KR), of which [kbase, kbase + span) exist
    auto block_keys = [&](int blk, int &kbase, int &span) {
        const int t0 = blk * TB, t1 = min(n, t0 + TB);
        kbase = (max(0, p0 + t0 - W + 1) / 16) * 16;
        span = p0 + t1 - kbase;
    };

    if (threadIdx.x == 0) {
        mbar_init(bar_qk, 1);
        mbar_init(bar_v, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_p, 128);
        mbar_init(bar_o, 1);
        mbar_init(&bar_oe[0], 128);
        mbar_init(&bar_oe[1], 128);
        mbar_init(done, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 4) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    volatile int *ab = abort_flag;
    auto give_up = [&]() {
        *abort_flag = 1;
        atomicExch(status, DS4G_ETIMEOUT);
    };

    if (warp == 4) {
        if (lane == 0) {
            // ---------------- TMA and MMA issue
            tma_prefetch_desc(&qhi);
            tma_prefetch_desc(&qlo);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            auto issue_qk = [&](int blk) {
                int kbase, span;
                block_keys(blk, kbase, span);
                mbar_expect_tx(bar_qk, 4 * kTaQBox + 2 * kvbox);
                tma_load_2d(sm + L.qhi, &qhi, 0, blk * kTaRows, bar_qk);
                tma_load_2d(sm + L.qhi + kTaQBox, &qhi, 64, blk * kTaRows, bar_qk);
                tma_load_2d(sm + L.qlo, &qlo, 0, blk * kTaRows, bar_qk);
                tma_load_2d(sm + L.qlo + kTaQBox, &qlo, 64, blk * kTaRows, bar_qk);
                tma_load_2d(sm + L.k, &kmap, 0, kbase, bar_qk);
                tma_load_2d(sm + L.k + kvbox, &kmap, 64, kbase, bar_qk);
            };
            auto issue_v = [&](int blk) {
                int kbase, span;
                block_keys(blk, kbase, span);
                mbar_expect_tx(bar_v, 2 * kvbox);
                tma_load_2d(sm + L.v, &vmap, 0, kbase, bar_v);
                tma_load_2d(sm + L.v + kvbox, &vmap, 64, kbase, bar_v);
            };
            unsigned nqk = 0, nv = 0;   // copies issued on bar_qk / bar_v
            int blk = blockIdx.x;
            if (blk < nblk) {
                issue_qk(blk);
                issue_v(blk);
                nqk = nv = 1;
            }
            const uint32_t id_o = idesc_bf16_f32_bmn(kTaRows, kTaHD);
            for (int it = 0; blk < nblk; blk += gridDim.x, ++it) {
                const int b = it & 1;
                int kbase, span;
                block_keys(blk, kbase, span);
                const int nk16 = (span + 15) / 16 * 16;
                if (!mbar_wait(bar_qk, it & 1, ab)) {
                    give_up();
                    break;
                }
                if (it >= 2 && !mbar_wait(&bar_oe[b], ((it >> 1) & 1) ^ 1, ab)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                const uint32_t acc = tmem + (uint32_t)(b * 256);
                // S = (Qhi + Qlo) K^T: 8 steps of 16 dims
                const uint32_t id_s = idesc_bf16_f32(kTaRows, nk16);
#pragma unroll
                for (int ks = 0; ks < kTaHD / 16; ++ks) {
                    const uint32_t qoff = (uint32_t)(ks >> 2) * kTaQBox + (uint32_t)(ks & 3) * 32;
                    const uint64_t kd = sdesc_kmajor_sw128(sbase + L.k + (uint32_t)(ks >> 2) * kvbox +
                                                           (uint32_t)(ks & 3) * 32);
                    tc_mma_bf16(acc, sdesc_kmajor_sw128(sbase + L.qhi + qoff), kd, id_s, ks > 0);
                    tc_mma_bf16(acc, sdesc_kmajor_sw128(sbase + L.qlo + qoff), kd, id_s, 1u);
                }
                tc_commit(bar_s);
                if (!mbar_wait(bar_s, it & 1, ab)) {
                    give_up();
                    break;
                }
                const int next = blk + gridDim.x;
                if (next < nblk) {   // the Q and K tiles are free: stage the next block's
                    issue_qk(next);
                    ++nqk;
                }
                if (!mbar_wait(bar_p, it & 1, ab)) {
                    give_up();
                    break;
                }
                tc_fence_after();
                // O = (Phi + Plo) V over 16-key steps, into the columns S held
                for (int ks = 0; ks < nk16 / 16; ++ks) {
                    const uint64_t vd = sdesc_mnmajor_sw128(sbase + L.v + (uint32_t)ks * 2048, kvbox, 1024);
                    const uint32_t poff = (uint32_t)ks * 256;
                    tc_mma_bf16(acc, sdesc_kmajor_plain(sbase + L.phi + poff, 128, (uint32_t)KR * 16), vd, id_o,
                                ks > 0);
                    tc_mma_bf16(acc, sdesc_kmajor_plain(sbase + L.plo + poff, 128, (uint32_t)KR * 16), vd, id_o, 1u);
                }
                tc_commit(bar_o);
                if (!mbar_wait(bar_o, it & 1, ab)) {
                    give_up();
                    break;
                }
                if (next < nblk) {   // V and P are free
                    issue_v(next);
                    ++nv;
                }
            }
            // nothing may be in flight when the CTA exits
            volatile int never = 0;
            if (nqk) mbar_wait(bar_qk, (nqk - 1) & 1, &never);
            if (nv) mbar_wait(bar_v, (nv - 1) & 1, &never);
            tc_commit(done);
            mbar_wait(done, 0, &never);
        }
    } else {
        // ---------------- softmax and output: thread = query row r of the block
        const int r = 32 * warp + lane;
        const float scale = rsqrtf((float)kTaHD);
        const uint32_t pbase = (uint32_t)(r >> 3) * ((uint32_t)KR * 16) + (uint32_t)(r & 7) * 16;
        int it = 0;
        for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++it) {
            const int b = it & 1;
            int kbase, span;
            block_keys(blk, kbase, span);
            const int nk16 = (span + 15) / 16 * 16;
            const int t = blk * TB + r / NH;
            const bool live = t < n;
            const int pos = p0 + t;
            const int lo = max(0, pos - W + 1) - kbase, hi = pos - kbase;   // the row's window, in columns
            if (!mbar_wait(bar_s, it & 1, ab)) {
                give_up();
                break;
            }
            tc_fence_after();
            const uint32_t row = tmem + ((uint32_t)(32 * warp) << 16) + (uint32_t)(b * 256);
            float mx = -INFINITY;
            for (int c0 = 0; c0 < nk16; c0 += 16) {
                float s[16];
                tmem_ld16(row + (uint32_t)c0, s);
#pragma unroll
                for (int j = 0; j < 16; ++j)
                    if (c0 + j >= lo && c0 + j <= hi) mx = fmaxf(mx, s[j]);
            }
            float sum = 0.f;
            for (int c0 = 0; c0 < nk16; c0 += 16) {
                float s[16];
                tmem_ld16(row + (uint32_t)c0, s);
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int j = 0; j < 16; j += 2) {
                    float p2[2];
#pragma unroll
                    for (int u = 0; u < 2; ++u) {
                        const int c = c0 + j + u;
                        p2[u] = live && c >= lo && c <= hi ? __expf((s[j + u] - mx) * scale) : 0.f;
                        sum += p2[u];
                    }
                    bf16 h0, l0, h1, l1;
                    split_hilo(p2[0], h0, l0);
                    split_hilo(p2[1], h1, l1);
                    wh[j / 2] = pack_bf16x2(h0, h1);
                    wl[j / 2] = pack_bf16x2(l0, l1);
                }
                // keys c0 .. c0+7 and c0+8 .. c0+15: two core matrices of the row's group
                const uint32_t off = pbase + (uint32_t)(c0 >> 3) * 128;
                *reinterpret_cast<uint4 *>(sm + L.phi + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4 *>(sm + L.phi + off + 128) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
                *reinterpret_cast<uint4 *>(sm + L.plo + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                *reinterpret_cast<uint4 *>(sm + L.plo + off + 128) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
            }
            // staged V rows past the last key are multiplied by P = 0: make them zeros
            if (!mbar_wait(bar_v, it & 1, ab)) {
                give_up();
                break;
            }
            for (int i = r; i < (nk16 - span) * 16; i += 128) {
                const int vr = span + (i >> 4), box = (i >> 3) & 1, ch = i & 7;
                *reinterpret_cast<uint4 *>(sm + L.v + (uint32_t)box * kvbox + (uint32_t)vr * 128 + ch * 16) =
                    make_uint4(0u, 0u, 0u, 0u);
            }
            fence_proxy_async_smem();   // P and the zeroed rows, before the MMAs read them
            tc_fence_before();          // this row's S reads, before O overwrites its columns
            mbar_arrive(bar_p);
            if (!mbar_wait(bar_o, it & 1, ab)) {
                give_up();
                break;
            }
            tc_fence_after();
            const float inv = live ? 1.f / sum : 0.f;
            bf16 *oh = o_hi + ((size_t)blk * kTaRows + r) * kTaHD;
            bf16 *ol = o_lo + ((size_t)blk * kTaRows + r) * kTaHD;
#pragma unroll 1
            for (int c0 = 0; c0 < kTaHD; c0 += 32) {
                float o[32];
                tmem_ld32(row + (uint32_t)c0, o);
                if (!live) continue;
#pragma unroll
                for (int v = 0; v < 4; ++v) {
                    uint32_t wh[4], wl[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        bf16 h0, l0, h1, l1;
                        split_hilo(o[8 * v + 2 * j] * inv, h0, l0);
                        split_hilo(o[8 * v + 2 * j + 1] * inv, h1, l1);
                        wh[j] = pack_bf16x2(h0, h1);
                        wl[j] = pack_bf16x2(l0, l1);
                    }
                    reinterpret_cast<uint4 *>(oh + c0)[v] = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                    reinterpret_cast<uint4 *>(ol + c0)[v] = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
            }
            tc_fence_before();
            mbar_arrive(&bar_oe[b]);
        }
    }
    tc_fence_before();
    __syncthreads();
    if (warp == 4) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

// ------------------------------------------------------------------ host side

cudaError_t attn_tc_setup(const Dims &d, int max_smem)
{
    if (!attn_tc_eligible(d)) return cudaSuccess;
    const size_t sm = attn_tc_smem(d);
    if (sm > (size_t)max_smem) return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(k_attn_prefill_tc, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)sm);
}

cudaError_t attn_tc_kv_maps(const Dims &d, const void *kc, const void *vc, int n_ctx, TcKVMaps &m)
{
    const int KR = ta_key_rows(d.W, d.NH);
    cudaError_t e = tc::make_map_bf16(&m.k, kc, n_ctx, kTaHD, kTaHD, KR);
    if (!e) e = tc::make_map_bf16(&m.v, vc, n_ctx, kTaHD, kTaHD, KR);
    return e;
}

cudaError_t attn_tc_q_maps(const Dims &d, int P, const bf16 *q_hi, const bf16 *q_lo, CUtensorMap &mhi,
                           CUtensorMap &mlo)
{
    cudaError_t e = tc::make_map_bf16(&mhi, q_hi, P * d.NH, kTaHD, kTaHD, kTaRows);
    if (!e) e = tc::make_map_bf16(&mlo, q_lo, P * d.NH, kTaHD, kTaHD, kTaRows);
    return e;
}

cudaError_t attn_prefill_tc(const Dims &d, const CUtensorMap &qhi, const CUtensorMap &qlo, const TcKVMaps &kv,
                            bf16 *o_hi, bf16 *o_lo, int p0, int n, int *status, cudaStream_t st, int nsm)
{
    const int TB = kTaRows / d.NH, nblk = (n + TB - 1) / TB;
    if (nblk <= 0) return cudaSuccess;
    const int KR = ta_key_rows(d.W, d.NH);
    const int grid = nblk < nsm ? nblk : nsm;
    k_attn_prefill_tc<<<grid, kTaThreads, attn_tc_smem(d), st>>>(qhi, qlo, kv.k, kv.v, o_hi, o_lo, p0, n, d.NH,
                                                                 d.W, KR, status);
    ++launch_count();
    return cudaGetLastError();
}

}  // namespace ds4g
