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
//                            query tiles into one FP32 accumulator in TMEM (with
//                            hilo = 0 the queries, probabilities and output are
//                            single BF16: no lo tiles, MMAs or stores);
//   softmax                  the warps of a row read its S from TMEM, mask it to
//                            the token's window, and write P = exp(scale (S - max))
//                            as BF16 hi/lo rows into shared memory (the row sum
//                            stays FP32);
//   O = (Phi + Plo) V        M 128 x N 128 dims x K keys, V read MN-major (its rows
//                            are keys) straight from the TMA tile;
//   out                      O / sum as BF16 hi/lo rows (the W_o GEMM's input),
//                            staged in shared memory and written by TMA stores.
// Keys are staged from an absolute position that is a multiple of 16 and every
// reduction runs over absolute 16-key steps (keys outside a row's window add exact
// zeros), so a token's result does not depend on how the prompt was cut into
// chunks or blocks.
//
// Roles (544 threads, one CTA per SM, persistent over blocks):
//   warps 0-15       softmax and output; warp w serves rows 32 (w % 4) .. +31 (its
//                    TMEM lanes) over every 4th 16-key chunk and one quarter of the
//                    128 output dims; the four parts of a row combine their maxima
//                    and sums through shared memory, in a fixed order;
//   warp 16 lane 0   TMA and MMA issue.  The next block's Q and K tiles load while
//                    this block's softmax runs and its S is issued as soon as they
//                    have landed (two TMEM buffers: S, then O in the same columns);
//                    its V tile loads once this block's O is complete.
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
static constexpr int kTaParts = 4;        // softmax warps per TMEM lane quarter (column parts)
static constexpr int kTaSoft = 128 * kTaParts;   // softmax / output threads
static constexpr int kTaCtl = kTaSoft / 32;      // the issuing warp
static constexpr int kTaThreads = kTaSoft + 32;
static constexpr uint32_t kTaQBox = kTaRows * 64 * 2;   // one 64-dim box of 128 query rows (16 KB)

// Staged key rows for NH heads: the union of 128 / NH windows, from a 16-aligned
// start, rounded up to 16.
static int ta_key_rows(int W, int NH) { return ((W + kTaRows / NH - 1 + 15) + 15) / 16 * 16; }

// Shared-memory layout of one CTA (offsets from the 1024-aligned base).
struct TaLayout {
    uint32_t qhi, qlo, k, v, phi, plo, red, bars, total;
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
        // the output's staging boxes reuse the P rows: at least 4 boxes of 16 KB
        red = phi + (2 * p > 4 * kTaQBox ? 2 * p : 4 * kTaQBox);   // [kTaParts][128] row maxima, then sums
        bars = red + kTaParts * kTaRows * 4;
        total = bars + 128;
    }
};

__device__ __forceinline__ float ex2_approx(float x)   // 2^x (hardware approximation)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

bool attn_tc_eligible(const Dims &d)
{
    const bool nh_ok = d.NH == 64 || d.NH == 128;   // 2 or 1 tokens per 128-row block
    return d.kvdt == DS4G_BF16 && d.HD == kTaHD && nh_ok && d.W >= 1 && d.W <= kTaMaxW;
}

size_t attn_tc_smem(const Dims &d) { return 1024 + TaLayout(ta_key_rows(d.W, d.NH)).total; }

__global__ void __launch_bounds__(kTaThreads, 1)
    k_attn_prefill_tc(const __grid_constant__ CUtensorMap qhi, const __grid_constant__ CUtensorMap qlo,
                      const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
                      const __grid_constant__ CUtensorMap ohi, const __grid_constant__ CUtensorMap olo, int p0,
                      int n, int NH, int W, int KR, int *status, int hilo)
{
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = reinterpret_cast<unsigned char *>(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const TaLayout L(KR);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L.bars);
    uint64_t *bar_qk = bar, *bar_v = bar + 1, *bar_p = bar + 2, *bar_o = bar + 3;
    uint64_t *bar_s = bar + 4;    // [2]: S of TMEM buffer b computed
    uint64_t *bar_oe = bar + 6;   // [2]: TMEM buffer b drained by the output threads
    uint64_t *done = bar + 8;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(bar + 9);
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
        mbar_init(&bar_s[0], 1);
        mbar_init(&bar_s[1], 1);
        mbar_init(bar_p, kTaSoft);
        mbar_init(bar_o, 1);
        mbar_init(&bar_oe[0], kTaSoft);
        mbar_init(&bar_oe[1], kTaSoft);
        mbar_init(done, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == kTaCtl) tmem_alloc(tslot, 512);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait();   // programmatic launch: the queries and K/V rows are complete past this point
    pdl_trigger();
    const uint32_t tmem = *tslot;
    volatile int *ab = abort_flag;
    auto give_up = [&]() {
        *abort_flag = 1;
        atomicExch(status, DS4G_ETIMEOUT);
    };

    if (warp == kTaCtl) {
        if (lane == 0) {
            // ---------------- TMA and MMA issue
            tma_prefetch_desc(&qhi);
            if (hilo) tma_prefetch_desc(&qlo);
            tma_prefetch_desc(&kmap);
            tma_prefetch_desc(&vmap);
            auto issue_qk = [&](int blk) {
                int kbase, span;
                block_keys(blk, kbase, span);
                mbar_expect_tx(bar_qk, (hilo ? 4 : 2) * kTaQBox + 2 * kvbox);
                tma_load_2d(sm + L.qhi, &qhi, 0, blk * kTaRows, bar_qk);
                tma_load_2d(sm + L.qhi + kTaQBox, &qhi, 64, blk * kTaRows, bar_qk);
                if (hilo) {
                    tma_load_2d(sm + L.qlo, &qlo, 0, blk * kTaRows, bar_qk);
                    tma_load_2d(sm + L.qlo + kTaQBox, &qlo, 64, blk * kTaRows, bar_qk);
                }
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
            const uint32_t id_o = idesc_bf16_f32_bmn(kTaRows, kTaHD);
            // S of block blk (the it-th of this CTA) into TMEM buffer it % 2
            auto issue_s = [&](int it, int blk) {
                int kbase, span;
                block_keys(blk, kbase, span);
                const uint32_t acc = tmem + (uint32_t)((it & 1) * 256);
                const uint32_t id_s = idesc_bf16_f32(kTaRows, (span + 15) / 16 * 16);
#pragma unroll
                for (int ks = 0; ks < kTaHD / 16; ++ks) {   // 16 dims a step
                    const uint32_t qoff = (uint32_t)(ks >> 2) * kTaQBox + (uint32_t)(ks & 3) * 32;
                    const uint64_t kd = sdesc_kmajor_sw128(sbase + L.k + (uint32_t)(ks >> 2) * kvbox +
                                                           (uint32_t)(ks & 3) * 32);
                    tc_mma_bf16(acc, sdesc_kmajor_sw128(sbase + L.qhi + qoff), kd, id_s, ks > 0);
                    if (hilo) tc_mma_bf16(acc, sdesc_kmajor_sw128(sbase + L.qlo + qoff), kd, id_s, 1u);
                }
                tc_commit(&bar_s[it & 1]);
            };
            // O of block blk over 16-key steps, into the columns its S held
            auto issue_pv = [&](int it, int blk) {
                int kbase, span;
                block_keys(blk, kbase, span);
                const uint32_t acc = tmem + (uint32_t)((it & 1) * 256);
                for (int ks = 0; ks < (span + 15) / 16; ++ks) {
                    const uint64_t vd = sdesc_mnmajor_sw128(sbase + L.v + (uint32_t)ks * 2048, kvbox, 1024);
                    const uint32_t poff = (uint32_t)ks * 256;
                    tc_mma_bf16(acc, sdesc_kmajor_plain(sbase + L.phi + poff, 128, (uint32_t)KR * 16), vd, id_o,
                                ks > 0);
                    if (hilo)
                        tc_mma_bf16(acc, sdesc_kmajor_plain(sbase + L.plo + poff, 128, (uint32_t)KR * 16), vd, id_o,
                                    1u);
                }
                tc_commit(bar_o);
            };
            unsigned nqk = 0, nv = 0;   // copies issued on bar_qk / bar_v
            int blk = blockIdx.x;
            bool ok = true;
            if (blk < nblk) {
                issue_qk(blk);
                issue_v(blk);
                nqk = nv = 1;
                ok = mbar_wait(bar_qk, 0, ab);
                if (ok) {
                    tc_fence_after();
                    issue_s(0, blk);
                } else {
                    give_up();
                }
            }
            for (int it = 0; ok && blk < nblk; blk += gridDim.x, ++it) {
                const int b = it & 1, next = blk + gridDim.x;
                const bool has_next = next < nblk;
                if (!mbar_wait(&bar_s[b], (it >> 1) & 1, ab)) {
                    give_up();
                    break;
                }
                if (has_next) {   // the Q and K tiles are free: stage the next block's
                    issue_qk(next);
                    ++nqk;
                }
                // whichever comes first: this block's P (then its O = P V), or the next
                // block's Q and K with a drained TMEM buffer (then its S)
                bool s_done = !has_next, pv_done = false;
                const long long t0 = clock64();
                while (!(s_done && pv_done)) {
                    if (!pv_done && mbar_try_wait(bar_p, it & 1)) {
                        tc_fence_after();
                        issue_pv(it, blk);
                        pv_done = true;
                    }
                    if (!s_done && mbar_try_wait(bar_qk, (it + 1) & 1) &&
                        (it < 1 || mbar_try_wait(&bar_oe[b ^ 1], (((it + 1) >> 1) & 1) ^ 1))) {
                        tc_fence_after();
                        issue_s(it + 1, next);
                        s_done = true;
                    }
                    if (*ab || clock64() - t0 > kWaitCycles) {
                        ok = false;
                        break;
                    }
                }
                if (!ok || !mbar_wait(bar_o, it & 1, ab)) {
                    give_up();
                    break;
                }
                if (has_next) {   // V and P are free
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
        // ---------------- softmax and output: warp w serves query rows r = 32 (w % 4) +
        // lane (its TMEM lanes) over every kTaParts-th 16-key chunk and one quarter of O
        const int q = warp & 3, part = warp >> 2;
        const int r = 32 * q + lane;
        const float scale = rsqrtf((float)kTaHD);
        const uint32_t pbase = (uint32_t)(r >> 3) * ((uint32_t)KR * 16) + (uint32_t)(r & 7) * 16;
        float *red = reinterpret_cast<float *>(sm + L.red);   // [part][row]
        // barrier of the softmax threads that also tells each of them whether any failed,
        // so that all leave the loop together
        auto soft_sync_any = [&](bool fail) -> bool {
            uint32_t any;
            asm volatile(
                "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, %2, q;\n"
                " selp.u32 %0, 1, 0, p;\n}\n"
                : "=r"(any)
                : "r"((uint32_t)fail), "n"(kTaSoft)
                : "memory");
            return any != 0;
        };
        auto soft_sync = [&]() { asm volatile("bar.sync 1, %0;" ::"n"(kTaSoft) : "memory"); };
        // a bounded wait whose outcome is the same for the whole warp
        auto warp_wait = [&](uint64_t *bar, uint32_t parity) {
            return __all_sync(0xffffffffu, mbar_wait(bar, parity, ab)) != 0;
        };
        int it = 0;
        for (int blk = blockIdx.x; blk < nblk; blk += gridDim.x, ++it) {
            const int b = it & 1;
            int kbase, span;
            block_keys(blk, kbase, span);
            const int nch = (span + 15) / 16;   // 16-key chunks
            const int t = blk * TB + r / NH;
            const bool live = t < n;
            const int pos = p0 + t;
            const int lo = max(0, pos - W + 1) - kbase, hi = pos - kbase;   // the row's window, in columns
            const uint32_t row = tmem + ((uint32_t)(32 * q) << 16) + (uint32_t)(b * 256);
            float mx = -INFINITY;
            bool ok = warp_wait(&bar_s[b], (it >> 1) & 1);
            if (ok) {
                tc_fence_after();
                for (int ch = part; ch < nch; ch += kTaParts) {
                    float s[16];
                    tmem_ld16(row + (uint32_t)(16 * ch), s);
#pragma unroll
                    for (int j = 0; j < 16; ++j)
                        if (16 * ch + j >= lo && 16 * ch + j <= hi) mx = fmaxf(mx, s[j]);
                }
            }
            red[part * kTaRows + r] = mx;
            if (soft_sync_any(!ok)) {
                give_up();
                break;
            }
#pragma unroll
            for (int u = 0; u < kTaParts; ++u) mx = fmaxf(mx, red[u * kTaRows + r]);
            if (threadIdx.x == 0) bulk_wait_read();   // the previous block's output has left the P region
            soft_sync();   // red is rewritten with the sums below, the P region with P
            // P = 2^(S scale / ln 2 - max scale / ln 2): one FMA and one exp2 per key
            const float c2 = scale * 1.44269504088896341f, moff = mx * c2;
            float sum = 0.f;
            for (int ch = part; ch < nch; ch += kTaParts) {
                const int c0 = 16 * ch;
                float s[16];
                tmem_ld16(row + (uint32_t)c0, s);
                const bool inside = live && c0 >= lo && c0 + 15 <= hi;   // the whole chunk is in the window
#pragma unroll
                for (int j = 0; j < 16; ++j) {
                    const bool in = inside || (live && c0 + j >= lo && c0 + j <= hi);
                    s[j] = in ? ex2_approx(fmaf(s[j], c2, -moff)) : 0.f;
                    sum += s[j];
                }
                uint32_t wh[8], wl[8];
#pragma unroll
                for (int j = 0; j < 8; ++j) split2_hilo(s[2 * j], s[2 * j + 1], wh[j], wl[j]);
                // keys c0 .. c0+7 and c0+8 .. c0+15: two core matrices of the row's group
                const uint32_t off = pbase + (uint32_t)(c0 >> 3) * 128;
                *reinterpret_cast<uint4 *>(sm + L.phi + off) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                *reinterpret_cast<uint4 *>(sm + L.phi + off + 128) = make_uint4(wh[4], wh[5], wh[6], wh[7]);
                if (hilo) {
                    *reinterpret_cast<uint4 *>(sm + L.plo + off) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                    *reinterpret_cast<uint4 *>(sm + L.plo + off + 128) = make_uint4(wl[4], wl[5], wl[6], wl[7]);
                }
            }
            red[part * kTaRows + r] = sum;
            // staged V rows past the last key are multiplied by P = 0: make them zeros
            ok = warp_wait(bar_v, it & 1);
            if (ok) {
                for (int i = threadIdx.x; i < (16 * nch - span) * 16; i += kTaSoft) {
                    const int vr = span + (i >> 4), box = (i >> 3) & 1, c16 = i & 7;
                    *reinterpret_cast<uint4 *>(sm + L.v + (uint32_t)box * kvbox + (uint32_t)vr * 128 + c16 * 16) =
                        make_uint4(0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();   // P and the zeroed rows, before the MMAs read them
                tc_fence_before();          // this thread's S reads, before O overwrites the columns
                mbar_arrive(bar_p);
            }
            if (soft_sync_any(!ok)) {   // (also: every part's row sum is in red)
                give_up();
                break;
            }
            sum = 0.f;
#pragma unroll
            for (int u = 0; u < kTaParts; ++u) sum += red[u * kTaRows + r];   // parts in a fixed order
            const float inv = live ? 1.f / sum : 0.f;
            const int c0 = 32 * part;   // this warp's quarter of O
            ok = warp_wait(bar_o, it & 1);
            if (ok) {
                tc_fence_after();
                float o[32];
                tmem_ld32(row + (uint32_t)c0, o);
                // this thread's 32 dims of O / sum as hi and lo BF16 into the P region (free
                // once O is complete), laid out as the 128-byte-swizzled 64-dim boxes that
                // the tensor store reads: boxes hi 0-63, hi 64-127, lo 0-63, lo 64-127
                unsigned char *bh = sm + L.phi + (uint32_t)(part >> 1) * kTaQBox, *bl = bh + 2 * kTaQBox;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t wh[4], wl[4];
#pragma unroll
                    for (int u = 0; u < 4; ++u)
                        split2_hilo(o[8 * j + 2 * u] * inv, o[8 * j + 2 * u + 1] * inv, wh[u], wl[u]);
                    const uint32_t cj = (uint32_t)r * 128 + (uint32_t)((((part & 1) * 4 + j) ^ (r & 7)) * 16);
                    *reinterpret_cast<uint4 *>(bh + cj) = make_uint4(wh[0], wh[1], wh[2], wh[3]);
                    if (hilo) *reinterpret_cast<uint4 *>(bl + cj) = make_uint4(wl[0], wl[1], wl[2], wl[3]);
                }
                fence_proxy_async_smem();   // the staged rows, before the tensor store reads them
                tc_fence_before();
                mbar_arrive(&bar_oe[b]);
            }
            if (soft_sync_any(!ok)) {
                give_up();
                break;
            }
            if (threadIdx.x == 0) {   // rows blk * 128 .. of the [token][head] output
                tma_store_2d(&ohi, sm + L.phi, 0, blk * kTaRows);
                tma_store_2d(&ohi, sm + L.phi + kTaQBox, 64, blk * kTaRows);
                if (hilo) {
                    tma_store_2d(&olo, sm + L.phi + 2 * kTaQBox, 0, blk * kTaRows);
                    tma_store_2d(&olo, sm + L.phi + 3 * kTaQBox, 64, blk * kTaRows);
                }
                bulk_commit();   // read out of the P region while the next block's S and maxima run
            }
        }
        if (threadIdx.x == 0) bulk_wait_all();
    }
    tc_fence_before();
    __syncthreads();
    if (warp == kTaCtl) {
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

cudaError_t attn_tc_row_map(const Dims &d, int P, const bf16 *base, CUtensorMap &m)
{
    return tc::make_map_bf16(&m, base, P * d.NH, kTaHD, kTaHD, kTaRows);
}

cudaError_t attn_prefill_tc(const Dims &d, const CUtensorMap &qhi, const CUtensorMap &qlo, const TcKVMaps &kv,
                            const CUtensorMap &ohi, const CUtensorMap &olo, int p0, int n, int *status,
                            cudaStream_t st, int nsm, bool hilo)
{
    const int TB = kTaRows / d.NH, nblk = (n + TB - 1) / TB;
    if (nblk <= 0) return cudaSuccess;
    const int KR = ta_key_rows(d.W, d.NH);
    const int grid = nblk < nsm ? nblk : nsm;
    return launch_pdl(k_attn_prefill_tc, dim3(grid), dim3(kTaThreads), attn_tc_smem(d), st, qhi, qlo, kv.k, kv.v, ohi,
                      olo, p0, n, (int)d.NH, (int)d.W, KR, status, hilo ? 1 : 0);
}

}  // namespace ds4g
