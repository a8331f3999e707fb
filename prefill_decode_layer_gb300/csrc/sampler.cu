// Sampler kernels: page "ds4.c 学习笔记 -- 端到端推理流程", 阶段四 4.3
// (sample_full_vocab / sample_top_p_min_p / sample_argmax).
//
// T > 0.  z_i = l_i / T and p_i = exp(z_i - max z) in f32 (the page's float
// arithmetic), then q_i = round(p_i * 2^40) as a
// 64-bit fixed-point integer.  All sums are integer sums, so every reduction
// order gives the same bits and the drawn token does not depend on timing.
//   pass 0   max of the logits (ordered-integer atomicMax)
//   pass 1-4 radix select, 8 bits at a time from the top, of the top-p
//            threshold tau on the f32 bit pattern of p (p >= 0, so the bit
//            pattern orders like the value): per digit, the sum of q over the
//            candidates; the last CTA of each pass picks the digit at which
//            the running sum from the top reaches ceil(top_p * total).
//            Ties at tau are kept in index order, as many as the target needs.
//   pass 5   per-chunk sums of kept q; the last CTA finds the chunk and then the
//            first token, in vocabulary order, whose running kept sum reaches
//            R = max(1, ceil(u * kept_total)) (u = k / 2^24 exactly).  With min-p,
//            a token of the top-p set is kept only if p >= min_p (p is relative to
//            the largest, which is exactly 1): the bit patterns compare the same way.
// T <= 0.   argmax: max of (ordered logit bits, inverted index) as one u64.
// Vocabularies up to 256 chunks run all passes in one cooperative launch
// (k_sample_one, below); larger ones, or a grid that cannot be resident at once,
// run one kernel per pass.  Both take the same decisions on the same integers.
#include "common.cuh"
#include <cstring>

#include "kernels.h"
#include "sm100.cuh"

namespace ds4g {

static constexpr int kChunk = 1024;   // tokens per CTA
static constexpr int kSThreads = 256;
static constexpr int kMaxChunks = 1024;   // chunk sums the last CTA of the draw keeps in shared memory

struct SampleWS {
    unsigned long long hist[4][256];   // per-pass digit sums of q
    unsigned long long total;          // sum of q over the vocabulary
    unsigned long long above;          // sum of q with p bits above the selected prefix
    unsigned long long target;         // ceil(top_p * total)
    unsigned long long keep_ties;      // tie tokens (p == tau) kept, in index order
    unsigned long long argmax_key;
    unsigned int max_key;              // ordered bits of max logit
    unsigned int prefix;               // selected high bits of tau so far
    unsigned int tickets[8];
    int result;
    int pad[3];
    // followed by: u64 chunk_above[nchunks], u32 chunk_ties[nchunks]
};

__device__ __forceinline__ unsigned ordered_bits(float f)
{
    const unsigned u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered(unsigned k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

__device__ __forceinline__ float prob(float l, float t, float zm)
{
    return expf(__fdiv_rn(l, t) - zm);
}

__device__ __forceinline__ unsigned long long fixed_q(float p)
{
    return (unsigned long long)__float2ll_rn(p * 1099511627776.0f);  // 2^40, exact scaling
}

// Ticket: returns true in the last CTA to arrive (all of its threads).
__device__ __forceinline__ bool last_cta(unsigned *ticket)
{
    __shared__ int s_last;
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        const unsigned t = atomicAdd(ticket, 1u);
        s_last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (s_last) __threadfence();
    return s_last != 0;
}

__global__ void __launch_bounds__(kSThreads) k_s_max(const float *logits, int n, SampleWS *ws,
                                                     int greedy)
{
    const int base = blockIdx.x * kChunk;
    unsigned mk = 0u;
    unsigned long long ak = 0ull;
    for (int i = base + threadIdx.x; i < min(base + kChunk, n); i += blockDim.x) {
        const unsigned k = ordered_bits(logits[i]);
        mk = max(mk, k);
        if (greedy) ak = max(ak, ((unsigned long long)k << 32) | (0xffffffffu - (unsigned)i));
    }
    for (int o = 16; o > 0; o >>= 1) {
        mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        ak = max(ak, __shfl_xor_sync(0xffffffffu, ak, o));
    }
    if ((threadIdx.x & 31) == 0) {
        atomicMax(&ws->max_key, mk);
        if (greedy) atomicMax(&ws->argmax_key, ak);
    }
    if (greedy && last_cta(&ws->tickets[0]) && threadIdx.x == 0) {
        ws->result = (int)(0xffffffffu - (unsigned)(ws->argmax_key & 0xffffffffull));
        ws->tickets[0] = 0u;
    }
}

// Digit-histogram pass d (0..3) over the candidates matching the prefix chosen so far.
__global__ void __launch_bounds__(kSThreads) k_s_hist(const float *logits, int n, float temp,
                                                      float top_p, SampleWS *ws, int d)
{
    __shared__ unsigned long long h[256];
    __shared__ unsigned long long s_tot;
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = 0ull;
    if (threadIdx.x == 0) s_tot = 0ull;
    __syncthreads();
    const float zm = __fdiv_rn(from_ordered(ws->max_key), temp);
    const unsigned prefix = ws->prefix;
    const int shift = 24 - 8 * d;
    const unsigned hi_mask = d == 0 ? 0u : (0xffffffffu << (32 - 8 * d));
    const int base = blockIdx.x * kChunk;
    unsigned long long tot = 0ull;
    for (int i = base + threadIdx.x; i < min(base + kChunk, n); i += blockDim.x) {
        const float p = prob(logits[i], temp, zm);
        const unsigned long long q = fixed_q(p);
        const unsigned bits = __float_as_uint(p);
        tot += q;
        if ((bits & hi_mask) == prefix && q) atomicAdd(&h[(bits >> shift) & 0xffu], q);
    }
    if (d == 0) {
        for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
        if ((threadIdx.x & 31) == 0) atomicAdd(&s_tot, tot);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += blockDim.x)
        if (h[i]) atomicAdd(&ws->hist[d][i], h[i]);
    if (d == 0 && threadIdx.x == 0) atomicAdd(&ws->total, s_tot);
    if (!last_cta(&ws->tickets[1 + d])) return;
    // the pass's 256 digit sums, loaded in parallel (a serial scan of global memory
    // would wait an L2 round trip per digit)
    for (int i = threadIdx.x; i < 256; i += blockDim.x) h[i] = __ldcg(&ws->hist[d][i]);
    __syncthreads();
    if (threadIdx.x == 0) {
        if (d == 0) {
            const double t = ceil((double)top_p * (double)ws->total);
            ws->target = t < 1.0 ? 1ull : (unsigned long long)t;  // keep at least one token
        }
        const unsigned long long target = ws->target;
        unsigned long long above = ws->above;
        int b = 255;
        for (; b > 0; --b) {
            const unsigned long long hb = h[b];
            if (above + hb >= target) break;
            above += hb;
        }
        ws->above = above;
        ws->prefix = prefix | ((unsigned)b << shift);
        ws->tickets[1 + d] = 0u;
    }
}

// Final pass: per-chunk kept sums, then the inverse-CDF search by the last CTA.
__global__ void __launch_bounds__(kSThreads) k_s_draw(const float *logits, int n, float temp,
                                                      int keep_all, unsigned mbits, unsigned u24, SampleWS *ws,
                                                      unsigned long long *chunk_above,
                                                      unsigned *chunk_ties)
{
    __shared__ unsigned long long s_sum;
    __shared__ unsigned s_ties;
    const float zm = __fdiv_rn(from_ordered(ws->max_key), temp);
    const unsigned tau = ws->prefix;
    const int base = blockIdx.x * kChunk;
    if (threadIdx.x == 0) { s_sum = 0ull; s_ties = 0u; }
    __syncthreads();
    unsigned long long sum = 0ull;
    unsigned ties = 0u;
    for (int i = base + threadIdx.x; i < min(base + kChunk, n); i += blockDim.x) {
        const float p = prob(logits[i], temp, zm);
        const unsigned bits = __float_as_uint(p);
        if (bits < mbits) continue;   // below min-p
        if (keep_all || bits > tau) sum += fixed_q(p);
        else if (bits == tau) ties += 1u;
    }
    for (int o = 16; o > 0; o >>= 1) {
        sum += __shfl_xor_sync(0xffffffffu, sum, o);
        ties += __shfl_xor_sync(0xffffffffu, ties, o);
    }
    if ((threadIdx.x & 31) == 0) { atomicAdd(&s_sum, sum); atomicAdd(&s_ties, ties); }
    __syncthreads();
    if (threadIdx.x == 0) { chunk_above[blockIdx.x] = s_sum; chunk_ties[blockIdx.x] = s_ties; }
    if (!last_cta(&ws->tickets[5])) return;

    // ---- last CTA: ties to keep, kept total, target R, chunk search, token search
    __shared__ unsigned long long s_qtau, s_keep, s_R, s_before;
    __shared__ unsigned s_ties_before;
    __shared__ int s_chunk;
    const int nch = gridDim.x;
    // the per-chunk sums, loaded in parallel for the serial scans below (vocabularies
    // up to kMaxChunks * kChunk tokens; beyond that the scans read global memory)
    __shared__ unsigned long long s_ca[kMaxChunks];
    __shared__ unsigned s_ct[kMaxChunks];
    const bool in_smem = nch <= kMaxChunks;
    if (in_smem)
        for (int c = threadIdx.x; c < nch; c += blockDim.x) {
            s_ca[c] = __ldcg(&chunk_above[c]);
            s_ct[c] = __ldcg(&chunk_ties[c]);
        }
    __syncthreads();
    auto ca = [&](int c) { return in_smem ? s_ca[c] : __ldcg(&chunk_above[c]); };
    auto ct = [&](int c) { return in_smem ? s_ct[c] : __ldcg(&chunk_ties[c]); };
    if (threadIdx.x == 0) {
        const unsigned long long qtau = keep_all ? 0ull : fixed_q(__uint_as_float(tau));
        unsigned long long keep = 0ull;
        if (!keep_all) {
            const unsigned long long need = ws->target > ws->above ? ws->target - ws->above : 0ull;
            keep = qtau ? (need + qtau - 1) / qtau : ~0ull;
        }
        unsigned long long kept_total = 0ull, tb = 0ull;
        for (int c = 0; c < nch; ++c) {
            const unsigned long long t = ct(c);
            const unsigned long long kt = keep_all ? 0ull : (tb >= keep ? 0ull : min(t, keep - tb));
            kept_total += ca(c) + kt * qtau;
            tb += t;
        }
        // R = max(1, ceil(u24 * kept_total / 2^24)), exact in 128-bit arithmetic
        const unsigned long long lo = (unsigned long long)u24 * (kept_total & 0xffffffull);
        const unsigned long long hi = (unsigned long long)u24 * (kept_total >> 24);
        unsigned long long R = hi + (lo >> 24) + ((lo & 0xffffffull) ? 1ull : 0ull);
        if (R == 0ull) R = 1ull;
        // the chunk in which the running kept sum reaches R
        unsigned long long run = 0ull;
        tb = 0ull;
        int chunk = nch - 1;
        unsigned long long before = 0ull, tbefore = 0ull;
        for (int c = 0; c < nch; ++c) {
            const unsigned long long t = ct(c);
            const unsigned long long kt = keep_all ? 0ull : (tb >= keep ? 0ull : min(t, keep - tb));
            const unsigned long long cs = ca(c) + kt * qtau;
            if (run + cs >= R) { chunk = c; before = run; tbefore = tb; break; }
            run += cs;
            tb += t;
            before = run;
            tbefore = tb;
        }
        s_qtau = qtau; s_keep = keep; s_R = R; s_before = before;
        s_ties_before = (unsigned)tbefore; s_chunk = chunk;
        ws->keep_ties = keep;
    }
    __syncthreads();
    // scan the chunk: threads take consecutive runs of tokens; block-wide ordered scan
    const int c0 = s_chunk * kChunk, c1 = min(c0 + kChunk, n);
    constexpr int per = kChunk / kSThreads;
    __shared__ unsigned long long s_part[kSThreads];
    __shared__ unsigned s_tpart[kSThreads];
    unsigned long long qv[per];
    unsigned char tie[per];
    unsigned long long psum = 0ull;
    unsigned tcount = 0u;
#pragma unroll
    for (int j = 0; j < per; ++j) {
        const int i = c0 + threadIdx.x * per + j;
        qv[j] = 0ull;
        tie[j] = 0;
        if (i < c1) {
            const float p = prob(logits[i], temp, zm);
            const unsigned bits = __float_as_uint(p);
            if (bits >= mbits) {
                if (keep_all || bits > tau) qv[j] = fixed_q(p);
                else if (bits == tau) { tie[j] = 1; tcount++; }
            }
        }
        psum += qv[j];
    }
    s_part[threadIdx.x] = psum;
    s_tpart[threadIdx.x] = tcount;
    __syncthreads();
    if (threadIdx.x == 0) {  // exclusive prefix over threads (fixed order)
        unsigned long long r = 0ull;
        unsigned t = 0u;
        for (int k = 0; k < kSThreads; ++k) {
            const unsigned long long a = s_part[k];
            const unsigned b = s_tpart[k];
            s_part[k] = r;
            s_tpart[k] = t;
            r += a;
            t += b;
        }
    }
    __syncthreads();
    // each thread walks its own tokens; ties count toward the kept set in index order
    unsigned long long run = s_before + s_part[threadIdx.x];
    unsigned long long tidx = (unsigned long long)s_ties_before + s_tpart[threadIdx.x];
    int found = 0x7fffffff;
    // running sum including ties requires the number of kept ties before this thread
    // (ties before it that were kept add q_tau each)
    {
        // recompute the kept-tie contribution preceding this thread's first token
        const unsigned long long keep = s_keep;
        const unsigned long long tb = (unsigned long long)s_ties_before;
        const unsigned long long ties_prior = tidx;  // global tie index of our first tie
        const unsigned long long kept_prior_in_chunk =
            keep_all ? 0ull
                     : (ties_prior >= keep ? (tb >= keep ? 0ull : keep - tb)
                                           : ties_prior - tb);
        run += kept_prior_in_chunk * s_qtau;
    }
#pragma unroll
    for (int j = 0; j < per; ++j) {
        unsigned long long q = qv[j];
        if (tie[j]) {
            q = tidx < s_keep ? s_qtau : 0ull;
            tidx++;
        }
        run += q;
        if (q && run >= s_R && found == 0x7fffffff) found = c0 + threadIdx.x * per + j;
    }
    __shared__ int s_found;
    if (threadIdx.x == 0) s_found = 0x7fffffff;
    __syncthreads();
    if (found != 0x7fffffff) atomicMin(&s_found, found);
    __syncthreads();
    if (threadIdx.x == 0) {
        int r = s_found;
        if (r == 0x7fffffff) {  // rounding guard: the last kept token of the chunk
            for (int i = c1 - 1; i >= c0; --i) {
                const float p = prob(logits[i], temp, zm);
                if (fixed_q(p) && __float_as_uint(p) >= mbits && (keep_all || __float_as_uint(p) >= tau)) {
                    r = i;
                    break;
                }
            }
        }
        ws->result = r;
        ws->tickets[5] = 0u;
    }
}

// ------------------------------------------------------------------ one-launch form
//
// The same passes and the same integer arithmetic in one cooperative launch of one
// CTA per 1024-token chunk (the grid must be resident at once; otherwise the
// separate kernels above run).  Thread t of CTA c holds the probabilities of
// tokens c * kChunk + t * 4 .. + 3 in registers from the first pass to the draw,
// so the vocabulary order is (CTA, thread, slot).  Grid barriers separate the
// passes.  A histogram pass adds each CTA's digit sums in shared memory
// (warp-aggregated: lanes holding the same digit add their q with two redux.sync on
// its 20-bit halves, one atomic per group), then one global add per non-empty bin;
// after the barrier every CTA reads the 256 sums and takes the same digit decision
// (no second barrier).  The draw: per-chunk kept sums, a barrier, then each CTA
// scans the chunk sums, and the CTA whose range holds the target R finds the token
// among its threads.  Waits are bounded: a barrier that gives up leaves the result
// DS4G_ETIMEOUT.
static constexpr int kTpt = kChunk / kSThreads;   // 4 tokens per thread

__device__ __forceinline__ bool s_grid_sync(unsigned *ctr, unsigned target, int *result)
{
    __shared__ int s_ok;
    __syncthreads();
    if (threadIdx.x == 0) {
        int ok = 1;
        asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(ctr) : "memory");
        const long long t0 = clock64();
        while ((int)(ld_acquire_gpu(ctr) - target) < 0) {
            if (clock64() - t0 > kWaitCycles) {
                atomicExch(result, DS4G_ETIMEOUT);
                ok = 0;
                break;
            }
        }
        s_ok = ok;
    }
    __syncthreads();
    return s_ok != 0;
}

// Exclusive scan of v over the CTA's threads in thread order; *total gets the sum.
__device__ __forceinline__ unsigned long long cta_exclusive_scan(unsigned long long v, unsigned long long *wtot,
                                                                 unsigned long long *total)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    unsigned long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        unsigned long long w = lane < nw ? wtot[lane] : 0ull;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned long long y = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += y;
        }
        if (lane < nw) wtot[lane] = w;   // inclusive warp totals
    }
    __syncthreads();
    *total = wtot[nw - 1];
    const unsigned long long r = x - v + (warp ? wtot[warp - 1] : 0ull);
    __syncthreads();   // wtot may be reused
    return r;
}

__global__ void __launch_bounds__(kSThreads) k_sample_one(const float *logits, int n, float temp, float top_p,
                                                          unsigned mbits, unsigned u24, int greedy, int keep_all,
                                                          SampleWS *ws, unsigned long long *chunk_above,
                                                          unsigned *chunk_ties)
{
    __shared__ unsigned long long h[256];
    __shared__ unsigned long long wtot[32];
    __shared__ unsigned long long s_tot;
    __shared__ unsigned s_prefix;
    __shared__ unsigned long long s_above, s_target;
    unsigned *bar = &ws->tickets[0];   // grid-barrier arrivals (zeroed with the workspace)
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int G = gridDim.x;
    const int t0 = blockIdx.x * kChunk + threadIdx.x * kTpt;
    unsigned nb = 0;   // barriers passed

    // ---- pass 0: max of the logits (and, greedy, the argmax key)
    float lg[kTpt];
    unsigned mk = 0u;
    unsigned long long ak = 0ull;
#pragma unroll
    for (int j = 0; j < kTpt; ++j) {
        const int i = t0 + j;
        lg[j] = i < n ? logits[i] : 0.f;
        if (i < n) {
            const unsigned k = ordered_bits(lg[j]);
            mk = max(mk, k);
            if (greedy) ak = max(ak, ((unsigned long long)k << 32) | (0xffffffffu - (unsigned)i));
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        mk = max(mk, __shfl_xor_sync(0xffffffffu, mk, o));
        ak = max(ak, __shfl_xor_sync(0xffffffffu, ak, o));
    }
    if (lane == 0) {
        atomicMax(&ws->max_key, mk);
        if (greedy) atomicMax(&ws->argmax_key, ak);
    }
    if (!s_grid_sync(bar, (++nb) * (unsigned)G, &ws->result)) return;
    if (greedy) {
        if (blockIdx.x == 0 && threadIdx.x == 0)
            ws->result = (int)(0xffffffffu - (unsigned)(__ldcg(&ws->argmax_key) & 0xffffffffull));
        return;
    }
    const float zm = __fdiv_rn(from_ordered(__ldcg(&ws->max_key)), temp);
    float pv[kTpt];
#pragma unroll
    for (int j = 0; j < kTpt; ++j) pv[j] = t0 + j < n ? prob(lg[j], temp, zm) : 0.f;

    // ---- passes 1-4: radix select of the top-p threshold on the bits of p
    unsigned prefix = 0u;
    unsigned long long above = 0ull, target = 0ull;
    if (!keep_all) {
        for (int d = 0; d < 4; ++d) {
            for (int b = threadIdx.x; b < 256; b += blockDim.x) h[b] = 0ull;
            if (threadIdx.x == 0) s_tot = 0ull;
            __syncthreads();
            const int shift = 24 - 8 * d;
            const unsigned hi_mask = d == 0 ? 0u : (0xffffffffu << (32 - 8 * d));
            unsigned long long tot = 0ull;
#pragma unroll
            for (int j = 0; j < kTpt; ++j) {
                const unsigned bits = __float_as_uint(pv[j]);
                const unsigned long long q = fixed_q(pv[j]);
                tot += q;
                const bool cand = (bits & hi_mask) == prefix && q;
                const unsigned key = cand ? (bits >> shift) & 0xffu : 256u + lane;
                const unsigned peers = __match_any_sync(0xffffffffu, key);
                if (cand) {
                    const unsigned hs = __reduce_add_sync(peers, (unsigned)(q >> 20));
                    const unsigned ls = __reduce_add_sync(peers, (unsigned)(q & 0xfffffull));
                    if (lane == __ffs(peers) - 1) atomicAdd(&h[key], ((unsigned long long)hs << 20) + ls);
                }
            }
            if (d == 0) {
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
                if (lane == 0) atomicAdd(&s_tot, tot);
            }
            __syncthreads();
            for (int b = threadIdx.x; b < 256; b += blockDim.x)
                if (h[b]) atomicAdd(&ws->hist[d][b], h[b]);
            if (d == 0 && threadIdx.x == 0) atomicAdd(&ws->total, s_tot);
            if (!s_grid_sync(bar, (++nb) * (unsigned)G, &ws->result)) return;
            if (warp == 0) {
                // lane L holds the sums of bins 255 - 8L - k, k = 0..7 (descending)
                unsigned long long v[8], ls = 0ull;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    v[k] = __ldcg(&ws->hist[d][255 - 8 * lane - k]);
                    ls += v[k];
                }
                unsigned long long incl = ls;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const unsigned long long y = __shfl_up_sync(0xffffffffu, incl, o);
                    if (lane >= o) incl += y;
                }
                if (d == 0) {
                    const double tg = ceil((double)top_p * (double)__ldcg(&ws->total));
                    target = tg < 1.0 ? 1ull : (unsigned long long)tg;   // keep at least one token
                }
                // the first bin from the top at which the running sum reaches the target;
                // bin 0 is taken when no higher bin does
                unsigned long long run = above + (incl - ls);
                int hit = -1;
                unsigned long long run_at = 0ull;
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int b = 255 - 8 * lane - k;
                    if (hit < 0 && (b == 0 || run + v[k] >= target)) {
                        hit = b;
                        run_at = run;
                    }
                    run += v[k];
                }
                const unsigned who = __ballot_sync(0xffffffffu, hit >= 0);
                const int src = __ffs(who) - 1;
                const int b = __shfl_sync(0xffffffffu, hit, src);
                above = __shfl_sync(0xffffffffu, run_at, src);
                if (lane == 0) {
                    s_prefix = prefix | ((unsigned)b << shift);
                    s_above = above;
                    s_target = target;
                }
            }
            __syncthreads();
            prefix = s_prefix;
            above = s_above;
            target = s_target;
        }
    }
    const unsigned tau = prefix;

    // ---- draw: kept sums in vocabulary order, the inverse-CDF target R, the token
    unsigned long long tsum = 0ull, tties = 0ull;
#pragma unroll
    for (int j = 0; j < kTpt; ++j) {
        const unsigned bits = __float_as_uint(pv[j]);
        if (t0 + j >= n || bits < mbits) continue;   // below min-p (or past the vocabulary)
        if (keep_all || bits > tau) tsum += fixed_q(pv[j]);
        else if (bits == tau) tties += 1ull;
    }
    unsigned long long csum, cties;
    const unsigned long long psum = cta_exclusive_scan(tsum, wtot, &csum);
    const unsigned long long pties = cta_exclusive_scan(tties, wtot, &cties);
    if (threadIdx.x == 0) {
        chunk_above[blockIdx.x] = csum;
        chunk_ties[blockIdx.x] = (unsigned)cties;
    }
    if (!s_grid_sync(bar, (++nb) * (unsigned)G, &ws->result)) return;
    const unsigned long long qtau = keep_all ? 0ull : fixed_q(__uint_as_float(tau));
    unsigned long long keep = 0ull;
    if (!keep_all) {
        const unsigned long long need = target > above ? target - above : 0ull;
        keep = qtau ? (need + qtau - 1) / qtau : ~0ull;
    }
    // the chunks' sums and ties before this CTA, and in all
    unsigned long long cs = 0ull, ct = 0ull;
    if (threadIdx.x < G) {   // one chunk per thread (G <= blockDim is required by the launch)
        cs = __ldcg(&chunk_above[threadIdx.x]);
        ct = __ldcg(&chunk_ties[threadIdx.x]);
    }
    unsigned long long sum_all, ties_all;
    const unsigned long long cs_pre = cta_exclusive_scan(cs, wtot, &sum_all);
    const unsigned long long ct_pre = cta_exclusive_scan(ct, wtot, &ties_all);
    __shared__ unsigned long long s_sum_before, s_ties_before;
    if (threadIdx.x == blockIdx.x) {
        s_sum_before = cs_pre;
        s_ties_before = ct_pre;
    }
    __syncthreads();
    auto kept_ties = [&](unsigned long long ties) { return keep_all ? 0ull : (ties < keep ? ties : keep); };
    const unsigned long long kept_total = sum_all + kept_ties(ties_all) * qtau;
    // R = max(1, ceil(u24 * kept_total / 2^24)), exact
    const unsigned long long lo = (unsigned long long)u24 * (kept_total & 0xffffffull);
    const unsigned long long hi = (unsigned long long)u24 * (kept_total >> 24);
    unsigned long long R = hi + (lo >> 24) + ((lo & 0xffffffull) ? 1ull : 0ull);
    if (R == 0ull) R = 1ull;
    // this thread's running kept sum before its first token, then its own tokens
    unsigned long long tie_idx = s_ties_before + pties;
    unsigned long long run = s_sum_before + psum + kept_ties(tie_idx) * qtau;
    if (run < R) {
#pragma unroll
        for (int j = 0; j < kTpt; ++j) {
            const unsigned bits = __float_as_uint(pv[j]);
            if (t0 + j >= n || bits < mbits) continue;
            unsigned long long q = 0ull;
            if (keep_all || bits > tau) q = fixed_q(pv[j]);
            else if (bits == tau) {
                q = tie_idx < keep ? qtau : 0ull;
                tie_idx += 1ull;
            }
            run += q;
            if (q && run >= R) {
                ws->result = t0 + j;
                break;
            }
        }
    }
}

// Whether the one-launch form applies: one CTA per chunk, all resident at once.
static bool sample_one_applies(int n, int *grid)
{
    const int nch = (n + kChunk - 1) / kChunk;
    if (n < 1 || nch > kSThreads) return false;   // the draw reads one chunk per thread
    int dev = 0, nsm = 0, per_sm = 0, coop = 0;
    if (cudaGetDevice(&dev) || cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) ||
        cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_sample_one, kSThreads, 0)) {
        cudaGetLastError();
        return false;
    }
    *grid = nch;
    return coop && (long long)per_sm * nsm >= nch;
}

static unsigned host_float_bits(float f)
{
    unsigned u;
    memcpy(&u, &f, 4);
    return u;
}

size_t sample_workspace_bytes(int n)
{
    const int nch = (n + kChunk - 1) / kChunk;
    return sizeof(SampleWS) + (size_t)nch * 12 + 256;
}

// Issues the sampler kernels; the token id is left at *result_dev.
cudaError_t sample_launch(const float *logits, int n, float temperature, float top_p, float min_p,
                          unsigned u24, void *ws_mem, cudaStream_t st, int **result_dev)
{
    SampleWS *ws = static_cast<SampleWS *>(ws_mem);
    const int nch = (n + kChunk - 1) / kChunk;
    unsigned long long *chunk_above = reinterpret_cast<unsigned long long *>(ws + 1);
    unsigned *chunk_ties = reinterpret_cast<unsigned *>(chunk_above + nch);
    *result_dev = &ws->result;
    const int greedy = temperature <= 0.f;
    const int keep_all_ = top_p >= 1.0f;
    // min-p as a bound on the bit pattern of p (p >= 0); 0 keeps everything
    const unsigned mbits_ = min_p > 0.f ? host_float_bits(min_p < 1.f ? min_p : 1.f) : 0u;
    cudaError_t e = cudaMemsetAsync(ws, 0, sizeof(SampleWS), st);
    if (e) return e;
    int grid = 0;
    if (sample_one_applies(n, &grid)) {   // one cooperative launch
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kSThreads);
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        ++launch_count();
        return cudaLaunchKernelEx(&cfg, k_sample_one, logits, n, temperature, top_p, mbits_, u24, greedy, keep_all_,
                                  ws, chunk_above, chunk_ties);
    }
    k_s_max<<<nch, kSThreads, 0, st>>>(logits, n, ws, greedy);
    ++launch_count();
    if ((e = cudaGetLastError())) return e;
    if (greedy) return cudaSuccess;
    const int keep_all = keep_all_;
    if (!keep_all) {
        for (int d = 0; d < 4; ++d) {
            k_s_hist<<<nch, kSThreads, 0, st>>>(logits, n, temperature, top_p, ws, d);
            ++launch_count();
            if ((e = cudaGetLastError())) return e;
        }
    }
    const unsigned mbits = mbits_;
    k_s_draw<<<nch, kSThreads, 0, st>>>(logits, n, temperature, keep_all, mbits, u24, ws, chunk_above,
                                         chunk_ties);
    ++launch_count();
    return cudaGetLastError();
}

// Fixed scratch for ds4g_sample_static: the workspace of the largest vocabulary it
// accepts, in device memory that exists from module load (no allocation).
static __device__ __align__(256) unsigned char g_sample_scratch[kSampleStaticBytes];
static_assert(kSampleStaticBytes >= sizeof(SampleWS) + ((kSampleStaticMaxVocab + kChunk - 1) / kChunk) * 12 + 256,
              "static sampler scratch too small for its maximum vocabulary");

// Device address of the fixed scratch on the current device, looked up on every
// call.  The lookup allocates nothing and is cheap once the module is loaded; a
// cached address would go stale if the caller reset the device or destroyed its
// primary context, after which the module (and the array) can be loaded elsewhere.
cudaError_t sample_static_scratch(void **p)
{
    void *a = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&a, g_sample_scratch);
    if (e) return e;
    *p = a;
    return cudaSuccess;
}

}  // namespace ds4g
