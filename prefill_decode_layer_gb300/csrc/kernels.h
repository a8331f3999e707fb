// Host-side entry points of the kernel files (internal to the library).
#pragma once

#include "common.cuh"

namespace ds4g {

// decode.cu
cudaError_t decode_setup(const Dims &d, int max_smem);
cudaError_t decode_layer(const StepArgs &a, cudaStream_t st, int nsm,
                         cudaEvent_t (*ev)[2] = nullptr);
cudaError_t decode_lm_head(const StepArgs &a, cudaStream_t st, int nsm);

// decode_persistent.cu
size_t persistent_smem(const Dims &d);
cudaError_t persistent_setup(const Dims &d, int max_smem, int nsm, bool *ok);
cudaError_t decode_persistent(const PersistArgs &a, cudaStream_t st, int nsm);

// sampler.cu
size_t sample_workspace_bytes(int n);
// Fixed sampler scratch (ds4g_sample_static): vocabularies up to kSampleStaticMaxVocab.
constexpr int kSampleStaticMaxVocab = 262144;
constexpr size_t kSampleStaticBytes = 16384;
cudaError_t sample_static_scratch(void **p);
cudaError_t sample_launch(const float *logits, int n, float temperature, float top_p, float min_p,
                          unsigned u24, void *ws, cudaStream_t st, int **result_dev);

// prefill.cu
// Positions whose per-layer residual a session records (ds4g_session_set_probe),
// plus the last prefilled token (DS4G_DBG_PREFILL_LAYER_X).
constexpr int kMaxProbe = 64;
constexpr int kMaxRec = kMaxProbe + 1;
// Parts of the tensor-core router GEMM's reduction (work items on twice the SMs;
// the parts' scores are summed in order by k_router_topk), when E <= 256.
constexpr int kRouterParts = 2;
inline int router_parts(int E) { return E <= 256 ? kRouterParts : 1; }
struct PrefillBufs {
    int P;            // chunk capacity (tokens)
    int *tok;         // [P]
    float *X;         // [P][H] residual
    void *XN;         // [P][H] normalised activations (activation type)
    float *XN32;      // [P][H] f32 copy of the MoE-side normalised activations (router)
    void *C;          // [P][RQ+RKV] latents
    void *Q;          // [P][QD] queries after RoPE
    void *O;          // [P][QD] attention output
    float *S;         // [kRouterParts][P][E] router scores (partial sums of the reduction's parts)
    char *end;        // one past the last byte laid out
    int *ids;         // [P][K]
    float *wts;       // [P][K]
    int *cnt;         // [E] tokens per expert
    int *off;         // [E+1] start of each expert's rows in the grouped order
    int *rows;        // [P*K] grouped order: token * K + slot
    int *segcnt;      // [ceil(P*K / kSortSeg)][E] per-segment expert counts, then bases
    int *tiles;       // [P*K/16 + E + 1] (expert, first row) work items; tiles[0] = count
    void *HG;         // [P*K][I] routed SwiGLU hidden, grouped order
    void *HS;         // [P][I] shared SwiGLU hidden
    float *YS;        // [P*K][H] routed expert outputs, token-slot order
    int *status;      // session status word (set after carving)
    // Side stream of the tensor-core form: the shared expert's GEMMs of a layer run
    // on it, forked after the FFN RMSNorm and joined before the combine (null: all
    // on the session stream).
    cudaStream_t side = nullptr;
    cudaEvent_t ev_fork = nullptr, ev_join = nullptr;
    // Timing mode (tensor-core form): an event after every launch of a chunk, with
    // the launch's kind (DS4G_K_P_*); ev[0] is recorded at the chunk's start.
    struct Timing {
        static constexpr int kMax = 1024;
        cudaEvent_t ev[kMax];
        int kind[kMax];
        int n;
    } *tm = nullptr;
    // Recorded rows: the residual of chunk row rec_row[i] entering each layer l, then
    // the final hidden state, is copied to rec_dst[i] + l * H ([L+1][H] each).
    int n_rec;
    int rec_row[kMaxRec];
    float *rec_dst[kMaxRec];
};
// Entries per segment of the counting sort that groups (token, slot) entries by expert.
static constexpr int kSortSeg = 512;
static inline size_t sort_segments(size_t nent) { return (nent + kSortSeg - 1) / kSortSeg; }
// Stable counting sort of pb.ids[0, nent) by expert into pb.rows, with the expert
// offsets pb.off[E + 1], counts pb.cnt[E] and the tile list pb.tiles (bm rows a tile).
cudaError_t group_by_expert(const PrefillBufs &pb, int nent, int E, int bm, cudaStream_t st);
size_t prefill_bytes(const Dims &d, int P);
void prefill_carve(const Dims &d, int P, char *base, PrefillBufs &pb);
cudaError_t prefill_setup(const Dims &d, int max_smem);
// Layer-major pass of tokens [0, n) of the chunk (already in pb.tok) at positions
// [p0, p0 + n): embed, every layer, and leaves the final hidden states in pb.X.
cudaError_t prefill_chunk(const Dims &d, const LayerPtrs *layers, void *const *kc,
                          void *const *vc, const float2 *rope, const uint16_t *tok_embd,
                          const PrefillBufs &pb, int p0, int n, cudaStream_t st, int nsm);

}  // namespace ds4g
