// Host-side launch interface shared by the library's translation units.
#pragma once

#include "common.cuh"

#include <utility>

namespace domino {

// Launch with programmatic dependent launch enabled (see pdl_wait()).
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args&&... args) {
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
    return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

struct RunArgs {
    const void* hidden;        // [B,16,H]
    const void* s;             // [B,15,F]
    const int32_t* verified;   // [B]
    int B;
    int K;                     // effective pool size: 0 = full vocabulary
    int n_prop;                // proposals produced (1..15): p_1 + n_prop-1 corrected steps
    void* s_out;               // non-null: compute s here ([B,15,F], input dtype); then s == s_out
    const int32_t* forced;     // nullable [B,15]
    domino_debug_bufs dbg;     // all-null when not debugging
    int32_t* out_tokens;       // [B,15]
    cudaStream_t st;
    int launches;              // incremented per kernel launch
};

// SIMT kernels (kernels_simt.cu)
constexpr int kPoolHistBits = 11;  // first radix digit of the pool select: the top 11 key bits
constexpr int kPoolHistBins = 1 << kPoolHistBits;
cudaError_t launch_reset(domino_ctx* c, RunArgs& r);
cudaError_t launch_lmhead_simt(domino_ctx* c, RunArgs& r);
cudaError_t launch_first_argmax(domino_ctx* c, RunArgs& r);
cudaError_t launch_pool_select(domino_ctx* c, RunArgs& r, bool score_ready);
cudaError_t launch_score(domino_ctx* c, RunArgs& r);  // pool scores from the base logits
// GRU update u (0..14): u = 0 consumes the verified token with h = 0,
// u >= 1 consumes proposal u-1 (or forced[:,u-1]).
cudaError_t launch_gru(domino_ctx* c, RunArgs& r, int u);
cudaError_t launch_fc1(domino_ctx* c, RunArgs& r, int k);
cudaError_t launch_correct_simt(domino_ctx* c, RunArgs& r, int k);
cudaError_t launch_finalize(domino_ctx* c, RunArgs& r);
cudaError_t prepare_simt_kernels(domino_ctx* c);

// tcgen05 / TMA kernels (lmhead_tc.cu)
cudaError_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows);
cudaError_t make_tmap_bf16_strided(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                                   uint32_t box_rows);
bool lmhead_tc_supported(const domino_ctx* c);
// also writes p_1's argmax word, when r.K > 0 the pool scores, and when
// r.s_out is set the per-step term s of projector layer 1
cudaError_t launch_lmhead_tc(domino_ctx* c, RunArgs& r);
// s from the backbone hidden on the CUDA cores (paths without the tcgen05 LM-head)
cudaError_t launch_backbone_s_simt(domino_ctx* c, RunArgs& r);

// tcgen05 correction over the full vocabulary (correct_tc.cu)
int correct_bn(int B);  // N tile of the batched tensor-core kernels
int pool_mask_words(int V);
// full vocabulary, or (with a pool membership mask) pools that cover much of it
bool correct_tc_supported(const domino_ctx* c, const RunArgs& r);
cudaError_t launch_pool_mask(domino_ctx* c, RunArgs& r);  // after the pool selection
cudaError_t prepare_correct_tc(domino_ctx* c, RunArgs& r, CUtensorMap* tmB);
cudaError_t launch_correct_tc(domino_ctx* c, RunArgs& r, const CUtensorMap& tmB, int k);

// cluster radix-select candidate pool (pool.cu)
bool pool_cluster_supported(const domino_ctx* c);
// hist: the LM-head epilogue's histogram of the scores' top kPoolHistBits key
// bits per request, or null (the select then builds its first pass itself)
cudaError_t launch_pool_cluster(domino_ctx* c, RunArgs& r, const unsigned* hist);
cudaError_t launch_pool_cluster_raw(const float* score, int32_t* pool, int B, int V, int K, cudaStream_t st);
bool pool_cluster_fits(int V);
// stage C of the tensor-parallel rollout on one GPU: P shard-local top-K, then the merge
bool pool_compact_supported(const domino_ctx* c, int P, int K);
cudaError_t launch_pool_compact(domino_ctx* c, RunArgs& r, int P);

// batched GRU / projector layer 1 for B >= 2 (kernels_batch.cu)
bool batch_kernels_supported(const domino_ctx* c);
// h16_out (nullable [B,G]): also store the new state as bf16 (tensor-core operand)
cudaError_t launch_gru_batch(domino_ctx* c, RunArgs& r, int u, __nv_bfloat16* h16_out = nullptr);
cudaError_t launch_fc1_batch(domino_ctx* c, RunArgs& r, int k);
// one fused launch per step for bf16 batches of up to eight requests
// (step_fused.cu): launch 0 forms W_hh h_0; launch u >= 1 updates to h_u and
// projects it (step k = u)
bool step_fused_supported(const domino_ctx* c, const RunArgs& r);
cudaError_t launch_step_fused(domino_ctx* c, RunArgs& r, int u);
bool pool_batch_supported(const domino_ctx* c);
cudaError_t launch_correct_pool_batch(domino_ctx* c, RunArgs& r, int k);

// input-side GRU pre-activations T[v, 3G] of every token (gi_table.cu)
cudaError_t build_gi_table(domino_ctx* c, cudaStream_t st);

// tcgen05 GRU update and projector layer 1 for batches (gru_tc.cu)
struct GruMaps {
    CUtensorMap h[2];    // the bf16 state copies H16[0], H16[1] (B operand of both contractions), 16-row boxes
    CUtensorMap h32[2];  // the same with 32-row boxes (32-column tiles of the joined projector)
    CUtensorMap fc1;
};
int gru_padded_units(int G);
bool gru_tc_shape_ok(const domino_config& g);
bool gru_tc_supported(const domino_ctx* c, const RunArgs& r);
cudaError_t pack_gru_weights(domino_ctx* c, cudaStream_t st);
cudaError_t prepare_gru_tc(domino_ctx* c, RunArgs& r, GruMaps* m);
cudaError_t launch_gru_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int u);
cudaError_t launch_fc1_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int k);
// the joined projector (fc1 rows of step k with the packed W_hh products for
// update k+1) and the element-wise update after the correction (gru_tc.cu)
cudaError_t launch_proj_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int k);
cudaError_t launch_update_tc(domino_ctx* c, RunArgs& r, int u);

// persistent driver of the GRU seed and the 14 corrected steps (persist.cu).
// Requests per GRU/projector staging group; the workspace's hidden-side
// products of the next update (domino_ctx::gh_next) hold one group.
constexpr int kPersistGruGroup = 4;
bool persist_supported(const domino_ctx* c, const RunArgs& r);
cudaError_t launch_persist(domino_ctx* c, RunArgs& r);

// persistent driver with tagged data exchanges for small batches (persist_ll.cu)
constexpr int kLLMaxBatch = 8;        // requests it covers
constexpr int kClaimCounters = 16;    // sync words 16..31: per-step shared-chunk counters (cleared per run)
constexpr int kRunEpochWord = 64;     // sync word 64: run counter (bumped per run, never cleared)
bool persist_ll_supported(const domino_ctx* c, const RunArgs& r);
cudaError_t launch_persist_ll(domino_ctx* c, RunArgs& r);

// index of the ping-pong h buffer written by GRU update u
__host__ __device__ inline int h_slot(int u) { return u & 1; }

}  // namespace domino
