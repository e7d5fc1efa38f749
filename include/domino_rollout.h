/*
 * domino_rollout.h - C ABI of the GB300 (sm_103a) Domino draft-block rollout.
 *
 * The operation (page "Add correctness-first Domino support to DFlash V2",
 * section "Design"; page "[Spec] Add Domino projector support to DFlash
 * speculative decoding (V2)", section "Implementation"): for each of B
 * independent requests, given the 16 draft hidden states of a DFlash block,
 *
 *   1. base logits  L[b,i,:] = lm_head @ hidden[b,i,:]  for the 16 rows i;
 *   2. p_1 = argmax of base row 1 over the full vocabulary (uncorrected);
 *   3. a bias-free GRU (gate rows r|z|n, h_0 = 0) is seeded with the
 *      embeddings of [verified_token, p_1];
 *   4. for corrected step k = 1..14:
 *        a = SiLU(fc1 @ h + s[b,k,:]),
 *        c[v] = fc2[v,:] . a + bias[v] + L[b,k+1,v]   (v in the pool),
 *        p_{k+1} = argmax_v c[v]  (lowest token id on ties),
 *        and, for k < 14, h = GRU(emb[p_{k+1}], h);
 *   5. out_tokens[b,:] = [p_1 .. p_15].
 *
 * The pool (page "Add correctness-first Domino support to DFlash V2",
 * section "Design": one per-request, block-shared candidate pool; size 0
 * means the full vocabulary) is, for 0 < K < V, the K token ids with the
 * largest max over base rows 1..15 (ties to the lower id).  K = 0 or K >= V
 * scores the full vocabulary.
 *
 * Threading: a context may be used from one host thread at a time.  All
 * calls taking a stream are asynchronous on that stream and make no host
 * synchronisation, except domino_rollout_status().  Every entry point
 * returns DOMINO_OK (0) or a negative status; nothing falls back to the CPU.
 */
#ifndef DOMINO_ROLLOUT_H
#define DOMINO_ROLLOUT_H

#include <stdint.h>

#if defined(__GNUC__)
#define DOMINO_API __attribute__((visibility("default")))
#else
#define DOMINO_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* status codes */
#define DOMINO_OK                 0
#define DOMINO_ERR_INVALID_ARG   -1  /* null pointer, B > max_B, K < 0, bad size   */
#define DOMINO_ERR_UNSUPPORTED   -2  /* block != 16, unknown dtype, misaligned dims */
#define DOMINO_ERR_NOT_LOADED    -3  /* run before load_weights                      */
#define DOMINO_ERR_CUDA          -4  /* a CUDA call or launch failed                 */
#define DOMINO_ERR_OOM           -5  /* workspace allocation failed                  */
#define DOMINO_ERR_TIMEOUT       -6  /* a device-side wait hit its iteration limit   */
#define DOMINO_ERR_BAD_TOKEN     -7  /* verified/forced token outside [0, V)         */
#define DOMINO_ERR_SCRATCH_LIMIT -8  /* request larger than the static scratch        */

#define DOMINO_DTYPE_FP32 0  /* fp32 weights/activations, fp32 arithmetic          */
#define DOMINO_DTYPE_BF16 1  /* bf16 weights/activations, fp32 accumulation        */

#define DOMINO_BLOCK 16      /* draft block size; 15 proposals per request         */

typedef struct domino_ctx domino_ctx;

/* Model dimensions fixed at init.  V vocabulary, H draft hidden size, E token
 * embedding size, G GRU state size, F projector width (fc1 rows, fc2 cols).
 * For DOMINO_DTYPE_BF16, H, E, G and F must be multiples of 8 (16-byte rows
 * for the bulk copies).  max_B / max_K size the workspace. */
typedef struct {
    int V, H, E, G, F;
    int block;   /* must be DOMINO_BLOCK */
    int max_B;   /* largest batch passed to run(), >= 1 */
    int max_K;   /* largest pool size passed to run() (0: full vocabulary only) */
    int dtype;   /* DOMINO_DTYPE_* */
} domino_config;

/* Create a context on CUDA device `device` and allocate its workspace there
 * in one allocation: base logits [max_B,16,V] fp32, pool scores [max_B,V],
 * pool [max_B,max_K], GRU/projector state, the per-step argmax words, and the
 * token table [V,3G] fp32 that load_weights fills (1.9 GB at V = 151,936,
 * G = 1024).  *out receives the context (NULL on failure).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA, OOM. */
DOMINO_API int domino_rollout_init(domino_ctx** out, const domino_config* cfg, int device);

/* Register the weights: DEVICE pointers, row-major, in the config's dtype,
 * BORROWED (the caller keeps them alive and unchanged until destroy or the
 * next load_weights).  Shapes: lm_head [V,H]; emb [V,E]; w_ih [3G,E] and
 * w_hh [3G,G] with gate rows r|z|n; fc1 [F,G]; fc2 [V,F]; bias [V].
 * Pointers must be 16-byte aligned.  Builds the TMA descriptors and derives,
 * on the legacy default stream and synchronously, the context's own copies:
 * the input-side GRU pre-activations of every token, T[v] = w_ih . emb[v]
 * (page "Add correctness-first Domino support to DFlash V2", section
 * "Design": the GRU consumes the embedding of the realised token, so this
 * half depends on the token alone), and for bf16 a packed w_hh for the
 * tensor-core GRU.  Changing emb, w_ih or w_hh afterwards requires calling
 * load_weights again.  Errors: INVALID_ARG, CUDA. */
DOMINO_API int domino_rollout_load_weights(domino_ctx* ctx, const void* lm_head, const void* emb,
                                const void* w_ih, const void* w_hh, const void* fc1,
                                const void* fc2, const void* bias);

/* Optional: the backbone-hidden half W_hid [F,H] of projector layer 1, a
 * DEVICE pointer in the config dtype, row-major, 16-byte aligned, BORROWED
 * like the other weights (NULL unregisters it).  The projector's first layer
 * acts on [backbone hidden | GRU state] (page "Add correctness-first Domino
 * support to DFlash V2", the Domino drafter training backend change), so its
 * per-step term is s[b,j,:] = W_hid . hidden[b,j+1,:]: the hidden row whose
 * base logits proposal j corrects.  With it registered, run/debug_run accept
 * s == NULL and compute s in the library (bf16: as extra rows of the LM-head
 * contraction, stored as bf16; fp32: on the CUDA cores).  No bias is added.
 * Errors: INVALID_ARG. */
DOMINO_API int domino_rollout_load_backbone_proj(domino_ctx* ctx, const void* w_hid);

/* Run one block rollout for B requests on `cuda_stream` (a cudaStream_t,
 * NULL = legacy default stream).  Asynchronous, with no host
 * synchronisation: after one ordinary call with the same B and K (which sets
 * kernel attributes once), a call can be captured into a CUDA graph and the
 * graph replayed with new contents in the same input buffers.  DEVICE pointers, owned by the caller:
 *   hidden       [B,16,H]  draft hidden states (config dtype, 16-B aligned)
 *   s            [B,15,F]  per-step additive term of projector layer 1
 *                          (row 0 is not read; row k serves corrected step k);
 *                          NULL = compute it from `hidden` with the weight given
 *                          to domino_rollout_load_backbone_proj (INVALID_ARG if
 *                          none was given)
 *   verified_tok [B] int32 the block's verified token
 *   out_tokens   [B,15] int32 proposals p_1..p_15 (written)
 * K: pool size; 0 (or >= V) = full-vocabulary correction; 0 < K < V needs
 * K <= max_K.  A verified token outside [0,V) is caught on the device: that
 * request's row of out_tokens becomes -1 and domino_rollout_status() reports
 * DOMINO_ERR_BAD_TOKEN.  Errors returned directly: INVALID_ARG,
 * NOT_LOADED, CUDA. */
DOMINO_API int domino_rollout_run(domino_ctx* ctx, const void* hidden, const void* s,
                       const int32_t* verified_tok, int B, int K,
                       int32_t* out_tokens, void* cuda_stream);

/* Optional dumps for domino_rollout_debug_run (each DEVICE pointer may be
 * NULL, caller-owned, fp32 unless noted). */
typedef struct {
    float*   logits;  /* [B,16,V] base logits                                   */
    int32_t* pool;    /* [B,K] pool ids, ascending (only when 0 < K < V)        */
    float*   h;       /* [B,15,G] GRU state after each of the 15 updates        */
    float*   z;       /* [B,14,F] projector pre-activation of each step         */
    float*   top1;    /* [B,15] winning score of each proposal                  */
    float*   scores;  /* [B,14,Kc] corrected scores, Kc = V (K0) or K (pool)    */
    unsigned long long* trace; /* [grid,DOMINO_TRACE_SLOTS] %globaltimer stamps (ns)
                                  of the persistent driver's phase boundaries per
                                  CTA (grid = SM count); untouched by the other
                                  driver */
} domino_debug_bufs;
#define DOMINO_TRACE_SLOTS 96

/* As domino_rollout_run, plus teacher forcing and dumps.  forced_tokens
 * (nullable DEVICE [B,15] int32): when given, the GRU is fed forced[b,k]
 * instead of p_{k+1}, while out_tokens still reports each step's own argmax.
 * A forced token outside [0,V) is a BAD_TOKEN fault like a verified one. */
DOMINO_API int domino_rollout_debug_run(domino_ctx* ctx, const void* hidden, const void* s,
                             const int32_t* verified_tok, int B, int K,
                             const int32_t* forced_tokens, const domino_debug_bufs* dbg,
                             int32_t* out_tokens, void* cuda_stream);

/* Driver of the 14 dependent steps.  The persistent drivers are one
 * cooperative launch (one CTA per SM).  The tagged-exchange one covers bf16,
 * B <= 8 (B = 1 for the full vocabulary), G, F <= 1024 and V < 2^18: its CTAs
 * pass activations, GRU state units and per-CTA bests through words that
 * carry the step they belong to, instead of meeting at grid barriers.
 * DOMINO_DRIVER_PERSISTENT takes it where it applies and the grid-barrier
 * kernel elsewhere; DOMINO_DRIVER_PERSISTENT_GRID always the latter.  A
 * persistent driver that does not cover the run gives UNSUPPORTED.  AUTO
 * takes a persistent driver for one request and the tagged-exchange one for
 * the pools it covers; other batches run one launch per phase. */
#define DOMINO_DRIVER_AUTO            0  /* pick per (B, K)                              */
#define DOMINO_DRIVER_KERNELS         1  /* one launch per phase, stream-ordered         */
#define DOMINO_DRIVER_PERSISTENT      2  /* one cooperative launch (see above)           */
#define DOMINO_DRIVER_PERSISTENT_GRID 3  /* one cooperative launch with grid barriers    */
DOMINO_API int domino_rollout_set_driver(domino_ctx* ctx, int driver);

/* Per-phase timing.  When enabled, run()/debug_run() record a pair of CUDA
 * events on the run's stream around every launch and tag it with its phase
 * (DOMINO_PHASE_*).  read_timing() waits for the recorded events, adds each
 * pair's elapsed time to ms[phase] and its launch to launches[phase] (both
 * caller-owned host arrays of DOMINO_N_PHASES entries, zeroed by the caller)
 * and forgets them.  At most 4096 pending pairs are kept; call read_timing()
 * after each run.  Errors: INVALID_ARG, CUDA. */
#define DOMINO_PHASE_LMHEAD     0  /* base LM-head (+ fused epilogue)                */
#define DOMINO_PHASE_ARGMAX     1  /* first-proposal argmax                          */
#define DOMINO_PHASE_POOL       2  /* candidate pool (score + select)                */
#define DOMINO_PHASE_GRU        3  /* GRU updates                                    */
#define DOMINO_PHASE_FC1        4  /* projector layer 1 + SiLU                       */
#define DOMINO_PHASE_CORRECT    5  /* correction + argmax                            */
#define DOMINO_PHASE_STEPS      6  /* persistent driver of the 14 steps              */
#define DOMINO_PHASE_OTHER      7  /* reset, write-out, debug copies                 */
#define DOMINO_N_PHASES         8
DOMINO_API int domino_rollout_enable_timing(domino_ctx* ctx, int enable);
DOMINO_API int domino_rollout_read_timing(domino_ctx* ctx, float* ms, int* launches);

/* Early stop: produce only the first n proposals (1 <= n <= 15; default 15)
 * with n-1 corrected steps, for a target that verifies only the first n+1
 * block positions (page "feat: support tensor-parallel Domino rollout",
 * section "Qwen3.6-27B checkpoint and full serving benchmark": the b8 run
 * keeps the block-16 draft and verifies 8 positions, i.e. n = 7).  The draft
 * itself is unchanged: the LM-head still covers all 16 rows and the pool
 * (K > 0) is still taken over the whole block, so the n tokens equal the
 * first n of the full rollout.  out_tokens keeps its [B,15] layout; entries
 * n..14 of each row are set to -1.  The setting applies to later runs of
 * this context.  Errors: INVALID_ARG (null ctx or n outside 1..15). */
DOMINO_API int domino_rollout_set_proposals(domino_ctx* ctx, int n);

/* Candidate-pool construction of the tensor-parallel stage C, on one GPU
 * (page "feat: support tensor-parallel Domino rollout", section
 * "Implementation": each rank takes a local top-K of its vocabulary shard and
 * the candidates are merged to the global top-K).  P > 1 splits the
 * vocabulary into P contiguous shards of ceil(V/P) ids: one cluster
 * radix-select per (request, shard), then one per request over the P*K
 * candidates.  The pool is the same as with P = 1 (the direct selection),
 * ties included; only the way it is built changes.  P = 1 (default) .. 8.
 * Pool modes with K > 0 only; ignored when the selection does not fit.
 * Errors: INVALID_ARG. */
#define DOMINO_MAX_VOCAB_PARTITIONS 8
DOMINO_API int domino_rollout_set_vocab_partitions(domino_ctx* ctx, int P);

/* Synchronise `cuda_stream`, then return and clear the device error word
 * (DOMINO_OK, DOMINO_ERR_BAD_TOKEN or DOMINO_ERR_TIMEOUT), or DOMINO_ERR_CUDA
 * if the stream reported an error. */
DOMINO_API int domino_rollout_status(domino_ctx* ctx, void* cuda_stream);

/* Test hook of the device-side timeout path (page "Add correctness-first
 * Domino support to DFlash V2", section "Supported and numerical scope":
 * clear errors, no silent fallback).  Off by default and one-shot: with
 * n >= 1, the next run that uses a persistent driver makes its first CTA
 * withhold its n-th synchronisation: its arrival at the n-th grid barrier
 * (barriers 1 and 2 follow the two seed updates; each corrected step then
 * has two, or three for more than four requests), or in the tagged-exchange
 * driver its n-th publication (1: its GRU units after the seed update; then
 * per step its activations, together with its units' hidden-side products
 * for one request, its best, and, for more than one request and unless the
 * step is the last, its GRU units after the next update).  Nothing replaces
 * it, so the bounded
 * wait of every CTA for it runs out after 200 ms, the kernel returns, the
 * run's tokens are meaningless and
 * domino_rollout_status() reports DOMINO_ERR_TIMEOUT.  Nothing faults or
 * hangs and the context stays usable; that run clears the hook (n = 0 clears
 * it by hand).  Errors: INVALID_ARG (null ctx, n < 0). */
DOMINO_API int domino_rollout_debug_drop_barrier_arrival(domino_ctx* ctx, int n);

/* Number of kernel launches the last run()/debug_run() enqueued. */
DOMINO_API int domino_rollout_last_launch_count(const domino_ctx* ctx);

/* Allocation-free candidate pool.  The method described by the pages has no
 * counterpart for this entry point: it exists for callers that must not
 * allocate device memory, e.g. code that runs while a memory planner owns
 * every byte of the device, or a process whose allocator is locked for the
 * lifetime of a captured workload.  It needs no context and calls no
 * cudaMalloc, cudaFree or allocating library routine.
 *
 * From base logits [B,16,V] fp32 (DEVICE, caller-owned; the layout that
 * domino_rollout_debug_run dumps), it forms score[b,v] = max over rows 1..15
 * in a scratch array that the library keeps in a file-scope __device__
 * buffer of DOMINO_STATIC_SCRATCH_FLOATS floats (8 MiB on every device that
 * loads the library, held until the process exits), then writes the K ids
 * with the largest scores (ties to the lower id), ascending, to pool_out
 * [B,K] int32 (DEVICE, caller-owned) on `cuda_stream`, for the current device.
 *
 * The first call on a device looks up the buffer's device address on that
 * device and keeps it for the life of the process; make that first call
 * before any stream capture.  A cudaDeviceReset() of that device afterwards
 * invalidates the kept address: do not call this entry point after one.  All calls share
 * the one buffer and every call overwrites it, so calls whose kernels can
 * overlap on the GPU (different streams without ordering) race and must be
 * serialised by the caller.  Requires 0 < K < V and V <= 431000.  Errors:
 * INVALID_ARG (null pointer, B < 1, K outside (0, V), V too large),
 * SCRATCH_LIMIT (B * V > DOMINO_STATIC_SCRATCH_FLOATS), CUDA. */
#define DOMINO_STATIC_SCRATCH_FLOATS (2u * 1024u * 1024u)
DOMINO_API int domino_candidate_pool_static(const float* base_logits, int B, int V, int K, int32_t* pool_out,
                                            void* cuda_stream);

/* Free the workspace and the context (NULL is ignored).  Synchronises the
 * context's device first.  Weights stay the caller's. */
DOMINO_API void domino_rollout_destroy(domino_ctx* ctx);

/* Static description of a status code. */
DOMINO_API const char* domino_rollout_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif /* DOMINO_ROLLOUT_H */
