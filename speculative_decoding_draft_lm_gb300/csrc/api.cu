// C ABI of the Domino draft-block rollout: argument checks, workspace, the
// sequence of launches for one block, status and teardown.
#include <stdlib.h>
#include <string.h>

#include "internal.h"

using namespace domino;

namespace {

struct DeviceGuard {
    int prev = -1;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) prev = -1;
        if (prev != dev) cudaSetDevice(dev);
    }
    ~DeviceGuard() {
        int cur;
        if (prev >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != prev) cudaSetDevice(prev);
    }
};

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

inline bool aligned16(const void* p) { return ((uintptr_t)p & 15u) == 0; }

int check_config(const domino_config* g) {
    if (!g) return DOMINO_ERR_INVALID_ARG;
    if (g->block != DOMINO_BLOCK) return DOMINO_ERR_UNSUPPORTED;
    if (g->dtype != DOMINO_DTYPE_FP32 && g->dtype != DOMINO_DTYPE_BF16) return DOMINO_ERR_UNSUPPORTED;
    if (g->V < 2 || g->H < 1 || g->E < 1 || g->G < 1 || g->F < 1 || g->max_B < 1 || g->max_K < 0)
        return DOMINO_ERR_INVALID_ARG;
    if (g->max_B > 4096) return DOMINO_ERR_INVALID_ARG;
    if (g->dtype == DOMINO_DTYPE_BF16 && ((g->H | g->E | g->G | g->F) & 7)) return DOMINO_ERR_UNSUPPORTED;
    return DOMINO_OK;
}

// Event pair around one launch when timing is on; returns the pair's slot
// (-1 when off or when the pending list is full).
int timing_begin(domino_ctx* c, cudaStream_t st, int phase) {
    if (!c->timing || c->n_pending >= 4096) return -1;
    int i = c->n_pending;
    while (c->n_events < 2 * (i + 1)) {
        if (cudaEventCreate(&c->ev[c->n_events]) != cudaSuccess) return -1;
        ++c->n_events;
    }
    if (cudaEventRecord(c->ev[2 * i], st) != cudaSuccess) return -1;
    c->pending_phase[i] = phase;
    c->n_pending = i + 1;
    return i;
}

cudaError_t timing_end(domino_ctx* c, cudaStream_t st, int slot) {
    if (slot < 0) return cudaSuccess;
    return cudaEventRecord(c->ev[2 * slot + 1], st);
}

int run_impl(domino_ctx* c, const void* hidden, const void* s, const int32_t* verified, int B, int K,
             const int32_t* forced, const domino_debug_bufs* dbg, int32_t* out, void* stream) {
    if (!c) return DOMINO_ERR_INVALID_ARG;
    if (!c->loaded) return DOMINO_ERR_NOT_LOADED;
    if (B < 0 || B > c->cfg.max_B || K < 0) return DOMINO_ERR_INVALID_ARG;
    if (B == 0) {
        c->last_launches = 0;
        return DOMINO_OK;
    }
    // s == null: derive it from the hidden rows with the loaded W_hid
    if (!hidden || !verified || !out || (!s && !c->fc1_hid)) return DOMINO_ERR_INVALID_ARG;
    const int Keff = (K >= c->cfg.V) ? 0 : K;
    if (Keff > c->cfg.max_K) return DOMINO_ERR_INVALID_ARG;
    if (c->cfg.dtype == DOMINO_DTYPE_BF16 && (!aligned16(hidden) || (s && !aligned16(s))))
        return DOMINO_ERR_INVALID_ARG;

    DeviceGuard guard(c->device);
    RunArgs r;
    memset(&r, 0, sizeof(r));
    r.hidden = hidden;
    r.s = s ? s : c->s_ws;
    r.s_out = s ? nullptr : c->s_ws;
    r.verified = verified;
    r.B = B;
    r.K = Keff;
    r.n_prop = c->n_proposals;
    r.forced = forced;
    if (dbg) r.dbg = *dbg;
    r.out_tokens = out;
    r.st = (cudaStream_t)stream;

    // 0: per-phase kernels, 1: grid-barrier persistent kernel, 2: tagged-exchange persistent kernel
    int persist_kind = 0;
    if (c->driver == DOMINO_DRIVER_PERSISTENT) {
        persist_kind = persist_ll_supported(c, r) ? 2 : persist_supported(c, r) ? 1 : -1;
    } else if (c->driver == DOMINO_DRIVER_PERSISTENT_GRID) {
        persist_kind = persist_supported(c, r) ? 1 : -1;
    } else if (c->driver == DOMINO_DRIVER_AUTO) {
        // one request: a persistent driver; pools of up to eight requests: the
        // tagged-exchange driver; other batches: the batched kernels
        if (r.B == 1) persist_kind = persist_ll_supported(c, r) ? 2 : persist_supported(c, r) ? 1 : 0;
        else if (r.K > 0 && persist_ll_supported(c, r)) persist_kind = 2;
    }
    if (persist_kind < 0) return DOMINO_ERR_UNSUPPORTED;
    const bool use_persist = persist_kind > 0;

    cudaError_t e;
#define STEP(phase, x)                                   \
    do {                                                 \
        int slot_ = timing_begin(c, r.st, phase);        \
        e = (x);                                         \
        if (e != cudaSuccess) goto fail;                 \
        e = timing_end(c, r.st, slot_);                  \
        if (e != cudaSuccess) goto fail;                 \
    } while (0)
    STEP(DOMINO_PHASE_OTHER, launch_reset(c, r));
    {
        const bool tc_path = lmhead_tc_supported(c) && (!r.s_out || c->has_fc1h_tmap);
        if (tc_path) {
            STEP(DOMINO_PHASE_LMHEAD, launch_lmhead_tc(c, r));  // s rides along when r.s_out is set
        } else {
            STEP(DOMINO_PHASE_LMHEAD, launch_lmhead_simt(c, r));
            if (r.s_out) STEP(DOMINO_PHASE_LMHEAD, launch_backbone_s_simt(c, r));
            STEP(DOMINO_PHASE_ARGMAX, launch_first_argmax(c, r));
        }
        if (r.K > 0) {
            if (c->partitions > 1 && pool_compact_supported(c, c->partitions, r.K)) {
                if (!tc_path) STEP(DOMINO_PHASE_POOL, launch_score(c, r));
                STEP(DOMINO_PHASE_POOL, launch_pool_compact(c, r, c->partitions));
            } else {
                STEP(DOMINO_PHASE_POOL, launch_pool_select(c, r, tc_path));
            }
        }
    }
    if (use_persist) {
        STEP(DOMINO_PHASE_STEPS, persist_kind == 2 ? launch_persist_ll(c, r) : launch_persist(c, r));
    } else {
    const bool batch = r.B >= 2 && batch_kernels_supported(c);
    // bf16 batches: GRU and projector layer 1 as tensor-core contractions
    const bool gru_tc = batch && gru_tc_supported(c, r);
    GruMaps gm;
    if (gru_tc) {
        e = prepare_gru_tc(c, r, &gm);
        if (e != cudaSuccess) goto fail;
    }
#define GRU(u) (gru_tc ? launch_gru_tc(c, r, gm, (u)) : batch ? launch_gru_batch(c, r, (u)) : launch_gru(c, r, (u)))
#define FC1(k) (gru_tc ? launch_fc1_tc(c, r, gm, (k)) : batch ? launch_fc1_batch(c, r, (k)) : launch_fc1(c, r, (k)))
    // bf16 batches of up to eight requests: one fused launch per step (the
    // GRU update and projector layer 1), after the seed update and W_hh h_0.
    // A block of one proposal has no step, but still the seed's second update.
    const bool fused = batch && !gru_tc && r.n_prop >= 2 && step_fused_supported(c, r);
    // tensor-core batches: per step one joined projector launch (fc1 rows and
    // W_hh h for the next update), the correction, then an element-wise update
    const bool joined = gru_tc && c->ghb;
    STEP(DOMINO_PHASE_GRU, GRU(0));
    if (joined) {
        STEP(DOMINO_PHASE_GRU, launch_proj_tc(c, r, gm, 0));
        STEP(DOMINO_PHASE_GRU, launch_update_tc(c, r, 1));
    } else {
        STEP(DOMINO_PHASE_GRU, fused ? launch_step_fused(c, r, 0) : GRU(1));
    }
    {
        // tensor cores once the full-vocabulary correction is a real
        // contraction (two or more requests); CUDA cores for B = 1 and pools
        const bool tc_corr = r.B >= 2 && correct_tc_supported(c, r);
        CUtensorMap tm_a;
        if (tc_corr && r.K > 0) STEP(DOMINO_PHASE_POOL, launch_pool_mask(c, r));
        if (tc_corr) {
            e = prepare_correct_tc(c, r, &tm_a);
            if (e != cudaSuccess) goto fail;
        }
        const int n_corr = r.n_prop - 1;
        for (int k = 1; k <= n_corr; ++k) {
            STEP(DOMINO_PHASE_FC1, fused ? launch_step_fused(c, r, k) : joined ? launch_proj_tc(c, r, gm, k) : FC1(k));
            if (tc_corr)
                STEP(DOMINO_PHASE_CORRECT, launch_correct_tc(c, r, tm_a, k));
            else if (r.K > 0 && batch && pool_batch_supported(c))
                STEP(DOMINO_PHASE_CORRECT, launch_correct_pool_batch(c, r, k));
            else
                STEP(DOMINO_PHASE_CORRECT, launch_correct_simt(c, r, k));
            if (k < n_corr && !fused) STEP(DOMINO_PHASE_GRU, joined ? launch_update_tc(c, r, k + 1) : GRU(k + 1));
        }
    }
#undef GRU
#undef FC1
    }
    STEP(DOMINO_PHASE_OTHER, launch_finalize(c, r));
    if (r.dbg.logits)
        STEP(DOMINO_PHASE_OTHER, cudaMemcpyAsync(r.dbg.logits, c->L, (size_t)B * kBlock * c->cfg.V * sizeof(float),
                                                 cudaMemcpyDeviceToDevice, r.st));
    if (r.dbg.pool && r.K > 0)
        STEP(DOMINO_PHASE_OTHER, cudaMemcpyAsync(r.dbg.pool, c->pool, (size_t)B * r.K * sizeof(int32_t),
                                                 cudaMemcpyDeviceToDevice, r.st));
#undef STEP
    c->last_launches = r.launches;
    return DOMINO_OK;
fail:
    c->last_launches = r.launches;
    return DOMINO_ERR_CUDA;
}

}  // namespace

extern "C" {

int domino_rollout_init(domino_ctx** out, const domino_config* cfg, int device) {
    if (!out) return DOMINO_ERR_INVALID_ARG;
    *out = nullptr;
    int st = check_config(cfg);
    if (st != DOMINO_OK) return st;
    int ndev = 0;
    if (cudaGetDeviceCount(&ndev) != cudaSuccess || device < 0 || device >= ndev) return DOMINO_ERR_CUDA;
    DeviceGuard guard(device);

    domino_ctx* c = (domino_ctx*)calloc(1, sizeof(domino_ctx));
    if (!c) return DOMINO_ERR_OOM;
    c->cfg = *cfg;
    c->device = device;
    if (cudaDeviceGetAttribute(&c->num_sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        free(c);
        return DOMINO_ERR_CUDA;
    }
    const domino_config& g = c->cfg;
    c->a_rows = (int)align_up((size_t)(g.max_B > 16 ? g.max_B : 16), 16);
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t o = off;
        off = align_up(off + bytes, 256);
        return o;
    };
    size_t oL = take((size_t)g.max_B * kBlock * g.V * sizeof(float));
    size_t oS = take(g.max_K > 0 ? (size_t)g.max_B * g.V * sizeof(float) : 0);
    size_t oP = take((size_t)g.max_B * (g.max_K > 0 ? g.max_K : 1) * sizeof(int32_t));
    size_t oSw = take((size_t)g.max_B * kProposals * g.F * (g.dtype == DOMINO_DTYPE_BF16 ? 2 : 4));
    size_t oH = take((size_t)2 * g.max_B * g.G * sizeof(float));
    size_t oA = take((size_t)g.max_B * g.F * sizeof(float));
    size_t oA16 = take((size_t)c->a_rows * g.F * sizeof(__nv_bfloat16));
    size_t oK = take((size_t)g.max_B * kBlock * sizeof(unsigned long long));
    size_t oBad = take((size_t)g.max_B * sizeof(int));
    size_t oErr = take(sizeof(int));
    size_t oSync = take(1024);
    const bool gru_tc = gru_tc_shape_ok(g);
    size_t oWp = take(gru_tc ? (size_t)4 * gru_padded_units(g.G) * g.G * 2 : 0);
    size_t oX = take(gru_tc ? (size_t)2 * c->a_rows * g.G * 2 : 0);
    size_t oT = take((size_t)g.V * 3 * g.G * sizeof(float));
    size_t oGh = take((size_t)kPersistGruGroup * 3 * g.G * sizeof(float));
    const bool pmask = g.max_K > 0 && g.dtype == DOMINO_DTYPE_BF16;
    size_t oM = take(pmask ? (size_t)g.max_B * pool_mask_words(g.V) * 4 : 0);
    size_t oHs = take(pmask ? (size_t)g.max_B * kPoolHistBins * 4 : 0);
    size_t oC = take(g.max_K > 0 ? (size_t)g.max_B * DOMINO_MAX_VOCAB_PARTITIONS * g.max_K * 4 : 0);
    const bool ll = g.dtype == DOMINO_DTYPE_BF16;  // tagged-exchange persistent driver
    size_t oXa = take(ll ? (size_t)2 * kLLMaxBatch * g.F * 8 : 0);
    size_t oXg = take(ll ? (size_t)2 * kLLMaxBatch * g.G * 8 : 0);
    size_t oXb = take(ll ? (size_t)2 * c->num_sms * kLLMaxBatch * 8 : 0);
    size_t oXq = take(ll ? (size_t)2 * 3 * g.G * 8 : 0);
    // hidden-side products of the batched paths: [2][max_B][3G] (fused step) or [2][max_B][4Gp] (packed)
    size_t oGb = take(ll ? (size_t)2 * g.max_B * 4 * gru_padded_units(g.G) * sizeof(float) : 0);
    c->ws_bytes = off;
    if (cudaMalloc(&c->ws_base, c->ws_bytes) != cudaSuccess) {
        cudaGetLastError();
        free(c);
        return DOMINO_ERR_OOM;
    }
    char* base = (char*)c->ws_base;
    c->L = (float*)(base + oL);
    c->score = (float*)(base + oS);
    c->pool = (int32_t*)(base + oP);
    c->s_ws = base + oSw;
    c->h = (float*)(base + oH);
    c->a = (float*)(base + oA);
    c->a16 = (__nv_bfloat16*)(base + oA16);
    c->keys = (unsigned long long*)(base + oK);
    c->bad = (int*)(base + oBad);
    c->err = (int*)(base + oErr);
    c->sync = (unsigned int*)(base + oSync);
    c->wp = gru_tc ? (__nv_bfloat16*)(base + oWp) : nullptr;
    c->h16 = gru_tc ? (__nv_bfloat16*)(base + oX) : nullptr;
    c->gi_table = (float*)(base + oT);
    c->gh_next = (float*)(base + oGh);
    c->pmask = pmask ? (uint32_t*)(base + oM) : nullptr;
    c->cand = g.max_K > 0 ? (int32_t*)(base + oC) : nullptr;
    c->xa = ll ? (unsigned long long*)(base + oXa) : nullptr;
    c->xh = ll ? (unsigned long long*)(base + oXg) : nullptr;
    c->xbest = ll ? (unsigned long long*)(base + oXb) : nullptr;
    c->xg = ll ? (unsigned long long*)(base + oXq) : nullptr;
    c->ghb = ll ? (float*)(base + oGb) : nullptr;
    c->hist = pmask ? (unsigned*)(base + oHs) : nullptr;
    // zero the small state (a16 padding rows must stay zero for the MMA path)
    if (cudaMemset(base + oH, 0, off - oH) != cudaSuccess || prepare_simt_kernels(c) != cudaSuccess ||
        cudaDeviceSynchronize() != cudaSuccess) {
        cudaFree(c->ws_base);
        free(c);
        return DOMINO_ERR_CUDA;
    }
    c->driver = DOMINO_DRIVER_AUTO;
    c->n_proposals = kProposals;
    c->partitions = 1;
    *out = c;
    return DOMINO_OK;
}

int domino_rollout_load_weights(domino_ctx* c, const void* lm_head, const void* emb, const void* w_ih,
                                const void* w_hh, const void* fc1, const void* fc2, const void* bias) {
    if (!c || !lm_head || !emb || !w_ih || !w_hh || !fc1 || !fc2 || !bias) return DOMINO_ERR_INVALID_ARG;
    const void* ps[] = {lm_head, emb, w_ih, w_hh, fc1, fc2, bias};
    for (const void* p : ps)
        if (!aligned16(p)) return DOMINO_ERR_INVALID_ARG;
    c->lm_head = lm_head;
    c->emb = emb;
    c->w_ih = w_ih;
    c->w_hh = w_hh;
    c->fc1 = fc1;
    c->fc2 = fc2;
    c->bias = bias;
    c->has_tma = false;
    if (c->cfg.dtype == DOMINO_DTYPE_BF16) {
        DeviceGuard guard(c->device);
        const domino_config& g = c->cfg;
        if (make_tmap_bf16(&c->tm_lm_head, lm_head, (uint64_t)g.V, (uint64_t)g.H, 128) != cudaSuccess ||
            make_tmap_bf16(&c->tm_fc2, fc2, (uint64_t)g.V, (uint64_t)g.F, 128) != cudaSuccess) {
            c->loaded = false;
            return DOMINO_ERR_CUDA;
        }
        c->has_tma = true;
        // the batched GRU contracts a packed copy of w_hh (built here, once)
        if (c->wp && pack_gru_weights(c, 0) != cudaSuccess) {
            c->loaded = false;
            return DOMINO_ERR_CUDA;
        }
    }
    {
        // input-side GRU pre-activations of every token (W_ih emb[v]), once
        DeviceGuard guard(c->device);
        int err_word = 0;
        if (build_gi_table(c, 0) != cudaSuccess || cudaStreamSynchronize(0) != cudaSuccess ||
            cudaMemcpy(&err_word, c->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess || err_word != 0) {
            c->loaded = false;
            return DOMINO_ERR_CUDA;
        }
    }
    c->loaded = true;
    return DOMINO_OK;
}

int domino_rollout_load_backbone_proj(domino_ctx* c, const void* w_hid) {
    if (!c) return DOMINO_ERR_INVALID_ARG;
    if (!w_hid) {
        c->fc1_hid = nullptr;
        c->has_fc1h_tmap = false;
        return DOMINO_OK;
    }
    if (!aligned16(w_hid)) return DOMINO_ERR_INVALID_ARG;
    c->fc1_hid = w_hid;
    c->has_fc1h_tmap = false;
    if (c->cfg.dtype == DOMINO_DTYPE_BF16) {
        DeviceGuard guard(c->device);
        // 16-byte TMA row stride; otherwise the CUDA-core path computes s
        if (c->cfg.H % 8 == 0 &&
            make_tmap_bf16(&c->tm_fc1h, w_hid, (uint64_t)c->cfg.F, (uint64_t)c->cfg.H, 128) == cudaSuccess)
            c->has_fc1h_tmap = true;
    }
    return DOMINO_OK;
}

int domino_rollout_run(domino_ctx* c, const void* hidden, const void* s, const int32_t* verified, int B, int K,
                       int32_t* out_tokens, void* stream) {
    return run_impl(c, hidden, s, verified, B, K, nullptr, nullptr, out_tokens, stream);
}

int domino_rollout_debug_run(domino_ctx* c, const void* hidden, const void* s, const int32_t* verified, int B, int K,
                             const int32_t* forced, const domino_debug_bufs* dbg, int32_t* out_tokens, void* stream) {
    return run_impl(c, hidden, s, verified, B, K, forced, dbg, out_tokens, stream);
}

int domino_rollout_set_driver(domino_ctx* c, int driver) {
    if (!c) return DOMINO_ERR_INVALID_ARG;
    if (driver != DOMINO_DRIVER_AUTO && driver != DOMINO_DRIVER_KERNELS && driver != DOMINO_DRIVER_PERSISTENT &&
        driver != DOMINO_DRIVER_PERSISTENT_GRID)
        return DOMINO_ERR_INVALID_ARG;
    c->driver = driver;
    return DOMINO_OK;
}

int domino_rollout_enable_timing(domino_ctx* c, int enable) {
    if (!c) return DOMINO_ERR_INVALID_ARG;
    c->timing = enable != 0;
    return DOMINO_OK;
}

int domino_rollout_read_timing(domino_ctx* c, float* ms, int* launches) {
    if (!c || !ms || !launches) return DOMINO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    for (int i = 0; i < c->n_pending; ++i) {
        float t = 0.f;
        if (cudaEventSynchronize(c->ev[2 * i + 1]) != cudaSuccess ||
            cudaEventElapsedTime(&t, c->ev[2 * i], c->ev[2 * i + 1]) != cudaSuccess) {
            c->n_pending = 0;
            return DOMINO_ERR_CUDA;
        }
        int p = c->pending_phase[i];
        if (p >= 0 && p < DOMINO_N_PHASES) {
            ms[p] += t;
            launches[p] += 1;
        }
    }
    c->n_pending = 0;
    return DOMINO_OK;
}

int domino_rollout_set_vocab_partitions(domino_ctx* c, int P) {
    if (!c || P < 1 || P > DOMINO_MAX_VOCAB_PARTITIONS) return DOMINO_ERR_INVALID_ARG;
    c->partitions = P;
    return DOMINO_OK;
}

int domino_rollout_set_proposals(domino_ctx* c, int n) {
    if (!c || n < 1 || n > kProposals) return DOMINO_ERR_INVALID_ARG;
    c->n_proposals = n;
    return DOMINO_OK;
}

int domino_rollout_debug_drop_barrier_arrival(domino_ctx* c, int n) {
    if (!c || n < 0) return DOMINO_ERR_INVALID_ARG;
    c->drop_barrier = n;
    return DOMINO_OK;
}

int domino_rollout_status(domino_ctx* c, void* stream) {
    if (!c) return DOMINO_ERR_INVALID_ARG;
    DeviceGuard guard(c->device);
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return DOMINO_ERR_CUDA;
    int word = 0;
    if (cudaMemcpy(&word, c->err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return DOMINO_ERR_CUDA;
    if (word && cudaMemset(c->err, 0, sizeof(int)) != cudaSuccess) return DOMINO_ERR_CUDA;
    if (word & kErrTimeout) return DOMINO_ERR_TIMEOUT;
    if (word & kErrBadToken) return DOMINO_ERR_BAD_TOKEN;
    return DOMINO_OK;
}

int domino_rollout_last_launch_count(const domino_ctx* c) { return c ? c->last_launches : 0; }

void domino_rollout_destroy(domino_ctx* c) {
    if (!c) return;
    {
        DeviceGuard guard(c->device);
        cudaDeviceSynchronize();
        cudaFree(c->ws_base);
        for (int i = 0; i < c->n_events; ++i) cudaEventDestroy(c->ev[i]);
    }
    free(c);
}

const char* domino_rollout_strerror(int st) {
    switch (st) {
        case DOMINO_OK: return "ok";
        case DOMINO_ERR_INVALID_ARG: return "invalid argument";
        case DOMINO_ERR_UNSUPPORTED: return "unsupported configuration";
        case DOMINO_ERR_NOT_LOADED: return "weights not loaded";
        case DOMINO_ERR_CUDA: return "CUDA error";
        case DOMINO_ERR_OOM: return "out of device memory";
        case DOMINO_ERR_TIMEOUT: return "device-side wait timed out";
        case DOMINO_ERR_BAD_TOKEN: return "token id outside [0, V)";
        case DOMINO_ERR_SCRATCH_LIMIT: return "request exceeds the static scratch buffer";
        default: return "unknown status";
    }
}

}  // extern "C"
