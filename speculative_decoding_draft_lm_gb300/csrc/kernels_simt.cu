// SIMT kernels of the rollout: reset, fp32 LM-head, first-proposal argmax,
// block-shared candidate pool, GRU update, projector layer 1 + SiLU,
// correction + argmax, and the token write-out.
//
// Method: page "Add correctness-first Domino support to DFlash V2", section
// "Design" (proposal chain, GRU seeding, pool) and page "[Spec] Add Domino
// projector support to DFlash speculative decoding (V2)", section
// "Implementation" (fused SiLU(z+s) @ fc2^T + bias + base-logits argmax,
// fused GRU cell).
#include "internal.h"

namespace domino {

namespace {

inline int grid_for(int items_per_block_unit, int units, int cap) {
    int g = (units + items_per_block_unit - 1) / items_per_block_unit;
    return g < 1 ? 1 : (g > cap ? cap : g);
}

// ---------------------------------------------------------------------------
__global__ void k_reset(unsigned long long* __restrict__ keys, int* __restrict__ bad, unsigned* __restrict__ sync,
                        unsigned long long* __restrict__ xbest, unsigned* __restrict__ hist, int n_keys, int B,
                        int n_xbest, int n_hist) {
    pdl_trigger();
    pdl_wait();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i < n_keys) keys[i] = 0ull;
    if (i < B) bad[i] = 0;
    if (i < 64) sync[i] = 0u;  // grid-barrier counter and the per-step chunk counters
    if (i < n_xbest) xbest[i] = 0ull;  // per-CTA bests of the tagged-exchange driver
    if (i < n_hist) hist[i] = 0u;      // the pool scores' first-digit histogram
    if (i == 0) sync[kRunEpochWord] += 1u;  // a new tag range for this run's exchange words
}

// ---------------------------------------------------------------------------
// LM-head on CUDA cores: one warp per vocabulary row, all 16 block rows of a
// request at once.  Used for the fp32 dtype (exact fp32 FMA) and as the
// reference-shaped path for bf16 when the tensor-core kernel is not taken.
template <typename T>
__global__ void __launch_bounds__(256) k_lmhead_simt(const T* __restrict__ X, const T* __restrict__ W,
                                                     float* __restrict__ L, int B, int V, int H) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int v = warp; v < V; v += nwarps) {
        const T* w = W + (size_t)v * H;
        for (int b = 0; b < B; ++b) {
            const T* x = X + (size_t)b * kBlock * H;
            float acc[kBlock];
#pragma unroll
            for (int r = 0; r < kBlock; ++r) acc[r] = 0.f;
            if ((H & 7) == 0) {
                for (int i = lane * 8; i < H; i += 256) {
                    float e[8];
                    load8(w + i, e);
#pragma unroll
                    for (int r = 0; r < kBlock; ++r) {
                        float f[8];
                        load8(x + (size_t)r * H + i, f);
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[r] = fmaf(e[j], f[j], acc[r]);
                    }
                }
            } else {
                for (int i = lane; i < H; i += 32) {
                    float e = to_f32(w[i]);
#pragma unroll
                    for (int r = 0; r < kBlock; ++r) acc[r] = fmaf(e, to_f32(x[(size_t)r * H + i]), acc[r]);
                }
            }
#pragma unroll
            for (int r = 0; r < kBlock; ++r) {
                float sum = warp_sum(acc[r]);
                if (lane == r) L[((size_t)b * kBlock + r) * V + v] = sum;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// p_1 = argmax over base row rho(0); one atomicMax per block.
__global__ void __launch_bounds__(256) k_first_argmax(const float* __restrict__ L,
                                                      unsigned long long* __restrict__ keys, int V) {
    __shared__ unsigned long long sw[8];
    const int b = blockIdx.y;
    const float* row = L + ((size_t)b * kBlock + kRowOffset) * V;
    unsigned long long best = 0ull;
    for (int v = blockIdx.x * blockDim.x + threadIdx.x; v < V; v += gridDim.x * blockDim.x) {
        unsigned long long k = pack_key(row[v], (uint32_t)v);
        best = k > best ? k : best;
    }
    best = warp_max_u64(best);
    if ((threadIdx.x & 31) == 0) sw[threadIdx.x >> 5] = best;
    __syncthreads();
    if (threadIdx.x == 0) {
        for (int w = 1; w < (int)(blockDim.x >> 5); ++w) best = sw[w] > best ? sw[w] : best;
        atomicMax(&keys[(size_t)b * kBlock + 0], best);
    }
}

// ---------------------------------------------------------------------------
// score[b,v] = max over the 15 base rows the proposals use.
__global__ void k_score(const float* __restrict__ L, float* __restrict__ score, int B, int V) {
    size_t n = (size_t)B * V;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        size_t b = i / V, v = i % V;
        const float* p = L + (b * kBlock + kRowOffset) * V + v;
        float m = p[0];
#pragma unroll
        for (int j = 1; j < kProposals; ++j) m = fmaxf(m, p[(size_t)j * V]);
        score[i] = m;
    }
}

// Exclusive block scan of one unsigned value per thread (blockDim = 1024).
__device__ __forceinline__ unsigned block_excl_scan(unsigned x, unsigned* warp_tot, unsigned* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        unsigned t = warp_tot[lane];
        unsigned ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            unsigned y = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += y;
        }
        warp_tot[lane] = ti - t;
        if (lane == 31) *total = ti;
    }
    __syncthreads();
    unsigned r = warp_tot[warp] + incl - x;
    __syncthreads();
    return r;
}

// Block-shared pool of one request: exact top-K of score by (score desc,
// id asc) through a 4-pass 8-bit radix select on the orderable key, then a
// stable compaction that writes the K ids in ascending order.
__global__ void __launch_bounds__(1024) k_pool_select(const float* __restrict__ score, int32_t* __restrict__ pool,
                                                      int V, int K) {
    __shared__ unsigned hist[256];
    __shared__ unsigned warp_tot[32];
    __shared__ unsigned s_prefix, s_remaining, s_total;
    const int b = blockIdx.x;
    const float* sc = score + (size_t)b * V;
    unsigned prefix = 0, mask = 0, remaining = (unsigned)K;
    for (int shift = 24; shift >= 0; shift -= 8) {
        for (int i = threadIdx.x; i < 256; i += blockDim.x) hist[i] = 0;
        __syncthreads();
        for (int v = threadIdx.x; v < V; v += blockDim.x) {
            unsigned k = ord_f32(sc[v]);
            if ((k & mask) == prefix) atomicAdd(&hist[(k >> shift) & 255u], 1u);
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned cum = 0;
            int d = 255;
            for (; d > 0; --d) {
                if (cum + hist[d] >= remaining) break;
                cum += hist[d];
            }
            s_prefix = prefix | ((unsigned)d << shift);
            s_remaining = remaining - cum;
        }
        __syncthreads();
        prefix = s_prefix;
        remaining = s_remaining;
        mask |= 255u << shift;
        __syncthreads();
    }
    const unsigned T = prefix, need = remaining;  // take `need` of the keys equal to T
    // each thread owns a contiguous run of ids, so the output stays ascending
    const int chunk = (V + blockDim.x - 1) / blockDim.x;
    const int v0 = threadIdx.x * chunk;
    const int v1 = min(V, v0 + chunk);
    unsigned gt = 0, eq = 0;
    for (int v = v0; v < v1; ++v) {
        unsigned k = ord_f32(sc[v]);
        gt += k > T;
        eq += k == T;
    }
    unsigned eq_before = block_excl_scan(eq, warp_tot, &s_total);
    unsigned eq_take = eq_before >= need ? 0u : min(eq, need - eq_before);
    unsigned pos = block_excl_scan(gt + eq_take, warp_tot, &s_total);
    int32_t* out = pool + (size_t)b * K;
    unsigned eq_used = 0;
    for (int v = v0; v < v1; ++v) {
        unsigned k = ord_f32(sc[v]);
        bool take = k > T;
        if (!take && k == T && eq_used < eq_take) {
            take = true;
            ++eq_used;
        }
        if (take && pos < (unsigned)K) out[pos++] = v;
    }
}

// ---------------------------------------------------------------------------
// One bias-free GRU update (gate rows r|z|n): one warp per state element j,
// looping over requests.  u = 0 consumes the verified token with h = 0;
// u >= 1 consumes proposal u-1 (teacher-forced token when `forced` is set).
// The input side W_ih emb[t] is row t of the table built at load time.
template <typename T>
__global__ void __launch_bounds__(256) k_gru(const float* __restrict__ gi_table,
                                             const T* __restrict__ w_hh, const float* __restrict__ h_in,
                                             float* __restrict__ h_out, const int32_t* __restrict__ verified,
                                             const int32_t* __restrict__ forced,
                                             const unsigned long long* __restrict__ keys, int* __restrict__ bad,
                                             int* __restrict__ err, float* __restrict__ dbg_h, int u, int B,
                                             int V, int E, int G) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int j = warp; j < G; j += nwarps) {
        for (int b = 0; b < B; ++b) {
            int t;
            if (u == 0) t = verified[b];
            else if (forced) t = forced[(size_t)b * kProposals + (u - 1)];
            else t = (int)key_index(keys[(size_t)b * kBlock + (u - 1)]);
            if (t < 0 || t >= V) {
                if (j == 0 && lane == 0) {
                    bad[b] = 1;
                    atomicOr(err, kErrBadToken);
                }
                t = 0;
            }
            const float* gi = gi_table + (size_t)t * 3 * G;
            const float gi_r = gi[j], gi_z = gi[G + j], gi_n = gi[2 * G + j];
            float gh_r = 0.f, gh_z = 0.f, gh_n = 0.f, hp = 0.f;
            if (u > 0) {
                const float* hv = h_in + (size_t)b * G;
                gh_r = warp_dot(w_hh + (size_t)j * G, hv, G, lane);
                gh_z = warp_dot(w_hh + (size_t)(G + j) * G, hv, G, lane);
                gh_n = warp_dot(w_hh + (size_t)(2 * G + j) * G, hv, G, lane);
                hp = hv[j];
            }
            if (lane == 0) {
                float r = sigmoidf_(gi_r + gh_r);
                float zg = sigmoidf_(gi_z + gh_z);
                float n = tanhf(gi_n + r * gh_n);
                float hn = (1.f - zg) * n + zg * hp;
                h_out[(size_t)b * G + j] = hn;
                if (dbg_h) dbg_h[((size_t)b * kProposals + u) * G + j] = hn;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Projector layer 1 + SiLU for corrected step k: a = SiLU(fc1 h + s[k]).
template <typename T>
__global__ void __launch_bounds__(256) k_fc1(const T* __restrict__ fc1, const float* __restrict__ h,
                                             const T* __restrict__ s, float* __restrict__ a,
                                             __nv_bfloat16* __restrict__ a16, float* __restrict__ dbg_z, int k,
                                             int B, int G, int F) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    for (int f = warp; f < F; f += nwarps) {
        for (int b = 0; b < B; ++b) {
            float z = warp_dot(fc1 + (size_t)f * G, h + (size_t)b * G, G, lane);
            if (lane == 0) {
                z += to_f32(s[((size_t)b * kProposals + k) * F + f]);
                float act = z * sigmoidf_(z);
                a[(size_t)b * F + f] = act;
                a16[(size_t)b * F + f] = __float2bfloat16_rn(act);
                if (dbg_z) dbg_z[((size_t)b * kCorrected + (k - 1)) * F + f] = z;
            }
        }
    }
}

// ---------------------------------------------------------------------------
// Correction + argmax over the full vocabulary for up to NB requests per
// block row group: c[v] = fc2[v] . a + bias[v] + L[b, k+1, v].
template <typename T, int NB>
__global__ void __launch_bounds__(256) k_correct_full(const T* __restrict__ fc2, const T* __restrict__ bias,
                                                      const float* __restrict__ L, const float* __restrict__ a,
                                                      unsigned long long* __restrict__ keys,
                                                      float* __restrict__ dbg_scores, int k, int B, int V, int F) {
    extern __shared__ float sa[];  // [NB][F]
    __shared__ unsigned long long sbest[NB];
    const int b0 = blockIdx.y * NB;
    const int nb = min(NB, B - b0);
    for (int i = threadIdx.x; i < nb * F; i += blockDim.x) sa[i] = a[(size_t)b0 * F + i];
    if (threadIdx.x < NB) sbest[threadIdx.x] = 0ull;
    __syncthreads();
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    unsigned long long best[NB];
#pragma unroll
    for (int r = 0; r < NB; ++r) best[r] = 0ull;
    for (int v = warp; v < V; v += nwarps) {
        const T* w = fc2 + (size_t)v * F;
        float acc[NB];
#pragma unroll
        for (int r = 0; r < NB; ++r) acc[r] = 0.f;
        if ((F & 7) == 0) {
            for (int i = lane * 8; i < F; i += 256) {
                float e[8];
                load8_stream(w + i, e);
#pragma unroll
                for (int r = 0; r < NB; ++r) {
                    if (r < nb) {
                        const float* x = sa + r * F + i;
#pragma unroll
                        for (int j = 0; j < 8; ++j) acc[r] = fmaf(e[j], x[j], acc[r]);
                    }
                }
            }
        } else {
            for (int i = lane; i < F; i += 32) {
                float e = to_f32(w[i]);
#pragma unroll
                for (int r = 0; r < NB; ++r)
                    if (r < nb) acc[r] = fmaf(e, sa[r * F + i], acc[r]);
            }
        }
        const float bv = to_f32(bias[v]);
#pragma unroll
        for (int r = 0; r < NB; ++r) {
            if (r < nb) {
                float c = warp_sum(acc[r]) + bv + L[((size_t)(b0 + r) * kBlock + kRowOffset + k) * V + v];
                unsigned long long key = pack_key(c, (uint32_t)v);
                best[r] = key > best[r] ? key : best[r];
                if (dbg_scores && lane == 0) dbg_scores[((size_t)(b0 + r) * kCorrected + (k - 1)) * V + v] = c;
            }
        }
    }
    if (lane == 0) {
#pragma unroll
        for (int r = 0; r < NB; ++r)
            if (r < nb && best[r]) atomicMax(&sbest[r], best[r]);
    }
    __syncthreads();
    if (threadIdx.x < nb && sbest[threadIdx.x]) atomicMax(&keys[(size_t)(b0 + threadIdx.x) * kBlock + k], sbest[threadIdx.x]);
}

// Correction + argmax over each request's pool: one warp per pool entry.
template <typename T>
__global__ void __launch_bounds__(256) k_correct_pool(const T* __restrict__ fc2, const T* __restrict__ bias,
                                                      const float* __restrict__ L, const float* __restrict__ a,
                                                      const int32_t* __restrict__ pool,
                                                      unsigned long long* __restrict__ keys,
                                                      float* __restrict__ dbg_scores, int k, int B, int V, int F,
                                                      int K) {
    const int lane = threadIdx.x & 31;
    const int warp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const long long items = (long long)B * K;
    // contiguous item range per warp so that the request rarely changes
    const long long per = (items + nwarps - 1) / nwarps;
    const long long i0 = (long long)warp * per;
    const long long i1 = min(items, i0 + per);
    int cur_b = -1;
    unsigned long long best = 0ull;
    for (long long it = i0; it < i1; ++it) {
        const int b = (int)(it / K);
        const int i = (int)(it % K);
        if (b != cur_b) {
            if (cur_b >= 0 && lane == 0 && best) atomicMax(&keys[(size_t)cur_b * kBlock + k], best);
            cur_b = b;
            best = 0ull;
        }
        const int v = pool[(size_t)b * K + i];
        float c = warp_dot(fc2 + (size_t)v * F, a + (size_t)b * F, F, lane) + to_f32(bias[v]) +
                  L[((size_t)b * kBlock + kRowOffset + k) * V + v];
        unsigned long long key = pack_key(c, (uint32_t)v);
        best = key > best ? key : best;
        if (dbg_scores && lane == 0) dbg_scores[((size_t)b * kCorrected + (k - 1)) * K + i] = c;
    }
    if (cur_b >= 0 && lane == 0 && best) atomicMax(&keys[(size_t)cur_b * kBlock + k], best);
}

// ---------------------------------------------------------------------------
__global__ void k_finalize(const unsigned long long* __restrict__ keys, const int* __restrict__ bad,
                           int32_t* __restrict__ out, float* __restrict__ dbg_top1, int B, int n_prop) {
    pdl_wait();
    int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * kProposals) return;
    int b = i / kProposals, j = i % kProposals;
    unsigned long long key = keys[(size_t)b * kBlock + j];
    const bool used = j < n_prop;
    out[i] = (bad[b] || !used) ? -1 : (int32_t)key_index(key);
    if (dbg_top1) dbg_top1[i] = used ? key_value(key) : 0.f;
}

}  // namespace

// ---------------------------------------------------------------------------
// Per-step term of projector layer 1 from the backbone hidden (page "Add
// correctness-first Domino support to DFlash V2": embed_proj over [backbone
// hidden | GRU state]): s[b, j, f] = W_hid[f, :] . hidden[b, j+1, :], one warp
// per output, stored in the input dtype.
__device__ __forceinline__ void store_as(float* p, float v) { *p = v; }
__device__ __forceinline__ void store_as(__nv_bfloat16* p, float v) { *p = __float2bfloat16_rn(v); }

template <typename T>
__global__ void __launch_bounds__(256) k_backbone_s(const T* __restrict__ hidden, const T* __restrict__ w,
                                                    T* __restrict__ s, int B, int H, int F) {
    const int lane = threadIdx.x & 31;
    const long long total = (long long)B * kProposals * F;
    const long long nwarps = (long long)gridDim.x * (blockDim.x >> 5);
    for (long long wid = (long long)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); wid < total;
         wid += nwarps) {
        const int f = (int)(wid % F);
        const long long bj = wid / F;
        const int b = (int)(bj / kProposals), j = (int)(bj % kProposals);
        const T* x = hidden + ((size_t)b * kBlock + kRowOffset + j) * H;
        const T* wr = w + (size_t)f * H;
        float acc = 0.f;
        for (int h = lane; h < H; h += 32) acc = fmaf(to_f32(x[h]), to_f32(wr[h]), acc);
        acc = warp_sum(acc);
        if (lane == 0) store_as(&s[((size_t)b * kProposals + j) * F + f], acc);
    }
}

// ===========================================================================
// host launchers
#define DOMINO_LAUNCH_CHECK()                      \
    do {                                           \
        ++r.launches;                              \
        cudaError_t e_ = cudaGetLastError();       \
        if (e_ != cudaSuccess) return e_;          \
    } while (0)

cudaError_t launch_reset(domino_ctx* c, RunArgs& r) {
    const int n = r.B * kBlock;
    const int nx = c->xbest ? 2 * c->num_sms * kLLMaxBatch : 0;
    const int nh = c->hist && r.K > 0 ? r.B * kPoolHistBins : 0;
    int m = n > nx ? n : nx;
    m = m > nh ? m : nh;
    ++r.launches;
    return launch_pdl(k_reset, dim3((m + 255) / 256), dim3(256), 0, r.st, c->keys, c->bad, c->sync, c->xbest, c->hist,
                      n, r.B, nx, nh);
}

cudaError_t launch_lmhead_simt(domino_ctx* c, RunArgs& r) {
    const domino_config& g = c->cfg;
    int grid = grid_for(8, g.V, c->num_sms * 8);
    if (g.dtype == DOMINO_DTYPE_FP32)
        k_lmhead_simt<float><<<grid, 256, 0, r.st>>>((const float*)r.hidden, (const float*)c->lm_head, c->L, r.B,
                                                     g.V, g.H);
    else
        k_lmhead_simt<__nv_bfloat16><<<grid, 256, 0, r.st>>>((const __nv_bfloat16*)r.hidden,
                                                             (const __nv_bfloat16*)c->lm_head, c->L, r.B, g.V, g.H);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_backbone_s_simt(domino_ctx* c, RunArgs& r) {
    const domino_config& g = c->cfg;
    const int grid = grid_for(8, r.B * kProposals * g.F, c->num_sms * 8);
    if (g.dtype == DOMINO_DTYPE_FP32)
        k_backbone_s<float><<<grid, 256, 0, r.st>>>((const float*)r.hidden, (const float*)c->fc1_hid,
                                                    (float*)r.s_out, r.B, g.H, g.F);
    else
        k_backbone_s<__nv_bfloat16><<<grid, 256, 0, r.st>>>((const __nv_bfloat16*)r.hidden,
                                                            (const __nv_bfloat16*)c->fc1_hid,
                                                            (__nv_bfloat16*)r.s_out, r.B, g.H, g.F);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_first_argmax(domino_ctx* c, RunArgs& r) {
    int gx = grid_for(256, c->cfg.V, c->num_sms);
    k_first_argmax<<<dim3(gx, r.B), 256, 0, r.st>>>(c->L, c->keys, c->cfg.V);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_score(domino_ctx* c, RunArgs& r) {
    int grid = grid_for(256, r.B * c->cfg.V, c->num_sms * 8);
    k_score<<<grid, 256, 0, r.st>>>(c->L, c->score, r.B, c->cfg.V);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_pool_select(domino_ctx* c, RunArgs& r, bool score_ready) {
    if (!score_ready) {
        cudaError_t e = launch_score(c, r);
        if (e != cudaSuccess) return e;
    }
    // the tensor-core LM-head also histograms the scores' first digit
    if (pool_cluster_supported(c)) return launch_pool_cluster(c, r, score_ready ? c->hist : nullptr);
    k_pool_select<<<r.B, 1024, 0, r.st>>>(c->score, c->pool, c->cfg.V, r.K);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_gru(domino_ctx* c, RunArgs& r, int u) {
    const domino_config& g = c->cfg;
    const float* h_in = c->h + (size_t)h_slot(u + 1) * g.max_B * g.G;  // = slot(u-1)
    float* h_out = c->h + (size_t)h_slot(u) * g.max_B * g.G;
    int grid = grid_for(8, g.G, c->num_sms * 4);
    if (g.dtype == DOMINO_DTYPE_FP32)
        k_gru<float><<<grid, 256, 0, r.st>>>(c->gi_table, (const float*)c->w_hh, h_in, h_out, r.verified, r.forced,
                                             c->keys, c->bad, c->err, r.dbg.h, u, r.B, g.V, g.E, g.G);
    else
        k_gru<__nv_bfloat16><<<grid, 256, 0, r.st>>>(c->gi_table, (const __nv_bfloat16*)c->w_hh, h_in, h_out,
                                                     r.verified, r.forced, c->keys, c->bad, c->err, r.dbg.h, u, r.B,
                                                     g.V, g.E, g.G);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_fc1(domino_ctx* c, RunArgs& r, int k) {
    const domino_config& g = c->cfg;
    const float* h = c->h + (size_t)h_slot(k) * g.max_B * g.G;
    int grid = grid_for(8, g.F, c->num_sms * 4);
    if (g.dtype == DOMINO_DTYPE_FP32)
        k_fc1<float><<<grid, 256, 0, r.st>>>((const float*)c->fc1, h, (const float*)r.s, c->a, c->a16, r.dbg.z, k,
                                             r.B, g.G, g.F);
    else
        k_fc1<__nv_bfloat16><<<grid, 256, 0, r.st>>>((const __nv_bfloat16*)c->fc1, h, (const __nv_bfloat16*)r.s,
                                                     c->a, c->a16, r.dbg.z, k, r.B, g.G, g.F);
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

template <typename T>
static cudaError_t correct_simt_t(domino_ctx* c, RunArgs& r, int k) {
    const domino_config& g = c->cfg;
    if (r.K == 0) {
        constexpr int NB = 8;
        int gy = (r.B + NB - 1) / NB;
        size_t smem = (size_t)NB * g.F * sizeof(float);
        int gx = grid_for(8, g.V, c->num_sms * 4);
        k_correct_full<T, NB><<<dim3(gx, gy), 256, smem, r.st>>>((const T*)c->fc2, (const T*)c->bias, c->L, c->a,
                                                                 c->keys, r.dbg.scores, k, r.B, g.V, g.F);
    } else {
        int grid = grid_for(8, r.B * r.K, c->num_sms * 4);
        k_correct_pool<T><<<grid, 256, 0, r.st>>>((const T*)c->fc2, (const T*)c->bias, c->L, c->a, c->pool, c->keys,
                                                  r.dbg.scores, k, r.B, g.V, g.F, r.K);
    }
    DOMINO_LAUNCH_CHECK();
    return cudaSuccess;
}

cudaError_t launch_correct_simt(domino_ctx* c, RunArgs& r, int k) {
    return c->cfg.dtype == DOMINO_DTYPE_FP32 ? correct_simt_t<float>(c, r, k) : correct_simt_t<__nv_bfloat16>(c, r, k);
}

cudaError_t launch_finalize(domino_ctx* c, RunArgs& r) {
    int n = r.B * kProposals;
    ++r.launches;
    return launch_pdl(k_finalize, dim3((n + 255) / 256), dim3(256), 0, r.st, (const unsigned long long*)c->keys,
                      (const int*)c->bad, r.out_tokens, r.dbg.top1, r.B, r.n_prop);
}

// The full-vocabulary correction kernel needs NB*F*4 bytes of dynamic shared
// memory; raise the opt-in limit once per context.
cudaError_t prepare_simt_kernels(domino_ctx* c) {
    size_t smem = (size_t)8 * c->cfg.F * sizeof(float);
    cudaError_t e = cudaFuncSetAttribute(k_correct_full<float, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(k_correct_full<__nv_bfloat16, 8>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)smem);
}

}  // namespace domino
