// GRU update and projector layer 1 on the tensor cores, for batches of
// independent requests (B >= 12, bf16 weights).
//
// GRU (page "Add correctness-first Domino support to DFlash V2", section
// "Design": bias-free prefix GRU in the ATen GRUCell form, gate rows r|z|n):
//   r = sigmoid(W_ir x + W_hr h), z = sigmoid(W_iz x + W_hz h),
//   n = tanh(W_in x + r * (W_hn h)), h' = (1 - z) * n + z * h.
// The input side W_i* x is a row of the token table built at load time; the
// hidden side is one contraction of a packed copy of W_hh with the bf16 state:
//   Wp row 4j + q = { W_hr[j], W_hz[j], W_hn[j], 0 }[q]
// for hidden unit j, so the three gates of a unit land in adjacent TMEM
// lanes of one epilogue warp, which finish the update with warp shuffles (no
// block-level exchange).  Units G..Gp-1 and the fourth row of every unit are
// zero.  Update u = 0 (h = 0) needs no contraction and runs on the CUDA cores.
//
// Projector layer 1 (page "[Spec] Add Domino projector support to DFlash
// speculative decoding (V2)", section "Implementation": SiLU(z + s)):
//   a[b, f] = SiLU(fc1[f, :] . h[b, :] + s[b, k, f]),
// with fc1 as the A operand and the bf16 state as the B operand.
//
// Operand rounding: the state enters both contractions as bf16; accumulation
// and the element-wise parts are fp32, and the fp32 state is what the update
// carries forward.  Buffers: H16[2] = [a_rows, G] bf16; update u writes
// H16[u & 1], which update u+1 and projector step k = u read.
#include "gemm_tc.cuh"
#include "internal.h"

namespace domino {

namespace {

// Wp row 4j + q for hidden unit j and gate q (q = 3: zero row).
__global__ void k_pack_gru(const __nv_bfloat16* __restrict__ w_hh, __nv_bfloat16* __restrict__ wp, int G, int Gp) {
    const size_t n = (size_t)4 * Gp * G;
    const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int prow = (int)(i / G), col = (int)(i % G);
        const int q = prow & 3, j = prow >> 2;
        wp[i] = (j < G && q < 3) ? w_hh[(size_t)(q * G + j) * G + col] : zero;
    }
}

struct EpiGru {
    static constexpr int kScratchWords = 1;
    static constexpr int kL2Ahead = 0;
    static constexpr int kPfChunk = 16;  // prefetch registers per 16-column chunk
    const float* gi_table;      // [V, 3G]
    const float* h_in;          // [B,G] state before the update
    float* h_out;               // [B,G]
    __nv_bfloat16* h16_out;     // [rows, G] bf16 copy of the new state
    const unsigned long long* keys;
    const int32_t* forced;      // nullable [B,15]
    int* bad;
    int* err;
    float* dbg_h;               // [B,15,G] or null
    int B, G, V, u;
    __device__ __forceinline__ void begin(unsigned long long*, int) const {}
    __device__ __forceinline__ void end(unsigned long long*, int) const {}
    // the token fed to this update, validated (an invalid one flags the request)
    __device__ __forceinline__ int token(int b) const {
        int t = forced ? forced[(size_t)b * kProposals + (u - 1)] : (int)key_index(keys[(size_t)b * kBlock + (u - 1)]);
        if (t < 0 || t >= V) {
            bad[b] = 1;
            atomicOr(err, kErrBadToken);
            t = 0;
        }
        return t;
    }
    // inputs of one output (b, j): previous state, then the three input-side
    // pre-activations of the request's token
    __device__ __forceinline__ void inputs(int b, int j, float* o) const {
        const float* gi = gi_table + (size_t)token(b) * 3 * G + j;
        o[0] = __ldg(&h_in[(size_t)b * G + j]);
        o[1] = __ldg(gi);
        o[2] = __ldg(gi + G);
        o[3] = __ldg(gi + 2 * G);
    }
    // accumulator row 4j + q; the lane of gate q finishes columns q, q+4, q+8,
    // q+12 of every 16-column chunk for unit j: prefetch their inputs
    template <int PF>
    __device__ __forceinline__ void prefetch(int col0, int row, float* pf) const {
        const int q = row & 3, j = row >> 2;
#pragma unroll
        for (int cc = 0; cc < PF / 16; ++cc)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int b = col0 + cc * 16 + q + 4 * i;
                if (b < B && j < G) inputs(b, j, pf + cc * 16 + 4 * i);
            }
    }
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int lane,
                                               unsigned long long*, const float* pf) const {
        if (col0 >= B) return;  // uniform over the warp
        const int q = row & 3, j = row >> 2;
        const int grp = lane & ~3;
        // g[gate][i]: hidden-side pre-activation `gate` of column q + 4i, from lane grp + gate
        float g[3][4];
#pragma unroll
        for (int c = 0; c < 16; ++c)
#pragma unroll
            for (int gate = 0; gate < 3; ++gate) {
                const float t = __shfl_sync(0xffffffffu, v[c], grp | gate);
                if ((c & 3) == q) g[gate][c >> 2] = t;
            }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = col0 + q + 4 * i;
            if (b < B && j < G) {
                float in[4];
                if (pf) {
#pragma unroll
                    for (int x = 0; x < 4; ++x) in[x] = pf[4 * i + x];
                } else {
                    inputs(b, j, in);
                }
                const float r = sigmoidf_(in[1] + g[0][i]), z = sigmoidf_(in[2] + g[1][i]);
                const float n = tanhf(in[3] + r * g[2][i]);
                const float out = (1.f - z) * n + z * in[0];
                h_out[(size_t)b * G + j] = out;
                h16_out[(size_t)b * G + j] = __float2bfloat16_rn(out);
                if (dbg_h) dbg_h[((size_t)b * kProposals + u) * G + j] = out;
            }
        }
    }
};

struct EpiFc1 {
    static constexpr int kScratchWords = 1;
    static constexpr int kL2Ahead = 0;
    static constexpr int kPfChunk = 16;  // prefetch registers per 16-column chunk
    const __nv_bfloat16* s;     // [B,15,F]
    float* a;                   // [B,F]
    __nv_bfloat16* a16;         // [a_rows,F]
    float* dbg_z;               // [B,14,F] or null
    int B, F, k;
    __device__ __forceinline__ void begin(unsigned long long*, int) const {}
    __device__ __forceinline__ void end(unsigned long long*, int) const {}
    template <int PF>
    __device__ __forceinline__ void prefetch(int col0, int row, float* pf) const {
#pragma unroll
        for (int c = 0; c < PF; ++c) {
            const int b = col0 + c;
            pf[c] = (b < B && row < F) ? __bfloat162float(s[((size_t)b * kProposals + k) * F + row]) : 0.f;
        }
    }
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int,
                                               unsigned long long*, const float* pf) const {
        if (row >= F) return;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int b = col0 + c;
            if (b < B) {
                const float sv = pf ? pf[c] : __bfloat162float(s[((size_t)b * kProposals + k) * F + row]);
                const float z = v[c] + sv;
                const float act = z * sigmoidf_(z);
                a[(size_t)b * F + row] = act;
                a16[(size_t)b * F + row] = __float2bfloat16_rn(act);
                if (dbg_z) dbg_z[((size_t)b * kCorrected + (k - 1)) * F + row] = z;
            }
        }
    }
};

// Projector layer 1 of step k and the hidden-side GRU products for update
// k+1 in one contraction of the same state h_k: A = [fc1 (rows 0..F-1, the
// tile rows past F zero-filled); Wp (packed W_hh rows 4j+q, from row fr
// on)], B = the bf16 state.  The fc1 rows finish as in EpiFc1; the packed
// rows are stored raw: W_hh h_k does not depend on the token the correction
// of step k picks, so only an element-wise update is left after it.
struct EpiProj {
    static constexpr int kScratchWords = 1;
    static constexpr int kL2Ahead = 0;
    static constexpr int kPfChunk = 16;
    EpiFc1 fc1;    // rows < fr (k >= 1)
    float* ghp;    // [B, 4Gp] products of the packed rows
    int fr, gp4;   // first packed row (a multiple of 128); 4Gp
    __device__ __forceinline__ void begin(unsigned long long*, int) const {}
    __device__ __forceinline__ void end(unsigned long long*, int) const {}
    template <int PF>
    __device__ __forceinline__ void prefetch(int col0, int row, float* pf) const {
        if (row < fr) fc1.template prefetch<PF>(col0, row, pf);
    }
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int lane, unsigned long long* sb,
                                               const float* pf) const {
        if (row < fr) {  // uniform over the warp: fr is a multiple of 128
            fc1(col0, row, v, lane, sb, pf);
            return;
        }
        const int pr = row - fr;
        if (pr >= gp4) return;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
            const int b = col0 + c;
            if (b < fc1.B) ghp[(size_t)b * gp4 + pr] = v[c];
        }
    }
};

// The update u >= 1 of every unit after the correction that picked its
// token: h = GRU(T[p_u], W_hh h_{u-1}, h_{u-1}) from the token-table row,
// the packed products of the projector launch and the previous state.
__global__ void __launch_bounds__(256) k_gru_update(const float* __restrict__ gi_table, const float* __restrict__ ghp,
                                                    const float* __restrict__ h_in, float* __restrict__ h_out,
                                                    __nv_bfloat16* __restrict__ h16_out,
                                                    const unsigned long long* __restrict__ keys,
                                                    const int32_t* __restrict__ forced, int* __restrict__ bad,
                                                    int* __restrict__ err, float* __restrict__ dbg_h, int u, int B,
                                                    int G, int gp4, int V) {
    pdl_trigger();
    pdl_wait();
    const int i = blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= B * G) return;
    const int b = i / G, j = i - b * G;
    int t = forced ? forced[(size_t)b * kProposals + (u - 1)] : (int)key_index(keys[(size_t)b * kBlock + (u - 1)]);
    if (t < 0 || t >= V) {
        if (j == 0) {
            bad[b] = 1;
            atomicOr(err, kErrBadToken);
        }
        t = 0;
    }
    const float* gi = gi_table + (size_t)t * 3 * G + j;
    const float4 gh = *reinterpret_cast<const float4*>(ghp + (size_t)b * gp4 + 4 * j);  // r, z, n, 0
    const float r = sigmoidf_(__ldg(gi) + gh.x);
    const float z = sigmoidf_(__ldg(gi + G) + gh.y);
    const float n = tanhf(__ldg(gi + 2 * G) + r * gh.z);
    const float h = (1.f - z) * n + z * h_in[(size_t)b * G + j];
    h_out[(size_t)b * G + j] = h;
    h16_out[(size_t)b * G + j] = __float2bfloat16_rn(h);
    if (dbg_h) dbg_h[((size_t)b * kProposals + u) * G + j] = h;
}

template <int BN, class Epi>
cudaError_t launch_gemm(domino_ctx* c, RunArgs& r, const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int K,
                        const Epi& epi) {
    using S = tc::GemmShape<BN, Epi::kScratchWords>;
    static bool attr_set[64] = {};
    auto kern = tc::k_gemm_tc<BN, Epi>;
    const int slot = c->device & 63;
    if (!attr_set[slot]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[slot] = true;
    }
    const int tiles = ((M + tc::kBM - 1) / tc::kBM) * ((r.B + BN - 1) / BN);
    const int grid = tiles < c->num_sms ? tiles : c->num_sms;
    ++r.launches;
    return launch_pdl(kern, dim3(grid), dim3(tc::kGemmThreads), S::SMEM, r.st, tmA, tmA, tmB, M, INT_MAX, r.B, K, epi,
                      c->err);
}

// two A matrices: tiles m < m_split from tmA, the rest from tmA2
template <int BN, class Epi>
cudaError_t launch_gemm2(domino_ctx* c, RunArgs& r, const CUtensorMap& tmA, const CUtensorMap& tmA2,
                         const CUtensorMap& tmB, int M, int m_split, int K, const Epi& epi) {
    using S = tc::GemmShape<BN, Epi::kScratchWords>;
    static bool attr_set[64] = {};
    auto kern = tc::k_gemm_tc<BN, Epi>;
    const int slot = c->device & 63;
    if (!attr_set[slot]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[slot] = true;
    }
    const int tiles = ((M + tc::kBM - 1) / tc::kBM) * ((r.B + BN - 1) / BN);
    const int grid = tiles < c->num_sms ? tiles : c->num_sms;
    ++r.launches;
    return launch_pdl(kern, dim3(grid), dim3(tc::kGemmThreads), S::SMEM, r.st, tmA, tmA2, tmB, M, m_split, r.B, K,
                      epi, c->err);
}

// 16 requests per tile for both contractions: their A matrices are small
// (W_hh 8 MB, fc1 2 MB), so a batch spreads over ceil(B/16) times as many
// CTAs, each with a short epilogue, and re-reads A from L2.
constexpr int kGruBN = 16;

template <class Epi>
cudaError_t launch_any_bn(domino_ctx* c, RunArgs& r, const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int K,
                          const Epi& epi) {
    return launch_gemm<kGruBN>(c, r, tmA, tmB, M, K, epi);
}

}  // namespace

int gru_padded_units(int G) { return (G + 31) / 32 * 32; }

bool gru_tc_shape_ok(const domino_config& g) {
    // 16-byte TMA row strides of the state copies and of fc1
    return g.dtype == DOMINO_DTYPE_BF16 && g.G % 8 == 0;
}

// Below this batch the CUDA-core batched kernels win: the contraction's few
// CTAs (one per 32 hidden units) stream the weights slower than the whole GPU.
constexpr int kGruTcMinBatch = 12;

bool gru_tc_supported(const domino_ctx* c, const RunArgs& r) {
    return c->has_tma && c->wp != nullptr && gru_tc_shape_ok(c->cfg) && r.B >= kGruTcMinBatch &&
           r.B <= c->a_rows;
}

cudaError_t pack_gru_weights(domino_ctx* c, cudaStream_t st) {
    const domino_config& g = c->cfg;
    const int Gp = gru_padded_units(g.G);
    k_pack_gru<<<4 * c->num_sms, 256, 0, st>>>((const __nv_bfloat16*)c->w_hh, c->wp, g.G, Gp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return make_tmap_bf16(&c->tm_wp, c->wp, (uint64_t)4 * Gp, (uint64_t)g.G, (uint32_t)tc::kBM);
}

cudaError_t prepare_gru_tc(domino_ctx* c, RunArgs& r, GruMaps* m) {
    const domino_config& g = c->cfg;
    const uint32_t bn = (uint32_t)kGruBN;  // box rows = the contractions' N tile
    for (int i = 0; i < 2; ++i) {
        cudaError_t e = make_tmap_bf16(&m->h[i], c->h16 + (size_t)i * c->a_rows * g.G, (uint64_t)c->a_rows,
                                       (uint64_t)g.G, bn);
        if (e != cudaSuccess) return e;
        e = make_tmap_bf16(&m->h32[i], c->h16 + (size_t)i * c->a_rows * g.G, (uint64_t)c->a_rows, (uint64_t)g.G,
                           32u);
        if (e != cudaSuccess) return e;
    }
    return make_tmap_bf16(&m->fc1, c->fc1, (uint64_t)g.F, (uint64_t)g.G, (uint32_t)tc::kBM);
}

cudaError_t launch_gru_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int u) {
    const domino_config& g = c->cfg;
    __nv_bfloat16* h16_out = c->h16 + (size_t)(u & 1) * c->a_rows * g.G;
    if (u == 0) return launch_gru_batch(c, r, 0, h16_out);  // h = 0: the token table alone
    const float* h_in = c->h + (size_t)h_slot(u - 1) * g.max_B * g.G;
    float* h_out = c->h + (size_t)h_slot(u) * g.max_B * g.G;
    EpiGru epi{c->gi_table, h_in, h_out, h16_out, (const unsigned long long*)c->keys, r.forced, c->bad, c->err,
               r.dbg.h, r.B, g.G, g.V, u};
    return launch_any_bn(c, r, c->tm_wp, m.h[(u - 1) & 1], 4 * gru_padded_units(g.G), g.G, epi);
}

// Launch k of the joined projector: k >= 1 projects h_k (fc1 rows), and
// unless k is the last step (or k = 0, the seed state alone) also forms the
// packed products W_hh h_k into GHP[k & 1] for update k+1.
cudaError_t launch_proj_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int k) {
    const domino_config& g = c->cfg;
    const int n_corr = r.n_prop - 1;
    const int gp4 = 4 * gru_padded_units(g.G);
    const bool gh = k < n_corr || k == 0;
    const int fr = k > 0 ? (g.F + tc::kBM - 1) / tc::kBM * tc::kBM : 0;
    EpiProj epi{EpiFc1{(const __nv_bfloat16*)r.s, c->a, c->a16, r.dbg.z, r.B, g.F, k},
                c->ghb + (size_t)(k & 1) * g.max_B * gp4, fr, gh ? gp4 : 0};
    const int M = fr + (gh ? gp4 : 0);
    const int m_split = fr / tc::kBM;
    // 16 requests per tile while the tiles fit one wave, else 32
    const int tiles16 = ((M + tc::kBM - 1) / tc::kBM) * ((r.B + 15) / 16);
    if (tiles16 <= c->num_sms)
        return launch_gemm2<16>(c, r, m.fc1, c->tm_wp, m.h[k & 1], M, m_split, g.G, epi);
    return launch_gemm2<32>(c, r, m.fc1, c->tm_wp, m.h32[k & 1], M, m_split, g.G, epi);
}

// Update u >= 1 after the correction of step u - 1 (token p_u): the packed
// products come from projector launch u - 1.
cudaError_t launch_update_tc(domino_ctx* c, RunArgs& r, int u) {
    const domino_config& g = c->cfg;
    const int gp4 = 4 * gru_padded_units(g.G);
    const float* ghp = c->ghb + (size_t)((u - 1) & 1) * g.max_B * gp4;
    const float* h_in = c->h + (size_t)h_slot(u - 1) * g.max_B * g.G;
    float* h_out = c->h + (size_t)h_slot(u) * g.max_B * g.G;
    __nv_bfloat16* h16_out = c->h16 + (size_t)(u & 1) * c->a_rows * g.G;
    const int n = r.B * g.G;
    ++r.launches;
    return launch_pdl(k_gru_update, dim3((n + 255) / 256), dim3(256), 0, r.st, (const float*)c->gi_table, ghp, h_in,
                      h_out, h16_out, (const unsigned long long*)c->keys, r.forced, c->bad, c->err, r.dbg.h, u, r.B,
                      g.G, gp4, g.V);
}

cudaError_t launch_fc1_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int k) {
    const domino_config& g = c->cfg;
    // the state after update k sits in H16[k & 1]
    EpiFc1 epi{(const __nv_bfloat16*)r.s, c->a, c->a16, r.dbg.z, r.B, g.F, k};
    return launch_any_bn(c, r, m.fc1, m.h[k & 1], g.F, g.G, epi);
}

}  // namespace domino
