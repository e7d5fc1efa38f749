// GRU update and projector layer 1 on the tensor cores, for batches of
// independent requests (B >= 12, bf16 weights).
//
// GRU (page "Add correctness-first Domino support to DFlash V2", section
// "Design": bias-free prefix GRU in the ATen GRUCell form, gate rows r|z|n):
//   r = sigmoid(W_ir x + W_hr h), z = sigmoid(W_iz x + W_hz h),
//   n = tanh(W_in x + r * (W_hn h)), h' = (1 - z) * n + z * h.
// The four pre-activations that the update needs (r and z summed over both
// inputs, the two halves of n kept apart) are one contraction of a packed
// weight matrix Wp [4*Gp, E+G] with the concatenated operand [x | h]:
//   Wp row 4j + q = { [W_ir | W_hr], [W_iz | W_hz], [W_in | 0], [0 | W_hn] }[q]
// for hidden unit j, so the four gates of a unit land in four adjacent TMEM
// lanes, i.e. four adjacent lanes of one epilogue warp, which finish the
// update with warp shuffles (no block-level exchange).  Wp is built once from
// w_ih / w_hh when the weights are loaded; units G..Gp-1 are zero rows.
//
// Projector layer 1 (page "[Spec] Add Domino projector support to DFlash
// speculative decoding (V2)", section "Implementation": SiLU(z + s)):
//   a[b, f] = SiLU(fc1[f, :] . h[b, :] + s[b, k, f]),
// with fc1 as the A operand and the bf16 state as the B operand.
//
// Operand rounding: the state h enters both contractions as bf16 (x is the
// bf16 embedding row itself); accumulation and the element-wise parts are
// fp32, and the fp32 state is what the update carries forward.
//
// Buffers: X[2] = [a_rows, E+G] bf16 operand rows [emb[token] | bf16(h)].
// Update u reads X[u & 1] and writes its new state into the h part of
// X[(u + 1) & 1], which projector step k = u reads; the embedding part of
// X[u & 1] is gathered by k_gru_x right before update u.
#include "gemm_tc.cuh"
#include "internal.h"

namespace domino {

namespace {

// Embedding rows of the tokens fed to GRU update u into the operand buffer:
// u = 0 the verified token (and h = 0), u >= 1 proposal u-1 (or forced[:,u-1]).
__global__ void __launch_bounds__(128) k_gru_x(const __nv_bfloat16* __restrict__ emb, __nv_bfloat16* __restrict__ x,
                                               const int32_t* __restrict__ verified,
                                               const int32_t* __restrict__ forced,
                                               const unsigned long long* __restrict__ keys, int* __restrict__ bad,
                                               int* __restrict__ err, int u, int V, int E, int G) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    int t;
    if (u == 0) t = verified[b];
    else if (forced) t = forced[(size_t)b * kProposals + (u - 1)];
    else t = (int)key_index(keys[(size_t)b * kBlock + (u - 1)]);
    if (t < 0 || t >= V) {
        if (threadIdx.x == 0) {
            bad[b] = 1;
            atomicOr(err, kErrBadToken);
        }
        t = 0;
    }
    const int ld = E + G;
    const uint4* src = reinterpret_cast<const uint4*>(emb + (size_t)t * E);
    uint4* dst = reinterpret_cast<uint4*>(x + (size_t)b * ld);
    for (int i = threadIdx.x; i < E / 8; i += blockDim.x) dst[i] = __ldg(src + i);
    if (u == 0) {
        uint4* hz = reinterpret_cast<uint4*>(x + (size_t)b * ld + E);
        for (int i = threadIdx.x; i < G / 8; i += blockDim.x) hz[i] = make_uint4(0u, 0u, 0u, 0u);
    }
}

// Wp row 4j + q for hidden unit j and gate block q.
__global__ void k_pack_gru(const __nv_bfloat16* __restrict__ w_ih, const __nv_bfloat16* __restrict__ w_hh,
                           __nv_bfloat16* __restrict__ wp, int E, int G, int Gp) {
    const int ld = E + G;
    const size_t n = (size_t)4 * Gp * ld;
    const __nv_bfloat16 zero = __float2bfloat16_rn(0.f);
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int prow = (int)(i / ld), col = (int)(i % ld);
        const int q = prow & 3, j = prow >> 2;
        __nv_bfloat16 v = zero;
        if (j < G) {
            const bool xin = col < E;
            if (q < 2 || (q == 2 && xin)) {
                v = xin ? w_ih[(size_t)(q * G + j) * E + col] : w_hh[(size_t)(q * G + j) * G + (col - E)];
            } else if (q == 3 && !xin) {
                v = w_hh[(size_t)(2 * G + j) * G + (col - E)];
            }
        }
        wp[i] = v;
    }
}

struct EpiGru {
    static constexpr int kScratchWords = 1;
    const float* h_in;          // [B,G] state before the update, null for u = 0
    float* h_out;               // [B,G]
    __nv_bfloat16* x_next;      // operand rows of the next update; the state goes at column E
    float* dbg_h;               // [B,15,G] or null
    int B, E, G, u;
    __device__ __forceinline__ void begin(unsigned long long*, int) const {}
    __device__ __forceinline__ void end(unsigned long long*, int) const {}
    // accumulator row 4j + q; the lane of gate q finishes columns q, q+4, q+8,
    // q+12 of every 16-column chunk for unit j: prefetch their previous state
    template <int PF>
    __device__ __forceinline__ void prefetch(int col0, int row, float* pf) const {
        const int q = row & 3, j = row >> 2;
#pragma unroll
        for (int cc = 0; cc < PF / 16; ++cc)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int b = col0 + cc * 16 + q + 4 * i;
                pf[cc * 16 + i] = (h_in && b < B && j < G) ? __ldg(&h_in[(size_t)b * G + j]) : 0.f;
            }
    }
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int lane,
                                               unsigned long long*, const float* pf) const {
        if (col0 >= B) return;  // uniform over the warp
        const int q = row & 3, j = row >> 2;
        const int grp = lane & ~3;
        // g[gate][i]: pre-activation `gate` of column q + 4i, from lane grp + gate
        float g[4][4];
#pragma unroll
        for (int c = 0; c < 16; ++c)
#pragma unroll
            for (int gate = 0; gate < 4; ++gate) {
                const float t = __shfl_sync(0xffffffffu, v[c], grp | gate);
                if ((c & 3) == q) g[gate][c >> 2] = t;
            }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int b = col0 + q + 4 * i;
            if (b < B && j < G) {
                const float r = sigmoidf_(g[0][i]), z = sigmoidf_(g[1][i]);
                const float n = tanhf(g[2][i] + r * g[3][i]);
                const float hp = pf ? pf[i] : (h_in ? h_in[(size_t)b * G + j] : 0.f);
                const float out = (1.f - z) * n + z * hp;
                h_out[(size_t)b * G + j] = out;
                x_next[(size_t)b * (E + G) + E + j] = __float2bfloat16_rn(out);
                if (dbg_h) dbg_h[((size_t)b * kProposals + u) * G + j] = out;
            }
        }
    }
};

struct EpiFc1 {
    static constexpr int kScratchWords = 1;
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

template <class Epi>
cudaError_t launch_any_bn(domino_ctx* c, RunArgs& r, const CUtensorMap& tmA, const CUtensorMap& tmB, int M, int K,
                          const Epi& epi) {
    switch (correct_bn(r.B)) {
        case 16: return launch_gemm<16>(c, r, tmA, tmB, M, K, epi);
        case 32: return launch_gemm<32>(c, r, tmA, tmB, M, K, epi);
        case 64: return launch_gemm<64>(c, r, tmA, tmB, M, K, epi);
        case 128: return launch_gemm<128>(c, r, tmA, tmB, M, K, epi);
        default: return launch_gemm<256>(c, r, tmA, tmB, M, K, epi);
    }
}

}  // namespace

int gru_padded_units(int G) { return (G + 31) / 32 * 32; }

bool gru_tc_shape_ok(const domino_config& g) {
    // 16-byte TMA strides and a 16-byte aligned state column inside X
    return g.dtype == DOMINO_DTYPE_BF16 && g.E % 8 == 0 && g.G % 8 == 0;
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
    k_pack_gru<<<4 * c->num_sms, 256, 0, st>>>((const __nv_bfloat16*)c->w_ih, (const __nv_bfloat16*)c->w_hh, c->wp,
                                                g.E, g.G, Gp);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return make_tmap_bf16(&c->tm_wp, c->wp, (uint64_t)4 * Gp, (uint64_t)(g.E + g.G), (uint32_t)tc::kBM);
}

cudaError_t prepare_gru_tc(domino_ctx* c, RunArgs& r, GruMaps* m) {
    const domino_config& g = c->cfg;
    const uint32_t bn = (uint32_t)correct_bn(r.B);
    for (int i = 0; i < 2; ++i) {
        const __nv_bfloat16* xb = c->xh16 + (size_t)i * c->a_rows * (g.E + g.G);
        cudaError_t e = make_tmap_bf16(&m->x[i], xb, (uint64_t)c->a_rows, (uint64_t)(g.E + g.G), bn);
        if (e != cudaSuccess) return e;
        // the state columns of X[i] alone: row stride E+G, first column E
        e = make_tmap_bf16_strided(&m->h[i], xb + g.E, (uint64_t)c->a_rows, (uint64_t)g.G, (uint64_t)(g.E + g.G),
                                   bn);
        if (e != cudaSuccess) return e;
    }
    return make_tmap_bf16(&m->fc1, c->fc1, (uint64_t)g.F, (uint64_t)g.G, (uint32_t)tc::kBM);
}

cudaError_t launch_gru_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int u) {
    const domino_config& g = c->cfg;
    const int ld = g.E + g.G;
    __nv_bfloat16* x_cur = c->xh16 + (size_t)(u & 1) * c->a_rows * ld;
    __nv_bfloat16* x_next = c->xh16 + (size_t)((u + 1) & 1) * c->a_rows * ld;
    ++r.launches;
    cudaError_t e = launch_pdl(k_gru_x, dim3(r.B), dim3(128), 0, r.st, (const __nv_bfloat16*)c->emb, x_cur,
                               r.verified, r.forced, (const unsigned long long*)c->keys, c->bad, c->err, u, g.V, g.E,
                               g.G);
    if (e != cudaSuccess) return e;
    const float* h_in = u > 0 ? c->h + (size_t)h_slot(u - 1) * g.max_B * g.G : nullptr;
    float* h_out = c->h + (size_t)h_slot(u) * g.max_B * g.G;
    EpiGru epi{h_in, h_out, x_next, r.dbg.h, r.B, g.E, g.G, u};
    return launch_any_bn(c, r, c->tm_wp, m.x[u & 1], 4 * gru_padded_units(g.G), ld, epi);
}

cudaError_t launch_fc1_tc(domino_ctx* c, RunArgs& r, const GruMaps& m, int k) {
    const domino_config& g = c->cfg;
    // the state after update k sits in X[(k + 1) & 1]
    EpiFc1 epi{(const __nv_bfloat16*)r.s, c->a, c->a16, r.dbg.z, r.B, g.F, k};
    return launch_any_bn(c, r, m.fc1, m.h[(k + 1) & 1], g.F, g.G, epi);
}

}  // namespace domino
