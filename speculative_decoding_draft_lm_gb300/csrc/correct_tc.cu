// Correction + argmax of one corrected step over the full vocabulary on the
// tensor cores, for batches of independent requests:
//   c[b, v] = fc2[v, :] . a[b, :] + bias[v] + L[b, k+1, v],
//   p_{k+1}[b] = argmax_v c[b, v]   (lowest id on ties).
// fc2 is streamed once per step as the MMA's A operand (128 vocabulary rows
// per tile); the bf16 activations a[b, :] of all requests form the N side.
//
// Method: page "[Spec] Add Domino projector support to DFlash speculative
// decoding (V2)", section "Implementation" (fused SiLU(z+s) @ fc2^T + bias +
// base_logits full-vocabulary argmax) and page "Add correctness-first Domino
// support to DFlash V2", section "Design" (full-vocabulary correction, K=0).
// The activations are rounded to bf16 for the MMA; accumulation is fp32.
//
// Pool mode at large B*K (page "Add correctness-first Domino support to
// DFlash V2", section "Design": block-shared top-K candidate pool): when the
// pools of the batch together cover a large part of the vocabulary, gathering
// B*K fc2 rows costs about as much as streaming fc2 once, so the same dense
// contraction runs and the argmax only admits each request's pool members
// (a [B, V/32] bit mask built from the pool).  The result is the pool argmax.
#include "gemm_tc.cuh"
#include "internal.h"

namespace domino {

namespace {

struct EpiCorrect {
    static constexpr int kScratchWords = tc::kEpiScratch;
    // A chunks beyond the first ring warmed into L2 before the dependent-launch
    // wait: fc2 streams while the GRU and projector kernels before it run
    // (24 chunks of 16 KB per CTA: 58 MB over 152 CTAs, about a fifth of fc2)
    static constexpr int kL2Ahead = 24;
    static constexpr int kPfChunk = 17;  // prefetch registers per 16-column chunk
    // fc2 is walked in reverse on even steps, and the last 4/10 of each walk
    // is loaded at normal L2 priority, so a step starts on the rows the step
    // before left in L2 (B=8 K0: 1067 -> 1051 us per block)
    static constexpr int kKeepTenths = 4;
    const __nv_bfloat16* bias;  // [V]
    const float* L;             // [B,16,V]
    unsigned long long* keys;   // [B,16]
    float* dbg_scores;          // [B,14,V] or null (never with a mask)
    const uint32_t* mask;       // [B, mask_words] pool membership bits, or null = full vocabulary
    int V, B, k, mask_words;
    bool rev;  // reversed walk over the fc2 tiles
    __device__ __forceinline__ void begin(unsigned long long* sb, int t) const {
        for (int i = t; i < tc::kEpiScratch; i += tc::kEpiThreads) sb[i] = 0ull;
    }
    __device__ __forceinline__ void end(unsigned long long* sb, int t) const {
        const int n = B < tc::kEpiScratch ? B : tc::kEpiScratch;
        for (int b = t; b < n; b += tc::kEpiThreads)
            if (sb[b]) atomicMax(&keys[(size_t)b * kBlock + k], sb[b]);
    }
    // per 16-column chunk: the base logits of its requests for this thread's
    // row, and (lane j < 16) the pool-membership word of request j for the
    // warp's 32 rows, kept as raw bits
    template <int PF>
    __device__ __forceinline__ void prefetch(int col0, int row, float* pf) const {
        const bool ok = row < V;
#pragma unroll
        for (int cc = 0; cc < PF / kPfChunk; ++cc) {
            float* p = pf + cc * kPfChunk;
            const int c0 = col0 + 16 * cc;
#pragma unroll
            for (int j = 0; j < 16; ++j)
                p[j] = (ok && c0 + j < B) ? __ldg(&L[((size_t)(c0 + j) * kBlock + kRowOffset + k) * V + row]) : 0.f;
            p[16] = __uint_as_float(mask_word(c0, row));
        }
    }
    // lane j < 16: membership bits of request col0 + j for the warp's rows
    // (row & ~31) .. +31; the word exists while the warp's first row is below
    // V, even when this lane's own row is past it
    __device__ __forceinline__ uint32_t mask_word(int col0, int row) const {
        const int j = row & 31;
        return (mask && j < 16 && col0 + j < B && (row >> 5) < mask_words)
                   ? __ldg(&mask[(size_t)(col0 + j) * mask_words + (row >> 5)])
                   : 0u;
    }
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int lane,
                                               unsigned long long* sb, const float* pf) const {
        if (col0 >= B) return;  // uniform: padding columns
        const bool ok = row < V;
        const int nb = B - col0 < 16 ? B - col0 : 16;
        float base[16];
        if (pf) {
#pragma unroll
            for (int j = 0; j < 16; ++j) base[j] = pf[j];
        } else {  // beyond the prefetch window: all loads of the chunk in flight at once
#pragma unroll
            for (int j = 0; j < 16; ++j)
                base[j] = (ok && j < nb) ? __ldg(&L[((size_t)(col0 + j) * kBlock + kRowOffset + k) * V + row]) : 0.f;
        }
        const float bv = ok ? __bfloat162float(bias[row]) : 0.f;
        uint32_t member = 0xffffu;  // bit j: column j may take this row
        if (mask) {  // uniform: every lane takes part in the shuffles
            const uint32_t w = pf ? __float_as_uint(pf[16]) : mask_word(col0, row);
            member = 0u;
#pragma unroll
            for (int j = 0; j < 16; ++j) member |= ((__shfl_sync(0xffffffffu, w, j) >> (row & 31)) & 1u) << j;
        }
        unsigned long long kk[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
            kk[j] = 0ull;
            if (ok && j < nb && ((member >> j) & 1u)) {
                const float c = v[j] + bv + base[j];
                kk[j] = pack_key(c, (uint32_t)row);
                if (dbg_scores) dbg_scores[((size_t)(col0 + j) * kCorrected + (k - 1)) * V + row] = c;
            }
        }
        // the 32 rows' best per request, one request per lane pair
        const unsigned long long key = warp_max16_u64(kk, lane);
        const int j = warp_max16_slot(lane);
        if ((lane & 1) == 0 && j < nb && key) {
            const int b = col0 + j;
            if (b < tc::kEpiScratch) atomicMax(&sb[b], key);
            else atomicMax(&keys[(size_t)b * kBlock + k], key);
        }
    }
};

template <int BN>
cudaError_t launch_bn(domino_ctx* c, RunArgs& r, const CUtensorMap& tmB, int k) {
    using S = tc::GemmShape<BN, EpiCorrect::kScratchWords>;
    static bool attr_set[64] = {};
    auto kern = tc::k_gemm_tc<BN, EpiCorrect>;
    const int slot = c->device & 63;
    if (!attr_set[slot]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[slot] = true;
    }
    const int tiles = ((c->cfg.V + tc::kBM - 1) / tc::kBM) * ((r.B + BN - 1) / BN);
    const int grid = tiles < c->num_sms ? tiles : c->num_sms;
    const bool pool = r.K > 0;
    EpiCorrect epi{(const __nv_bfloat16*)c->bias, c->L, c->keys, pool ? nullptr : r.dbg.scores,
                   pool ? c->pmask : nullptr, c->cfg.V, r.B, k, pool_mask_words(c->cfg.V), (k & 1) == 0};
    ++r.launches;
    return launch_pdl(kern, dim3(grid), dim3(tc::kGemmThreads), S::SMEM, r.st, c->tm_fc2, c->tm_fc2, tmB, c->cfg.V,
                      INT_MAX, r.B, c->cfg.F, epi, c->err);
}

}  // namespace

int correct_bn(int B) { return B <= 16 ? 16 : B <= 32 ? 32 : B <= 64 ? 64 : B <= 128 ? 128 : 256; }

int pool_mask_words(int V) { return (V + 31) / 32; }

bool correct_tc_supported(const domino_ctx* c, const RunArgs& r) {
    if (!c->has_tma || c->cfg.dtype != DOMINO_DTYPE_BF16 || r.B > c->a_rows) return false;
    if (r.K == 0) return true;
    // pools covering at least half a vocabulary's worth of rows between them;
    // score dumps keep the gathering path (they are indexed by pool position)
    return c->pmask != nullptr && 2LL * r.B * r.K >= (long long)c->cfg.V && r.dbg.scores == nullptr;
}

namespace {

__global__ void __launch_bounds__(256) k_pool_mask(const int32_t* __restrict__ pool, uint32_t* __restrict__ mask,
                                                   int K, int words) {
    pdl_trigger();
    pdl_wait();
    const int b = blockIdx.x;
    uint32_t* m = mask + (size_t)b * words;
    for (int i = threadIdx.x; i < words; i += blockDim.x) m[i] = 0u;
    __syncthreads();
    const int32_t* p = pool + (size_t)b * K;
    for (int i = threadIdx.x; i < K; i += blockDim.x) {
        const int v = p[i];
        atomicOr(&m[v >> 5], 1u << (v & 31));
    }
}

}  // namespace

cudaError_t launch_pool_mask(domino_ctx* c, RunArgs& r) {
    ++r.launches;
    return launch_pdl(k_pool_mask, dim3(r.B), dim3(256), 0, r.st, (const int32_t*)c->pool, c->pmask, r.K,
                      pool_mask_words(c->cfg.V));
}

cudaError_t prepare_correct_tc(domino_ctx* c, RunArgs& r, CUtensorMap* tmB) {
    return make_tmap_bf16(tmB, c->a16, (uint64_t)c->a_rows, (uint64_t)c->cfg.F, (uint32_t)correct_bn(r.B));
}

cudaError_t launch_correct_tc(domino_ctx* c, RunArgs& r, const CUtensorMap& tmB, int k) {
    switch (correct_bn(r.B)) {
        case 16: return launch_bn<16>(c, r, tmB, k);
        case 32: return launch_bn<32>(c, r, tmB, k);
        case 64: return launch_bn<64>(c, r, tmB, k);
        case 128: return launch_bn<128>(c, r, tmB, k);
        default: return launch_bn<256>(c, r, tmB, k);
    }
}

}  // namespace domino
