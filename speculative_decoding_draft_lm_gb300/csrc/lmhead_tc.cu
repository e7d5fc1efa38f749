// Base LM-head on the tensor cores (bf16 in, fp32 accumulate):
//   L[b, i, v] = sum_h hidden[b, i, h] * lm_head[v, h]   for all 16 block rows,
// with the first-proposal argmax (row 1) and, in pool mode, the per-request
// pool score max_{i=1..15} L[b, i, v] fused into the epilogue, so the logits
// are written to HBM once and never re-read for those two reductions.
//
// Method: page "support tensor-parallel Domino rollout", section "Rollout
// performance" (step-major base LM-head) and page "Add correctness-first
// Domino support to DFlash V2", section "Design" (full-vocabulary base
// projection, first proposal = its argmax, block-shared pool).
//
// Orientation: vocabulary rows are the MMA's M (128 per tile, A = lm_head,
// streamed once), the B*16 draft rows are N (B operand, L2-resident).
//
// When the per-step term s of projector layer 1 is computed in the library,
// its weight W_hid [F, H] (the backbone-hidden half of that layer, page "Add
// correctness-first Domino support to DFlash V2": embed_proj acts on
// [backbone hidden | GRU state]) rides along as extra A rows after the
// vocabulary, sharing the hidden-state operand:
//   s[b, j, f] = sum_h hidden[b, j+1, h] * W_hid[f, h],  j = 0..14,
// stored in the input dtype (bf16).
#include "gemm_tc.cuh"
#include "internal.h"

#include <cudaTypedefs.h>

namespace domino {

namespace {

struct EpiLmHead {
    static constexpr int kScratchWords = tc::kEpiScratch;
    static constexpr int kL2Ahead = 0;
    static constexpr int kPfChunk = 16;  // prefetch registers per 16-column chunk
    float* L;                  // [B,16,V]
    unsigned long long* keys;  // [B,16], slot 0 = p_1
    float* score;              // [B,V] or null
    unsigned* hist;            // [B, kPoolHistBins] counts of the scores' top key bits, or null
    __nv_bfloat16* s_out;      // [B,15,F] or null: rows from s_row0 on are W_hid rows
    int V, B, s_row0, F;
    __device__ __forceinline__ void begin(unsigned long long* sb, int t) const {
        for (int i = t; i < tc::kEpiScratch; i += tc::kEpiThreads) sb[i] = 0ull;
    }
    __device__ __forceinline__ void end(unsigned long long* sb, int t) const {
        const int n = B < tc::kEpiScratch ? B : tc::kEpiScratch;
        for (int b = t; b < n; b += tc::kEpiThreads)
            if (sb[b]) atomicMax(&keys[(size_t)b * kBlock], sb[b]);
    }
    template <int PF>
    __device__ __forceinline__ void prefetch(int, int, float*) const {}
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int lane,
                                               unsigned long long* sb, const float*) const {
        const int b = col0 >> 4;  // 16 columns = the 16 block rows of request b
        if (b >= B) return;       // uniform across the warp
        if (row >= s_row0) {      // uniform: s_row0 is a multiple of 128
            const int f = row - s_row0;
            if (f < F) {
#pragma unroll
                for (int i = kRowOffset; i < kRowOffset + kProposals; ++i)
                    s_out[((size_t)b * kProposals + (i - kRowOffset)) * F + f] = __float2bfloat16_rn(v[i]);
            }
            return;
        }
        const bool ok = row < V;
        float m = 0.f;  // the score: max over the 15 used rows
        if (ok) {
            float* dst = L + (size_t)b * kBlock * V + row;
#pragma unroll
            for (int i = 0; i < kBlock; ++i) dst[(size_t)i * V] = v[i];
            if (score) {
                m = v[kRowOffset];
#pragma unroll
                for (int i = kRowOffset + 1; i < kRowOffset + kProposals; ++i) m = fmaxf(m, v[i]);
                score[(size_t)b * V + row] = m;
            }
        }
        if (hist) {  // set only with score
            // the pool select's first radix pass: warp-aggregated counts of the
            // top key bits (lanes with equal digits add once)
            const unsigned okm = __ballot_sync(0xffffffffu, ok);
            if (ok) {
                const unsigned d = ord_f32(m) >> (32 - kPoolHistBits);
                const unsigned peers = __match_any_sync(okm, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&hist[(size_t)b * kPoolHistBins + d], (unsigned)__popc(peers));
            }
        }
        unsigned long long key = ok ? pack_key(v[kRowOffset], (uint32_t)row) : 0ull;
        key = warp_max_u64(key);
        if (lane == 0 && key) {
            if (b < tc::kEpiScratch) atomicMax(&sb[b], key);
            else atomicMax(&keys[(size_t)b * kBlock], key);
        }
    }
};

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }
    return fn;
}

template <int BN>
cudaError_t launch_bn(domino_ctx* c, RunArgs& r, const CUtensorMap& tmB, float* score) {
    using S = tc::GemmShape<BN, EpiLmHead::kScratchWords>;
    static bool attr_set[64] = {};
    auto kern = tc::k_gemm_tc<BN, EpiLmHead>;
    const int slot = c->device & 63;
    if (!attr_set[slot]) {
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
        attr_set[slot] = true;
    }
    const int N = r.B * kBlock;
    const int v_tiles = (c->cfg.V + tc::kBM - 1) / tc::kBM;
    const bool with_s = r.s_out != nullptr;
    const int m_tiles = v_tiles + (with_s ? (c->cfg.F + tc::kBM - 1) / tc::kBM : 0);
    const int tiles = m_tiles * ((N + BN - 1) / BN);
    const int grid = tiles < c->num_sms ? tiles : c->num_sms;
    const int s_row0 = with_s ? v_tiles * tc::kBM : INT_MAX;
    EpiLmHead epi{c->L, c->keys, score, score ? c->hist : nullptr, (__nv_bfloat16*)r.s_out, c->cfg.V, r.B, s_row0,
                  c->cfg.F};
    ++r.launches;
    const int M = with_s ? s_row0 + c->cfg.F : c->cfg.V;
    return launch_pdl(kern, dim3(grid), dim3(tc::kGemmThreads), S::SMEM, r.st, c->tm_lm_head,
                      with_s ? c->tm_fc1h : c->tm_lm_head, tmB, M, with_s ? v_tiles : INT_MAX, N, c->cfg.H, epi,
                      c->err);
}

}  // namespace

// 2-D bf16 tensor map over a row-major [rows, cols] matrix whose rows are
// `ld` elements apart, box {64, box_rows}, 128-byte swizzle, zero fill
// outside the matrix.
cudaError_t make_tmap_bf16_strided(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint64_t ld,
                                   uint32_t box_rows) {
    PFN_cuTensorMapEncodeTiled_v12000 enc = get_encode();
    if (!enc) return cudaErrorNotSupported;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {ld * 2};
    cuuint32_t box[2] = {(cuuint32_t)tc::kBK, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult res = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
                       CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                       CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return res == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t make_tmap_bf16(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
    return make_tmap_bf16_strided(m, base, rows, cols, cols, box_rows);
}

bool lmhead_tc_supported(const domino_ctx* c) { return c->has_tma && c->cfg.dtype == DOMINO_DTYPE_BF16; }

int lmhead_bn(int B) {
    const int N = B * kBlock;
    return N <= 16 ? 16 : N <= 32 ? 32 : N <= 64 ? 64 : N <= 128 ? 128 : 256;
}

cudaError_t launch_lmhead_tc(domino_ctx* c, RunArgs& r) {
    const int BN = lmhead_bn(r.B);
    CUtensorMap tmB;
    cudaError_t e = make_tmap_bf16(&tmB, r.hidden, (uint64_t)r.B * kBlock, (uint64_t)c->cfg.H, (uint32_t)BN);
    if (e != cudaSuccess) return e;
    float* score = r.K > 0 ? c->score : nullptr;
    switch (BN) {
        case 16: return launch_bn<16>(c, r, tmB, score);
        case 32: return launch_bn<32>(c, r, tmB, score);
        case 64: return launch_bn<64>(c, r, tmB, score);
        case 128: return launch_bn<128>(c, r, tmB, score);
        default: return launch_bn<256>(c, r, tmB, score);
    }
}

}  // namespace domino
