// Input-side GRU pre-activations of every vocabulary token, built once when
// the weights are loaded:
//   T[v, g*G + j] = sum_e emb[v, e] * w_ih[g*G + j, e],   g = r|z|n,
// so that each GRU update reads one 3G-vector per request instead of
// contracting w_ih with the embedding row (page "Add correctness-first Domino
// support to DFlash V2", section "Design": the bias-free GRU consumes the
// embedding of the realised token; W_ih x depends on the token alone).  The
// table is fp32 (the same fp32 accumulation the contraction would give) and
// takes V * 3G * 4 bytes of device memory (1.9 GB at V = 151,936, G = 1024):
// memory traded for the per-step weight traffic and latency of W_ih x.
//
// bf16 weights: one tcgen05 contraction (A = emb [V, E], B = w_ih [3G, E]);
// fp32 weights: a CUDA-core kernel.
#include "gemm_tc.cuh"
#include "internal.h"

namespace domino {

namespace {

struct EpiTable {
    static constexpr int kScratchWords = 1;
    static constexpr int kL2Ahead = 0;
    static constexpr int kPfChunk = 16;  // prefetch registers per 16-column chunk
    float* T;  // [V, N]
    int V, N;
    __device__ __forceinline__ void begin(unsigned long long*, int) const {}
    __device__ __forceinline__ void end(unsigned long long*, int) const {}
    template <int PF>
    __device__ __forceinline__ void prefetch(int, int, float*) const {}
    __device__ __forceinline__ void operator()(int col0, int row, const float* v, int, unsigned long long*,
                                               const float*) const {
        if (row >= V || col0 >= N) return;
        float* dst = T + (size_t)row * N + col0;
        if (col0 + 16 <= N) {  // N % 8 == 0 and col0 % 16 == 0: 16-byte aligned
#pragma unroll
            for (int q = 0; q < 4; ++q)
                reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int j = 0; j < 16; ++j)
                if (col0 + j < N) dst[j] = v[j];
        }
    }
};

template <typename T>
__global__ void __launch_bounds__(256) k_gi_table(const T* __restrict__ emb, const T* __restrict__ w_ih,
                                                  float* __restrict__ table, int V, int E, int N) {
    const size_t n = (size_t)V * N;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const int v = (int)(i / N), c = (int)(i % N);
        const T* x = emb + (size_t)v * E;
        const T* w = w_ih + (size_t)c * E;
        float acc = 0.f;
        for (int e = 0; e < E; ++e) acc = fmaf(to_f32(x[e]), to_f32(w[e]), acc);
        table[i] = acc;
    }
}

}  // namespace

cudaError_t build_gi_table(domino_ctx* c, cudaStream_t st) {
    const domino_config& g = c->cfg;
    const int N = 3 * g.G;
    if (c->has_tma && g.dtype == DOMINO_DTYPE_BF16) {
        constexpr int BN = 256;
        using S = tc::GemmShape<BN, EpiTable::kScratchWords>;
        auto kern = tc::k_gemm_tc<BN, EpiTable>;
        cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)S::SMEM);
        if (e != cudaSuccess) return e;
        CUtensorMap tm_emb, tm_wih;
        e = make_tmap_bf16(&tm_emb, c->emb, (uint64_t)g.V, (uint64_t)g.E, (uint32_t)tc::kBM);
        if (e != cudaSuccess) return e;
        e = make_tmap_bf16(&tm_wih, c->w_ih, (uint64_t)N, (uint64_t)g.E, (uint32_t)BN);
        if (e != cudaSuccess) return e;
        const int tiles = ((g.V + tc::kBM - 1) / tc::kBM) * ((N + BN - 1) / BN);
        const int grid = tiles < c->num_sms ? tiles : c->num_sms;
        EpiTable epi{c->gi_table, g.V, N};
        kern<<<grid, tc::kGemmThreads, S::SMEM, st>>>(tm_emb, tm_emb, tm_wih, g.V, INT_MAX, N, g.E, epi, c->err);
        return cudaGetLastError();
    }
    const int grid = 8 * c->num_sms;
    if (g.dtype == DOMINO_DTYPE_FP32)
        k_gi_table<float><<<grid, 256, 0, st>>>((const float*)c->emb, (const float*)c->w_ih, c->gi_table, g.V, g.E,
                                                N);
    else
        k_gi_table<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16*)c->emb,
                                                        (const __nv_bfloat16*)c->w_ih, c->gi_table, g.V, g.E, N);
    return cudaGetLastError();
}

}  // namespace domino
