// Allocation-free candidate pool: the pool selection with its score scratch
// in a file-scope device array instead of a context workspace, for callers
// that may not allocate device memory at call time.
#include <mutex>

#include "internal.h"

namespace domino {

namespace {

// Scratch for the per-request scores: DOMINO_STATIC_SCRATCH_FLOATS floats on
// every device that loads the library, alive until the process exits.
__device__ __align__(256) float g_pool_scratch[DOMINO_STATIC_SCRATCH_FLOATS];

constexpr int kMaxDevices = 64;
float* g_scratch_addr[kMaxDevices];  // device address of g_pool_scratch, per device
std::mutex g_scratch_mu;

// score[b, v] = max over the 15 base rows the proposals use (rows 1..15)
__global__ void k_score_static(const float* __restrict__ L, float* __restrict__ score, int B, int V) {
    const size_t n = (size_t)B * V;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (size_t)gridDim.x * blockDim.x) {
        const size_t b = i / V, v = i % V;
        const float* p = L + (b * kBlock + kRowOffset) * V + v;
        float m = p[0];
#pragma unroll
        for (int j = 1; j < kProposals; ++j) m = fmaxf(m, p[(size_t)j * V]);
        score[i] = m;
    }
}

// Device address of the scratch on the current device; looked up once per
// device (host code cannot use the symbol itself as a device pointer).
cudaError_t scratch_on_current_device(float** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (!g_scratch_addr[dev]) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_pool_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_addr[dev] = static_cast<float*>(p);
    }
    *out = g_scratch_addr[dev];
    return cudaSuccess;
}

}  // namespace

}  // namespace domino

extern "C" int domino_candidate_pool_static(const float* base_logits, int B, int V, int K, int32_t* pool_out,
                                            void* cuda_stream) {
    using namespace domino;
    if (!base_logits || !pool_out || B < 1 || V < 2 || K <= 0 || K >= V) return DOMINO_ERR_INVALID_ARG;
    if (!pool_cluster_fits(V)) return DOMINO_ERR_INVALID_ARG;
    if ((unsigned long long)B * (unsigned long long)V > (unsigned long long)DOMINO_STATIC_SCRATCH_FLOATS)
        return DOMINO_ERR_SCRATCH_LIMIT;
    float* score = nullptr;
    if (scratch_on_current_device(&score) != cudaSuccess) return DOMINO_ERR_CUDA;
    const cudaStream_t st = (cudaStream_t)cuda_stream;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return DOMINO_ERR_CUDA;
    const size_t n = (size_t)B * V;
    int grid = (int)((n + 255) / 256);
    if (grid > sms * 8) grid = sms * 8;
    k_score_static<<<grid, 256, 0, st>>>(base_logits, score, B, V);
    if (cudaGetLastError() != cudaSuccess) return DOMINO_ERR_CUDA;
    if (launch_pool_cluster_raw(score, pool_out, B, V, K, st) != cudaSuccess) return DOMINO_ERR_CUDA;
    return DOMINO_OK;
}
