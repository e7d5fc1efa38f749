// One launch per corrected step for small batches (2 <= B <= 8, bf16): the
// GRU update fed by the step's token and projector layer 1 on the new state,
// fused (page "[Spec] Add Domino projector support to DFlash speculative
// decoding (V2)", section "Implementation": the fused GRU cell and the fused
// projector; page "Add correctness-first Domino support to DFlash V2",
// section "Design": bias-free GRU in the ATen GRUCell form, gate rows r|z|n).
//
// Launch u (update u >= 1, corrected step k = u):
//   h_u[b] = GRU(T[p_u(b)], W_hh h_{u-1}[b], h_{u-1}[b])          (every cluster)
//   a_k[b, f] = SiLU(fc1[f] . h_u[b] + s[b, k, f])                (fc1 rows)
//   W_hh h_u[b]  for the next launch's update                     (W_hh rows)
// The hidden-side products W_hh h_{u-1} come from the previous launch, so
// an update is element-wise: one cluster of 8 CTAs splits the G units among
// its CTAs, each CTA computes its eighth for every request from the
// token-table row T[p_u] (input side, built at load time), the products and
// h_{u-1}, and the CTAs then copy each other's eighths through distributed
// shared memory, so every CTA holds the whole state after one cluster
// barrier.  Launch 0 (after the seed update) has no update and no fc1 rows:
// it forms W_hh h_0 from the seed state.
//
// The rows: each CTA owns a contiguous range of the items [fc1 rows; W_hh
// rows], staged in shared memory (padded row stride, for ldmatrix without
// bank conflicts) before the kernel waits for the previous one.  Products on
// the tensor cores: 16-row tiles, mma m16n8k16 with one column per request;
// the fp32 state enters as bf16 leading parts and remainders (two products
// per k-step, |error| <= 2^-16 |w h| before the fp32 accumulation); the 16
// warps take (tile, k-range) units and their partial tiles are summed
// through shared memory.
#include <cooperative_groups.h>

#include "internal.h"
#include "persist_util.cuh"

namespace cg = cooperative_groups;

namespace domino {

using namespace persist;

namespace {

constexpr int kSThreads = 512;
constexpr int kSWarps = kSThreads / 32;
constexpr int kSCluster = 8;   // CTAs that share one update
constexpr int kSCols = 8;      // requests: one mma column tile
constexpr int kSPad = 8;       // elements after each staged row and each state row

struct StepParams {
    const __nv_bfloat16 *w_hh, *fc1, *s;
    const float* gi_table;     // [V, 3G]
    const float* h_prev;       // [B, G]  h_{u-1}, or (u = 0) the state to project
    const float* gh_prev;      // [B, 3G] W_hh h_{u-1} (u >= 1)
    float* h_out;              // [B, G]  h_u (u >= 1), written by cluster 0
    float* gh_out;             // [B, 3G] W_hh h_u, or null
    float* a;                  // [B, F]
    __nv_bfloat16* a16;        // [a_rows, F]
    float *dbg_h, *dbg_z;
    const unsigned long long* keys;
    const int32_t* forced;
    int *bad, *err;
    int B, V, G, F;
    int u;    // update index (1..14), or 0: project the given state
    int ipc;  // items per CTA
};

__host__ __device__ inline int step_rows_bytes(int ipc, int G) { return ((ipc * (G + kSPad) * 2) + 127) & ~127; }
__host__ __device__ inline int step_state_bytes(int G) { return kSCols * (G + kSPad) * 4; }
__host__ __device__ inline int step_part_bytes(int ipc) {
    const int mt = (ipc + 15) / 16;
    return 128 * 4 * (mt > kSWarps ? mt : kSWarps);
}

__global__ void __launch_bounds__(kSThreads, 1) k_step_fused(StepParams p) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ int stok[kSCols];
    cg::cluster_group cluster = cg::this_cluster();
    const int G = p.G, F = p.F, B = p.B, RS = G + kSPad;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int nF = p.u > 0 ? F : 0;
    const int n_items = nF + (p.gh_out ? 3 * G : 0);
    const int it0 = min(n_items, (int)blockIdx.x * p.ipc), nit = min(n_items, it0 + p.ipc) - it0;
    __nv_bfloat16* sw = reinterpret_cast<__nv_bfloat16*>(sm);
    float* sh = reinterpret_cast<float*>(sm + step_rows_bytes(p.ipc, G));  // [kSCols][RS]
    float* spart = sh + kSCols * RS;

    pdl_trigger();
    // the rows do not depend on the previous kernel: stage them first
    {
        const int per_row = G / 8;
        for (int i = tid; i < nit * per_row; i += kSThreads) {
            const int rr = i / per_row, e = (i % per_row) * 8, it = it0 + rr;
            const __nv_bfloat16* src = it < nF ? p.fc1 + (size_t)it * G : p.w_hh + (size_t)(it - nF) * G;
            cp_async16(sw + (size_t)rr * RS + e, src + e);
        }
        cp_async_commit();
        for (int i = tid; i < nit + kSCols; i += kSThreads) {
            if (i < nit) {
                *reinterpret_cast<uint4*>(sw + (size_t)i * RS + G) = make_uint4(0u, 0u, 0u, 0u);
            } else {
                float4* z = reinterpret_cast<float4*>(sh + (size_t)(i - nit) * RS + G);
                z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    pdl_wait();

    if (p.u == 0) {
        // the given state, whole, in every CTA
        for (int b = 0; b < B; ++b)
            for (int j = tid * 4; j < G; j += kSThreads * 4)
                *reinterpret_cast<float4*>(sh + (size_t)b * RS + j) =
                    *reinterpret_cast<const float4*>(p.h_prev + (size_t)b * G + j);
    } else {
        // the token fed to update u, validated (an invalid one flags the request)
        if (tid < B) {
            int t = p.forced ? p.forced[(size_t)tid * kProposals + (p.u - 1)]
                             : (int)key_index(p.keys[(size_t)tid * kBlock + (p.u - 1)]);
            if (t < 0 || t >= p.V) {
                if (blockIdx.x == 0) {
                    p.bad[tid] = 1;
                    atomicOr(p.err, kErrBadToken);
                }
                t = 0;
            }
            stok[tid] = t;
        }
        __syncthreads();
        // this CTA's eighth of the units, for every request
        const int rank = (int)cluster.block_rank();
        const int per = (G / 8 + kSCluster - 1) / kSCluster * 8;  // units per rank, a multiple of 8
        const int ju0 = min(G, rank * per), ju1 = min(G, ju0 + per);
        const bool writer = blockIdx.x < kSCluster;  // the first cluster stores h_u
        for (int i = tid; i < B * (ju1 - ju0); i += kSThreads) {
            const int b = i / (ju1 - ju0), j = ju0 + i % (ju1 - ju0);
            const float* gi = p.gi_table + (size_t)stok[b] * 3 * G + j;
            const float* gh = p.gh_prev + (size_t)b * 3 * G + j;
            const float r = sigmoidf_(__ldg(gi) + gh[0]);
            const float zg = sigmoidf_(__ldg(gi + G) + gh[G]);
            const float n = tanhf(__ldg(gi + 2 * G) + r * gh[2 * G]);
            const float h = (1.f - zg) * n + zg * p.h_prev[(size_t)b * G + j];
            sh[(size_t)b * RS + j] = h;
            if (writer) {
                p.h_out[(size_t)b * G + j] = h;
                if (p.dbg_h) p.dbg_h[((size_t)b * kProposals + p.u) * G + j] = h;
            }
        }
        cluster.sync();  // every CTA's eighth is complete
        // the other CTAs' eighths, 16 bytes at a time
        for (int q = 1; q < kSCluster; ++q) {
            const int src = (rank + q) % kSCluster;
            const int q0 = min(G, src * per), q1 = min(G, q0 + per), nq = (q1 - q0) / 4;
            const float* rsh = cluster.map_shared_rank(sh, src);
            for (int i = tid; i < B * nq; i += kSThreads) {
                const int b = i / nq, j = q0 + (i % nq) * 4;
                *reinterpret_cast<float4*>(sh + (size_t)b * RS + j) =
                    *reinterpret_cast<const float4*>(rsh + (size_t)b * RS + j);
            }
        }
        cluster.sync();  // no CTA reads another's shared memory after this
    }
    cp_async_wait_all();
    __syncthreads();

    // ---- the CTA's items against the state: (tile, k-range) units
    if (nit > 0) {
        const int mt = (nit + 15) / 16;
        const int nkr = mt >= kSWarps ? 1 : kSWarps / mt;
        const int ks = (G + 15) / 16;
        const int mi = lane >> 3, rl = (lane & 7) + (mi & 1) * 8, kofs = (mi >> 1) * 8;
        const float* xrow = sh + (size_t)min(lane >> 2, B - 1) * RS + (lane & 3) * 2;
        for (int un = warp; un < mt * nkr; un += kSWarps) {
            const int m = un / nkr, r = un % nkr;
            const int rr = min(m * 16 + rl, nit - 1);  // rows past the items repeat the last one
            const uint32_t abase = tc::smem_u32(sw + (size_t)rr * RS + kofs);
            const int kq1 = (r + 1) * ks / nkr;
            float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kq = r * ks / nkr; kq < kq1; ++kq) {
                uint32_t a[4];
                ldmatrix_x4(abase + (uint32_t)kq * 32u, a);
                const float2 x01 = *reinterpret_cast<const float2*>(xrow + kq * 16);
                const float2 x23 = *reinterpret_cast<const float2*>(xrow + kq * 16 + 8);
                uint32_t h0, l0, h1, l1;
                split_bf16x2(x01.x, x01.y, h0, l0);
                split_bf16x2(x23.x, x23.y, h1, l1);
                mma_16816(d0, a, h0, h1);
                mma_16816(d1, a, l0, l1);
            }
            float* pt = spart + (size_t)un * 128;
            const int row = lane >> 2, col = (lane & 3) * 2;
            *reinterpret_cast<float2*>(pt + row * 8 + col) = make_float2(d0[0] + d1[0], d0[1] + d1[1]);
            *reinterpret_cast<float2*>(pt + (row + 8) * 8 + col) = make_float2(d0[2] + d1[2], d0[3] + d1[3]);
        }
        __syncthreads();
        for (int o = tid; o < mt * 128; o += kSThreads) {
            const int m = o >> 7, row = (o >> 3) & 15, b = o & 7, rr = m * 16 + row;
            if (rr < nit && b < B) {
                const float* pt = spart + (size_t)m * nkr * 128 + row * 8 + b;
                float v = 0.f;
                for (int r = 0; r < nkr; ++r) v += pt[r * 128];
                const int it = it0 + rr;
                if (it < nF) {
                    const int k = p.u;  // corrected step fed by update u
                    const float z = v + __bfloat162float(p.s[((size_t)b * kProposals + k) * F + it]);
                    const float act = z * sigmoidf_(z);
                    p.a[(size_t)b * F + it] = act;
                    p.a16[(size_t)b * F + it] = __float2bfloat16_rn(act);
                    if (p.dbg_z) p.dbg_z[((size_t)b * kCorrected + (k - 1)) * F + it] = z;
                } else {
                    p.gh_out[(size_t)b * 3 * G + (it - nF)] = v;
                }
            }
        }
    }
}

size_t step_smem_for(const domino_ctx* c, int grid) {
    const int ipc = (c->cfg.F + 3 * c->cfg.G + grid - 1) / grid;
    return (size_t)step_rows_bytes(ipc, c->cfg.G) + step_state_bytes(c->cfg.G) + step_part_bytes(ipc);
}

// Few CTAs: the SMs they leave free take the correction kernel that follows
// early (programmatic dependent launch), which then warms its first fc2 tiles
// while the step runs (B=8 K0: 1097 us per block on 152 CTAs of 8-CTA
// clusters, 1067 on 64, 1064 on 48).  Enough CTAs that the rows of one fit
// its shared memory; 0 if none does.
int step_grid(const domino_ctx* c) {
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    for (int n = 64; n <= c->num_sms / kSCluster * kSCluster; n += kSCluster)
        if (step_smem_for(c, n) + 1024 <= (size_t)max_smem) return n;
    return 0;
}

}  // namespace

bool step_fused_supported(const domino_ctx* c, const RunArgs& r) {
    const domino_config& g = c->cfg;
    if (g.dtype != DOMINO_DTYPE_BF16 || !c->ghb) return false;
    return r.B >= 2 && r.B <= kSCols && (g.G & 7) == 0 && (g.F & 7) == 0 && step_grid(c) >= kSCluster;
}

// Launch u: u = 0 forms W_hh h_0 from the seed state; u >= 1 updates to h_u
// with the token of update u and projects it (corrected step k = u), and
// forms W_hh h_u unless u is the last update.
cudaError_t launch_step_fused(domino_ctx* c, RunArgs& r, int u) {
    const domino_config& g = c->cfg;
    const int n_corr = r.n_prop - 1;
    StepParams p;
    p.w_hh = (const __nv_bfloat16*)c->w_hh;
    p.fc1 = (const __nv_bfloat16*)c->fc1;
    p.s = (const __nv_bfloat16*)r.s;
    p.gi_table = c->gi_table;
    p.h_prev = c->h + (size_t)h_slot(u == 0 ? 0 : u - 1) * g.max_B * g.G;
    p.gh_prev = u == 0 ? nullptr : c->ghb + (size_t)((u - 1) & 1) * g.max_B * 3 * g.G;
    p.h_out = u == 0 ? nullptr : c->h + (size_t)h_slot(u) * g.max_B * g.G;
    p.gh_out = u < n_corr ? c->ghb + (size_t)(u & 1) * g.max_B * 3 * g.G : nullptr;
    p.a = c->a;
    p.a16 = c->a16;
    p.dbg_h = r.dbg.h;
    p.dbg_z = r.dbg.z;
    p.keys = c->keys;
    p.forced = r.forced;
    p.bad = c->bad;
    p.err = c->err;
    p.B = r.B;
    p.V = g.V;
    p.G = g.G;
    p.F = g.F;
    p.u = u;
    const int grid = step_grid(c);
    p.ipc = ((u > 0 ? g.F : 0) + (p.gh_out ? 3 * g.G : 0) + grid - 1) / grid;
    const size_t smem = step_smem_for(c, grid);  // sized for the largest launch
    cudaError_t e = cudaFuncSetAttribute(k_step_fused, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kSThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = r.st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSCluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    ++r.launches;
    return cudaLaunchKernelEx(&cfg, k_step_fused, p);
}

}  // namespace domino
