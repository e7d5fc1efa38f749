// Batched GRU update and projector layer 1 for several requests at once
// (the per-phase driver with B >= 2).
//
// GRU (page "Add correctness-first Domino support to DFlash V2", section
// "Design": bias-free GRU; gate rows r|z|n, PyTorch GRUCell algebra):
//   r = sigmoid(W_ir x + W_hr h), u = sigmoid(W_iz x + W_hz h),
//   n = tanh(W_in x + r * (W_hn h)), h' = (1 - u) * n + u * h.
// Projector layer 1 (page "[Spec] Add Domino projector support to DFlash
// speculative decoding (V2)", section "Implementation"): a = SiLU(fc1 h + s).
//
// Layout: a CTA owns JT consecutive state elements j (3 gate rows of W_hh),
// staged once in shared memory; each warp takes requests in turn, holds the
// request's state in registers (lane l owns elements (l + 32c)*8 .. +7) and
// forms the 3*JT hidden-side dot products from them.  The input side W_ih x
// is row x of the table of every token's input pre-activations.
#include "internal.h"

namespace domino {

namespace {

constexpr int kJT = 4;        // GRU state elements per CTA
constexpr int kFT = 8;        // projector outputs per CTA
constexpr int kBatchThreads = 256;

template <typename T, int NCH>
struct VecRegs {
    float v[NCH][8];
    __device__ __forceinline__ void load_f(const float* p, int n, int lane) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int e = (lane + 32 * c) * 8;
            if (e < n) {
                const float4 x = *reinterpret_cast<const float4*>(p + e);
                const float4 y = *reinterpret_cast<const float4*>(p + e + 4);
                v[c][0] = x.x; v[c][1] = x.y; v[c][2] = x.z; v[c][3] = x.w;
                v[c][4] = y.x; v[c][5] = y.y; v[c][6] = y.z; v[c][7] = y.w;
            } else {
#pragma unroll
                for (int i = 0; i < 8; ++i) v[c][i] = 0.f;
            }
        }
    }
};

__device__ __forceinline__ void sm8(const float* p, float* o) {
    const float4 x = reinterpret_cast<const float4*>(p)[0], y = reinterpret_cast<const float4*>(p)[1];
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
}
__device__ __forceinline__ void sm8(const __nv_bfloat16* p, float* o) {
    const uint4 q = *reinterpret_cast<const uint4*>(p);
    bf16x2_to_f32(q.x, o[0], o[1]);
    bf16x2_to_f32(q.y, o[2], o[3]);
    bf16x2_to_f32(q.z, o[4], o[5]);
    bf16x2_to_f32(q.w, o[6], o[7]);
}

// lane-partial dot of a shared-memory row with register-resident elements
template <typename T, int NCH>
__device__ __forceinline__ float part_dot(const T* row, const VecRegs<T, NCH>& x, int n, int lane) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int e = (lane + 32 * c) * 8;
        if (e < n) {
            float w[8];
            sm8(row + e, w);
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                a0 = fmaf(w[i], x.v[c][i], a0);
                a1 = fmaf(w[i + 1], x.v[c][i + 1], a1);
            }
        }
    }
    return a0 + a1;
}

// 16-byte asynchronous global -> shared copies: every copy of a staging loop
// is in flight at once (no register round trip); cp_wait() completes them.
__device__ __forceinline__ void cp16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src)
                 : "memory");
}
__device__ __forceinline__ void cp_wait() {
    asm volatile("cp.async.commit_group;\ncp.async.wait_all;" ::: "memory");
}

// Stage gate rows: for gate g < 3 and jj < nrows, source row
// g*gate_rows + row0 + jj (n elements) -> shared row g*nrows + jj.
template <typename T>
__device__ __forceinline__ void stage_rows(T* dst, const T* src_base, int row0, int nrows, int gate_rows, int n) {
    const int per_row = n * (int)sizeof(T) / 16;
    for (int i = threadIdx.x; i < 3 * nrows * per_row; i += blockDim.x) {
        const int rr = i / per_row, e = (i % per_row) * (16 / (int)sizeof(T));
        const int g = rr / nrows, jj = rr % nrows;
        cp16(dst + (size_t)rr * n + e, src_base + (size_t)(g * gate_rows + row0 + jj) * n + e);
    }
}

template <typename T, int NCH>
__global__ void __launch_bounds__(kBatchThreads) k_gru_batch(
    const float* __restrict__ gi_table, const T* __restrict__ w_hh, const float* __restrict__ h_in,
    float* __restrict__ h_out, __nv_bfloat16* __restrict__ h16_out, const int32_t* __restrict__ verified,
    const int32_t* __restrict__ forced, const unsigned long long* __restrict__ keys, int* __restrict__ bad,
    int* __restrict__ err, float* __restrict__ dbg_h, int u, int B, int V, int G) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int j0 = blockIdx.x * kJT;
    const int jn = min(kJT, G - j0);
    T* s_hh = reinterpret_cast<T*>(smem);  // [3*jn][G]
    pdl_trigger();
    // weights do not depend on the previous kernel: stage them before waiting
    if (u > 0) stage_rows(s_hh, w_hh, j0, jn, G, G);
    cp_wait();
    __syncthreads();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = warp; b < B; b += kBatchThreads / 32) {
        int t;
        if (u == 0) t = verified[b];
        else if (forced) t = forced[(size_t)b * kProposals + (u - 1)];
        else t = (int)key_index(keys[(size_t)b * kBlock + (u - 1)]);
        if (t < 0 || t >= V) {
            if (blockIdx.x == 0 && lane == 0) {
                bad[b] = 1;
                atomicOr(err, kErrBadToken);
            }
            t = 0;
        }
        // the token's input-side values, requested before the hidden-side products
        const int j = j0 + lane;
        const float* gi = gi_table + (size_t)t * 3 * G;
        float gir = 0.f, giz = 0.f, gin = 0.f, hp = 0.f;
        if (lane < jn) {
            gir = __ldg(gi + j);
            giz = __ldg(gi + G + j);
            gin = __ldg(gi + 2 * G + j);
            if (u > 0) hp = h_in[(size_t)b * G + j];
        }
        float gh[3 * kJT];
#pragma unroll
        for (int i = 0; i < 3 * kJT; ++i) gh[i] = 0.f;
        if (u > 0) {
            VecRegs<T, NCH> hv;
            hv.load_f(h_in + (size_t)b * G, G, lane);
#pragma unroll
            for (int i = 0; i < 3 * kJT; ++i)
                if (i % kJT < jn) gh[i] = warp_sum(part_dot(s_hh + (size_t)((i / kJT) * jn + i % kJT) * G, hv, G, lane));
        }
        if (lane < jn) {
            float hr = 0, hz = 0, hn = 0;
#pragma unroll
            for (int jj = 0; jj < kJT; ++jj)
                if (jj == lane) {
                    hr = gh[0 * kJT + jj]; hz = gh[1 * kJT + jj]; hn = gh[2 * kJT + jj];
                }
            const float r = sigmoidf_(gir + hr);
            const float zg = sigmoidf_(giz + hz);
            const float n = tanhf(gin + r * hn);
            const float out = (1.f - zg) * n + zg * hp;
            h_out[(size_t)b * G + j] = out;
            if (h16_out) h16_out[(size_t)b * G + j] = __float2bfloat16_rn(out);
            if (dbg_h) dbg_h[((size_t)b * kProposals + u) * G + j] = out;
        }
    }
}

template <typename T, int NCH>
__global__ void __launch_bounds__(kBatchThreads) k_fc1_batch(const T* __restrict__ fc1, const float* __restrict__ h,
                                                             const T* __restrict__ s, float* __restrict__ a,
                                                             __nv_bfloat16* __restrict__ a16, float* __restrict__ dbg_z,
                                                             int k, int B, int G, int F) {
    extern __shared__ __align__(16) uint8_t smem[];
    const int f0 = blockIdx.x * kFT;
    const int fn = min(kFT, F - f0);
    T* s_w = reinterpret_cast<T*>(smem);  // [fn][G]
    pdl_trigger();
    const int per_row = G * (int)sizeof(T) / 16;
    for (int i = threadIdx.x; i < fn * per_row; i += blockDim.x) {
        const int rr = i / per_row, e = (i % per_row) * (16 / (int)sizeof(T));
        cp16(s_w + (size_t)rr * G + e, fc1 + (size_t)(f0 + rr) * G + e);
    }
    cp_wait();
    __syncthreads();
    pdl_wait();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    for (int b = warp; b < B; b += kBatchThreads / 32) {
        VecRegs<T, NCH> hv;
        hv.load_f(h + (size_t)b * G, G, lane);
        float z[kFT];
#pragma unroll
        for (int i = 0; i < kFT; ++i) z[i] = i < fn ? warp_sum(part_dot(s_w + (size_t)i * G, hv, G, lane)) : 0.f;
        if (lane < fn) {
            float zz = 0.f;
#pragma unroll
            for (int i = 0; i < kFT; ++i)
                if (i == lane) zz = z[i];
            const int f = f0 + lane;
            zz += to_f32(s[((size_t)b * kProposals + k) * F + f]);
            const float act = zz * sigmoidf_(zz);
            a[(size_t)b * F + f] = act;
            a16[(size_t)b * F + f] = __float2bfloat16_rn(act);
            if (dbg_z) dbg_z[((size_t)b * kCorrected + (k - 1)) * F + f] = zz;
        }
    }
}

// Correction + argmax over each request's candidate pool (B >= 2): a warp
// takes 4 pool entries at a time, requests all 4 gathered fc2 rows before
// using any (16-byte loads that bypass L1), keeps its request's activations
// in registers, and finishes the 4 rows on 4 lanes after one transposed warp
// reduction.  c = fc2[v] . a[b] + bias[v] + L[b, k+1, v], lowest id on ties.
constexpr int kPoolRows = 4;

__device__ __forceinline__ uint4 ldg_stream(const void* p) {
    uint4 q;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w)
                 : "l"(p));
    return q;
}

// each of 4 per-lane values summed over the warp (6 shuffles); lane l holds
// the total of value ((l >> 4) & 1) * 2 + ((l >> 3) & 1)
__device__ __forceinline__ float warp_sum4_t(float v0, float v1, float v2, float v3, int lane) {
    const bool hi16 = (lane & 16) != 0;
    float a = hi16 ? v2 : v0, b = hi16 ? v3 : v1;
    const float c = hi16 ? v0 : v2, d = hi16 ? v1 : v3;
    a += __shfl_xor_sync(0xffffffffu, c, 16);
    b += __shfl_xor_sync(0xffffffffu, d, 16);
    const bool hi8 = (lane & 8) != 0;
    float keep = hi8 ? b : a;
    const float send = hi8 ? a : b;
    keep += __shfl_xor_sync(0xffffffffu, send, 8);
    keep += __shfl_xor_sync(0xffffffffu, keep, 4);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    keep += __shfl_xor_sync(0xffffffffu, keep, 1);
    return keep;
}

template <int NCH>
__global__ void __launch_bounds__(kBatchThreads) k_correct_pool_batch(
    const __nv_bfloat16* __restrict__ fc2, const __nv_bfloat16* __restrict__ bias, const float* __restrict__ L,
    const float* __restrict__ a, const int32_t* __restrict__ pool, unsigned long long* __restrict__ keys,
    float* __restrict__ dbg_scores, int k, int B, int V, int F, int K, int items_per_block) {
    __shared__ unsigned long long sbest[64];
    pdl_trigger();
    pdl_wait();
    const long long items = (long long)B * K;
    const long long i0 = (long long)blockIdx.x * items_per_block;
    const long long i1 = min(items, i0 + items_per_block);
    if (i0 >= i1) return;
    const int b_first = (int)(i0 / K);
    const int nreq = (int)((i1 - 1) / K) - b_first + 1;  // <= 64 by the launch
    for (int i = threadIdx.x; i < 64; i += blockDim.x) sbest[i] = 0ull;
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nwarps = kBatchThreads / 32;
    float areg[NCH][8];
    int areg_b = -1;
    unsigned long long best = 0ull;
    int cur = -1;
    for (long long g = i0 + (long long)warp * kPoolRows; g < i1; g += (long long)nwarps * kPoolRows) {
        const int nr = (int)min((long long)kPoolRows, i1 - g);
        int v[kPoolRows];
#pragma unroll
        for (int rr = 0; rr < kPoolRows; ++rr) v[rr] = rr < nr ? pool[g + rr] : 0;
        uint4 w[kPoolRows][NCH];
#pragma unroll
        for (int rr = 0; rr < kPoolRows; ++rr)
#pragma unroll
            for (int cc = 0; cc < NCH; ++cc) {
                const int e = (lane + 32 * cc) * 8;
                w[rr][cc] = (rr < nr && e < F) ? ldg_stream(fc2 + (size_t)v[rr] * F + e) : make_uint4(0, 0, 0, 0);
            }
        // the finishing lane of each row fetches its bias and base logit early
        const int rsel = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
        const bool fin = (lane & 7) == 0 && rsel < nr;
        float tail = 0.f;
        int rb = 0, rv = 0;
        if (fin) {
            rb = (int)((g + rsel) / K);
            rv = pool[g + rsel];
            tail = __bfloat162float(bias[rv]) + L[((size_t)rb * kBlock + kRowOffset + k) * V + rv];
        }
        float part[kPoolRows];
#pragma unroll
        for (int rr = 0; rr < kPoolRows; ++rr) {
            part[rr] = 0.f;
            if (rr < nr) {
                const int b = (int)((g + rr) / K);
                if (b != areg_b) {  // warp-uniform, once per request run
#pragma unroll
                    for (int cc = 0; cc < NCH; ++cc) {
                        const int e = (lane + 32 * cc) * 8;
                        if (e < F) {
                            const float4 x = __ldg(reinterpret_cast<const float4*>(a + (size_t)b * F + e));
                            const float4 y = __ldg(reinterpret_cast<const float4*>(a + (size_t)b * F + e) + 1);
                            areg[cc][0] = x.x; areg[cc][1] = x.y; areg[cc][2] = x.z; areg[cc][3] = x.w;
                            areg[cc][4] = y.x; areg[cc][5] = y.y; areg[cc][6] = y.z; areg[cc][7] = y.w;
                        }
                    }
                    areg_b = b;
                }
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    const int e = (lane + 32 * cc) * 8;
                    if (e < F) {
                        float x[8];
                        bf16x2_to_f32(w[rr][cc].x, x[0], x[1]);
                        bf16x2_to_f32(w[rr][cc].y, x[2], x[3]);
                        bf16x2_to_f32(w[rr][cc].z, x[4], x[5]);
                        bf16x2_to_f32(w[rr][cc].w, x[6], x[7]);
#pragma unroll
                        for (int i = 0; i < 8; i += 2) {
                            a0 = fmaf(x[i], areg[cc][i], a0);
                            a1 = fmaf(x[i + 1], areg[cc][i + 1], a1);
                        }
                    }
                }
                part[rr] = a0 + a1;
            }
        }
        const float tot = warp_sum4_t(part[0], part[1], part[2], part[3], lane);
        if (fin) {
            const float cv = tot + tail;
            const unsigned long long key = pack_key(cv, (uint32_t)rv);
            const int bl = rb - b_first;
            if (bl != cur) {
                if (cur >= 0 && best) atomicMax(&sbest[cur], best);
                cur = bl;
                best = 0ull;
            }
            best = key > best ? key : best;
            if (dbg_scores) dbg_scores[((size_t)rb * kCorrected + (k - 1)) * K + (int)((g + rsel) % K)] = cv;
        }
    }
    if (best) atomicMax(&sbest[cur], best);
    __syncthreads();
    for (int i = threadIdx.x; i < nreq; i += blockDim.x)
        if (sbest[i]) atomicMax(&keys[(size_t)(b_first + i) * kBlock + k], sbest[i]);
}

template <typename T>
using GruKern = void (*)(const float*, const T*, const float*, float*, __nv_bfloat16*, const int32_t*,
                         const int32_t*, const unsigned long long*, int*, int*, float*, int, int, int, int);
template <typename T>
using Fc1Kern = void (*)(const T*, const float*, const T*, float*, __nv_bfloat16*, float*, int, int, int, int);

template <typename T>
GruKern<T> pick_gru(int nch) {
    return nch <= 1 ? k_gru_batch<T, 1> : nch <= 2 ? k_gru_batch<T, 2> : nch <= 4 ? k_gru_batch<T, 4>
         : nch <= 6 ? k_gru_batch<T, 6> : nch <= 8 ? k_gru_batch<T, 8> : nullptr;
}
template <typename T>
Fc1Kern<T> pick_fc1(int nch) {
    return nch <= 1 ? k_fc1_batch<T, 1> : nch <= 2 ? k_fc1_batch<T, 2> : nch <= 4 ? k_fc1_batch<T, 4>
         : nch <= 6 ? k_fc1_batch<T, 6> : nch <= 8 ? k_fc1_batch<T, 8> : nullptr;
}

inline int nch_of(int n) { return (n + 255) / 256; }

template <int NCH>
cudaError_t launch_pool_nch(domino_ctx* c, RunArgs& r, int k) {
    const domino_config& g = c->cfg;
    // items per block: about four blocks per SM (every warp's gathered rows in
    // flight at once), whole 4-row groups per warp, at most 8 groups per warp
    // and at most 64 requests a block
    long long items = (long long)r.B * r.K;
    const int group = (kBatchThreads / 32) * kPoolRows;  // one 4-row group per warp
    long long want = (items + 4LL * c->num_sms - 1) / (4LL * c->num_sms);
    want = (want + group - 1) / group * group;
    int ipb = (int)(want < group ? group : want > 8 * group ? 8 * group : want);
    if ((long long)ipb > 62LL * r.K) ipb = (int)(62LL * r.K);
    if (ipb < 1) ipb = 1;
    const long long blocks = (items + ipb - 1) / ipb;
    ++r.launches;
    return launch_pdl(k_correct_pool_batch<NCH>, dim3((unsigned)blocks), dim3(kBatchThreads), 0, r.st,
                      (const __nv_bfloat16*)c->fc2, (const __nv_bfloat16*)c->bias, (const float*)c->L,
                      (const float*)c->a, (const int32_t*)c->pool, c->keys, r.dbg.scores, k, r.B, g.V, g.F, r.K,
                      ipb);
}

}  // namespace

bool pool_batch_supported(const domino_ctx* c) {
    return c->cfg.dtype == DOMINO_DTYPE_BF16 && (c->cfg.F & 7) == 0 && nch_of(c->cfg.F) <= 8;
}

cudaError_t launch_correct_pool_batch(domino_ctx* c, RunArgs& r, int k) {
    const int nch = nch_of(c->cfg.F);
    return nch <= 1 ? launch_pool_nch<1>(c, r, k) : nch <= 2 ? launch_pool_nch<2>(c, r, k)
         : nch <= 4 ? launch_pool_nch<4>(c, r, k) : nch <= 6 ? launch_pool_nch<6>(c, r, k)
                    : launch_pool_nch<8>(c, r, k);
}

bool batch_kernels_supported(const domino_ctx* c) {
    const domino_config& g = c->cfg;
    if (g.dtype != DOMINO_DTYPE_BF16) return false;
    if ((g.E | g.G | g.F) & 7) return false;
    const int mx = g.E > g.G ? (g.E > g.F ? g.E : g.F) : (g.G > g.F ? g.G : g.F);
    if (nch_of(mx) > 8) return false;
    const size_t gru_smem = (size_t)3 * kJT * g.G * 2;
    return gru_smem <= 200 * 1024;
}

cudaError_t launch_gru_batch(domino_ctx* c, RunArgs& r, int u, __nv_bfloat16* h16_out) {
    using T = __nv_bfloat16;
    const domino_config& g = c->cfg;
    const float* h_in = c->h + (size_t)h_slot(u + 1) * g.max_B * g.G;
    float* h_out = c->h + (size_t)h_slot(u) * g.max_B * g.G;
    GruKern<T> kern = pick_gru<T>(nch_of(g.G));
    const size_t smem = (size_t)3 * kJT * g.G * sizeof(T);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = (g.G + kJT - 1) / kJT;
    ++r.launches;
    return launch_pdl(kern, dim3(grid), dim3(kBatchThreads), smem, r.st, (const float*)c->gi_table,
                      (const T*)c->w_hh, h_in, h_out, h16_out, r.verified, r.forced,
                      (const unsigned long long*)c->keys, c->bad, c->err, r.dbg.h, u, r.B, g.V, g.G);
}

cudaError_t launch_fc1_batch(domino_ctx* c, RunArgs& r, int k) {
    using T = __nv_bfloat16;
    const domino_config& g = c->cfg;
    const float* h = c->h + (size_t)h_slot(k) * g.max_B * g.G;
    Fc1Kern<T> kern = pick_fc1<T>(nch_of(g.G));
    const size_t smem = (size_t)kFT * g.G * sizeof(T);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int grid = (g.F + kFT - 1) / kFT;
    ++r.launches;
    return launch_pdl(kern, dim3(grid), dim3(kBatchThreads), smem, r.st, (const T*)c->fc1, h, (const T*)r.s, c->a,
                      c->a16, r.dbg.z, k, r.B, g.G, g.F);
}

}  // namespace domino
