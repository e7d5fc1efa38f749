// Shared device helpers and the library's internal context.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <climits>

#include "domino_rollout.h"

namespace domino {

constexpr int kBlock = DOMINO_BLOCK;       // draft positions per request
constexpr int kProposals = kBlock - 1;     // p_1 .. p_15
constexpr int kCorrected = kProposals - 1; // corrected steps k = 1..14
// Base row used by proposal j (0-based): block position 0 holds the verified
// token, so proposal j reads row j + 1.
constexpr int kRowOffset = 1;

// Device error word bits.
constexpr int kErrBadToken = 1;
constexpr int kErrTimeout = 2;

// ---------------------------------------------------------------------------
// argmax keys: (orderable(value) << 32) | ~index.  A larger key is a larger
// value, and among equal values the lower index.  -0.0 is folded into +0.0 so
// that signed zeros compare equal, as they do as numbers.
__device__ __forceinline__ uint32_t ord_f32(float f) {
    uint32_t u = __float_as_uint(f + 0.0f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float unord_f32(uint32_t o) {
    uint32_t u = (o & 0x80000000u) ? (o & 0x7FFFFFFFu) : ~o;
    return __uint_as_float(u);
}
__device__ __forceinline__ unsigned long long pack_key(float v, uint32_t idx) {
    return ((unsigned long long)ord_f32(v) << 32) | (unsigned long long)(~idx);
}
__device__ __forceinline__ uint32_t key_index(unsigned long long k) {
    return ~(uint32_t)(k & 0xFFFFFFFFull);
}
__device__ __forceinline__ float key_value(unsigned long long k) {
    return unord_f32((uint32_t)(k >> 32));
}

__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long k) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        unsigned long long other = __shfl_xor_sync(0xffffffffu, k, o);
        k = other > k ? other : k;
    }
    return k;
}
// Per-slot maxima of 16 keys over the warp with a transposed butterfly
// (16 64-bit shuffles instead of 16 separate 5-level reductions).  Returns
// the maximum of slot ((l>>4)&1)*8 + ((l>>3)&1)*4 + ((l>>2)&1)*2 + ((l>>1)&1)
// in lane l (lanes l and l^1 hold the same slot).
__device__ __forceinline__ unsigned long long warp_max16_u64(unsigned long long* v, int lane) {
#pragma unroll
    for (int level = 0; level < 4; ++level) {
        const int mask = 16 >> level, half = 8 >> level;
        const bool up = (lane & mask) != 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            if (i < half) {
                const unsigned long long send = up ? v[i] : v[i + half];
                const unsigned long long keep = up ? v[i + half] : v[i];
                const unsigned long long got = __shfl_xor_sync(0xffffffffu, send, mask);
                v[i] = got > keep ? got : keep;
            }
        }
    }
    const unsigned long long other = __shfl_xor_sync(0xffffffffu, v[0], 1);
    return other > v[0] ? other : v[0];
}
__device__ __forceinline__ int warp_max16_slot(int lane) {
    return ((lane >> 4) & 1) * 8 + ((lane >> 3) & 1) * 4 + ((lane >> 2) & 1) * 2 + ((lane >> 1) & 1);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

// Programmatic dependent launch: a kernel launched with the programmatic
// stream-serialization attribute may start while the previous kernel of the
// stream is still running.  pdl_wait() blocks until that kernel has completed
// and its memory is visible (a no-op for a normal launch); pdl_trigger() lets
// the next kernel start early.  Everything before pdl_wait() may only touch
// data no earlier kernel of the run writes.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// element loads: 8 consecutive elements widened to fp32
__device__ __forceinline__ void load8(const float* p, float* o) {
    float4 a = __ldg(reinterpret_cast<const float4*>(p));
    float4 b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
    o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void bf16x2_to_f32(uint32_t w, float& lo, float& hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xFFFF0000u);
}
__device__ __forceinline__ void load8(const __nv_bfloat16* p, float* o) {
    uint4 q = __ldg(reinterpret_cast<const uint4*>(p));
    bf16x2_to_f32(q.x, o[0], o[1]);
    bf16x2_to_f32(q.y, o[2], o[3]);
    bf16x2_to_f32(q.z, o[4], o[5]);
    bf16x2_to_f32(q.w, o[6], o[7]);
}
// streaming variant: do not keep the line in L1
__device__ __forceinline__ void load8_stream(const __nv_bfloat16* p, float* o) {
    uint4 q;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(q.x), "=r"(q.y), "=r"(q.z), "=r"(q.w) : "l"(p));
    bf16x2_to_f32(q.x, o[0], o[1]);
    bf16x2_to_f32(q.y, o[2], o[3]);
    bf16x2_to_f32(q.z, o[4], o[5]);
    bf16x2_to_f32(q.w, o[6], o[7]);
}
__device__ __forceinline__ void load8_stream(const float* p, float* o) { load8(p, o); }

__device__ __forceinline__ float to_f32(float x) { return x; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 x) { return __bfloat162float(x); }

// Warp-cooperative dot product of one weight row (n elements of T) with a
// fp32 vector; every lane returns the full sum.
template <typename T>
__device__ __forceinline__ float warp_dot(const T* __restrict__ w, const float* __restrict__ x, int n, int lane) {
    float acc = 0.f;
    if ((n & 7) == 0) {
        for (int i = lane * 8; i < n; i += 256) {
            float e[8];
            load8(w + i, e);
#pragma unroll
            for (int j = 0; j < 8; ++j) acc = fmaf(e[j], x[i + j], acc);
        }
    } else {
        for (int i = lane; i < n; i += 32) acc = fmaf(to_f32(w[i]), x[i], acc);
    }
    return warp_sum(acc);
}

}  // namespace domino

// ---------------------------------------------------------------------------
// Library context (opaque to callers).
struct domino_ctx {
    domino_config cfg;
    int device;
    int num_sms;
    int driver;
    int n_proposals;  // early stop: proposals per block (1..15)
    int partitions;   // vocabulary shards of the compact pool construction (1 = direct)
    int last_launches;
    int drop_barrier;  // test hook of the timeout path (0 = off): see domino_rollout_debug_drop_barrier_arrival
    bool loaded;
    // borrowed weights
    const void *lm_head, *emb, *w_ih, *w_hh, *fc1, *fc2, *bias;
    const void* fc1_hid;      // [F,H] backbone-hidden half of projector layer 1, or null
    // workspace (owned)
    float* L;                 // [max_B,16,V]
    float* score;             // [max_B,V]
    int32_t* pool;            // [max_B,max_K]
    void* s_ws;               // [max_B,15,F] input dtype: s computed from the backbone hidden
    int32_t* cand;            // [max_B, DOMINO_MAX_VOCAB_PARTITIONS*max_K] stage-C candidates, or null
    uint32_t* pmask;          // [max_B, ceil(V/32)] pool membership bits (bf16, max_K > 0), or null
    float* h;                 // [2][max_B,G] ping-pong
    float* a;                 // [max_B,F]
    __nv_bfloat16* a16;       // [a_rows,F] bf16 copy of a, zero padded
    int a_rows;
    unsigned long long* keys; // [max_B,16] argmax words, one per proposal
    int* bad;                 // [max_B] request saw an invalid token
    int* err;                 // device error word
    unsigned int* sync;       // grid-barrier words, per-step claim counters and the run counter
    unsigned long long* xa;     // [2][kLLMaxBatch,F] tagged activations (tagged-exchange driver)
    unsigned long long* xh;     // [2][kLLMaxBatch,G] tagged GRU state
    unsigned long long* xbest;  // [2][num_sms,kLLMaxBatch] per-CTA best of a step
    unsigned long long* xg;     // [2][3G] tagged hidden-side products of every unit (one request)
    float* gi_table;          // [V, 3G] input-side GRU pre-activations of every token (built at load)
    float* gh_next;           // [kPersistGruGroup][3G] hidden-side pre-activations of the next GRU update (persistent driver)
    unsigned* hist;           // [max_B, 2048] histogram of the pool scores' top 11 key bits (LM-head epilogue), or null
    float* ghb;               // [2][max_B,3G] hidden-side products W_hh h of the fused per-step launches (bf16 batches), or null
    __nv_bfloat16* wp;        // [4*Gp, G] packed hidden-side GRU weights (bf16 batches), or null
    __nv_bfloat16* h16;       // [2][a_rows, G] bf16 copies of the GRU state (tensor-core operands)
    void* ws_base;            // single workspace allocation
    size_t ws_bytes;
    // TMA descriptors (bf16 path)
    CUtensorMap tm_lm_head;
    CUtensorMap tm_fc2;
    CUtensorMap tm_wp;
    CUtensorMap tm_fc1h;
    bool has_fc1h_tmap;
    bool has_tma;
    // per-phase timing (host side)
    bool timing;
    int n_pending;
    int pending_phase[4096];
    cudaEvent_t ev[2 * 4096];
    int n_events;  // created so far
};
