// Device helpers shared by the persistent drivers of the rollout: the
// consumer-warp barrier, asynchronous 4-byte copies, shared-memory and
// register-held weight rows widened to fp32, and transposed warp sums.
#pragma once

#include "tc_common.cuh"

namespace domino {
namespace persist {

// 15 consumer warps + 1 producer warp: the consumers synchronise among
// themselves on named barrier 1
constexpr int kConsumerWarps = 15;
constexpr int kThreads = (kConsumerWarps + 1) * 32;

__device__ __forceinline__ void cons_sync() { asm volatile("bar.sync 1, 480;" ::: "memory"); }

__device__ __forceinline__ unsigned ld_acquire(const unsigned* p) {
    unsigned v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void cp_async4(float* dst, const float* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// 8 consecutive elements of a shared-memory row widened to fp32
__device__ __forceinline__ void lds8(const float* p, float* o) {
    float4 x = reinterpret_cast<const float4*>(p)[0], y = reinterpret_cast<const float4*>(p)[1];
    o[0] = x.x; o[1] = x.y; o[2] = x.z; o[3] = x.w; o[4] = y.x; o[5] = y.y; o[6] = y.z; o[7] = y.w;
}
__device__ __forceinline__ void lds8(const __nv_bfloat16* p, float* o) {
    uint4 q = *reinterpret_cast<const uint4*>(p);
    bf16x2_to_f32(q.x, o[0], o[1]);
    bf16x2_to_f32(q.y, o[2], o[3]);
    bf16x2_to_f32(q.z, o[4], o[5]);
    bf16x2_to_f32(q.w, o[6], o[7]);
}

// One weight row held in registers: lane l owns elements (l + 32 c) * 8 .. +7
// for c < NCH (NCH * 256 >= row length).  All chunks are requested before any
// is used, with an L2 evict-last hint (these small matrices are re-read every
// step while fc2 streams past them).
template <typename T, int NCH>
struct RegRow;
template <int NCH>
struct RegRow<__nv_bfloat16, NCH> {
    uint4 q[NCH];
    __device__ __forceinline__ void load(const __nv_bfloat16* row, int n, int lane, uint64_t pol) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int e = (lane + 32 * c) * 8;
            if (e < n)
                asm volatile("ld.global.nc.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
                             : "=r"(q[c].x), "=r"(q[c].y), "=r"(q[c].z), "=r"(q[c].w)
                             : "l"(row + e), "l"(pol));
            else
                q[c] = make_uint4(0, 0, 0, 0);
        }
    }
    __device__ __forceinline__ void get(int c, float* o) const {
        bf16x2_to_f32(q[c].x, o[0], o[1]);
        bf16x2_to_f32(q[c].y, o[2], o[3]);
        bf16x2_to_f32(q[c].z, o[4], o[5]);
        bf16x2_to_f32(q[c].w, o[6], o[7]);
    }
};
template <int NCH>
struct RegRow<float, NCH> {
    float4 q[2 * NCH];
    __device__ __forceinline__ void load(const float* row, int n, int lane, uint64_t pol) {
#pragma unroll
        for (int c = 0; c < NCH; ++c) {
            const int e = (lane + 32 * c) * 8;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (e < n)
                    asm volatile("ld.global.nc.L2::cache_hint.v4.f32 {%0,%1,%2,%3}, [%4], %5;"
                                 : "=f"(q[2 * c + h].x), "=f"(q[2 * c + h].y), "=f"(q[2 * c + h].z),
                                   "=f"(q[2 * c + h].w)
                                 : "l"(row + e + 4 * h), "l"(pol));
                else
                    q[2 * c + h] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    __device__ __forceinline__ void get(int c, float* o) const {
        o[0] = q[2 * c].x; o[1] = q[2 * c].y; o[2] = q[2 * c].z; o[3] = q[2 * c].w;
        o[4] = q[2 * c + 1].x; o[5] = q[2 * c + 1].y; o[6] = q[2 * c + 1].z; o[7] = q[2 * c + 1].w;
    }
};

// dot of a register row with a shared-memory fp32 vector (same element map)
template <typename T, int NCH>
__device__ __forceinline__ float row_dot_smem(const RegRow<T, NCH>& w, const float* x, int n, int lane) {
    float a0 = 0.f, a1 = 0.f;
#pragma unroll
    for (int c = 0; c < NCH; ++c) {
        const int e = (lane + 32 * c) * 8;
        if (e < n) {
            float ww[8], xx[8];
            w.get(c, ww);
            lds8(x + e, xx);
#pragma unroll
            for (int i = 0; i < 8; i += 2) {
                a0 = fmaf(ww[i], xx[i], a0);
                a1 = fmaf(ww[i + 1], xx[i + 1], a1);
            }
        }
    }
    return a0 + a1;
}

// Sum each of 4 per-lane values over the warp with 6 shuffles (a transposed
// butterfly).  Lane l ends with the total of value ((l >> 4) & 1) * 2 +
// ((l >> 3) & 1).
__device__ __forceinline__ float warp_sum4(float v0, float v1, float v2, float v3, int lane) {
    const bool hi16 = (lane & 16) != 0;
    float a = hi16 ? v2 : v0, b = hi16 ? v3 : v1;          // keep
    float c = hi16 ? v0 : v2, d = hi16 ? v1 : v3;          // send
    a += __shfl_xor_sync(0xffffffffu, c, 16);
    b += __shfl_xor_sync(0xffffffffu, d, 16);
    const bool hi8 = (lane & 8) != 0;
    float keep = hi8 ? b : a, send = hi8 ? a : b;
    keep += __shfl_xor_sync(0xffffffffu, send, 8);
    keep += __shfl_xor_sync(0xffffffffu, keep, 4);
    keep += __shfl_xor_sync(0xffffffffu, keep, 2);
    keep += __shfl_xor_sync(0xffffffffu, keep, 1);
    return keep;
}

// 16-byte asynchronous global -> shared copy (both 16-byte aligned)
__device__ __forceinline__ void cp_async16(void* dst, const void* src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(dst)), "l"(src) : "memory");
}

// Named-barrier sync of the consumer warps that also ORs a predicate over
// them: every thread gets the same answer, so a decision taken on it (e.g.
// to stop after a timed-out wait) is uniform.
__device__ __forceinline__ bool cons_sync_or(bool x) {
    uint32_t r;
    asm volatile(
        "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, 1, 480, p;\n selp.u32 %0, 1, 0, q;\n}"
        : "=r"(r)
        : "r"((uint32_t)x)
        : "memory");
    return r != 0;
}

// A bf16 row in the conflict-free lane layout: lane l holds elements
// 128c + 4l .. +3 (c < NC) as two packed bf16 pairs.
template <int NC>
struct Row4 {
    uint2 q[NC];
    __device__ __forceinline__ void load_smem(const __nv_bfloat16* row, int n, int lane) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int e = c * 128 + 4 * lane;
            q[c] = e < n ? *reinterpret_cast<const uint2*>(row + e) : make_uint2(0u, 0u);
        }
    }
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int c = 0; c < NC; ++c) q[c] = make_uint2(0u, 0u);
    }
    __device__ __forceinline__ void load_global(const __nv_bfloat16* row, int n, int lane, uint64_t pol) {
#pragma unroll
        for (int c = 0; c < NC; ++c) {
            const int e = c * 128 + 4 * lane;
            if (e < n)
                asm volatile("ld.global.nc.L2::cache_hint.v2.u32 {%0,%1}, [%2], %3;"
                             : "=r"(q[c].x), "=r"(q[c].y)
                             : "l"(row + e), "l"(pol));
            else
                q[c] = make_uint2(0u, 0u);
        }
    }
};

// fp32 shared-memory vector chunk c of this lane (zero past n)
__device__ __forceinline__ float4 vec4(const float* x, int c, int n, int lane) {
    const int e = c * 128 + 4 * lane;
    return e < n ? *reinterpret_cast<const float4*>(x + e) : make_float4(0.f, 0.f, 0.f, 0.f);
}
__device__ __forceinline__ void fma4(uint2 w, float4 x, float& a0, float& a1) {
    float w0, w1, w2, w3;
    bf16x2_to_f32(w.x, w0, w1);
    bf16x2_to_f32(w.y, w2, w3);
    a0 = fmaf(w0, x.x, a0);
    a1 = fmaf(w1, x.y, a1);
    a0 = fmaf(w2, x.z, a0);
    a1 = fmaf(w3, x.w, a1);
}

// Two warp sums at once (their shuffles interleaved).
__device__ __forceinline__ void warp_sum2(float& a, float& b) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a += __shfl_xor_sync(0xffffffffu, a, o);
        b += __shfl_xor_sync(0xffffffffu, b, o);
    }
}

// Sum each of N per-lane values (N a power of two, N <= 32) over the warp
// with a transposed butterfly: N - 1 + (5 - log2 N) shuffles instead of
// 5 N.  At each halving step a lane keeps the half of its values selected
// by one bit of its lane id and sends the other half to its partner.  Lane l
// ends with the total of value tr_index<N>(l), which lanes that differ only
// in the bits below the selecting ones hold as well.
template <int N>
__device__ __forceinline__ float warp_sum_tr(float (&v)[N], int lane) {
#pragma unroll
    for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int i = 0; i < n / 2; ++i) {
            const float keep = up ? v[i + n / 2] : v[i];
            const float send = up ? v[i] : v[i + n / 2];
            v[i] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
    }
    float t = v[0];
#pragma unroll
    for (int o = 16 / N; o > 0; o >>= 1) t += __shfl_xor_sync(0xffffffffu, t, o);
    return t;
}
template <int N>
__device__ __forceinline__ int tr_index(int lane) {
    int idx = 0;
#pragma unroll
    for (int n = N, o = 16; n > 1; n >>= 1, o >>= 1)
        if (lane & o) idx += n / 2;
    return idx;
}
// The lanes that report the values of warp_sum_tr<N>: one per value.
template <int N>
__device__ __forceinline__ bool tr_reporter(int lane) {
    return (lane & (32 / N - 1)) == 0;
}

// ---- warp-level bf16 tensor-core products (m16n8k16, fp32 accumulate)
// Four 8x8 bf16 matrices from shared memory; lane l gives the address of row
// l % 8 of matrix l / 8 (16-byte aligned) and receives in register i the
// elements (row l / 4, columns 2 (l % 4) and 2 (l % 4) + 1) of matrix i.
__device__ __forceinline__ void ldmatrix_x4(uint32_t addr, uint32_t (&r)[4]) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(addr));
}
// d += A (16x16, row-major fragments) * B (16x8, column fragments)
__device__ __forceinline__ void mma_16816(float (&d)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}
// Two fp32 values as a pair of bf16 leading parts (hi, round to nearest) and
// a pair of bf16 remainders (lo = x - hi, rounded; x - hi itself is exact):
// |x - hi - lo| <= 2^-16 |x|, and the products of a bf16 weight with hi and
// with lo are exact in fp32, so w*hi + w*lo differs from w*x by at most
// 2^-16 |w x| before the accumulation's own rounding.
__device__ __forceinline__ void split_bf16x2(float x0, float x1, uint32_t& hi, uint32_t& lo) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(x0, x1);
    const __nv_bfloat162 l = __floats2bfloat162_rn(x0 - __low2float(h), x1 - __high2float(h));
    hi = *reinterpret_cast<const uint32_t*>(&h);
    lo = *reinterpret_cast<const uint32_t*>(&l);
}

}  // namespace persist
}  // namespace domino
