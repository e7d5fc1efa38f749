// Persistent tcgen05 "skinny" GEMM core: D[128 x BN] tiles of A[M,K] . B[N,K]^T
// with A streamed from HBM and B (a few activation rows) re-read from L2.
//
//   warp 0      TMA producer (one elected thread): A box {64, 128} and B box
//               {64, BN} per k-chunk into a STAGES-deep ring, 128-byte swizzle
//   warp 1      TMEM allocator + MMA issuer (one thread): 4 x tcgen05.mma
//               (M=128, N=BN, K=16) per k-chunk into one of two TMEM
//               accumulators, tcgen05.commit frees the ring slot
//   warps 2..9  epilogue: tcgen05.ld of the accumulator (one TMEM lane = one
//               row of A), handed to the Epi functor 16 columns at a time;
//               warp w reads TMEM lanes 32*(w%4).., warps 2..5 take the first
//               half of the tile's 16-column chunks and warps 6..9 the second,
//               so that a wide tile's epilogue keeps pace with its MMAs
//
// Epi provides begin(scratch, t) / prefetch(col0, row, pf) /
// operator()(col0, row, v[16], lane, scratch, pf + Epi::kPfChunk * c) / end(scratch, t),
// t = epilogue thread 0..kEpiThreads-1; `scratch` is Epi::kScratchWords per-block
// 64-bit words in shared memory (per-request argmax words); operator() must
// not wait on the other epilogue warps (after a timed-out wait they may have
// left the tile loop); `pf` holds up to kPrefetch
// values per thread that the epilogue may load for the next tile while the
// MMAs of that tile are still running.
//
// A second A matrix may follow the first: tiles m >= m_split read their 128
// rows from tmA2 at row (m - m_split) * 128, so that two weight matrices that
// share the B operand run in one launch (the epilogue sees the virtual row
// m * 128 + r).
//
// Tiles are visited m-major (tile t -> m = t / n_tiles, n = t % n_tiles), grid
// stride over a persistent grid of one CTA per SM, so CTAs that share an A
// tile run at the same time.  An Epi with a `rev` member set walks the m tiles
// in reverse (m = m_tiles - 1 - t / n_tiles); one with a kKeepTenths constant
// loads the A tiles of the last kKeepTenths/10 of its walk at normal L2
// priority instead of evict-first.  A launch per step over the same A that
// alternates `rev` then finds in L2 the tiles the previous launch read last.
// Every wait is bounded (tc::mbar_wait); on a timeout the block drains its
// copies and MMAs, frees TMEM and returns with the device error word set.
#pragma once

#include "tc_common.cuh"

namespace domino {
namespace tc {

constexpr int kBM = 128;          // rows of A per tile (MMA M)
constexpr int kBK = 64;           // K elements per chunk (128 bytes of bf16)
constexpr int kEpiWarps = 8;
constexpr int kEpiThreads = 32 * kEpiWarps;
constexpr int kGemmThreads = 64 + kEpiThreads;
constexpr int kEpiScratch = 256;  // 64-bit words
constexpr int kPrefetch = 64;     // per-thread epilogue prefetch registers

__device__ __forceinline__ void epi_bar() { asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory"); }

// optional Epi members: `rev` (reversed m-tile walk) and kKeepTenths (see above)
template <class E>
__device__ __forceinline__ auto tile_rev(const E& e, int) -> decltype(bool(e.rev)) {
    return e.rev;
}
template <class E>
__device__ __forceinline__ bool tile_rev(const E&, long) {
    return false;
}
template <class E>
__device__ __forceinline__ auto tile_keep(const E&, int) -> decltype(int(E::kKeepTenths)) {
    return E::kKeepTenths;
}
template <class E>
__device__ __forceinline__ int tile_keep(const E&, long) {
    return 0;
}

template <int BN, int SCRATCH_WORDS = kEpiScratch>
struct GemmShape {
    static constexpr int A_BYTES = kBM * kBK * 2;
    static constexpr int B_BYTES = BN * kBK * 2;
    static constexpr int STAGE = A_BYTES + B_BYTES;
    static constexpr int STAGES = (196608 / STAGE) > 12 ? 12 : (196608 / STAGE);
    static constexpr int TMEM_COLS = (2 * BN) < 32 ? 32 : 2 * BN;
    static constexpr size_t SMEM = (size_t)STAGES * STAGE + 1024 + 512 + 8 * SCRATCH_WORDS;
};

template <int BN, class Epi>
__global__ void __launch_bounds__(kGemmThreads, 1)
    k_gemm_tc(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmA2,
              const __grid_constant__ CUtensorMap tmB, int M, int m_split, int N, int K, Epi epi, int* err) {
    using S = GemmShape<BN, Epi::kScratchWords>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + (size_t)S::STAGES * S::STAGE);
    // bars: full[STAGES], empty[STAGES], tfull[2], tempty[2], drain
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S::STAGES + 5);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* consumed_ptr = reinterpret_cast<volatile int*>(tmem_slot + 2);
    unsigned long long* scratch = reinterpret_cast<unsigned long long*>(smem + (size_t)S::STAGES * S::STAGE + 512);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t full0 = smem_u32(bars), empty0 = smem_u32(bars + S::STAGES);
    const uint32_t tfull0 = smem_u32(bars + 2 * S::STAGES), tempty0 = tfull0 + 16, drain = tfull0 + 32;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S::STAGES; ++s) {
            mbar_init(full0 + 8 * s, 1);
            mbar_init(empty0 + 8 * s, 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(tfull0 + 8 * b, 1);
            mbar_init(tempty0 + 8 * b, kEpiThreads);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        *consumed_ptr = 0;
        fence_barrier_init();
        fence_proxy_async();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), S::TMEM_COLS);
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        tma_prefetch_desc(&tmA);
        if (m_split < (M + kBM - 1) / kBM) tma_prefetch_desc(&tmA2);
        tma_prefetch_desc(&tmB);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    // setup above overlaps the previous kernel.  The A operand is a weight
    // matrix that no kernel writes, so the producer requests the first
    // ring-full of A tiles before waiting for the previous kernel; everything
    // else waits for it here.
    pdl_trigger();
    if (warp != 0) pdl_wait();

    const int m_tiles = (M + kBM - 1) / kBM;
    const int n_tiles = (N + BN - 1) / BN;
    const int k_iters = (K + kBK - 1) / kBK;
    const int tiles = m_tiles * n_tiles;
    int issued = 0;
    const bool rev = tile_rev(epi, 0);
    auto m_of = [&](int t) {
        const int m = t / n_tiles;
        return rev ? m_tiles - 1 - m : m;
    };
    const int t_keep = tiles - (tile_keep(epi, 0) * tiles + 5) / 10;  // tiles t >= t_keep: normal priority

    if (warp == 0) {
        if (lane == 0) {
            const uint64_t pol_a = policy_evict_first();
            const uint64_t pol_a_keep = policy_evict_normal();
            const uint64_t pol_b = policy_evict_last();
            const int my_tiles = (int)blockIdx.x < tiles ? (tiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
            const int total = my_tiles * k_iters;
            const int pre = total < S::STAGES ? total : S::STAGES;  // chunk i sits in stage i
            auto a_row = [&](int t, const CUtensorMap*& ta) {
                const int m = m_of(t);
                const bool second = m >= m_split;
                ta = second ? &tmA2 : &tmA;
                return (second ? m - m_split : m) * kBM;
            };
            for (int i = 0; i < pre; ++i) {  // fresh ring: no slot to wait for
                const int t = blockIdx.x + (i / k_iters) * gridDim.x, kk = i % k_iters;
                const CUtensorMap* ta;
                const int arow = a_row(t, ta);
                mbar_arrive_expect_tx(full0 + 8 * i, S::STAGE);
                tma_load_2d(smem_u32(smem + (size_t)i * S::STAGE), ta, kk * kBK, arow, full0 + 8 * i,
                            t >= t_keep ? pol_a_keep : pol_a);
            }
            if (Epi::kL2Ahead > 0) {
                const uint64_t pol_l2 = policy_evict_normal();
                const int ahead = total < pre + Epi::kL2Ahead ? total : pre + Epi::kL2Ahead;
                for (int i = pre; i < ahead; ++i) {
                    const int t = blockIdx.x + (i / k_iters) * gridDim.x, kk = i % k_iters;
                    const CUtensorMap* ta;
                    const int arow = a_row(t, ta);
                    tma_prefetch_2d(ta, kk * kBK, arow, pol_l2);
                }
            }
            pdl_wait();
            int stage = 0;
            uint32_t phase = 0;
            int i = 0;
            // the pre-issued stages always get their B half (so that every copy
            // in flight belongs to a stage the abort drain below can wait for)
            for (int t = blockIdx.x; t < tiles && (i < pre || !*abort_flag); t += gridDim.x) {
                const int n = t % n_tiles;
                const CUtensorMap* ta;
                const int arow = a_row(t, ta);
                for (int kk = 0; kk < k_iters; ++kk, ++i) {
                    const uint32_t sa = smem_u32(smem + (size_t)stage * S::STAGE);
                    if (i >= pre) {
                        if (!mbar_wait(empty0 + 8 * stage, phase ^ 1, abort_flag, err)) break;
                        mbar_arrive_expect_tx(full0 + 8 * stage, S::STAGE);
                        tma_load_2d(sa, ta, kk * kBK, arow, full0 + 8 * stage, t >= t_keep ? pol_a_keep : pol_a);
                    }
                    tma_load_2d(sa + S::A_BYTES, &tmB, kk * kBK, n * BN, full0 + 8 * stage, pol_b);
                    ++issued;
                    if (++stage == S::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            constexpr uint32_t idesc = idesc_bf16_f32(kBM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            int consumed = 0;
            for (int t = blockIdx.x; t < tiles && !*abort_flag; t += gridDim.x) {
                if (!mbar_wait(tempty0 + 8 * acc, acc_phase ^ 1, abort_flag, err)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                bool ok = true;
                for (int kk = 0; kk < k_iters; ++kk) {
                    if (!mbar_wait(full0 + 8 * stage, phase, abort_flag, err)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sa = smem_u32(smem + (size_t)stage * S::STAGE);
                    const uint32_t sb = sa + S::A_BYTES;
#pragma unroll
                    for (int j = 0; j < kBK / 16; ++j)
                        mma_bf16(d, sdesc_sw128(sa + 32 * j), sdesc_sw128(sb + 32 * j), idesc, (kk | j) != 0);
                    mma_commit(empty0 + 8 * stage);
                    *consumed_ptr = ++consumed;
                    if (++stage == S::STAGES) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                mma_commit(tfull0 + 8 * acc);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            // all MMAs issued by this thread are complete once `drain` fires
            mma_commit(drain);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(drain, 0)) {
                if (globaltimer() - t0 > kWaitLimitNs) {
                    *abort_flag = 1;
                    atomicOr(err, kErrTimeout);
                    break;
                }
            }
        }
    } else {
        const int quarter = warp & 3;
        const int et = threadIdx.x - 64;
        // chunks [c_lo, c_hi) of every tile belong to this half of the epilogue warps
        constexpr int NC = BN / 16, HC = (NC + 1) / 2;
        const int half = et / 128;
        const int c_lo = half * HC, c_hi = (half + 1) * HC < NC ? (half + 1) * HC : NC;
        int acc = 0;
        uint32_t acc_phase = 0;
        epi.begin(scratch, et);
        epi_bar();
        // Epi::kPfChunk prefetch registers per 16-column chunk, for the
        // first kPrefetch / 16 chunks of this half
        constexpr int PFC = Epi::kPfChunk;
        constexpr int PF_CHUNKS = HC < kPrefetch / 16 ? HC : kPrefetch / 16;
        constexpr int PF = PFC * PF_CHUNKS;
        float pf[PF];
        if ((int)blockIdx.x < tiles && c_lo < c_hi) {
            const int t0 = blockIdx.x;
            epi.template prefetch<PF>((t0 % n_tiles) * BN + 16 * c_lo, m_of(t0) * kBM + quarter * 32 + lane, pf);
        }
        for (int t = blockIdx.x; t < tiles; t += gridDim.x) {
            if (!mbar_wait(tfull0 + 8 * acc, acc_phase, abort_flag, err)) break;
            tc_fence_after();
            const int m = m_of(t), n = t % n_tiles;
            const int row = m * kBM + quarter * 32 + lane;
            const uint32_t tbase = tmem_base + ((uint32_t)(quarter * 32) << 16) + (uint32_t)(acc * BN);
#pragma unroll
            for (int i = 0; i < HC; ++i) {
                const int c = c_lo + i;
                if (c < c_hi) {  // uniform over the warp
                    float v[16];
                    tmem_ld16(tbase + 16 * c, v);
                    epi(n * BN + 16 * c, row, v, lane, scratch, i < PF_CHUNKS ? pf + PFC * i : nullptr);
                }
            }
            const int tn = t + gridDim.x;  // the next tile's epilogue inputs, during its MMAs
            if (tn < tiles && c_lo < c_hi)
                epi.template prefetch<PF>((tn % n_tiles) * BN + 16 * c_lo, m_of(tn) * kBM + quarter * 32 + lane,
                                          pf);
            tc_fence_before();
            mbar_arrive(tempty0 + 8 * acc);
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
        epi_bar();
        epi.end(scratch, et);
    }
    __syncthreads();
    if (*abort_flag && warp == 0 && lane == 0) {
        // let every copy this block issued land before the block exits
        const int consumed = *consumed_ptr;
        for (int i = consumed; i < issued; ++i) {
            const int s = i % S::STAGES;
            const uint32_t par = (uint32_t)((i / S::STAGES) & 1);
            const unsigned long long t0 = globaltimer();
            while (!mbar_try_wait(full0 + 8 * s, par) && globaltimer() - t0 < 2000000ull) {
            }
        }
    }
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, S::TMEM_COLS);
    }
}

}  // namespace tc
}  // namespace domino
