// Persistent single-launch driver of the rollout after the LM-head: the two
// GRU seed updates and the 14 dependent corrected steps (fewer with an early
// stop) run in one cooperative kernel (one CTA per SM) separated by software
// grid barriers.
//
// Per corrected step k (page "Add correctness-first Domino support to DFlash
// V2", section "Design"; page "[Spec] Add Domino projector support to DFlash
// speculative decoding (V2)", section "Implementation"):
//   phase B  a = SiLU(fc1 h + s[k])        each CTA: a slice of the F outputs
//   -- grid barrier --
//   phase C  c[v] = fc2[v].a + bias[v] + L[b,k+1,v], argmax   each CTA: a
//            contiguous slice of fc2 rows (full vocabulary) or of the pool
//            entries; per-CTA best folded into the step's argmax word
//   -- grid barrier --
//   phase A  h = GRU(emb[p_{k+1}], h)      each CTA: a slice of the G outputs;
//            the input side W_ih emb[p] is a row of the token table built at
//            load time, the hidden side W_hh h is computed during phase C
//   -- grid barrier --
//
// A producer warp streams the fc2 rows (contiguous slices, or one row per
// pool entry) with cp.async.bulk into a ring of shared-memory slots.  The rows
// are the same at every step, so the producer runs ahead across phases and
// steps: while the CTA computes the GRU and fc1 phases and waits at barriers
// the ring refills.  Successive steps walk the slice in opposite directions,
// so a step starts on the rows the previous one read last (still in L2).
//
// The correction here runs on CUDA cores (a consumer warp takes a whole
// 4-row slot and keeps the activations in registers, fp32 FMA; row totals go
// to shared memory and an epilogue adds bias and base logits and takes the
// argmax), which suits one request per row: B = 1 over the full vocabulary,
// or pool entries of any request.  Every wait (grid barrier, ring slot) is
// bounded; on a timeout the kernel raises the device error word and returns.
#include "internal.h"
#include "persist_util.cuh"
#include "tc_common.cuh"

namespace domino {

namespace {

using namespace persist;
// 15 consumer warps + 1 producer warp: 16 warps leave 128 registers a thread
constexpr int kPersistThreads = persist::kThreads;
constexpr int kRowsPerSlot = 4;    // rows per ring slot; one warp consumes a whole slot
constexpr int kMaxSlots = 48;
// Ring slot q % n_slots is consumed by warp q % n_cons alone (n_cons divides
// n_slots): each slot has one waiting consumer and the producer, so a parity
// wait can never observe a fill that belongs to a later pass over the ring.
constexpr int kMaxReq = 8;         // requests a CTA may touch in phase C
constexpr int kGruGroup = kPersistGruGroup;  // requests per GRU/fc1 staging group
constexpr int kMaxSeg = 2048;      // rows (or pool entries) per CTA

template <typename T>
struct PersistParams {
    const T *w_hh, *fc1, *fc2, *bias, *s;
    const float* gi_table;  // [V, 3G] input-side GRU pre-activations of every token
    const int32_t *verified, *forced, *pool;
    const float* L;
    float* h;       // [2][max_B*G]
    float* gh;      // [kGruGroup][3][G] W_hh h of the next update, all units
    float* a;       // [max_B*F]
    unsigned long long* keys;
    int *bad, *err;
    unsigned int* sync;
    float *dbg_h, *dbg_z, *dbg_scores;
    unsigned long long* trace;  // [grid][DOMINO_TRACE_SLOTS] or null
    int B, K, V, E, G, F, max_B;
    int n_corr;     // corrected steps (early stop: fewer than 14)
    int seg;        // rows (K0) or pool entries per CTA
    int n_slots;
    int n_cons;     // consumer warps of the correction phase (divides n_slots)
    int slot_bytes;
    int drop_barrier;  // test hook: CTA 0 skips its arrival at this grid barrier (0 = never)
};

// Grid barrier among the consumer warps of every CTA.  `n` counts barriers
// passed so far; the counter was zeroed before the launch.  drop_at == n
// (a test hook for the timeout path) withholds this CTA's arrival, so every
// CTA's bounded wait at that barrier runs out.
__device__ bool grid_sync(unsigned* counter, unsigned& n, volatile int* abort_flag, int* err, int drop_at) {
    cons_sync();
    ++n;
    if (threadIdx.x == 0) {
        if (drop_at != (int)n) asm volatile("red.release.gpu.global.add.u32 [%0], 1;" ::"l"(counter) : "memory");
        const unsigned target = n * gridDim.x;
        const unsigned long long t0 = tc::globaltimer();
        while (ld_acquire(counter) < target) {
            if (*abort_flag) break;
            if (tc::globaltimer() - t0 > tc::kWaitLimitNs) {
                *abort_flag = 1;
                atomicOr(err, kErrTimeout);
                break;
            }
        }
    }
    cons_sync();
    return !*abort_flag;
}

// Shared-memory layout (bytes, all offsets 128-aligned)
// Requests whose activations one CTA needs in phase C.
__host__ __device__ inline int phase_c_requests(int B, int K, int seg) {
    if (K == 0) return B;
    const int n = seg / K + 2;
    return n < B ? n : B;
}

struct Layout {
    int ring, bars, sa, sh, sg, sL, sbias, stot, sbest, stok, misc, total;
    __host__ __device__ Layout(int n_slots, int slot_bytes, int E, int G, int F, int seg, int B, int K) {
        auto up = [](int x) { return (x + 127) & ~127; };
        const int nreq = phase_c_requests(B, K, seg), ngru = B < kGruGroup ? B : kGruGroup;
        int o = 0;
        ring = o; o = up(o + n_slots * slot_bytes);
        bars = o; o = up(o + 16 * n_slots);
        sa = o;   o = up(o + 4 * nreq * F);
        sh = o;   o = up(o + 4 * ngru * G);
        sg = o;   o = up(o + 4 * 3 * kGruGroup * 64);   // hidden-side products of one request group
        sL = o;   o = up(o + 4 * seg);
        sbias = o; o = up(o + 4 * seg);
        stot = o; o = up(o + 4 * seg);
        sbest = o; o = up(o + 8 * kMaxReq);
        stok = o; o = up(o + 4 * 256);
        misc = o; o = up(o + 64);
        total = o;
    }
};

template <typename T, int NCH>
__global__ void __launch_bounds__(kPersistThreads, 1) k_rollout_persist(PersistParams<T> p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const Layout lay(p.n_slots, p.slot_bytes, p.E, p.G, p.F, p.seg, p.B, p.K);
    uint8_t* ring = sm + lay.ring;
    const uint32_t full0 = tc::smem_u32(sm + lay.bars), empty0 = full0 + 8 * p.n_slots;
    float* sa = reinterpret_cast<float*>(sm + lay.sa);
    float* sh = reinterpret_cast<float*>(sm + lay.sh);
    float* sg = reinterpret_cast<float*>(sm + lay.sg);
    float* sL = reinterpret_cast<float*>(sm + lay.sL);
    float* sbias = reinterpret_cast<float*>(sm + lay.sbias);
    float* stot = reinterpret_cast<float*>(sm + lay.stot);  // fc2 row . a of each row of the slice
    unsigned long long* sbest = reinterpret_cast<unsigned long long*>(sm + lay.sbest);
    int* stok = reinterpret_cast<int*>(sm + lay.stok);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + lay.misc);
    volatile int* consumed_ptr = abort_flag + 1;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const bool full_vocab = p.K == 0;
    const int B = p.B, V = p.V, E = p.E, G = p.G, F = p.F;
    const size_t row_bytes = (size_t)F * sizeof(T);

    // this CTA's slice of correction work: rows [w0, w1) of fc2 (full
    // vocabulary) or entries [w0, w1) of the flattened [B, K] pool
    const long long work = full_vocab ? (long long)V : (long long)B * p.K;
    const long long w0 = min(work, (long long)blockIdx.x * p.seg);
    const long long w1 = min(work, w0 + p.seg);
    const int nw = (int)(w1 - w0);
    const int n_chunks = (nw + kRowsPerSlot - 1) / kRowsPerSlot;
    const int b_first = full_vocab ? 0 : (nw > 0 ? (int)(w0 / p.K) : 0);
    const int b_count = full_vocab ? B : (nw > 0 ? (int)((w1 - 1) / p.K) - b_first + 1 : 0);

    if (tid == 0) {
        for (int s = 0; s < p.n_slots; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        *consumed_ptr = 0;
        tc::fence_barrier_init();
        tc::fence_proxy_async();
    }
    __syncthreads();

    // This kernel may start while the previous kernel of the stream (the
    // LM-head, or the pool selection) still runs: pdl_wait() separates what
    // only reads weights and inputs from what reads that kernel's output.
    pdl_trigger();
    // ------------------------------------------------------------------ producer
    if (warp == kConsumerWarps) {
        if (!full_vocab) pdl_wait();  // pool ids come from the previous kernel
        if (lane < 4) {
            // full vocabulary: normal priority, so that the rows a step reads last
            // are still in L2 when the next step (walking backwards) starts;
            // pool rows are re-read every step: keep them
            const uint64_t pol = full_vocab ? tc::policy_evict_normal() : tc::policy_evict_last();
            int q = 0;
            for (int k = 1; k <= p.n_corr && !*abort_flag; ++k) {
                const bool fwd = (k & 1) != 0;
                for (int ci = 0; ci < n_chunks; ++ci) {
                    const int c = fwd ? ci : n_chunks - 1 - ci;
                    const int slot = q % p.n_slots;
                    const uint32_t par = (uint32_t)((q / p.n_slots) & 1);
                    if ((q & 3) != lane) {  // four producer lanes share the issue work
                        ++q;
                        continue;
                    }
                    if (!tc::mbar_wait(empty0 + 8 * slot, par ^ 1, abort_flag, p.err)) break;
                    const int r0 = c * kRowsPerSlot;
                    const int nr = min(kRowsPerSlot, nw - r0);
                    const uint32_t dst = tc::smem_u32(ring + (size_t)slot * p.slot_bytes);
                    tc::mbar_arrive_expect_tx(full0 + 8 * slot, (uint32_t)(nr * row_bytes));
                    if (full_vocab) {
                        tc::bulk_load(dst, p.fc2 + (size_t)(w0 + r0) * F, (uint32_t)(nr * row_bytes), full0 + 8 * slot,
                                      pol);
                    } else {
                        for (int r = 0; r < nr; ++r) {
                            const int v = p.pool[w0 + r0 + r];
                            tc::bulk_load(dst + (uint32_t)(r * row_bytes), p.fc2 + (size_t)v * F, (uint32_t)row_bytes,
                                          full0 + 8 * slot, pol);
                        }
                    }
                    ++q;
                }
            }
            if (lane != 0) return;
            // every copy issued must land before the block exits
            const unsigned long long t0 = tc::globaltimer();
            while (*consumed_ptr < q && !*abort_flag && tc::globaltimer() - t0 < tc::kWaitLimitNs) {
            }
            if (*consumed_ptr < q) {  // aborted: the last ring-full of copies may still be landing
                for (int i = q > p.n_slots ? q - p.n_slots : 0; i < q; ++i) {
                    const int s = i % p.n_slots;
                    const unsigned long long t1 = tc::globaltimer();
                    while (!tc::mbar_try_wait(full0 + 8 * s, (uint32_t)((i / p.n_slots) & 1)) &&
                           tc::globaltimer() - t1 < 2000000ull) {
                    }
                }
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    if (!full_vocab) pdl_wait();
    unsigned nsync = 0;
    unsigned* counter = p.sync;
    const int drop_at = blockIdx.x == 0 ? p.drop_barrier : 0;
    // static per-CTA bias values of the slice
    for (int i = tid; i < nw; i += kConsumerWarps * 32) {
        const int v = full_vocab ? (int)(w0 + i) : p.pool[w0 + i];
        sbias[i] = to_f32(p.bias[v]);
    }
    if (tid < kMaxReq) sbest[tid] = 0ull;

    const int jpc = (G + gridDim.x - 1) / gridDim.x;   // GRU outputs per CTA (<= 64)
    const int j0 = min(G, (int)blockIdx.x * jpc), j1 = min(G, j0 + jpc), jn = j1 - j0;
    const int fpc = (F + gridDim.x - 1) / gridDim.x;
    const int f0 = min(F, (int)blockIdx.x * fpc), f1 = min(F, f0 + fpc);

    const uint64_t pol_keep = tc::policy_evict_last();
    // W_hh h of the next GRU update is computed during the correction phase
    // (its warps have slack while fc2 streams) when all requests fit one group
    const bool pre_gh = B <= kGruGroup;

    // ---- one GRU update u for every request; writes h[slot(u)]
    auto gru = [&](int u) {
        const float* h_in = p.h + (size_t)h_slot(u + 1) * p.max_B * G;
        float* h_out = p.h + (size_t)h_slot(u) * p.max_B * G;
        if (tid < B) {
            int t;
            if (u == 0) t = p.verified[tid];
            else if (p.forced) t = p.forced[(size_t)tid * kProposals + (u - 1)];
            else t = (int)key_index(__ldcg(&p.keys[(size_t)tid * kBlock + (u - 1)]));
            if (t < 0 || t >= V) {
                if (blockIdx.x == 0) {
                    p.bad[tid] = 1;
                    atomicOr(p.err, kErrBadToken);
                }
                t = 0;
            }
            stok[tid] = t;
        }
        const bool need_gh = u > 0;
        for (int g0 = 0; g0 < B; g0 += kGruGroup) {
            const int ng = min(kGruGroup, B - g0);
            // the input side W_ih x of every request is a row of the token table;
            // only the hidden side W_hh h is contracted here (unless precomputed)
            RegRow<T, NCH> wh;
            int it = warp;
            if (need_gh && it < jn * 3) {  // first item's weight row before the staging loads
                const int jj = it / 3, gate = it % 3;
                wh.load(p.w_hh + (size_t)(gate * G + j0 + jj) * G, G, lane, pol_keep);
            }
            cons_sync();  // stok visible
            if (need_gh) {
                for (int i = tid; i < ng * G; i += kConsumerWarps * 32) {
                    const int b = i / G, e = i % G;
                    sh[b * G + e] = __ldcg(&h_in[(size_t)(g0 + b) * G + e]);
                }
                cons_sync();
                for (; it < jn * 3; it += kConsumerWarps) {
                    const int jj = it / 3, gate = it % 3;
                    if (it != warp) wh.load(p.w_hh + (size_t)(gate * G + j0 + jj) * G, G, lane, pol_keep);
#pragma unroll
                    for (int b = 0; b < kGruGroup; ++b) {
                        if (b < ng) {
                            const float gh = warp_sum(row_dot_smem(wh, sh + b * G, G, lane));
                            if (lane == 0) sg[(jj * 3 + gate) * kGruGroup + b] = gh;
                        }
                    }
                }
                cons_sync();
            }
            for (int i = tid; i < jn * ng; i += kConsumerWarps * 32) {
                const int jj = i / ng, b = i % ng;
                const float* gi = p.gi_table + (size_t)stok[g0 + b] * 3 * G + j0 + jj;
                float gh[3];
#pragma unroll
                for (int q = 0; q < 3; ++q) gh[q] = need_gh ? sg[(jj * 3 + q) * kGruGroup + b] : 0.f;
                const float r = sigmoidf_(__ldg(gi) + gh[0]);
                const float zg = sigmoidf_(__ldg(gi + G) + gh[1]);
                const float n = tanhf(__ldg(gi + 2 * G) + r * gh[2]);
                const float hp = u > 0 ? sh[b * G + j0 + jj] : 0.f;
                const float hn = (1.f - zg) * n + zg * hp;
                h_out[(size_t)(g0 + b) * G + j0 + jj] = hn;
                if (p.dbg_h) p.dbg_h[((size_t)(g0 + b) * kProposals + u) * G + j0 + jj] = hn;
            }
            cons_sync();
        }
    };

    // ---- W_hh h_k of the next GRU update (one request group, h_k staged in
    // sh by the projector phase of step k): this CTA's units, into p.gh
    auto hidden_products = [&](int k) {
        if (!(pre_gh && k < p.n_corr) || *abort_flag) return;
        for (int it = warp; it < jn * 3; it += kConsumerWarps) {
            const int jj = it / 3, gate = it % 3;
            RegRow<T, NCH> wh;
            wh.load(p.w_hh + (size_t)(gate * G + j0 + jj) * G, G, lane, pol_keep);
#pragma unroll
            for (int b = 0; b < kGruGroup; ++b) {
                if (b < B) {
                    const float gh = warp_sum(row_dot_smem(wh, sh + b * G, G, lane));
                    if (lane == 0) p.gh[((size_t)b * 3 + gate) * G + j0 + jj] = gh;
                }
            }
        }
    };

    // ---- GRU update u for one request group (B <= kGruGroup), computed in
    // full by every CTA from the token table row, the hidden-side products
    // p.gh (written by all CTAs during the previous correction) and h_{u-1}
    // (still staged in sh): the new state replaces sh in place and this CTA
    // publishes its own slice.  Saves the GRU phase and its grid barrier.
    auto gru_local = [&](int u) {
        float* h_out = p.h + (size_t)h_slot(u) * p.max_B * G;
        if (tid < B) {
            int t = p.forced ? p.forced[(size_t)tid * kProposals + (u - 1)]
                             : (int)key_index(__ldcg(&p.keys[(size_t)tid * kBlock + (u - 1)]));
            if (t < 0 || t >= V) {
                if (blockIdx.x == 0) {
                    p.bad[tid] = 1;
                    atomicOr(p.err, kErrBadToken);
                }
                t = 0;
            }
            stok[tid] = t;
        }
        cons_sync();
        constexpr int kNT = kConsumerWarps * 32, kPer = 2;  // elements a thread keeps in flight
        for (int base = 0; base < B * G; base += kPer * kNT) {
            float in[kPer][6];
#pragma unroll
            for (int e = 0; e < kPer; ++e) {  // every load of the round before any use
                const int i = base + e * kNT + tid;
                if (i < B * G) {
                    const int b = i / G, j = i % G;
                    const float* gi = p.gi_table + (size_t)stok[b] * 3 * G + j;
                    const float* gh = p.gh + (size_t)b * 3 * G + j;
                    in[e][0] = __ldg(gi);
                    in[e][1] = __ldg(gi + G);
                    in[e][2] = __ldg(gi + 2 * G);
                    in[e][3] = __ldcg(gh);
                    in[e][4] = __ldcg(gh + G);
                    in[e][5] = __ldcg(gh + 2 * G);
                }
            }
#pragma unroll
            for (int e = 0; e < kPer; ++e) {
                const int i = base + e * kNT + tid;
                if (i < B * G) {
                    const int b = i / G, j = i % G;
                    const float r = sigmoidf_(in[e][0] + in[e][3]);
                    const float zg = sigmoidf_(in[e][1] + in[e][4]);
                    const float n = tanhf(in[e][2] + r * in[e][5]);
                    const float hn = (1.f - zg) * n + zg * sh[b * G + j];
                    sh[b * G + j] = hn;
                    if (j >= j0 && j < j1) {
                        h_out[(size_t)b * G + j] = hn;
                        if (p.dbg_h) p.dbg_h[((size_t)b * kProposals + u) * G + j] = hn;
                    }
                }
            }
        }
        cons_sync();
    };

    // ---- projector layer 1 + SiLU for step k; writes a.  Leaves h_k staged
    // in sh (single group) for the hidden-side GRU products.
    auto fc1 = [&](int k, bool merged) {
        const float* hv = p.h + (size_t)h_slot(k) * p.max_B * G;
        for (int g0 = 0; g0 < B; g0 += kGruGroup) {
            const int ng = min(kGruGroup, B - g0);
            RegRow<T, NCH> w;
            int f = f0 + warp;
            if (f < f1) w.load(p.fc1 + (size_t)f * G, G, lane, pol_keep);
            if (merged) gru_local(k);  // one group: h_k computed into sh, the weight row in flight
            else
                for (int i = tid; i < ng * G; i += kConsumerWarps * 32) {
                    const int b = i / G, e = i % G;
                    sh[b * G + e] = __ldcg(&hv[(size_t)(g0 + b) * G + e]);
                }
            cons_sync();
            for (; f < f1; f += kConsumerWarps) {
                if (f != f0 + warp) w.load(p.fc1 + (size_t)f * G, G, lane, pol_keep);
#pragma unroll
                for (int b = 0; b < kGruGroup; ++b) {
                    if (b < ng) {
                        float z = warp_sum(row_dot_smem(w, sh + b * G, G, lane));
                        if (lane == 0) {
                            z += to_f32(p.s[((size_t)(g0 + b) * kProposals + k) * F + f]);
                            p.a[(size_t)(g0 + b) * F + f] = z * sigmoidf_(z);
                            if (p.dbg_z) p.dbg_z[((size_t)(g0 + b) * kCorrected + (k - 1)) * F + f] = z;
                        }
                    }
                }
            }
            cons_sync();
        }
    };

    // ---- correction + argmax of step k over this CTA's slice.  Ring slot q
    // (kRowsPerSlot rows) is consumed by warp q % n_cons alone.
    auto correct = [&](int k) {
        // activations of the requests this slice touches
        for (int i = tid; i < b_count * F; i += kConsumerWarps * 32) {
            const int b = i / F, f = i % F;
            sa[b * F + f] = __ldcg(&p.a[(size_t)(b_first + b) * F + f]);
        }
        cp_async_wait_all();
        cons_sync();
        float areg[NCH][8];
        int areg_b = -1;
        unsigned long long best = 0ull;  // running best of the rows this lane finalises
        int cur = -1;
        const bool fwd = (k & 1) != 0;
        const int qb = (k - 1) * n_chunks;
        const int nc = p.n_cons;
        int q = warp < nc ? qb + ((warp - qb) % nc + nc) % nc : qb + n_chunks;
        for (; q < qb + n_chunks; q += nc) {
            const int ci = q - qb;
            const int c = fwd ? ci : n_chunks - 1 - ci;
            const int slot = q % p.n_slots;
            if (!tc::mbar_wait(full0 + 8 * slot, (uint32_t)((q / p.n_slots) & 1), abort_flag, p.err)) break;
            const int r0 = c * kRowsPerSlot;
            const int nr = min(kRowsPerSlot, nw - r0);
            // requests of the slot's first and last rows (a slot spans two only
            // at a request boundary of the pool)
            const int bl0 = full_vocab ? 0 : (int)((w0 + r0) / p.K) - b_first;
            const int bl1 = full_vocab ? 0 : (int)((w0 + r0 + nr - 1) / p.K) - b_first;
            const T* srow = reinterpret_cast<const T*>(ring + (size_t)slot * p.slot_bytes);
            float part[kRowsPerSlot];
            if (bl0 == bl1) {
                if (bl0 != areg_b) {  // warp-uniform; once per step (full vocabulary)
#pragma unroll
                    for (int cc = 0; cc < NCH; ++cc) {
                        const int e = (lane + 32 * cc) * 8;
                        if (e < F) lds8(sa + bl0 * F + e, areg[cc]);
                    }
                    areg_b = bl0;
                }
                // the slot's rows as independent FMA chains
                float acc[kRowsPerSlot][2];
#pragma unroll
                for (int rr = 0; rr < kRowsPerSlot; ++rr) acc[rr][0] = acc[rr][1] = 0.f;
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    const int e = (lane + 32 * cc) * 8;
                    if (e < F) {
#pragma unroll
                        for (int rr = 0; rr < kRowsPerSlot; ++rr) {
                            if (rr < nr) {
                                float w[8];
                                lds8(srow + (size_t)rr * F + e, w);
#pragma unroll
                                for (int i = 0; i < 8; i += 2) {
                                    acc[rr][0] = fmaf(w[i], areg[cc][i], acc[rr][0]);
                                    acc[rr][1] = fmaf(w[i + 1], areg[cc][i + 1], acc[rr][1]);
                                }
                            }
                        }
                    }
                }
#pragma unroll
                for (int rr = 0; rr < kRowsPerSlot; ++rr) part[rr] = acc[rr][0] + acc[rr][1];
            } else {
                // rows of two requests: one row at a time with its own activations
#pragma unroll
                for (int rr = 0; rr < kRowsPerSlot; ++rr) {
                    part[rr] = 0.f;
                    if (rr < nr) {
                        const int bl = (int)((w0 + r0 + rr) / p.K) - b_first;
                        if (bl != areg_b) {
#pragma unroll
                            for (int cc = 0; cc < NCH; ++cc) {
                                const int e = (lane + 32 * cc) * 8;
                                if (e < F) lds8(sa + bl * F + e, areg[cc]);
                            }
                            areg_b = bl;
                        }
                        float a0 = 0.f, a1 = 0.f;
#pragma unroll
                        for (int cc = 0; cc < NCH; ++cc) {
                            const int e = (lane + 32 * cc) * 8;
                            if (e < F) {
                                float w[8];
                                lds8(srow + (size_t)rr * F + e, w);
#pragma unroll
                                for (int i = 0; i < 8; i += 2) {
                                    a0 = fmaf(w[i], areg[cc][i], a0);
                                    a1 = fmaf(w[i + 1], areg[cc][i + 1], a1);
                                }
                            }
                        }
                        part[rr] = a0 + a1;
                    }
                }
            }
            __syncwarp();
            if (lane == 0) tc::mbar_arrive(empty0 + 8 * slot);  // the slot is read: hand it back
            const float tot = warp_sum4(part[0], part[1], part[2], part[3], lane);
            const int rsel = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);
            if ((lane & 7) == 0 && rsel < nr) stot[r0 + rsel] = tot;  // finished after the loop
            if (lane == 0) atomicAdd((int*)consumed_ptr, 1);
        }
        // hidden-side GRU products for the next update while the ring refills
        hidden_products(k);
        cons_sync();
        // finish every row of the slice: bias, base logit, argmax key
        for (int r = tid; r < nw; r += kConsumerWarps * 32) {
            const long long item = w0 + r;
            const int bl = full_vocab ? 0 : (int)(item / p.K) - b_first;
            const int v = full_vocab ? (int)item : p.pool[item];
            const float cv = stot[r] + sbias[r] + sL[r];
            const unsigned long long key = pack_key(cv, (uint32_t)v);
            if (bl != cur) {
                if (cur >= 0 && best) atomicMax(&sbest[cur], best);
                cur = bl;
                best = 0ull;
            }
            best = key > best ? key : best;
            if (p.dbg_scores) {
                const int b = b_first + bl;
                if (full_vocab) p.dbg_scores[((size_t)b * kCorrected + (k - 1)) * V + v] = cv;
                else p.dbg_scores[((size_t)b * kCorrected + (k - 1)) * p.K + (int)(item % p.K)] = cv;
            }
        }
        if (full_vocab) {  // one request: reduce over the warp first
            best = warp_max_u64(best);
            if (lane == 0 && best) atomicMax(&sbest[0], best);
        } else if (best) {
            atomicMax(&sbest[cur], best);
        }
        cons_sync();
        if (tid < b_count) {
            if (sbest[tid]) atomicMax(&p.keys[(size_t)(b_first + tid) * kBlock + k], sbest[tid]);
            sbest[tid] = 0ull;
        }
    };

    // base-logit values of step k for the slice, fetched asynchronously
    auto prefetch_L = [&](int k) {
        for (int r = tid; r < nw; r += kConsumerWarps * 32) {
            const long long item = w0 + r;
            const int b = full_vocab ? 0 : (int)(item / p.K);
            const int v = full_vocab ? (int)item : p.pool[item];
            cp_async4(&sL[r], p.L + ((size_t)b * kBlock + kRowOffset + k) * V + v);
        }
        cp_async_commit();
    };

    // optional trace: stamp s of this CTA = time at the end of phase s
    unsigned long long* tr = p.trace ? p.trace + (size_t)blockIdx.x * DOMINO_TRACE_SLOTS : nullptr;
    int ts = 0;
    auto stamp = [&]() {
        if (tr && tid == 0 && ts < DOMINO_TRACE_SLOTS) tr[ts] = tc::globaltimer();
        ++ts;
    };
    auto body = [&]() {
        stamp();                                                     // 0: start
        gru(0);  // the verified token: independent of the previous kernel
        stamp();                                                     // 1
        pdl_wait();     // base logits, p_1 and the cleared argmax words are ready
        if (!grid_sync(counter, nsync, abort_flag, p.err, drop_at)) return;
        stamp();                                                     // 2
        gru(1);
        stamp();                                                     // 3
        if (!grid_sync(counter, nsync, abort_flag, p.err, drop_at)) return;
        stamp();                                                     // 4
        for (int k = 1; k <= p.n_corr; ++k) {                        // 5 + 6 (k-1) + ...
            prefetch_L(k);
            // one request group: GRU update k joins the projector phase
            fc1(k, pre_gh && k > 1);
            stamp();                                                 // +0 projector done
            if (!grid_sync(counter, nsync, abort_flag, p.err, drop_at)) return;
            stamp();                                                 // +1 barrier
            correct(k);
            stamp();                                                 // +2 correction done
            if (!grid_sync(counter, nsync, abort_flag, p.err, drop_at)) return;
            stamp();                                                 // +3 barrier
            if (k < p.n_corr) {
                if (pre_gh) {  // the next update runs in the next projector phase
                    stamp();                                         // +4
                    stamp();                                         // +5
                } else {
                    gru(k + 1);
                    stamp();                                         // +4 GRU done
                    if (!grid_sync(counter, nsync, abort_flag, p.err, drop_at)) return;
                    stamp();                                         // +5 barrier
                }
            }
        }
    };
    body();
}

struct Plan {
    int seg, slot_bytes, n_slots, n_cons, smem;
};

inline int gcd_int(int a, int b) { return b == 0 ? a : gcd_int(b, a % b); }

// Per-CTA slice, ring slot size and ring depth: the ring gets what the rest
// of the layout leaves of the opt-in shared-memory maximum (n_slots < 2: no).
Plan make_plan(const domino_ctx* c, int B, int K) {
    const domino_config& g = c->cfg;
    const int grid = c->num_sms;
    const long long work = K == 0 ? (long long)g.V : (long long)B * K;
    int seg = (int)((work + grid - 1) / grid);
    seg = (seg + kRowsPerSlot - 1) / kRowsPerSlot * kRowsPerSlot;
    const int esize = g.dtype == DOMINO_DTYPE_BF16 ? 2 : 4;
    const int slot_bytes = kRowsPerSlot * g.F * esize;
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    Layout base(0, slot_bytes, g.E, g.G, g.F, seg, B, K);
    int n_slots = (max_smem - base.total - 1024) / (slot_bytes + 16);
    if (n_slots > kMaxSlots) n_slots = kMaxSlots;
    // four producer lanes own the slots q % 4: keep the ring a multiple of 4;
    // consumer warps: the count (<= kConsumerWarps) whose multiple uses the most slots
    int n_cons = n_slots < kConsumerWarps ? n_slots : kConsumerWarps;
    int best = n_cons > 0 ? n_slots / n_cons * n_cons : 0;
    best = 0;
    for (int w = n_cons; w >= 4; --w) {
        const int l = w * 4 / gcd_int(w, 4);  // lcm(w, 4)
        if (n_slots / l * l > best) {
            best = n_slots / l * l;
            n_cons = w;
        }
    }
    Plan pl{seg, slot_bytes, best, n_cons, 0};
    n_slots = best;
    if (n_slots >= 2) pl.smem = Layout(n_slots, slot_bytes, g.E, g.G, g.F, seg, B, K).total;
    return pl;
}

// Register-row widths compiled per dtype (bf16 up to rows of 2048; fp32,
// used by the small fp32 workloads, up to rows of 512).
template <typename T>
void (*pick_kernel(int nch))(PersistParams<T>);
template <>
void (*pick_kernel<__nv_bfloat16>(int nch))(PersistParams<__nv_bfloat16>) {
    using T = __nv_bfloat16;
    return nch <= 1 ? k_rollout_persist<T, 1>
         : nch <= 2 ? k_rollout_persist<T, 2>
         : nch <= 4 ? k_rollout_persist<T, 4>
         : nch <= 6 ? k_rollout_persist<T, 6>
         : nch <= 8 ? k_rollout_persist<T, 8> : nullptr;
}
template <>
void (*pick_kernel<float>(int nch))(PersistParams<float>) {
    return nch <= 1 ? k_rollout_persist<float, 1> : nch <= 2 ? k_rollout_persist<float, 2> : nullptr;
}

template <typename T>
cudaError_t launch_t(domino_ctx* c, RunArgs& r) {
    const domino_config& g = c->cfg;
    const int grid = c->num_sms;
    const Plan pl = make_plan(c, r.B, r.K);
    if (pl.n_slots < 2) return cudaErrorNotSupported;
    const int seg = pl.seg, slot_bytes = pl.slot_bytes, n_slots = pl.n_slots, n_cons = pl.n_cons;
    struct {
        int total;
    } lay{pl.smem};

    PersistParams<T> p;
    p.gi_table = c->gi_table;
    p.w_hh = (const T*)c->w_hh;
    p.fc1 = (const T*)c->fc1;
    p.fc2 = (const T*)c->fc2;
    p.bias = (const T*)c->bias;
    p.s = (const T*)r.s;
    p.verified = r.verified;
    p.forced = r.forced;
    p.pool = c->pool;
    p.L = c->L;
    p.h = c->h;
    p.gh = c->gh_next;
    p.a = c->a;
    p.keys = c->keys;
    p.bad = c->bad;
    p.err = c->err;
    p.sync = c->sync;
    p.dbg_h = r.dbg.h;
    p.dbg_z = r.dbg.z;
    p.dbg_scores = r.dbg.scores;
    p.trace = r.dbg.trace;
    p.B = r.B;
    p.K = r.K;
    p.V = g.V;
    p.E = g.E;
    p.G = g.G;
    p.F = g.F;
    p.max_B = g.max_B;
    p.n_corr = r.n_prop - 1;
    p.seg = seg;
    p.n_slots = n_slots;
    p.n_cons = n_cons;
    p.slot_bytes = slot_bytes;
    p.drop_barrier = c->drop_barrier;  // one-shot test hook
    c->drop_barrier = 0;

    const int mx = g.E > g.G ? (g.E > g.F ? g.E : g.F) : (g.G > g.F ? g.G : g.F);
    const int nch = (mx + 255) / 256;
    void (*kern)(PersistParams<T>) = pick_kernel<T>(nch);
    if (!kern) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, lay.total);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kPersistThreads);
    cfg.dynamicSmemBytes = lay.total;
    cfg.stream = r.st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    ++r.launches;
    return e;
}

}  // namespace

// Whether the persistent driver covers this run: one request over the full
// vocabulary, or a pool whose per-CTA slice touches at most kMaxReq requests;
// rows must be whole 16-byte units and the per-CTA slice must fit the tables.
bool persist_supported(const domino_ctx* c, const RunArgs& r) {
    const domino_config& g = c->cfg;
    const int esize = g.dtype == DOMINO_DTYPE_BF16 ? 2 : 4;
    const int max_row = esize == 2 ? 2048 : 512;
    if (((g.E | g.G | g.F) & 7) || (g.F * esize) % 16 != 0 || g.F > max_row || g.E > max_row || g.G > max_row)
        return false;
    if ((g.G + c->num_sms - 1) / c->num_sms > 64) return false;
    if (r.B > 256) return false;
    const int grid = c->num_sms;
    if (r.K == 0) {
        if (r.B != 1) return false;
        const int seg = (g.V + grid - 1) / grid;
        return seg + kRowsPerSlot <= kMaxSeg && make_plan(c, r.B, r.K).n_slots >= 2;
    }
    const long long work = (long long)r.B * r.K;
    const long long seg = (work + grid - 1) / grid + kRowsPerSlot;
    if (seg > kMaxSeg) return false;
    if (seg / r.K + 2 > kMaxReq && r.B > kMaxReq) return false;
    return make_plan(c, r.B, r.K).n_slots >= 2;
}

cudaError_t launch_persist(domino_ctx* c, RunArgs& r) {
    return c->cfg.dtype == DOMINO_DTYPE_BF16 ? launch_t<__nv_bfloat16>(c, r) : launch_t<float>(c, r);
}

}  // namespace domino
