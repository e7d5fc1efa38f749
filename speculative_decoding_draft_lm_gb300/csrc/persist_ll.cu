// Persistent driver for small batches (B <= 8, bf16) whose CTAs exchange
// data through step-tagged words instead of meeting at grid barriers.
//
// Per corrected step k (page "Add correctness-first Domino support to DFlash
// V2", section "Design"; page "[Spec] Add Domino projector support to DFlash
// speculative decoding (V2)", section "Implementation"), every CTA holds the
// whole GRU state h_k in shared memory and
//   P_k  computes its slice of a = SiLU(fc1 h_k + s[k]) and publishes it, and
//        the hidden-side products W_hh h_k of its own GRU units (kept);
//   C_k  reads all of a, scores its slice of fc2 rows (full vocabulary,
//        B = 1) or of the pool entries, c[v] = fc2[v].a + bias[v] +
//        L[b,k+1,v], and publishes its best (value, id) per request;
//   X_k  reads every CTA's best, takes p_{k+1} (lowest id on ties), updates
//        its own units, h_{k+1}[j] = GRU(emb[p_{k+1}], h_k)[j], from the
//        token-table row's three entries and its kept products, and
//        publishes them;
//   H_k  reads the whole new state.
// For one request the hidden-side products of every unit are published
// with the activations and read while the bests come in; X_k then updates
// every unit in each CTA, and H_k (one exchange per step) is not needed.
//
// Exchange words are 64 bits: a 32-bit payload with a 32-bit tag (run epoch
// * 16 + step), or for the per-CTA bests the packed key (orderable value, low
// id first) with the step in the low bits.  One 8-byte store publishes value
// and tag together, and a reader polls the word until its tag is the one it
// waits for, so a read of the data is also the synchronisation (no separate
// barrier round trip).  Each word has one writer per step.  Every exchange
// is double-buffered by step parity: a CTA that publishes nothing another
// waits for (e.g. one without projector rows) may still be reading step k's
// words when a faster CTA publishes step k+1, but no CTA can publish step
// k+2 before every CTA has published something that follows its reading of
// step k, so a buffer is never overwritten while it is read.  A reader
// loads several words at once and reads the ones without the tag again
// together, so a late word costs one more L2 round trip, not one per word.
//
// The fc1 rows of a CTA, and for pools its W_hh rows (and its pool rows
// when they fit), stay in shared memory for the whole launch.  With all its
// rows resident, a CTA's projector runs on the tensor cores (16-row tiles,
// one column per request, the fp32 state split into bf16 leading parts and
// remainders); over the full vocabulary, where W_hh is read from L2, a warp
// keeps two rows in registers and streams the state from shared memory in a
// lane layout without bank conflicts (lane l holds elements 128c + 4l ..
// 128c + 4l + 3), reducing all its (row, request) dots in one transposed
// butterfly.  Over the full vocabulary a producer warp streams fc2 with bulk
// copies into a ring (walking the slice in alternating directions so a step
// starts on the rows the last one read); the last seventh of every slice is
// shared: producers that finish their own part early claim those chunks
// through a per-step counter, which absorbs the per-step spread of the CTAs'
// streaming rates.  Pool rows that do not fit are gathered through the ring
// step by step, with a fixed chunk count per step.  A pool CTA reads only the
// activations of the requests its slice covers, and with several requests
// the bests only of the CTAs that cover each request (and of those past the
// pool's end, so that every CTA's word is still read by all).
//
// Every wait (exchange word, ring slot) is bounded; on a timeout the kernel
// raises the device error word, and all consumer warps leave together (the
// decision is taken with a barrier that ORs their flags).
#include <type_traits>

#include "internal.h"
#include "persist_util.cuh"

namespace domino {

using namespace persist;

namespace {

constexpr int kRows = 4;           // fc2 rows per ring slot
constexpr int kMaxSlots = 64;
constexpr int kShareDiv = 7;       // a seventh of each full-vocabulary slice is shared
constexpr int kKeepTenths = 4;     // last 4/10 of a full-vocabulary walk: normal L2 priority
constexpr int kProducerLanes = 4;  // lanes of the producer warp that issue copies
constexpr int kMaxSeg = 2048;
constexpr int kPad = 8;            // elements after each resident row and each state row (bank spread)
constexpr unsigned kBestTagMask = 0x3FFFu;  // low 14 bits of a best word: the step
constexpr int kBestIdShift = 14;            // next 18 bits: ~id

struct LLParams {
    const __nv_bfloat16 *w_hh, *fc1, *fc2, *bias, *s;
    const float* gi_table;  // [V, 3G]
    const int32_t *verified, *forced, *pool;
    const float* L;
    unsigned long long* keys;
    int *bad, *err;
    unsigned* claim;        // [16] per-step shared-chunk counters, zeroed per run
    const unsigned* epoch;  // run counter, bumped per run before this kernel
    unsigned long long* xa;     // [2][kLLMaxBatch][F]   activations, by step parity
    unsigned long long* xh;     // [2][kLLMaxBatch][G]   GRU state, by update parity
    unsigned long long* xbest;  // [2][grid][kLLMaxBatch] per-CTA bests, by step parity, zeroed per run
    unsigned long long* xg;     // [2][3G] hidden-side products of every unit (one request), by step parity
    float *dbg_h, *dbg_z, *dbg_scores;
    unsigned long long* trace;
    int B, K, V, G, F;
    int n_corr;
    int seg;        // rows (K0) or pool entries per CTA, a multiple of kRows
    int jpc, fpc;   // GRU units / fc1 rows per CTA
    int n_slots, n_cons, resident, pin_gi;
    int ra;         // requests whose activations a CTA keeps (its slice spans at most this many)
    int wh_res;     // W_hh rows of the CTA's units kept in shared memory (else read from L2 each step)
    int drop_at;    // test hook: CTA 0 withholds its publication number drop_at (0 = never)
};

struct LLLayout {
    int ring, bars, srow, swhh, sfc1, sh, spart, sa, sL, sbias, spid, sqid, ss, sgh, sgall, sred, stok, misc, total;
    // ra: requests whose activations a CTA keeps (those its correction slice covers);
    // wh_res: W_hh rows resident, which is the case exactly for pools
    __host__ __device__ LLLayout(int n_slots, int slot_bytes, int G, int F, int jpc, int fpc, int seg, int B, int ra,
                                 bool wh_res) {
        const bool pools = wh_res;
        auto up = [](int x) { return (x + 127) & ~127; };
        const int rs = G + kPad;                       // row stride of the resident rows and of the state
        const int mt = (fpc + 3 * jpc + 15) / 16;      // 16-row tiles of the tensor-core projector
        int o = 0;
        ring = o;  o = up(o + n_slots * slot_bytes);
        bars = o;  o = up(o + 16 * n_slots);
        srow = o;  o = up(o + 4 * n_slots);
        swhh = o;  o = up(o + (wh_res ? 3 * jpc * rs * 2 : 0));
        sfc1 = o;  o = up(o + fpc * rs * 2);
        sh = o;    o = up(o + 4 * B * rs);
        spart = o; o = up(o + (wh_res ? 4 * 128 * (mt > kConsumerWarps ? mt : kConsumerWarps) : 0));
        sa = o;    o = up(o + 4 * ra * F);
        sL = o;    o = up(o + 4 * seg);
        sbias = o; o = up(o + 4 * seg);
        spid = o;  o = up(o + (pools ? 4 * seg : 0));     // pool ids of the slice
        sqid = o;  o = up(o + (pools ? 4 * seg : 0));     // the same, for the producer warp
        ss = o;    o = up(o + 4 * B * kProposals * fpc);  // s entries of the CTA's projector outputs
        sgh = o;   o = up(o + 4 * B * 3 * jpc);           // hidden-side products of the CTA's units
        sgall = o; o = up(o + (B == 1 ? 4 * 3 * G : 0));  // one request: those of every unit
        sred = o;  o = up(o + 8 * 2 * kLLMaxBatch);
        stok = o;  o = up(o + 4 * kLLMaxBatch);
        misc = o;  o = up(o + 64);
        total = o;
    }
};

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ unsigned long long tagged(float x, unsigned tag) {
    return ((unsigned long long)tag << 32) | __float_as_uint(x);
}

// Does word w carry `tag`?  Mode 0: in its high 32 bits (tagged payloads);
// mode 1: in its low 14 bits (per-CTA bests).
__device__ __forceinline__ bool has_tag(unsigned long long w, unsigned tag, int mode) {
    return mode == 0 ? (unsigned)(w >> 32) == tag : (unsigned)(w & kBestTagMask) == tag;
}

// NC: 128-element chunks of a row per lane; MB: requests a lane tracks bests for
template <int NC, int MB>
__global__ void __launch_bounds__(kThreads, 1) k_rollout_ll(LLParams p) {
    extern __shared__ __align__(128) uint8_t sm[];
    const int B = p.B, V = p.V, G = p.G, F = p.F;
    const size_t row_bytes = (size_t)F * sizeof(__nv_bfloat16);
    const int slot_bytes = kRows * F * (int)sizeof(__nv_bfloat16);
    const LLLayout lay(p.n_slots, slot_bytes, G, F, p.jpc, p.fpc, p.seg, B, p.ra, p.wh_res != 0);
    uint8_t* ring = sm + lay.ring;
    const uint32_t full0 = tc::smem_u32(sm + lay.bars), empty0 = full0 + 8 * p.n_slots;
    volatile int* srow = reinterpret_cast<volatile int*>(sm + lay.srow);
    const __nv_bfloat16* swhh = reinterpret_cast<const __nv_bfloat16*>(sm + lay.swhh);
    const __nv_bfloat16* sfc1 = reinterpret_cast<const __nv_bfloat16*>(sm + lay.sfc1);
    float* sh = reinterpret_cast<float*>(sm + lay.sh);  // [B][SS] the state (fp32)
    float* spart = reinterpret_cast<float*>(sm + lay.spart);
    const int RS = G + kPad, SS = G + kPad;
    float* sa = reinterpret_cast<float*>(sm + lay.sa);
    float* sL = reinterpret_cast<float*>(sm + lay.sL);
    float* sbias = reinterpret_cast<float*>(sm + lay.sbias);
    int* spid = reinterpret_cast<int*>(sm + lay.spid);
    float* ss = reinterpret_cast<float*>(sm + lay.ss);
    float* sgh = reinterpret_cast<float*>(sm + lay.sgh);
    float* sgall = reinterpret_cast<float*>(sm + lay.sgall);
    unsigned long long* sred = reinterpret_cast<unsigned long long*>(sm + lay.sred);
    int* stok = reinterpret_cast<int*>(sm + lay.stok);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(sm + lay.misc);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, tid = threadIdx.x;
    const bool full_vocab = p.K == 0;
    const int grid = gridDim.x, cta = blockIdx.x;

    // this CTA's correction slice: fc2 rows [w0, w1) or pool entries [w0, w1)
    const long long work = full_vocab ? (long long)V : (long long)B * p.K;
    const long long w0 = min(work, (long long)cta * p.seg);
    const long long w1 = min(work, w0 + p.seg);
    const int nw = (int)(w1 - w0);
    const int n_chunks = (nw + kRows - 1) / kRows;
    // the requests of the slice (a pool slice covers consecutive requests)
    const int rb0 = full_vocab || nw == 0 ? 0 : (int)(w0 / p.K);
    const int nra = full_vocab ? 1 : nw == 0 ? 0 : (int)((w1 - 1) / p.K) - rb0 + 1;
    const int n_share = full_vocab ? n_chunks / kShareDiv : 0;
    const int n_static = n_chunks - n_share;
    // GRU units and fc1 rows of this CTA
    const int j0 = min(G, cta * p.jpc), jn = min(G, j0 + p.jpc) - j0;
    const int f0 = min(F, cta * p.fpc), fn = min(F, f0 + p.fpc) - f0;

    if (tid == 0) {
        for (int s = 0; s < p.n_slots; ++s) {
            tc::mbar_init(full0 + 8 * s, 1);
            tc::mbar_init(empty0 + 8 * s, 1);
        }
        *abort_flag = 0;
        tc::fence_barrier_init();
        tc::fence_proxy_async();
    }
    __syncthreads();
    pdl_trigger();

    // ------------------------------------------------------------------ producer
    // Four lanes issue the ring's bulk copies in lockstep rounds: each round
    // hands consecutive slot numbers to the lanes that have an item, so every
    // lane keeps the same count of slots issued while the copies (and the
    // waits for free slots) of a round proceed in parallel.
    if (warp == kConsumerWarps) {
        int* sqid = reinterpret_cast<int*>(sm + lay.sqid);
        if (!full_vocab) {
            pdl_wait();  // the pool ids come from the previous kernel
            // the slice's pool ids, read from global memory once (not before every copy)
            for (int i = lane; i < nw; i += 32) sqid[i] = p.pool[w0 + i];
            __syncwarp();
        }
        if (lane >= kProducerLanes) return;
        constexpr unsigned kLanes = (1u << kProducerLanes) - 1u;
        const uint64_t pol = full_vocab ? tc::policy_evict_normal() : tc::policy_evict_last();
        // Full vocabulary: the walk reverses every step, so the rows a step reads
        // last are the next step's first. The walk's head is loaded evict-first
        // and its last kKeepTenths/10 (the shared tails included) at normal
        // priority, so that the head's misses evict one another rather than the
        // tail a slower CTA has yet to re-read (B=1 K0: 883.7 -> 877.6 us per block).
        const uint64_t pol_head = tc::policy_evict_first();
        const int n_head = n_static - max(0, (kKeepTenths * n_chunks + 5) / 10 - n_share);
        uint64_t pol_fc2 = pol;
        int q = 0;        // slots issued so far (same in every lane)
        bool ok = true;   // same in every lane
        // fill slot number qq with rows/entries [item0, item0 + nr); item0 < 0: end of a step
        auto issue_at = [&](int qq, long long item0, int nr) {
            const int slot = qq % p.n_slots;
            if (!tc::mbar_wait(empty0 + 8 * slot, (uint32_t)(((qq / p.n_slots) & 1) ^ 1), abort_flag, p.err))
                return false;
            srow[slot] = (int)item0;
            if (item0 < 0) {
                tc::mbar_arrive(full0 + 8 * slot);
            } else {
                const uint32_t dst = tc::smem_u32(ring + (size_t)slot * slot_bytes);
                tc::mbar_arrive_expect_tx(full0 + 8 * slot, (uint32_t)(nr * row_bytes));
                if (full_vocab) {
                    tc::bulk_load(dst, p.fc2 + (size_t)item0 * F, (uint32_t)(nr * row_bytes), full0 + 8 * slot, pol_fc2);
                } else {
                    for (int r = 0; r < nr; ++r)
                        tc::bulk_load(dst + (uint32_t)(r * row_bytes), p.fc2 + (size_t)sqid[item0 - w0 + r] * F,
                                      (uint32_t)row_bytes, full0 + 8 * slot, pol);
                }
            }
            return true;
        };
        auto round = [&](bool have, long long item0, int nr) {
            const unsigned vm = __ballot_sync(kLanes, have);
            bool mine = true;
            if (have) mine = issue_at(q + __popc(vm & ((1u << lane) - 1u)), item0, nr);
            q += __popc(vm);
            ok = __all_sync(kLanes, mine) != 0;
        };
        if (p.resident) {
            // pool rows loaded once: chunk c stays in slot c for the whole launch
            for (int c0 = 0; c0 < n_chunks && ok; c0 += kProducerLanes) {
                const int c = c0 + lane;
                round(c < n_chunks, w0 + c * kRows, min(kRows, nw - c * kRows));
            }
        } else if (!full_vocab) {
            // pools: step k's chunks are sequence numbers (k-1) n_chunks + i,
            // and lane l issues i = l, l + 4, ... on its own, so a slot that
            // frees early is refilled without waiting for the other lanes
            for (int k = 1; k <= p.n_corr && ok && !*abort_flag; ++k) {
                const bool fwd = (k & 1) != 0;
                for (int i = lane; i < n_chunks && ok; i += kProducerLanes) {
                    const int c = fwd ? i : n_chunks - 1 - i;
                    ok = issue_at((k - 1) * n_chunks + i, w0 + c * kRows, min(kRows, nw - c * kRows));
                }
            }
            q = p.n_corr * n_chunks;
        } else {
            const unsigned total_claims = (unsigned)((p.seg / kRows) / kShareDiv + 1) * (unsigned)grid;
            for (int k = 1; k <= p.n_corr; ++k) {
                ok = __all_sync(kLanes, ok && !*abort_flag) != 0;
                if (!ok) break;
                const bool fwd = (k & 1) != 0;
                for (int ci0 = 0; ci0 < n_static && ok; ci0 += kProducerLanes) {
                    const int ci = ci0 + lane;
                    const int c = fwd ? ci : n_chunks - 1 - ci;
                    pol_fc2 = ci < n_head ? pol_head : pol;
                    round(ci < n_static, w0 + c * kRows, min(kRows, nw - c * kRows));
                }
                if (full_vocab && ok) {
                    // shared tails of every slice, kProducerLanes chunks per claim;
                    // the counters are cleared by the run's first kernel
                    if (k == 1) pdl_wait();
                    pol_fc2 = pol;
                    unsigned* ctr = p.claim + k;
                    unsigned base = lane == 0 ? atomicAdd(ctr, (unsigned)kProducerLanes) : 0u;
                    base = __shfl_sync(kLanes, base, 0);
                    while (base < total_claims && ok) {
                        unsigned next = total_claims;  // the next claim is requested before this one is issued
                        if (lane == 0 && base + kProducerLanes < total_claims)
                            next = atomicAdd(ctr, (unsigned)kProducerLanes);
                        const unsigned i = base + (unsigned)lane;
                        bool have = false;
                        long long item0 = 0;
                        int nr = 0;
                        if (i < total_claims) {
                            const int owner = (int)(i % (unsigned)grid), j = (int)(i / (unsigned)grid);
                            const long long ow0 = min(work, (long long)owner * p.seg);
                            const int onw = (int)(min(work, ow0 + p.seg) - ow0);
                            const int och = (onw + kRows - 1) / kRows, osh = och / kShareDiv;
                            if (j < osh) {
                                const int oc = fwd ? och - osh + j : osh - 1 - j;
                                have = true;
                                item0 = ow0 + oc * kRows;
                                nr = min(kRows, onw - oc * kRows);
                            }
                        }
                        round(have, item0, nr);
                        base = __shfl_sync(kLanes, next, 0);
                    }
                }
                // full vocabulary: the per-step count of a CTA's chunks varies with
                // the claims, so an end marker per consumer warp closes the step
                // (pools: every step has n_chunks, and the consumers count them)
                if (full_vocab)
                    for (int e0 = 0; e0 < p.n_cons && ok; e0 += kProducerLanes) round(e0 + lane < p.n_cons, -1, 0);
            }
        }
        if (lane != 0) return;
        // the copies issued last must land before the block may exit
        for (int i = q > p.n_slots ? q - p.n_slots : 0; i < q; ++i) {
            const unsigned long long t1 = tc::globaltimer();
            while (!tc::mbar_try_wait(full0 + 8 * (i % p.n_slots), (uint32_t)((i / p.n_slots) & 1)) &&
                   tc::globaltimer() - t1 < 2000000ull) {
            }
        }
        return;
    }

    // ------------------------------------------------------------------ consumers
    bool failed = false;
    const uint64_t pol_keep = tc::policy_evict_last();
    // resident weights: this CTA's fc1 rows and (pools) its units' W_hh rows
    {
        const int per_row = G / 8;  // 16-byte pieces of a row
        for (int i = tid; i < (p.wh_res ? 3 * jn * per_row : 0); i += kConsumerWarps * 32) {
            const int rr = i / per_row, e = (i % per_row) * 8;
            const int gate = rr / jn, jj = rr % jn;
            cp_async16((void*)(swhh + ((size_t)gate * p.jpc + jj) * RS + e),
                       p.w_hh + ((size_t)gate * G + j0 + jj) * G + e);
        }
        for (int i = tid; i < fn * per_row; i += kConsumerWarps * 32) {
            const int rr = i / per_row, e = (i % per_row) * 8;
            cp_async16((void*)(sfc1 + (size_t)rr * RS + e), p.fc1 + (size_t)(f0 + rr) * G + e);
        }
        cp_async_commit();
        // zero padding after every resident row and state row (a tensor-core
        // k-step may run past G when G is not a multiple of 16)
        __nv_bfloat16* zw = reinterpret_cast<__nv_bfloat16*>(sm + lay.swhh);
        __nv_bfloat16* zf = reinterpret_cast<__nv_bfloat16*>(sm + lay.sfc1);
        for (int i = tid; i < (p.wh_res ? 3 * p.jpc : 0) + p.fpc + B; i += kConsumerWarps * 32) {
            const int n1 = p.wh_res ? 3 * p.jpc : 0;
            if (i < n1) *reinterpret_cast<uint4*>(zw + (size_t)i * RS + G) = make_uint4(0u, 0u, 0u, 0u);
            else if (i < n1 + p.fpc) *reinterpret_cast<uint4*>(zf + (size_t)(i - n1) * RS + G) = make_uint4(0u, 0u, 0u, 0u);
            else {
                float4* z = reinterpret_cast<float4*>(sh + (size_t)(i - n1 - p.fpc) * SS + G);
                z[0] = make_float4(0.f, 0.f, 0.f, 0.f);
                z[1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    if (full_vocab)
        for (int i = tid; i < nw; i += kConsumerWarps * 32) sbias[i] = __bfloat162float(p.bias[w0 + i]);

    // trace stamps (thread 0): slot s = time at the end of phase s
    unsigned long long* tr = p.trace ? p.trace + (size_t)cta * DOMINO_TRACE_SLOTS : nullptr;
    int ts = 0;
    auto stamp = [&]() {
        if (tr && tid == 0 && ts < DOMINO_TRACE_SLOTS) tr[ts] = tc::globaltimer();
        ++ts;
    };
    stamp();  // 0

    // token of GRU update u (1..14) for request b, from p_u; checked
    auto fed_token = [&](int b, int u, int p_u) {
        int t = p.forced ? p.forced[(size_t)b * kProposals + (u - 1)] : p_u;
        if (t < 0 || t >= V) {
            if (cta == 0) {
                p.bad[b] = 1;
                atomicOr(p.err, kErrBadToken);
            }
            t = 0;
        }
        return t;
    };

    // ---- projector items of this CTA: its fc1 rows (item < fn, k > 0) and
    // its units' W_hh rows (item >= fn, when gh is set).  With all of them
    // resident (pools) they run on the tensor cores (tc_pass).  Otherwise
    // (the full vocabulary, W_hh rows read from L2) a warp takes two
    // consecutive items with the rows in registers, forms the lane-partial
    // dots with every request's state (streamed from shared memory once per
    // chunk for both rows), reduces all of them in one transposed butterfly
    // and finishes them on as many lanes at once; the fc1 pairs run on warps
    // of their own, the W_hh pairs (requested as early as possible) on the
    // others.  xg_k: where the hidden-side products are published as well
    // (one request), or null.
    auto project = [&](int k, bool gh, bool pub_a, unsigned tag_a, unsigned long long* xa_k, unsigned long long* xg_k) {
        const int nf = k > 0 ? fn : 0;
        const int n_items = nf + (gh ? 3 * jn : 0);
        auto load = [&](int it, Row4<NC>& r) {
            if (it < nf) {
                r.load_smem(sfc1 + (size_t)it * RS, G, lane);
            } else {
                const int g = it - nf, gate = g / jn, jj = g % jn;
                if (p.wh_res) r.load_smem(swhh + ((size_t)gate * p.jpc + jj) * RS, G, lane);
                else r.load_global(p.w_hh + ((size_t)gate * G + j0 + jj) * G, G, lane, pol_keep);
            }
        };
        auto finish = [&](int it, int b, float v) {
            if (it < nf) {
                const int f = f0 + it;
                const float z = v + ss[(b * kProposals + k) * p.fpc + it];
                if (pub_a) st_relaxed_u64(xa_k + (size_t)b * F + f, tagged(z * sigmoidf_(z), tag_a));
                if (p.dbg_z) p.dbg_z[((size_t)b * kCorrected + (k - 1)) * F + f] = z;
            } else {
                const int g = it - nf, gate = g / jn, jj = g % jn;
                sgh[(b * 3 + gate) * p.jpc + jj] = v;
                if (xg_k && pub_a) st_relaxed_u64(xg_k + (size_t)gate * G + j0 + jj, tagged(v, tag_a));
            }
        };
        // items [lo, hi), one (TWO = false) or two per warp
        // items [lo, hi) on warps [wa, wa + nwa), one (TWO = false) or two per warp
        auto pass = [&](auto two_c, int lo, int hi, int wa, int nwa) {
            constexpr bool TWO = decltype(two_c)::value;
            constexpr int NR = TWO ? 2 : 1;
            constexpr int NV = NR * MB;  // v[r * MB + b]: row r of the warp's items, request b
            if (warp < wa || warp >= wa + nwa) return;  // the same for the whole warp
            for (int it0 = lo + NR * (warp - wa); it0 < hi; it0 += NR * nwa) {
                const bool two = TWO && it0 + 1 < hi;
                Row4<NC> r[NR];
                load(it0, r[0]);
                if (TWO) {
                    if (two) load(it0 + 1, r[NR - 1]);
                    else r[NR - 1].zero();
                }
                float v[NV];
#pragma unroll
                for (int i = 0; i < NV; ++i) v[i] = 0.f;
#pragma unroll
                for (int c = 0; c < NC; ++c) {
                    float w[NR][4];
#pragma unroll
                    for (int rr = 0; rr < NR; ++rr) {
                        bf16x2_to_f32(r[rr].q[c].x, w[rr][0], w[rr][1]);
                        bf16x2_to_f32(r[rr].q[c].y, w[rr][2], w[rr][3]);
                    }
#pragma unroll
                    for (int b = 0; b < MB; ++b) {
                        if (b < B) {
                            const float4 x = vec4(sh + b * SS, c, G, lane);
#pragma unroll
                            for (int rr = 0; rr < NR; ++rr)
                                v[rr * MB + b] = fmaf(w[rr][0], x.x,
                                                      fmaf(w[rr][1], x.y,
                                                           fmaf(w[rr][2], x.z, fmaf(w[rr][3], x.w, v[rr * MB + b]))));
                        }
                    }
                }
                const float t = warp_sum_tr<NV>(v, lane);
                if (tr_reporter<NV>(lane)) {
                    const int idx = tr_index<NV>(lane), rr = idx / MB, b = idx % MB;
                    if (b < B && (rr == 0 || two)) finish(it0 + rr, b, t);
                }
            }
        };
        // All rows resident: the items as 16-row tiles on the tensor cores
        // (mma m16n8k16, one column per request).  A warp takes a (tile,
        // k-range) unit: the rows come from shared memory with ldmatrix, the
        // state as bf16 leading parts and remainders (two products per
        // k-step, fp32 accumulation); the units' partial tiles are summed
        // through shared memory and finished one output per thread.
        auto tc_pass = [&]() {
            if (n_items == 0) return;  // the same in every warp of the CTA
            const int mt = (n_items + 15) / 16;
            const int nkr = mt >= kConsumerWarps ? 1 : kConsumerWarps / mt;
            const int ks = (G + 15) / 16;
            const int mi = lane >> 3, rl = (lane & 7) + (mi & 1) * 8, kofs = (mi >> 1) * 8;
            const float* xrow = sh + (size_t)min(lane >> 2, B - 1) * SS + (lane & 3) * 2;
            for (int u = warp; u < mt * nkr; u += kConsumerWarps) {
                const int m = u / nkr, r = u % nkr;
                const int it = min(m * 16 + rl, n_items - 1);  // rows past the items repeat the last one
                const __nv_bfloat16* arow;
                if (it < nf) {
                    arow = sfc1 + (size_t)it * RS;
                } else {
                    const int g = it - nf, gate = g / jn, jj = g % jn;
                    arow = swhh + ((size_t)gate * p.jpc + jj) * RS;
                }
                const uint32_t abase = tc::smem_u32(arow + kofs);
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
                float* pt = spart + (size_t)u * 128;
                const int row = lane >> 2, col = (lane & 3) * 2;
                *reinterpret_cast<float2*>(pt + row * 8 + col) = make_float2(d0[0] + d1[0], d0[1] + d1[1]);
                *reinterpret_cast<float2*>(pt + (row + 8) * 8 + col) = make_float2(d0[2] + d1[2], d0[3] + d1[3]);
            }
            cons_sync();
            for (int o = tid; o < mt * 128; o += kConsumerWarps * 32) {
                const int m = o >> 7, row = (o >> 3) & 15, col = o & 7, it = m * 16 + row;
                if (it < n_items && col < B) {
                    const float* pt = spart + (size_t)m * nkr * 128 + row * 8 + col;
                    float v = 0.f;
                    for (int r = 0; r < nkr; ++r) v += pt[r * 128];
                    finish(it, col, v);
                }
            }
        };
        if constexpr (MB > 1) {
            tc_pass();  // batches run only on pools, whose rows are all resident
        } else {
            if (p.wh_res) {
                tc_pass();
            } else {
                // fc1 pairs on warps of their own, so that no activation waits
                // for a W_hh row's L2 read (B=1 K0: 899 -> 879 us per block)
                const int fw = nf == 0 ? 0 : min(kConsumerWarps - 1, (nf + 1) / 2);
                pass(std::true_type{}, 0, nf, 0, fw > 0 ? fw : 1);
                pass(std::true_type{}, nf, n_items, fw, kConsumerWarps - fw);
            }
        }
    };

    // ---- update u of this CTA's units: h[j] = GRU(token-table row, kept
    // hidden-side products, h_prev[j]) for j in [j0, j0+jn); published
    auto update_own = [&](int u, bool pub, unsigned tag, unsigned long long* xh_u) {
        for (int i = tid; i < B * jn; i += kConsumerWarps * 32) {
            const int b = i / jn, jj = i % jn, j = j0 + jj;
            const float* gi = p.gi_table + (size_t)stok[b] * 3 * G + j;
            const float gr = __ldg(gi), gz = __ldg(gi + G), gn = __ldg(gi + 2 * G);
            const float* gh = sgh + b * 3 * p.jpc + jj;
            const float r = sigmoidf_(gr + gh[0]);
            const float zg = sigmoidf_(gz + gh[p.jpc]);
            const float n = tanhf(gn + r * gh[2 * p.jpc]);
            const float h = (1.f - zg) * n + zg * sh[b * SS + j];
            if (pub) st_relaxed_u64(xh_u + (size_t)b * G + j, tagged(h, tag));
            if (p.dbg_h) p.dbg_h[((size_t)b * kProposals + u) * G + j] = h;
        }
    };
    // ---- `count` tagged words, word i at addr(i): four loads per thread in
    // flight (eight for more than four requests); the words that do not carry
    // the tag yet are read again together (one L2 round trip per retry round
    // for all of them), with a short back-off between rounds; bounded.
    // consume(i, word) for each.
    auto gather = [&](int count, auto addr, unsigned tag, int mode, auto consume) {
        constexpr int kNT = kConsumerWarps * 32, kDepth = MB > 4 ? 8 : 4;
        for (int base = 0; base < count; base += kDepth * kNT) {
            unsigned long long w[kDepth];
            const unsigned long long* pw[kDepth];  // addresses, formed once
            unsigned miss = 0u;
#pragma unroll
            for (int e = 0; e < kDepth; ++e) {
                const int i = base + e * kNT + tid;
                w[e] = 0ull;
                pw[e] = nullptr;
                if (i < count) {
                    pw[e] = addr(i);
                    w[e] = ld_relaxed_u64(pw[e]);
                    miss |= 1u << e;
                }
            }
            unsigned long long t0 = 0ull;
            for (unsigned round = 0;; ++round) {
#pragma unroll
                for (int e = 0; e < kDepth; ++e)
                    if (((miss >> e) & 1u) && has_tag(w[e], tag, mode)) miss &= ~(1u << e);
                if (!miss) break;
                if ((round & 15u) == 15u) {  // the abort flag and the clock, every 16 rounds
                    if (*abort_flag) {
                        failed = true;
                        break;
                    }
                    const unsigned long long now = tc::globaltimer();
                    if (t0 == 0ull) {
                        t0 = now;
                    } else if (now - t0 > tc::kWaitLimitNs) {
                        *abort_flag = 1;
                        atomicOr(p.err, kErrTimeout);
                        failed = true;
                        break;
                    }
                }
                __nanosleep(32);  // every waiting thread of every CTA polls L2: keep its request rate down
#pragma unroll
                for (int e = 0; e < kDepth; ++e)
                    if ((miss >> e) & 1u) w[e] = ld_relaxed_u64(pw[e]);
            }
#pragma unroll
            for (int e = 0; e < kDepth; ++e) {
                const int i = base + e * kNT + tid;
                if (i < count && !((miss >> e) & 1u)) consume(i, w[e]);
            }
        }
    };
    // n tagged fp32 payloads into dst
    auto read_tagged = [&](const unsigned long long* src, float* dst, int n, unsigned tag) {
        gather(
            n, [&](int i) { return src + i; }, tag, 0,
            [&](int i, unsigned long long w) { dst[i] = __uint_as_float((unsigned)w); });
    };
    // ---- one request, update u of every unit from the token-table row and
    // every unit's hidden-side products (sgall), in place: each element is
    // read and written by one thread
    auto update_all = [&](int u) {
        constexpr int kNT = kConsumerWarps * 32;
        const float* gi = p.gi_table + (size_t)stok[0] * 3 * G;
        for (int j0_ = tid; j0_ < G; j0_ += 4 * kNT) {
            float gr[4], gz[4], gn[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0_ + e * kNT;
                if (j < G) {
                    gr[e] = __ldg(gi + j);
                    gz[e] = __ldg(gi + G + j);
                    gn[e] = __ldg(gi + 2 * G + j);
                }
            }
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0_ + e * kNT;
                if (j < G) {
                    const float r = sigmoidf_(gr[e] + sgall[j]);
                    const float zg = sigmoidf_(gz[e] + sgall[G + j]);
                    const float n = tanhf(gn[e] + r * sgall[2 * G + j]);
                    const float h = (1.f - zg) * n + zg * sh[j];
                    sh[j] = h;
                    if (p.dbg_h && j >= j0 && j < j0 + jn) p.dbg_h[(size_t)u * G + j] = h;
                }
            }
        }
    };
    // ---- the whole state after update u, from every CTA's published units
    // (word i of the exchange is element i % G of request i / G; the quotient
    // by a multiply-high with ceil(2^32 / G), exact for i < 2^32 / G)
    const unsigned g_magic = (unsigned)((0x100000000ull + (unsigned)G - 1u) / (unsigned)G);
    auto read_state = [&](unsigned tag, const unsigned long long* xh_u) {
        gather(
            B * G, [&](int i) { return xh_u + i; }, tag, 0,
            [&](int i, unsigned long long w) {
                const int b = (int)__umulhi((unsigned)i, g_magic);
                sh[b * SS + (i - b * G)] = __uint_as_float((unsigned)w);
            });
    };

    // ---- seed update 0 (h_{-1} = 0): the verified token only, independent
    // of the previous kernel; every CTA computes the whole state
    if (tid < B) {
        int t = p.verified[tid];
        if (t < 0 || t >= V) {
            if (cta == 0) {
                p.bad[tid] = 1;
                atomicOr(p.err, kErrBadToken);
            }
            t = 0;
        }
        stok[tid] = t;
    }
    cons_sync();
    for (int i = tid; i < B * G; i += kConsumerWarps * 32) {
        const int b = i / G, j = i % G;
        const float* gi = p.gi_table + (size_t)stok[b] * 3 * G + j;
        // h = 0: the reset gate multiplies W_hn h = 0 and drops out
        const float zg = sigmoidf_(__ldg(gi + G));
        const float n = tanhf(__ldg(gi + 2 * G));
        const float h = (1.f - zg) * n;
        sh[b * SS + j] = h;
        if (p.dbg_h && j >= j0 && j < j0 + jn) p.dbg_h[((size_t)b * kProposals + 0) * G + j] = h;
    }
    cp_async_wait_all();
    cons_sync();
    project(0, true, false, 0u, nullptr, nullptr);  // hidden-side products of update 1
    stamp();  // 1
    pdl_wait();  // base logits, p_1 and the pool are ready; the run counter is bumped
    const unsigned ep16 = *p.epoch * 16u;
    int pub = 0;  // publications so far (for the timeout test hook)
    auto publish_ok = [&]() { return !(cta == 0 && ++pub == p.drop_at); };
    // the buffers of update u / step k
    auto xh_of = [&](int u) { return p.xh + (size_t)(u & 1) * kLLMaxBatch * G; };
    auto xa_of = [&](int k) { return p.xa + (size_t)(k & 1) * kLLMaxBatch * F; };
    auto xbest_of = [&](int k) { return p.xbest + (size_t)(k & 1) * grid * kLLMaxBatch; };
    auto xg_of = [&](int k) { return p.xg + (size_t)(k & 1) * 3 * G; };
    if (!full_vocab)
        for (int i = tid; i < nw; i += kConsumerWarps * 32) {
            const int v = p.pool[w0 + i];
            spid[i] = v;
            sbias[i] = __bfloat162float(p.bias[v]);
            // the candidates' token-table rows: every fed token of a pool run is one of them
            if (p.pin_gi) tc::bulk_prefetch_l2(p.gi_table + (size_t)v * 3 * G, (uint32_t)(3 * G * 4), pol_keep);
        }
    // this CTA's entries of s (they may come from the previous kernel)
    for (int i = tid; i < B * kProposals * fn; i += kConsumerWarps * 32) {
        const int b = i / (kProposals * fn), r = i % (kProposals * fn), j = r / fn, f = r % fn;
        ss[(b * kProposals + j) * p.fpc + f] = __bfloat162float(p.s[((size_t)b * kProposals + j) * F + f0 + f]);
    }
    // update 1 consumes p_1 (the LM-head's argmax of base row 1)
    if (tid < B) stok[tid] = fed_token(tid, 1, (int)key_index(__ldcg(&p.keys[(size_t)tid * kBlock])));
    // per-request best of this CTA's rows (sbest_c) and of every CTA's bests
    // (sbest_x), folded with shared-memory atomics; cleared after each read
    unsigned long long* sbest_c = sred;
    unsigned long long* sbest_x = sred + kLLMaxBatch;
    if (tid < 2 * kLLMaxBatch) sred[tid] = 0ull;
    cons_sync();
    update_own(1, publish_ok(), ep16 + 1, xh_of(1));
    cons_sync();  // every read of the old state is done
    read_state(ep16 + 1, xh_of(1));
    if (cons_sync_or(failed)) return;
    stamp();  // 2

    // correction: lane l holds elements (l + 32c)*8 .. +7 of a row (16-byte
    // shared loads of the ring's rows); the activations of one request in registers
    constexpr int NCH = (NC + 1) / 2;  // 256-element chunks
    float areg[NCH][8];
    int areg_b = -1;
    auto load_areg = [&](int b) {
#pragma unroll
        for (int cc = 0; cc < NCH; ++cc) {
            const int e = (lane + 32 * cc) * 8;
            if (e < F) lds8(sa + (b - rb0) * F + e, areg[cc]);
        }
        areg_b = b;
    };
    // the rows of one slot (entries item0 .. item0+nr-1) dotted with the
    // activations of their request(s); lane-partial sums in part[]
    auto slot_dots = [&](const __nv_bfloat16* srows, long long item0, int nr, float* part) {
        const int bl0 = full_vocab ? 0 : (int)(item0 / p.K);
        const int bl1 = full_vocab ? 0 : (int)((item0 + nr - 1) / p.K);
        if (bl0 == bl1) {
            if (bl0 != areg_b) load_areg(bl0);
            // all rows of the slot, also those past nr (in the slot's memory;
            // their totals are not used): the four 16-byte loads of a chunk
            // are issued together, then their products
            float acc[kRows][2];
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) acc[rr][0] = acc[rr][1] = 0.f;
#pragma unroll
            for (int cc = 0; cc < NCH; ++cc) {
                const int e = (lane + 32 * cc) * 8;
                if (e < F) {
                    uint4 raw[kRows];
#pragma unroll
                    for (int rr = 0; rr < kRows; ++rr) raw[rr] = *reinterpret_cast<const uint4*>(srows + (size_t)rr * F + e);
#pragma unroll
                    for (int rr = 0; rr < kRows; ++rr) {
                        float wv[8];
                        bf16x2_to_f32(raw[rr].x, wv[0], wv[1]);
                        bf16x2_to_f32(raw[rr].y, wv[2], wv[3]);
                        bf16x2_to_f32(raw[rr].z, wv[4], wv[5]);
                        bf16x2_to_f32(raw[rr].w, wv[6], wv[7]);
#pragma unroll
                        for (int i = 0; i < 8; i += 2) {
                            acc[rr][0] = fmaf(wv[i], areg[cc][i], acc[rr][0]);
                            acc[rr][1] = fmaf(wv[i + 1], areg[cc][i + 1], acc[rr][1]);
                        }
                    }
                }
            }
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) part[rr] = acc[rr][0] + acc[rr][1];
        } else {  // a slot across a request boundary of the pool
#pragma unroll
            for (int rr = 0; rr < kRows; ++rr) {
                part[rr] = 0.f;
                if (rr < nr) {
                    const int bl = (int)((item0 + rr) / p.K);
                    if (bl != areg_b) load_areg(bl);
                    float a0 = 0.f, a1 = 0.f;
#pragma unroll
                    for (int cc = 0; cc < NCH; ++cc) {
                        const int e = (lane + 32 * cc) * 8;
                        if (e < F) {
                            float wv[8];
                            lds8(srows + (size_t)rr * F + e, wv);
#pragma unroll
                            for (int i = 0; i < 8; i += 2) {
                                a0 = fmaf(wv[i], areg[cc][i], a0);
                                a1 = fmaf(wv[i + 1], areg[cc][i + 1], a1);
                            }
                        }
                    }
                    part[rr] = a0 + a1;
                }
            }
        }
    };
    // best word of an exchange: orderable value, then ~id (lower id wins), then the step
    auto best_key = [](float c, int v) {
        return ((unsigned long long)ord_f32(c) << 32) |
               ((unsigned long long)(~(uint32_t)v & 0x3FFFFu) << kBestIdShift);
    };

    const int rsel = ((lane >> 4) & 1) * 2 + ((lane >> 3) & 1);  // the slot row this lane finishes
    int qw = warp;  // ring: sequence number of this warp's next slot (slot q is consumed by warp q % n_cons)
    for (int k = 1; k <= p.n_corr; ++k) {
        const unsigned tag_k = ep16 + (unsigned)k;
        const bool fwd = (k & 1) != 0;
        // rows of the slice this CTA finishes itself (full vocabulary: the
        // static part, whose end alternates with the walking direction)
        const int st_lo = full_vocab ? (fwd ? 0 : n_share * kRows) : 0;
        const int st_hi = full_vocab ? (fwd ? min(nw, n_static * kRows) : nw) : nw;
        for (int r = st_lo + tid; r < st_hi; r += kConsumerWarps * 32) {
            const long long item = w0 + r;
            const int b = full_vocab ? 0 : (int)(item / p.K);
            const int v = full_vocab ? (int)item : spid[r];
            cp_async4(&sL[r], p.L + ((size_t)b * kBlock + kRowOffset + k) * V + v);
        }
        cp_async_commit();

        // ---- P_k: the projector slice (published), and the next update's
        // hidden-side products of this CTA's units (kept)
        project(k, k < p.n_corr, publish_ok(), tag_k, xa_of(k), MB == 1 && k < p.n_corr ? xg_of(k) : nullptr);
        stamp();  // 3 + 4(k-1): projector published
        // ---- C_k: all activations, then this CTA's slice
        read_tagged(xa_of(k) + (size_t)rb0 * F, sa, nra * F, tag_k);
        cp_async_wait_all();
        if (cons_sync_or(failed)) return;
        areg_b = -1;
        stamp();  // 4 + 4(k-1): activations in
        unsigned long long m[MB];  // this lane's best per request of the rows it finishes
#pragma unroll
        for (int b = 0; b < MB; ++b) m[b] = 0ull;
        // a small resident slice (at most two rows per warp): one row per warp
        // at a time, so that every warp shares the dot products
        const bool row_mode = p.resident && nw <= 2 * kConsumerWarps;
        if (row_mode) {
            for (int rr = warp; rr < nw; rr += kConsumerWarps) {
                const int slot = rr / kRows;
                if (k == 1 && !tc::mbar_wait(full0 + 8 * slot, 0u, abort_flag, p.err)) {
                    failed = true;
                    break;
                }
                const int item = (int)w0 + rr;
                const int b = item / p.K;
                if (b != areg_b) load_areg(b);
                const __nv_bfloat16* row =
                    reinterpret_cast<const __nv_bfloat16*>(ring + (size_t)slot * slot_bytes) + (size_t)(rr % kRows) * F;
                float a0 = 0.f, a1 = 0.f;
#pragma unroll
                for (int cc = 0; cc < NCH; ++cc) {
                    const int e = (lane + 32 * cc) * 8;
                    if (e < F) {
                        float wv[8];
                        lds8(row + e, wv);
#pragma unroll
                        for (int i = 0; i < 8; i += 2) {
                            a0 = fmaf(wv[i], areg[cc][i], a0);
                            a1 = fmaf(wv[i + 1], areg[cc][i + 1], a1);
                        }
                    }
                }
                float tot = a0 + a1;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, o);
                if (lane == 0) {
                    const int v = spid[rr];
                    const float cv = tot + sbias[rr] + sL[rr];
                    const unsigned long long key = best_key(cv, v);
#pragma unroll
                    for (int bb = 0; bb < MB; ++bb)
                        if (bb == b) m[bb] = max(m[bb], key);
                    if (p.dbg_scores) p.dbg_scores[((size_t)b * kCorrected + (k - 1)) * p.K + item % p.K] = cv;
                }
            }
        }
        // one loop for both layouts (a single copy of the slot code): resident
        // pool rows, chunk c in slot c; or ring slots, slot q for warp q % n_cons
        if (!row_mode) {
            int c_res = warp;
            const bool active = p.resident ? true : warp < p.n_cons;
            while (active) {
                int slot;
                long long item0;
                if (p.resident) {
                    if (c_res >= n_chunks) break;
                    slot = c_res;
                    c_res += kConsumerWarps;
                    if (k == 1 && !tc::mbar_wait(full0 + 8 * slot, 0u, abort_flag, p.err)) {
                        failed = true;
                        break;
                    }
                    item0 = w0 + slot * kRows;
                } else {
                    if (!full_vocab && qw >= k * n_chunks) break;  // this warp's chunks of the step are done
                    const int q = qw;
                    qw += p.n_cons;
                    slot = q % p.n_slots;
                    if (!tc::mbar_wait(full0 + 8 * slot, (uint32_t)((q / p.n_slots) & 1), abort_flag, p.err)) {
                        failed = true;
                        break;
                    }
                    item0 = srow[slot];
                    if (item0 < 0) {  // end of this step for this warp
                        __syncwarp();
                        if (lane == 0) tc::mbar_arrive(empty0 + 8 * slot);
                        break;
                    }
                }
                const int nr = full_vocab ? min(kRows, V - (int)item0) : min(kRows, (int)(w1 - item0));
                const bool own = item0 >= w0 + st_lo && item0 < w0 + st_hi;
                // a shared row: this lane fetches its bias and base logit before the dots
                float tail = 0.f;
                if (!own && (lane & 7) == 0 && rsel < nr)
                    tail = __bfloat162float(p.bias[item0 + rsel]) +
                           __ldg(p.L + (size_t)(kRowOffset + k) * V + item0 + rsel);
                float part[kRows];
                slot_dots(reinterpret_cast<const __nv_bfloat16*>(ring + (size_t)slot * slot_bytes), item0, nr, part);
                if (!p.resident) {
                    __syncwarp();
                    if (lane == 0) tc::mbar_arrive(empty0 + 8 * slot);  // the slot is read
                }
                const float tot = warp_sum4(part[0], part[1], part[2], part[3], lane);
                if ((lane & 7) == 0 && rsel < nr) {
                    // finish the row: bias and base logit (own rows: staged; shared rows: fetched above)
                    const int item = (int)item0 + rsel, r = item - (int)w0;
                    const int b = full_vocab ? 0 : item / p.K;
                    const int v = full_vocab ? item : spid[r];
                    const float cv = own ? tot + sbias[r] + sL[r] : tot + tail;
                    const unsigned long long key = best_key(cv, v);
#pragma unroll
                    for (int bb = 0; bb < MB; ++bb)
                        if (bb == b) m[bb] = max(m[bb], key);
                    if (p.dbg_scores) {
                        if (full_vocab) p.dbg_scores[(size_t)(k - 1) * V + v] = cv;
                        else p.dbg_scores[((size_t)b * kCorrected + (k - 1)) * p.K + item % p.K] = cv;
                    }
                }
            }
        }
        // the requests of the slice (at most nra of them hold a value)
#pragma unroll
        for (int b = 0; b < MB; ++b) {
            if (b >= B) break;
            if (b < rb0 || b >= rb0 + nra) continue;
            const unsigned long long w = warp_max_u64(m[b]);
            if (lane == 0 && w) atomicMax(&sbest_c[b], w);
        }
        if (cons_sync_or(failed)) return;
        {
            const bool pub_b = publish_ok();
            if (tid < B) {
                if (pub_b)
                    st_relaxed_u64(xbest_of(k) + (size_t)cta * kLLMaxBatch + tid, sbest_c[tid] | (unsigned long long)k);
                sbest_c[tid] = 0ull;
            }
        }
        stamp();  // 5 + 4(k-1): best published
        if (k == p.n_corr && cta != 0) return;  // only CTA 0 reports the last step
        // one request: every unit's hidden-side products (published with the
        // activations, long since) while the other CTAs finish their bests
        if (MB == 1 && k < p.n_corr) read_tagged(xg_of(k), sgall, 3 * G, tag_k);
        // ---- X_k: every CTA's best of step k gives p_{k+1} for every request
        {
            const unsigned kk = (unsigned)k;
            const unsigned long long* xb = xbest_of(k);
            if (full_vocab || B == 1) {
                gather(
                    grid * B, [&](int i) { return xb + (size_t)(i / B) * kLLMaxBatch + i % B; }, kk, 1,
                    [&](int i, unsigned long long w) {
                        if (w > kBestTagMask) atomicMax(&sbest_x[i % B], w & ~(unsigned long long)kBestTagMask);
                    });
            } else {
                // pools of several requests: request b's entries lie in the
                // slices of CTAs b K / seg .. ((b+1) K - 1) / seg, at most `span` of them
                // (a shorter run repeats its last CTA: a harmless second max).
                // The CTAs past the pool's end have no entries, but their
                // (empty) words are read too: every CTA's word of a step is
                // read by every CTA, which is what keeps any CTA from running
                // two steps ahead of another (the exchanges' double buffering)
                const int span = (p.K + p.seg - 1) / p.seg + 1;
                const int n_cover = (B * p.K + p.seg - 1) / p.seg;
                gather(
                    B * span + (grid - n_cover),
                    [&](int i) {
                        if (i >= B * span) return xb + (size_t)(n_cover + i - B * span) * kLLMaxBatch;
                        const int b = i / span;  // b K < B * K <= grid * seg: 32-bit products
                        const int c_lo = b * p.K / p.seg;
                        const int c_hi = ((b + 1) * p.K - 1) / p.seg;
                        return xb + (size_t)min(c_lo + i % span, c_hi) * kLLMaxBatch + b;
                    },
                    kk, 1,
                    [&](int i, unsigned long long w) {
                        if (i < B * span && w > kBestTagMask)
                            atomicMax(&sbest_x[i / span], w & ~(unsigned long long)kBestTagMask);
                    });
            }
            cons_sync();
            if (tid < B) {
                const unsigned long long w = sbest_x[tid];
                sbest_x[tid] = 0ull;
                const int id = (int)(~(uint32_t)(w >> kBestIdShift) & 0x3FFFFu);
                if (cta == 0) p.keys[(size_t)tid * kBlock + k] = pack_key(unord_f32((uint32_t)(w >> 32)), (uint32_t)id);
                if (k < p.n_corr) stok[tid] = fed_token(tid, k + 1, id);
            }
        }
        if (cons_sync_or(failed)) return;
        if (k < p.n_corr) {
            if constexpr (MB == 1) {
                // ---- one request: the whole h_{k+1} here, no exchange
                update_all(k + 1);
                cons_sync();
            } else {
                // ---- this CTA's units of h_{k+1}, then (H_k) the whole state
                update_own(k + 1, publish_ok(), ep16 + (unsigned)(k + 1), xh_of(k + 1));
                cons_sync();  // every read of the old state is done
                read_state(ep16 + (unsigned)(k + 1), xh_of(k + 1));
                if (cons_sync_or(failed)) return;
            }
        }
        stamp();  // 6 + 4(k-1): next state built
    }
}

struct LLPlan {
    int seg, jpc, fpc, n_slots, n_cons, resident, wh_res, ra, smem;
};

LLPlan make_ll_plan(const domino_ctx* c, int B, int K) {
    const domino_config& g = c->cfg;
    const int grid = c->num_sms;
    const long long work = K == 0 ? (long long)g.V : (long long)B * K;
    LLPlan pl{};
    pl.seg = (int)((work + grid - 1) / grid);
    pl.seg = (pl.seg + kRows - 1) / kRows * kRows;
    pl.jpc = (g.G + grid - 1) / grid;
    pl.fpc = (g.F + grid - 1) / grid;
    const int slot_bytes = kRows * g.F * 2;
    int max_smem = 0;
    cudaDeviceGetAttribute(&max_smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, c->device);
    // over the full vocabulary the correction phase leaves the hidden-side
    // products plenty of time to read W_hh from L2, and the ring gets the room
    pl.wh_res = K > 0;
    // a slice of seg consecutive pool entries spans at most (seg - 1) / K + 2 requests
    pl.ra = K == 0 ? 1 : ((pl.seg - 1) / K + 2 < B ? (pl.seg - 1) / K + 2 : B);
    const LLLayout base(0, slot_bytes, g.G, g.F, pl.jpc, pl.fpc, pl.seg, B, pl.ra, pl.wh_res != 0);
    const int avail = max_smem - base.total - 1024;
    const int per_slot = slot_bytes + 20;
    const int chunks = pl.seg / kRows;
    if (K > 0 && chunks * per_slot <= avail && chunks <= kMaxSlots) {
        pl.resident = 1;  // pool rows loaded once
        pl.n_slots = chunks;
        pl.n_cons = kConsumerWarps;
    } else {
        int n = avail / per_slot;
        if (n > kMaxSlots) n = kMaxSlots;
        // consumer warps: the count whose multiple uses the most of the ring (at least 8);
        // slot q is consumed by warp q % n_cons
        int best = 0, nc = 0;
        for (int w = kConsumerWarps; w >= 8; --w)
            if (n / w * w > best) {
                best = n / w * w;
                nc = w;
            }
        pl.n_slots = best;
        pl.n_cons = nc;
    }
    if (pl.n_slots < 1) return pl;
    pl.smem = LLLayout(pl.n_slots, slot_bytes, g.G, g.F, pl.jpc, pl.fpc, pl.seg, B, pl.ra, pl.wh_res != 0).total;
    return pl;
}

}  // namespace

// One request over the full vocabulary, or pools of up to kLLMaxBatch
// requests; bf16 rows of at most 1024 elements, ids that fit the 18 id bits
// of an exchange word, and a slice that fits the per-CTA tables.
bool persist_ll_supported(const domino_ctx* c, const RunArgs& r) {
    const domino_config& g = c->cfg;
    if (g.dtype != DOMINO_DTYPE_BF16 || !c->xbest) return false;
    if (g.G > 1024 || g.F > 1024 || (g.G & 7) || (g.F & 7)) return false;
    if (g.V >= (1 << 18) || r.B < 1 || r.B > kLLMaxBatch) return false;
    if (r.K == 0 && r.B != 1) return false;
    const LLPlan pl = make_ll_plan(c, r.B, r.K);
    if (pl.seg > kMaxSeg || pl.jpc > 64 || pl.fpc > 64) return false;
    if (pl.resident) return pl.smem > 0;
    return pl.n_slots >= 8 && pl.smem > 0;
}

cudaError_t launch_persist_ll(domino_ctx* c, RunArgs& r) {
    const domino_config& g = c->cfg;
    const LLPlan pl = make_ll_plan(c, r.B, r.K);
    LLParams p;
    p.w_hh = (const __nv_bfloat16*)c->w_hh;
    p.fc1 = (const __nv_bfloat16*)c->fc1;
    p.fc2 = (const __nv_bfloat16*)c->fc2;
    p.bias = (const __nv_bfloat16*)c->bias;
    p.s = (const __nv_bfloat16*)r.s;
    p.gi_table = c->gi_table;
    p.verified = r.verified;
    p.forced = r.forced;
    p.pool = c->pool;
    p.L = c->L;
    p.keys = c->keys;
    p.bad = c->bad;
    p.err = c->err;
    p.claim = c->sync + kClaimCounters;
    p.epoch = c->sync + kRunEpochWord;
    p.xa = c->xa;
    p.xh = c->xh;
    p.xbest = c->xbest;
    p.xg = c->xg;
    p.dbg_h = r.dbg.h;
    p.dbg_z = r.dbg.z;
    p.dbg_scores = r.dbg.scores;
    p.trace = r.dbg.trace;
    p.B = r.B;
    p.K = r.K;
    p.V = g.V;
    p.G = g.G;
    p.F = g.F;
    p.n_corr = r.n_prop - 1;
    p.seg = pl.seg;
    p.jpc = pl.jpc;
    p.fpc = pl.fpc;
    p.n_slots = pl.n_slots;
    p.n_cons = pl.n_cons;
    p.ra = pl.ra;
    p.resident = pl.resident;
    p.wh_res = pl.wh_res;
    // the candidates' token-table rows stay in L2 when they are a modest share of it
    p.pin_gi = r.K > 0 && (long long)r.B * r.K * 3 * g.G * 4 <= (48ll << 20);
    p.drop_at = c->drop_barrier;  // one-shot test hook
    c->drop_barrier = 0;

    const int mx = g.G > g.F ? g.G : g.F;
    // rows of up to 256, 512 or 1024 elements; one, up to four or up to eight requests
    auto pick = [&](auto mb) -> void (*)(LLParams) {
        constexpr int MB = decltype(mb)::value;
        return mx <= 256 ? k_rollout_ll<2, MB> : mx <= 512 ? k_rollout_ll<4, MB> : k_rollout_ll<8, MB>;
    };
    void (*kern)(LLParams) = r.B == 1   ? pick(std::integral_constant<int, 1>{})
                             : r.B <= 4 ? pick(std::integral_constant<int, 4>{})
                                        : pick(std::integral_constant<int, kLLMaxBatch>{});
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, pl.smem);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(c->num_sms);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem;
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

}  // namespace domino
