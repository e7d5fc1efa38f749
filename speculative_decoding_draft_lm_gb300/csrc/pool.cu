// Block-shared candidate pool (page "Add correctness-first Domino support to
// DFlash V2", section "Design": one per-request pool shared by all steps of
// the block; page "support tensor-parallel Domino rollout", section
// "Implementation", stage B): the K token ids with the largest
//   score[b, v] = max_{i=1..15} L[b, i, v],
// ties at the cutoff to the lower id, stored in ascending id order.
//
// One thread-block cluster of R CTAs per request (R = 16, a non-portable
// cluster size, for a single row; else 8: at B = 8 eight clusters of 16
// measured slower than eight of 8, 51 us against 32 us).  Each CTA caches its
// contiguous slice of the vocabulary as 32-bit orderable keys in shared
// memory.  An exact radix select over three digit passes (11, 11, 10 bits)
// finds the K-th largest key T: each pass builds per-CTA histograms with
// warp-aggregated shared-memory atomics, merges them through distributed
// shared memory, and locates the digit holding the K-th key.  The ids with
// key > T and the lowest-id `need` ids with key == T are then written, each
// CTA at the offset given by the counts of the CTAs before it, so the pool
// comes out in ascending order without a sort.
//
// The same kernel runs the two passes of the tensor-parallel compact pool
// (page "feat: support tensor-parallel Domino rollout", section
// "Implementation", stage C), emulated on one GPU with P vocabulary shards:
//   pass 1, one row per (request, shard): the shard-local top-K of the
//           shard's scores [p*S, min(V, (p+1)*S)), S = ceil(V/P); a shard
//           shorter than K gives all its ids and pads its K slots with -1;
//   pass 2, one row per request: the top-K of the P*K candidates, whose
//           scores are gathered through their ids (padding ranks lowest).
// Both order by (score desc, id asc), and the candidates of a request are in
// ascending id order, so pass 2 returns exactly the direct pool.
#include <cooperative_groups.h>

#include "internal.h"

namespace cg = cooperative_groups;

namespace domino {

namespace {

constexpr int kRanksPortable = 8;  // CTAs per request (portable cluster size)
constexpr int kRanksWide = 16;     // non-portable cluster size for small batches
constexpr int kPoolThreads = 1024;
constexpr int kBins = 2048;

template <int R>
struct PoolShared {
    unsigned hist[kBins];
    unsigned merged[kBins / R];
    unsigned warp_tot[32];
    unsigned total;          // this CTA's merged-bin total / block scan total
    unsigned gt, eq;         // compaction counts of this CTA
    unsigned digit, rem;     // result of a pass, written by the CTA that found it
};

__device__ __forceinline__ unsigned block_scan_excl(unsigned x, unsigned* warp_tot, unsigned* total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    unsigned incl = x;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const unsigned y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const unsigned t = warp_tot[lane];
        unsigned ti = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const unsigned y = __shfl_up_sync(0xffffffffu, ti, o);
            if (lane >= o) ti += y;
        }
        warp_tot[lane] = ti - t;
        if (lane == 31) *total = ti;
    }
    __syncthreads();
    const unsigned r = warp_tot[warp] + incl - x;
    __syncthreads();
    return r;
}

// Row y of the grid: request b = y / shards, shard p = y % shards.
// cand == null: select among score[b*stride + p*shard_len + i], i < min(shard_len, V - p*shard_len),
//               writing vocabulary ids to pool[b*out_stride + p*K + j];
// cand != null: (shards == 1) select among the V candidates cand[b*V + i] (id -1 = none) by
//               score[b*stride + id], writing the candidate ids to pool[b*out_stride + j].
// Bounded to 32 registers so two CTAs share an SM: with 64 requests the 512
// CTAs then fit in one wave (B = 64, K = 2048: 1975 -> 1913 us per block).
template <int R>
__global__ void __launch_bounds__(kPoolThreads, 2) k_pool_cluster(const float* __restrict__ score, long long stride,
                                                                 const int32_t* __restrict__ cand, int shards,
                                                                 int shard_len, int32_t* __restrict__ pool,
                                                                 int out_stride, int V, int K, int chunk,
                                                                 const unsigned* __restrict__ ghist) {
    extern __shared__ __align__(16) uint8_t smem[];
    PoolShared<R>& S = *reinterpret_cast<PoolShared<R>*>(smem);
    unsigned* keys = reinterpret_cast<unsigned*>(smem + sizeof(PoolShared<R>));
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = (int)cluster.block_rank();
    const int b = blockIdx.y / shards, shard = blockIdx.y % shards;
    const int lane = threadIdx.x & 31;
    const int lo = shard * shard_len;
    const int n_row = min(shard_len, V - lo);
    const int Kr = min(K, n_row);
    const int v0 = min(n_row, rank * chunk), v1 = min(n_row, v0 + chunk), n = v1 - v0;

    // An ordinary launch (no early trigger): releasing the kernels after it
    // early let a chain of waiting batched kernels occupy the SMs and measured
    // slower (B=8 K2048: 0.75 -> 0.82 ms).
    const float* srow = score + (size_t)b * stride;
    const int32_t* crow = cand ? cand + (size_t)b * V + v0 : nullptr;
    if (cand) {
        // key 0 is below every finite score's key: padding never outranks a real id
        for (int i = threadIdx.x; i < n; i += kPoolThreads) {
            const int id = crow[i];
            keys[i] = id >= 0 ? ord_f32(srow[id]) : 0u;
        }
    } else {
        for (int i = threadIdx.x; i < n; i += kPoolThreads) keys[i] = ord_f32(srow[lo + v0 + i]);
    }
    int32_t* out = pool + (size_t)b * out_stride + (size_t)shard * K;
    if (rank == 0)
        for (int j = (Kr > 0 ? Kr : 0) + threadIdx.x; j < K; j += kPoolThreads) out[j] = -1;
    if (Kr <= 0) return;  // an empty shard: the whole cluster (one row) leaves together

    unsigned prefix = 0, pmask = 0, remaining = (unsigned)Kr;
    const int shifts[3] = {21, 10, 0};
    const int widths[3] = {11, 11, 10};
    int pass0 = 0;
    if (ghist) {
        // the first pass from the counts the LM-head epilogue made (the same
        // data in every CTA, so each finds the digit without the cluster):
        // thread t holds bins kBins-1-2t and kBins-2-2t, and a block scan
        // gives the keys in the bins above them
        static_assert(kBins == 2 * kPoolThreads && kBins == kPoolHistBins, "two bins per thread");
        const unsigned* gh = ghist + (size_t)b * kBins;
        const int t = threadIdx.x;
        const unsigned c_hi = gh[kBins - 1 - 2 * t], c_lo = gh[kBins - 2 - 2 * t];
        const unsigned above = block_scan_excl(c_hi + c_lo, S.warp_tot, &S.total);
        if (above < remaining && above + c_hi >= remaining) {
            S.digit = (unsigned)(kBins - 1 - 2 * t);
            S.rem = remaining - above;
        } else if (above + c_hi < remaining && above + c_hi + c_lo >= remaining) {
            S.digit = (unsigned)(kBins - 2 - 2 * t);
            S.rem = remaining - above - c_hi;
        }
        __syncthreads();
        prefix = S.digit << shifts[0];
        pmask = (unsigned)(kBins - 1) << shifts[0];
        remaining = S.rem;
        pass0 = 1;
    }
#pragma unroll 1
    for (int pass = pass0; pass < 3; ++pass) {
        const int shift = shifts[pass];
        const unsigned nb = 1u << widths[pass];
        const unsigned dmask = nb - 1;
        for (unsigned i = threadIdx.x; i < nb; i += kPoolThreads) S.hist[i] = 0;
        __syncthreads();
        const int n_round = (n + 31) & ~31;
        for (int i = threadIdx.x; i < n_round; i += kPoolThreads) {
            const unsigned k = i < n ? keys[i] : 0u;
            const bool part = i < n && (k & pmask) == prefix;
            const unsigned m = __ballot_sync(0xffffffffu, part);
            if (part) {
                const unsigned d = (k >> shift) & dmask;
                const unsigned peers = __match_any_sync(m, d);
                if (lane == __ffs(peers) - 1) atomicAdd(&S.hist[d], (unsigned)__popc(peers));
            }
        }
        cluster.sync();  // every CTA's histogram is complete
        // this CTA merges the bins [rank*per, (rank+1)*per) of all CTAs
        const unsigned per = nb / R;
        unsigned mine = 0;
        for (unsigned t = threadIdx.x; t < per; t += kPoolThreads) {
            unsigned s = 0;
#pragma unroll
            for (int r = 0; r < R; ++r) s += cluster.map_shared_rank(S.hist, r)[rank * per + t];
            S.merged[t] = s;
            mine += s;
        }
        // block total of the merged slice
        for (int o = 16; o > 0; o >>= 1) mine += __shfl_xor_sync(0xffffffffu, mine, o);
        if (lane == 0) S.warp_tot[threadIdx.x >> 5] = mine;
        __syncthreads();
        if (threadIdx.x == 0) {
            unsigned t = 0;
            for (int w = 0; w < kPoolThreads / 32; ++w) t += S.warp_tot[w];
            S.total = t;
        }
        cluster.sync();  // merged slices and their totals are visible
        // the K-th largest key lies in the highest slice whose suffix reaches
        // `remaining`, then in the highest bin of that slice that does: one
        // warp scans the slice totals and the slice's bins in parallel
        if (threadIdx.x < 32) {
            const unsigned t = lane < R ? *cluster.map_shared_rank(&S.total, lane) : 0u;
            unsigned suf = t;  // inclusive suffix over ranks lane..R-1
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_down_sync(0xffffffffu, suf, o);
                if (lane + o < 32) suf += y;
            }
            const unsigned hit = __ballot_sync(0xffffffffu, lane < R && suf >= remaining);
            const int hr = 31 - __clz(hit);  // highest rank whose suffix reaches `remaining`
            const unsigned above = __shfl_sync(0xffffffffu, suf, hr) - __shfl_sync(0xffffffffu, t, hr);
            const unsigned rem = remaining - above;
            const unsigned* mg = cluster.map_shared_rank(S.merged, hr);
            const int ppl = (int)per / 32;  // bins per lane (8, 4 or 2)
            unsigned vals[8];
            unsigned lsum = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                vals[i] = i < ppl ? mg[lane * ppl + i] : 0u;
                lsum += vals[i];
            }
            unsigned lsuf = lsum;  // inclusive suffix of lane sums
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const unsigned y = __shfl_down_sync(0xffffffffu, lsuf, o);
                if (lane + o < 32) lsuf += y;
            }
            unsigned acc = lsuf - lsum;  // keys in the bins of higher lanes
#pragma unroll
            for (int i = 7; i >= 0; --i) {
                if (i < ppl) {
                    const unsigned before = acc;  // keys in bins above bin (lane*ppl + i)
                    acc += vals[i];
                    if (before < rem && acc >= rem) {
                        S.digit = (unsigned)hr * per + (unsigned)(lane * ppl + i);
                        S.rem = rem - before;
                    }
                }
            }
        }
        cluster.sync();  // remote reads done before the histograms are reused
        prefix |= S.digit << shift;
        pmask |= dmask << shift;
        remaining = S.rem;
    }
    const unsigned T = prefix, need = remaining;  // take `need` of the ids whose key equals T

    // ordered compaction: each thread owns a contiguous run of this CTA's slice
    const int per_t = (n + kPoolThreads - 1) / kPoolThreads;
    const int i0 = min(n, (int)threadIdx.x * per_t), i1 = min(n, i0 + per_t);
    unsigned gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
        gt += keys[i] > T;
        eq += keys[i] == T;
    }
    const unsigned eq_before_t = block_scan_excl(eq, S.warp_tot, &S.total);
    const unsigned eq_cta = S.total;
    const unsigned gt_before_t = block_scan_excl(gt, S.warp_tot, &S.total);
    const unsigned gt_cta = S.total;
    if (threadIdx.x == 0) {
        S.gt = gt_cta;
        S.eq = eq_cta;
    }
    cluster.sync();
    // the counts of the CTAs before this one: one warp reads them in parallel
    // (lane r from rank r) and sums them, instead of a chain of remote reads
    if (threadIdx.x < 32) {
        unsigned g = 0, e = 0;
        if (lane < rank) {
            g = *cluster.map_shared_rank(&S.gt, lane);
            e = *cluster.map_shared_rank(&S.eq, lane);
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            g += __shfl_xor_sync(0xffffffffu, g, o);
            e += __shfl_xor_sync(0xffffffffu, e, o);
        }
        if (lane == 0) {
            S.digit = g;  // the selection's scratch words are free again: reused for the sums
            S.rem = e;
        }
    }
    __syncthreads();
    const unsigned gt_before_r = S.digit, eq_before_r = S.rem;
    const unsigned eq_before = eq_before_r + eq_before_t;
    const unsigned eq_take = eq_before >= need ? 0u : min(eq, need - eq_before);
    // ids written before this thread: all greater ones, and the equal ones taken so far
    unsigned pos = gt_before_r + gt_before_t + min(need, eq_before);
    unsigned eq_used = 0;
    for (int i = i0; i < i1; ++i) {
        const unsigned k = keys[i];
        bool take = k > T;
        if (!take && k == T && eq_used < eq_take) {
            take = true;
            ++eq_used;
        }
        if (take && pos < (unsigned)Kr) out[pos++] = cand ? crow[i] : lo + v0 + i;
    }
    cluster.sync();  // no CTA leaves while others may still read its shared memory
}

}  // namespace

namespace {

template <int R>
cudaError_t launch_rows_r(const float* score, long long stride, const int32_t* cand, int shards, int shard_len,
                          int32_t* pool, int out_stride, int B, int V, int K, cudaStream_t st, const unsigned* ghist) {
    const int chunk = (shard_len + R - 1) / R;
    const size_t smem = sizeof(PoolShared<R>) + (size_t)chunk * 4;
    cudaError_t e = cudaFuncSetAttribute(k_pool_cluster<R>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    if (R > kRanksPortable) {
        e = cudaFuncSetAttribute(k_pool_cluster<R>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
        if (e != cudaSuccess) return e;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(R, B * shards);
    cfg.blockDim = dim3(kPoolThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = R;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, k_pool_cluster<R>, score, stride, cand, shards, shard_len, pool, out_stride, V, K,
                              chunk, ghist);
}

// R = 16 for a single row when the GPU has room for it (num_sms = 0: never)
// ghist: first-digit counts of the rows (direct pool only), or null
cudaError_t launch_rows(const float* score, long long stride, const int32_t* cand, int shards, int shard_len,
                        int32_t* pool, int out_stride, int B, int V, int K, cudaStream_t st, int num_sms = 0,
                        const unsigned* ghist = nullptr) {
    if (num_sms >= kRanksWide && B * shards == 1) {
        cudaError_t e =
            launch_rows_r<kRanksWide>(score, stride, cand, shards, shard_len, pool, out_stride, B, V, K, st, ghist);
        if (e == cudaSuccess) return e;
        cudaGetLastError();  // wide clusters unavailable: the portable size
    }
    return launch_rows_r<kRanksPortable>(score, stride, cand, shards, shard_len, pool, out_stride, B, V, K, st, ghist);
}

bool fits(int row_len) {
    return sizeof(PoolShared<kRanksPortable>) + (size_t)((row_len + kRanksPortable - 1) / kRanksPortable) * 4 <=
           220 * 1024;
}

}  // namespace

// Pool selection from caller-given scores: the same kernel, pointers passed in.
cudaError_t launch_pool_cluster_raw(const float* score, int32_t* pool, int B, int V, int K, cudaStream_t st) {
    return launch_rows(score, V, nullptr, 1, V, pool, K, B, V, K, st);
}

bool pool_cluster_fits(int V) { return fits(V); }

bool pool_cluster_supported(const domino_ctx* c) { return fits(c->cfg.V); }

cudaError_t launch_pool_cluster(domino_ctx* c, RunArgs& r, const unsigned* hist) {
    ++r.launches;
    return launch_rows(c->score, c->cfg.V, nullptr, 1, c->cfg.V, c->pool, r.K, r.B, c->cfg.V, r.K, r.st, c->num_sms,
                       hist);
}

bool pool_compact_supported(const domino_ctx* c, int P, int K) {
    return P >= 2 && P <= DOMINO_MAX_VOCAB_PARTITIONS && c->cand != nullptr && K <= c->cfg.max_K &&
           fits((c->cfg.V + P - 1) / P) && fits(P * K);
}

cudaError_t launch_pool_compact(domino_ctx* c, RunArgs& r, int P) {
    const int V = c->cfg.V, K = r.K;
    const int S = (V + P - 1) / P;
    // pass 1: shard-local top-K of every (request, shard) into cand [B, P*K]
    ++r.launches;
    cudaError_t e = launch_rows(c->score, V, nullptr, P, S, c->cand, P * K, r.B, V, K, r.st, c->num_sms);
    if (e != cudaSuccess) return e;
    // pass 2: the global top-K among each request's P*K candidates
    ++r.launches;
    return launch_rows(c->score, V, c->cand, 1, P * K, c->pool, K, r.B, P * K, K, r.st, c->num_sms);
}

}  // namespace domino
