// Step 2 of the CSA2 decode path in one launch: indexer scoring of every
// candidate and the exact Top-K of each selection row.
//
// Helmcode "DeepSeek V4.1 Flash" explainer, "03 · CSA2": a Full layer scores
// every position, a Reindex layer rescores a Full layer's keys with its own
// query; Louis Bouchard's KV-cache report, "Share the cache and the search
// work": the first indexing layer keeps a candidate pool that later indexing
// layers search.  Order: score descending, ties to the lower position; the
// output is ascending positions, -1 padded (include/csa2.h).
//
// One *group* of G CTAs takes one (job, sequence); a job is one key cache
// scored by up to two queries (a Full layer and a pool-free Reindex layer
// over the same keys share the pass), each query a selection row with up to
// two targets (its Top-K and, for a Full layer, its pool).  CTA g owns the
// contiguous candidates [g chunk, (g+1) chunk):
//   scan     its key tiles arrive by bulk copy (a ring of up to 4 batches of 16 tiles)
//            or, for a pool, by per-key gathers; each thread scores two
//            candidates at a time (exact integer block products); each
//            score becomes an order-preserving uint32 key kept in shared
//            memory and counted in the CTA's histogram of the keys' top 11
//            bits, added into the group's after the scan;
//   rounds   after each group barrier every CTA reads the same global state
//            and takes the same decisions: the threshold bin of each target;
//            when that bin holds at most CAP candidates, every CTA appends
//            its candidates of the bin (key, index) to a global list and
//            publishes how many of its keys lie above the bin; otherwise the
//            next 11 (then 10) key bits are histogrammed the same way; when
//            all 32 bits are fixed and the ties exceed CAP, each CTA
//            publishes its counts above and at the threshold key;
//   output   after the last barrier each CTA resolves the candidate list
//            exactly (radix passes over the list's remaining key bits, then
//            over the candidate indices of the threshold key), derives every
//            CTA's output offset from the published counts, and writes its
//            own winners in position order.
// The common case takes two group barriers (histogram, candidate list).
// Barrier counters and histograms live in the caller's workspace, which must
// be zero at the first call; every launch leaves them zero again.  The
// launch is co-resident (all CTAs of the grid fit on the device at once);
// group barriers are bounded spins that raise the timeout flag when they
// give up.  The Full layer's appended main-KV row and indexer key (position
// L-1) are quantised here, the key patched into the scanning CTA's copy.
// Inside a decode step each winner's main-KV row is brought into L2 as its
// index is written: the attention launch that follows gathers those rows
// right after its wait for this kernel.
#include <algorithm>
#include <cstring>
#include <vector>

#include "internal.h"
#include "scan.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kThreads = 512;                       // 16 warps: the scoring loop is latency-bound
constexpr int kWarps = kThreads / 32;
constexpr int kBatchKeys = 1024;                    // candidates per bulk-copy batch
constexpr int kBatchTiles = kBatchKeys / kIdxTile;  // 16 tiles
constexpr int kBatchBytes = kBatchTiles * kIdxTileBytes;
constexpr int kMaxSel = 4;                          // (row, target) selections per group
constexpr int kCandCap = 1024;                      // candidate list capacity per selection (every CTA resolves the
                                                    // whole list: a larger threshold bin takes a refining round)
constexpr int kMaxG = 1024;
constexpr int kMaxChunk = 8192;
constexpr int kMaxRing = 4;                          // bulk-copy ring slots at most
constexpr size_t kMaxSmem = 232448;                  // dynamic shared memory per CTA at most

enum : int32_t { kRefine = 0, kPubCand = 1, kPubCount = 2, kDone = 3 };

// Global state of one group (zero at launch, left zero).
struct GroupHdr {
    uint32_t bar;
    uint32_t exit;
    uint32_t cand_n[kMaxSel];
    uint32_t pad[58];
};
static_assert(sizeof(GroupHdr) == 256, "group header");

struct GroupState {
    GroupHdr hdr;
    uint32_t hist1[2][kHistBins];          // per row: top 11 bits
    uint32_t hist2[kMaxSel][kHistBins];    // per selection: next 11 bits
    uint32_t hist3[kMaxSel][1024];         // per selection: last 10 bits
    uint32_t cnt[kMaxSel][kMaxG][2];       // per CTA: keys above the threshold prefix, ties at it
    uint2 cand[kMaxSel][kCandCap];         // (key, candidate index)
};

using FusedJob = FusedJobDesc;
constexpr int kMaxFusedJobs = 8;

struct FusedParams {
    FusedJob jobs[kMaxFusedJobs];
    const int32_t *seq_lens;
    uint8_t *state;           // GroupState per (job, sequence)
    int64_t scores_stride;
    int32_t batch, topk, pool_out, max_len;
    int32_t G, chunk, cap;    // CTAs per group, candidates per CTA, candidate capacity
    int32_t ring_slots;       // bulk-copy ring slots (1 .. kMaxRing)
    uint32_t spin_limit;      // group-barrier polls before giving up
    uint32_t first_wait_limit;  // polls of the first tile wait (test hook; normally the mbarrier limit)
    int32_t keys_ready;         // the key caches predate the previous kernel: copies go out before the wait
};

struct Sel {
    int32_t state;
    uint32_t K;
    uint32_t prefix;   // top nb bits of the threshold
    int32_t nb;
    uint32_t need;     // still wanted among keys with that prefix
    uint32_t above;    // keys of the group above the prefix
    uint32_t at;       // keys of the group at the prefix
    int32_t all_valid; // fewer candidates than K: take every valid one
};

struct Misc {
    scan::QuerySet qs;
    float sk_lut[256];
    Sel sel[kMaxSel];
    uint32_t scratch[48];
    uint32_t warp_a[kWarps], warp_t[kWarps];
    uint32_t app_key[9];       // appended indexer key: 32 B codes + 4 B scales
    int32_t app_local;         // its candidate index within this CTA's range, or -1
    int32_t ok;
    uint32_t bcast[8];
    uint32_t tile_ok[kMaxRing];  // per ring slot: tiles whose copy was issued
    uint64_t bar[kMaxRing];
};

// ---- block-wide helpers (kThreads threads) ---------------------------------------------

// Finds bin d with above(d) < need <= above(d) + h[d] (above = count in bins
// > d, bins taken from the top).  Returns bin -1 (above = total) when the
// total is below need.  nbins % kThreads == 0.
struct Thresh {
    int bin;
    uint32_t above;
    uint32_t at;
};

__device__ __noinline__ Thresh find_threshold(const uint32_t *h, int nbins, uint32_t need, uint32_t *scratch)
{
    // bins by rank from the top (rank k = bin nbins-1-k); warp w sums ranks
    // [w seg, (w+1) seg) with coalesced reads, a prefix over the warps finds
    // the segment holding the need-th key, and that warp walks it 32 at a time
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int seg = nbins / kWarps;
    uint32_t wsum = 0;
    for (int k = lane; k < seg; k += 32) wsum += h[nbins - 1 - (warp * seg + k)];
    wsum = __reduce_add_sync(0xFFFFFFFFu, wsum);
    if (lane == 0) scratch[warp] = wsum;
    __syncthreads();
    if (tid == 0) {
        uint32_t run = 0;
        int wsel = -1;
        uint32_t before = 0;
        for (int w = 0; w < kWarps; ++w) {
            if (wsel < 0 && run + scratch[w] >= need) {
                wsel = w;
                before = run;
            }
            run += scratch[w];
        }
        scratch[kWarps] = run;                      // total
        scratch[kWarps + 3] = (uint32_t)wsel;       // warp holding the threshold, or -1
        scratch[kWarps + 4] = before;               // count above its segment
        scratch[kWarps + 1] = 0xFFFFFFFFu;
        scratch[kWarps + 2] = run;
    }
    __syncthreads();
    if (warp == (int)scratch[kWarps + 3]) {
        uint32_t above = scratch[kWarps + 4];
        for (int k0 = 0; k0 < seg; k0 += 32) {
            const int rk = warp * seg + k0 + lane;
            const uint32_t c = h[nbins - 1 - rk];
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
                if (lane >= o) incl += v;
            }
            const uint32_t hit = __ballot_sync(0xFFFFFFFFu, above + incl >= need);
            if (hit) {
                const int first = __ffs(hit) - 1;
                if (lane == first) {
                    scratch[kWarps + 1] = (uint32_t)(nbins - 1 - rk);
                    scratch[kWarps + 2] = above + incl - c;
                }
                break;
            }
            above += __shfl_sync(0xFFFFFFFFu, incl, 31);
        }
    }
    __syncthreads();
    Thresh r;
    r.bin = (int)scratch[kWarps + 1];
    r.above = scratch[kWarps + 2];
    r.at = (r.bin >= 0) ? h[r.bin] : 0u;
    __syncthreads();
    return r;
}

// Exclusive prefix of v[0..n) in place (n <= kMaxG); returns the total.
__device__ __noinline__ uint32_t block_exclusive_scan(uint32_t *v, int n, uint32_t *scratch)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int per = (n + kThreads - 1) / kThreads;
    const int i0 = tid * per;
    uint32_t local = 0;
    for (int i = i0; i < min(n, i0 + per); ++i) local += v[i];
    uint32_t incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += u;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t x = (lane < kWarps) ? scratch[lane] : 0u;
        uint32_t s = x;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += u;
        }
        if (lane < kWarps) scratch[lane] = s - x;
        if (lane == kWarps - 1) scratch[kWarps] = s;
    }
    __syncthreads();
    uint32_t run = scratch[warp] + incl - local;
    for (int i = i0; i < min(n, i0 + per); ++i) {
        const uint32_t x = v[i];
        v[i] = run;
        run += x;
    }
    const uint32_t total = scratch[kWarps];
    __syncthreads();
    return total;
}

// dst[0..n) = src[0..n) (global, L2) by the CTA, eight independent loads in
// flight per thread before any is stored.
template <typename T>
__device__ __forceinline__ void load_to_smem(T *dst, const T *src, int n)
{
    for (int base = 0; base < n; base += 8 * kThreads) {
        T v[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = base + k * kThreads + (int)threadIdx.x;
            if (i < n) v[k] = __ldcg(src + i);
        }
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const int i = base + k * kThreads + (int)threadIdx.x;
            if (i < n) dst[i] = v[k];
        }
    }
}

// Bounded group barrier: counter `bar` reaches `target` (G per round).  The
// CTA barrier orders every thread's writes before thread 0's fence, whose
// gpu-scope ordering is cumulative; thread 0 alone arrives, polls (relaxed)
// and fences again before the CTA barrier releases the others.
__device__ __forceinline__ void group_barrier(uint32_t *bar, uint32_t target, uint32_t limit, Misc &M)
{
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        asm volatile("red.relaxed.gpu.global.add.u32 [%0], 1;\n" ::"l"(bar) : "memory");
        uint32_t v = 0, i = 0;
        do {
            asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];\n" : "=r"(v) : "l"(bar) : "memory");
        } while (v < target && ++i < limit);
        if (v < target) M.ok = 0;
        __threadfence();
    }
    __syncthreads();
}

__device__ __forceinline__ uint32_t prefix_of(uint32_t key, int nb) { return nb >= 32 ? key : key >> (32 - nb); }

// ---- the kernel ------------------------------------------------------------------------

// Brings the main-KV row of (sequence b, position pos) into L2: the attention
// launch that follows gathers it, and its gather waits on the index kernel.
__device__ __forceinline__ void warm_row(const CacheView &kv, int b, int32_t pos)
{
    if (pos < 0) return;
    const int64_t slot = slot_of(kv, b, pos);
    if (slot < 0) return;
    const uint8_t *row = kv.data + slot * kKvRow;
    tc::prefetch_l2(row);
    tc::prefetch_l2(row + 128);
    tc::prefetch_l2(row + 256);
    tc::prefetch_l2(row + kKvRow - 1);
}

__global__ void __launch_bounds__(kThreads) index_fused_kernel(const __grid_constant__ FusedParams P, int *flags)
{
    extern __shared__ __align__(128) uint8_t smem[];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = blockIdx.x, b = blockIdx.y, jz = blockIdx.z;
    const int G = P.G;
    const FusedJob &job = P.jobs[jz];
    const int n_rows = job.n_q;
    // shared memory: ring | keys[n_rows][chunk] | hist[2][2048] | misc
    uint8_t *ring = smem;
    uint32_t *keys = reinterpret_cast<uint32_t *>(smem + (size_t)P.ring_slots * kBatchBytes);
    uint32_t *hist = keys + (size_t)2 * P.chunk;
    Misc &M = *reinterpret_cast<Misc *>(hist + 2 * kHistBins);
    GroupState &GS = *reinterpret_cast<GroupState *>(P.state + ((size_t)jz * P.batch + b) * sizeof(GroupState));

    if (tid == 0) {
        for (int i = 0; i < kMaxRing; ++i) tc::mbar_init(&M.bar[i], 1);
        tc::mbar_init_fence();
        M.ok = 1;
        M.app_local = -1;
    }
    if (tid < 256) M.sk_lut[tid] = e4m3_value((uint32_t)tid);
    for (int i = tid; i < 2 * kHistBins; i += kThreads) hist[i] = 0u;
    __syncthreads();

    const bool direct = job.pool == nullptr;
    const int64_t c0 = (int64_t)g * P.chunk;
    auto load_len = [&]() {
        int v = __ldcg(P.seq_lens + b);
        if (v < 0 || v > P.max_len) {
            if (tid == 0 && g == 0) raise_flag(flags, kFlagBounds);
            v = v < 0 ? 0 : P.max_len;
        }
        return v;
    };
    // contiguous caches: the tile copies cover the candidates up to max_len and go
    // out before the sequence length is known (positions past it are ignored);
    // paged caches map only the sequence's own pages, so they wait for it
    const bool early = direct && job.keys.page_size == 0;
    // when the keys predate the previous kernel, the copies go out while it runs
    const bool pre = early && P.keys_ready;
    if (!pre) tc::pdl_wait();
    int L = (early && !pre) ? -1 : load_len();  // with pre, the lengths predate the previous kernel too
    const int64_t c1_max = min((int64_t)(direct ? (early ? P.max_len : L) : job.pool_len), c0 + P.chunk);
    const int nb_max = (int)max((int64_t)0, (c1_max - c0 + kBatchKeys - 1) / kBatchKeys);

    auto issue_batch = [&](int k) {
        // thread 0: the bulk copies of batch k's tiles into ring slot k % slots
        const int slot = k % P.ring_slots;
        uint32_t bytes = 0, okm = 0;
        const uint8_t *src[kBatchTiles];
        for (int i = 0; i < kBatchTiles; ++i) {
            src[i] = nullptr;
            const int64_t p0 = c0 + (int64_t)k * kBatchKeys + (int64_t)i * kIdxTile;
            if (p0 < c1_max) {
                const int64_t s = slot_of(job.keys, b, p0);
                // a 64-aligned position block is one whole tile (page and stride are multiples of 64)
                if (s >= 0 && s + kIdxTile <= job.keys.n_slots) {
                    src[i] = job.keys.data + (s / kIdxTile) * kIdxTileBytes;
                    bytes += kIdxTileBytes;
                    okm |= 1u << i;
                } else {
                    raise_flag(flags, kFlagBounds);
                }
            }
        }
        M.tile_ok[slot] = okm;
        tc::mbar_expect_tx(&M.bar[slot], bytes);
        // runs of tiles adjacent in memory (always, in a contiguous cache) go as one copy
        for (int i = 0; i < kBatchTiles;) {
            if (!src[i]) {
                ++i;
                continue;
            }
            int n = 1;
            while (i + n < kBatchTiles && src[i + n] == src[i] + (size_t)n * kIdxTileBytes) ++n;
            tc::bulk_g2s(ring + (size_t)slot * kBatchBytes + i * kIdxTileBytes, src[i], (uint32_t)n * kIdxTileBytes,
                         &M.bar[slot]);
            i += n;
        }
    };
    if (direct && tid == 0) {
        for (int k = 0; k < min(nb_max, P.ring_slots); ++k) issue_batch(k);
    }
    if (pre) tc::pdl_wait();
    if (L < 0) L = load_len();
    const int64_t n_cand = direct ? L : job.pool_len;
    const int64_t c1 = min(n_cand, c0 + P.chunk);
    const int nk = (int)max((int64_t)0, c1 - c0);
    const int32_t *pool = direct ? nullptr : job.pool + (int64_t)b * job.pool_len;

    // appends of a Full layer: the new main-KV row (warp 0 of the last CTA) and
    // the new indexer key (warp 1 of the CTA that scans position L-1)
    if (L > 0 && job.new_kv && g == G - 1 && warp == 0) {
        float x[16];
        const float4 *src = reinterpret_cast<const float4 *>(job.new_kv + (int64_t)b * kDim + 16 * lane);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const float4 v = __ldcg(src + k);
            x[4 * k] = v.x, x[4 * k + 1] = v.y, x[4 * k + 2] = v.z, x[4 * k + 3] = v.w;
        }
        uint2 codes;
        uint32_t sc;
        fp4_block16(x, codes, sc);
        const int64_t slot = slot_of(job.kv, b, (int64_t)L - 1);
        if (slot < 0) {
            if (lane == 0) raise_flag(flags, kFlagBounds);
        } else {
            uint8_t *row = job.kv.data + slot * kKvRow;
            *reinterpret_cast<uint2 *>(row + 8 * lane) = codes;
            row[kKvCodes + lane] = (uint8_t)sc;
        }
    }
    if (L > 0 && job.new_key && direct && (int64_t)(L - 1) >= c0 && (int64_t)(L - 1) < c1 && warp == 1) {
        uint2 codes = make_uint2(0u, 0u);
        uint32_t sc = 0;
        if (lane < 4) {
            float x[16];
            const float4 *src = reinterpret_cast<const float4 *>(job.new_key + (int64_t)b * kIdxDim + 16 * lane);
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const float4 v = __ldcg(src + k);
                x[4 * k] = v.x, x[4 * k + 1] = v.y, x[4 * k + 2] = v.z, x[4 * k + 3] = v.w;
            }
            fp4_block16(x, codes, sc);
            M.app_key[2 * lane] = codes.x;
            M.app_key[2 * lane + 1] = codes.y;
        }
        const uint32_t scales = __shfl_sync(0xFFFFFFFFu, sc, 0) | (__shfl_sync(0xFFFFFFFFu, sc, 1) << 8) |
                                (__shfl_sync(0xFFFFFFFFu, sc, 2) << 16) | (__shfl_sync(0xFFFFFFFFu, sc, 3) << 24);
        const int64_t slot = slot_of(job.keys, b, (int64_t)L - 1);
        if (lane == 0) {
            M.app_key[8] = scales;
            M.app_local = (int32_t)((int64_t)L - 1 - c0);
            if (slot < 0) {
                raise_flag(flags, kFlagBounds);
            } else {
                uint8_t *tile = job.keys.data + (slot / kIdxTile) * kIdxTileBytes;
                const int rr = (int)(slot % kIdxTile);
                *reinterpret_cast<uint32_t *>(tile + kIdxTile * 32 + rr * 4) = scales;
            }
        }
        if (lane < 4 && slot >= 0) {
            uint8_t *tile = job.keys.data + (slot / kIdxTile) * kIdxTileBytes;
            const int rr = (int)(slot % kIdxTile);
            *reinterpret_cast<uint2 *>(tile + rr * 32 + 8 * lane) = codes;
        }
    }

    if (tid < 256) scan::prep_query_set(tid, job.n_q, job.q_idx, job.w, b, M.qs);  // 256 threads
    __syncthreads();

    // ---- scan: one thread scores whole keys (all of this job's queries)
    // every issued batch is waited for, also those past the sequence's end
    const int nb_loop = direct ? nb_max : (nk + kBatchKeys - 1) / kBatchKeys;
    for (int k = 0; k < nb_loop; ++k) {
        const int slot = direct ? k % P.ring_slots : 0;
        bool have = true;
        if (direct) {
            const uint32_t lim = (k == 0) ? P.first_wait_limit : tc::kWaitLimit;
            bool got = false;
            for (uint32_t i = 0; i < lim && !got; ++i) got = tc::mbar_try_wait(&M.bar[slot], (k / P.ring_slots) & 1);
            if (!got) {
                if (tid == 0) M.ok = 0;
                got = tc::mbar_wait(&M.bar[slot], (k / P.ring_slots) & 1);  // drain: copies land before reuse
            }
            have = got;
            // the appended key replaces its stale copy in the ring
            const int al = M.app_local;
            if (al >= k * kBatchKeys && al < (k + 1) * kBatchKeys && tid < 9) {
                const int li = al - k * kBatchKeys;
                uint8_t *tile = ring + (size_t)slot * kBatchBytes + (li / kIdxTile) * kIdxTileBytes;
                const int rr = li % kIdxTile;
                if (tid < 8) reinterpret_cast<uint32_t *>(tile + rr * 32)[tid] = M.app_key[tid];
                else *reinterpret_cast<uint32_t *>(tile + kIdxTile * 32 + rr * 4) = M.app_key[8];
            }
            __syncthreads();
        }
        const uint8_t *tiles = ring + (size_t)slot * kBatchBytes;
        const int base = k * kBatchKeys;  // local index of the batch's first candidate
        // candidate i of the batch: its codes as int8 words and its block scales; false when absent
        auto fetch = [&](int i, uint32_t (&kw)[16], float (&sk)[4]) -> bool {
            const int li = base + i;
            bool ok = li < nk;
            uint4 c0v = make_uint4(0u, 0u, 0u, 0u), c1v = c0v;
            uint32_t scw = 0u;
            if (ok && direct) {
                const int ti = i / kIdxTile, rr = i % kIdxTile;
                ok = have && ((M.tile_ok[slot] >> ti) & 1u);
                const uint8_t *tile = tiles + ti * kIdxTileBytes;
                c0v = *reinterpret_cast<const uint4 *>(tile + rr * 32);
                c1v = *reinterpret_cast<const uint4 *>(tile + rr * 32 + 16);
                scw = *reinterpret_cast<const uint32_t *>(tile + kIdxTile * 32 + rr * 4);
            } else if (ok) {
                int64_t pos = (int64_t)__ldcg(pool + c0 + li);
                ok = pos >= 0 && pos < L;
                if (ok) {
                    const int64_t slotk = slot_of(job.keys, b, pos);
                    if (slotk < 0) {
                        raise_flag(flags, kFlagBounds);
                        ok = false;
                    } else {
                        const uint8_t *tile = job.keys.data + (slotk / kIdxTile) * kIdxTileBytes;
                        const int rr = (int)(slotk % kIdxTile);
                        c0v = __ldcg(reinterpret_cast<const uint4 *>(tile + rr * 32));
                        c1v = __ldcg(reinterpret_cast<const uint4 *>(tile + rr * 32 + 16));
                        scw = __ldcg(reinterpret_cast<const uint32_t *>(tile + kIdxTile * 32 + rr * 4));
                    }
                }
            }
            scan::unpack_key(c0v, c1v, scw, M.sk_lut, kw, sk);
            return ok;
        };
        // candidate i's score for row q: its key in shared memory and one
        // shared atomic into the histogram of the keys' top bits
        auto record = [&](int i, bool ok, float sc, int q) {
            const int li = base + i;
            const uint32_t key = ok ? score_key(sc) : 0u;
            if (li < nk) keys[(size_t)q * P.chunk + li] = key;
            if (key) atomicAdd(&hist[q * kHistBins + (key >> (32 - kHistBits))], 1u);
            if (key && job.out_scores[q]) job.out_scores[q][(int64_t)b * P.scores_stride + c0 + li] = sc;
        };
        // two candidates per thread at a time (i and i + kThreads), their scores'
        // dependent chains interleaved
        static_assert(kBatchKeys % (2 * kThreads) == 0, "two candidates per step");
#pragma unroll 1
        for (int i = tid; i < kBatchKeys && base < nk; i += 2 * kThreads) {
            uint32_t kwa[16], kwb[16];
            float ska[4], skb[4];
            const bool oka = fetch(i, kwa, ska), okb = fetch(i + kThreads, kwb, skb);
#pragma unroll 1
            for (int q = 0; q < n_rows; ++q) {
                float sa, sb;
                scan::score_pair(kwa, ska, kwb, skb, M.qs, q, sa, sb);
                record(i, oka, sa, q);
                record(i + kThreads, okb, sb, q);
            }
        }
        __syncthreads();
        if (direct && tid == 0 && k + P.ring_slots < nb_max) {
            asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
            issue_batch(k + P.ring_slots);
        }
    }
    // this CTA's histograms into the group's
    for (int r = 0; r < n_rows; ++r)
        for (int i = tid; i < kHistBins; i += kThreads) {
            const uint32_t c = hist[r * kHistBins + i];
            if (c) atomicAdd(&GS.hist1[r][i], c);
        }

    // ---- selection rounds ------------------------------------------------------------
    if (tid < kMaxSel) {
        const int r = tid >> 1, tg = tid & 1;
        Sel &S = M.sel[tid];
        const bool act = r < n_rows && (tg == 0 || (job.out_pool[r] && P.pool_out > 0));
        S.state = act ? kRefine : kDone;
        S.K = (uint32_t)(tg == 0 ? P.topk : P.pool_out);
        S.prefix = 0;
        S.nb = 0;
        S.need = S.K;
        S.above = 0;
        S.at = 0;
        S.all_valid = 0;
    }
    const int cap = P.cap;
    uint32_t round = 0;
    bool pending = true;
    while (pending) {
        group_barrier(&GS.hdr.bar, (uint32_t)G * ++round, P.spin_limit, M);
        if (round == 1) tc::pdl_launch_dependents();  // every CTA of the grid is resident by now
        pending = false;
        for (int si = 0; si < kMaxSel; ++si) {
            const int st = M.sel[si].state;
            if (st == kDone) continue;
            const int r = si >> 1, tg = si & 1;
            const uint32_t *rk = keys + (size_t)r * P.chunk;
            if (st == kPubCand || st == kPubCount) {
                // ---- output of a terminal selection
                Sel S = M.sel[si];
                uint32_t *cnt_sel = reinterpret_cast<uint32_t *>(ring);  // [G] (ring is idle now)
                uint2 *cands = reinterpret_cast<uint2 *>(ring + 4 * kMaxG);
                uint32_t T = 0, ties_total = 0;
                int64_t cut = INT64_MAX;
                uint32_t ties_need = 0;
                if (st == kPubCand) {
                    // every CTA's published count above the prefix goes out with the
                    // list's length and the list, one round trip to L2
                    uint32_t cnt_pub[kMaxG / kThreads];
#pragma unroll
                    for (int j = 0; j < kMaxG / kThreads; ++j) {
                        const int i = tid + j * kThreads;
                        cnt_pub[j] = i < G ? __ldcg(&GS.cnt[si][i][0]) : 0u;
                    }
                    const uint32_t n = min(__ldcg(&GS.hdr.cand_n[si]), (uint32_t)cap);
                    load_to_smem(cands, &GS.cand[si][0], (int)n);
                    for (int i = tid; i < G; i += kThreads) cnt_sel[i] = 0u;
                    __syncthreads();
                    // the need-th largest key among the candidates (they share the top nb bits)
                    uint32_t need = S.need, pfx = S.prefix;
                    int nb = S.nb;
                    uint32_t *h = hist;  // scratch histogram (4,096 bins)
                    while (nb < 32) {
                        const int bits = min(11, 32 - nb);
                        const int shift = 32 - nb - bits;
                        const int nbins = 1 << bits;
                        for (int i = tid; i < 2048; i += kThreads) h[i] = 0u;
                        __syncthreads();
                        for (uint32_t i = tid; i < n; i += kThreads) {
                            const uint32_t kk = cands[i].x;
                            if (prefix_of(kk, nb) == pfx) atomicAdd(&h[(kk >> shift) & (nbins - 1)], 1u);
                        }
                        __syncthreads();
                        const Thresh th = find_threshold(h, nbins < kThreads ? kThreads : nbins, need, M.scratch);
                        need -= th.above;
                        pfx = (pfx << bits) | (uint32_t)(th.bin < 0 ? 0 : th.bin);
                        nb += bits;
                    }
                    T = pfx;
                    ties_need = need;
                    // ties at T: the ties_need lowest candidate indices
                    uint32_t nt = 0;
                    for (uint32_t i = tid; i < n; i += kThreads) nt += (cands[i].x == T);
                    nt = __reduce_add_sync(0xFFFFFFFFu, nt);
                    if (lane == 0) M.warp_t[warp] = nt;
                    __syncthreads();
                    ties_total = 0;
                    for (int w = 0; w < kWarps; ++w) ties_total += M.warp_t[w];
                    __syncthreads();
                    if (ties_need < ties_total) {
                        // radix over the (24-bit) candidate index, smallest first (digit mirrored)
                        uint32_t ipfx = 0, ineed = ties_need;
                        for (int pass = 0; pass < 2; ++pass) {
                            const int shift = pass == 0 ? 12 : 0;
                            for (int i = tid; i < 4096; i += kThreads) h[i] = 0u;
                            __syncthreads();
                            for (uint32_t i = tid; i < n; i += kThreads) {
                                const uint2 cd = cands[i];
                                if (cd.x == T && (pass == 0 || (cd.y >> 12) == ipfx))
                                    atomicAdd(&h[4095u - ((cd.y >> shift) & 4095u)], 1u);
                            }
                            __syncthreads();
                            const Thresh th = find_threshold(h, 4096, ineed, M.scratch);
                            ineed -= th.above;
                            ipfx = (ipfx << (pass == 0 ? 0 : 12)) | (4095u - (uint32_t)th.bin);
                            if (pass == 0) ipfx = 4095u - (uint32_t)th.bin;
                        }
                        cut = (int64_t)ipfx;
                    }
                    // selected candidates per owning CTA
                    for (uint32_t i = tid; i < n; i += kThreads) {
                        const uint2 cd = cands[i];
                        if (cd.x > T || (cd.x == T && (int64_t)cd.y <= cut))
                            atomicAdd(&cnt_sel[min((int)(cd.y / (uint32_t)P.chunk), G - 1)], 1u);
                    }
                    __syncthreads();
#pragma unroll
                    for (int j = 0; j < kMaxG / kThreads; ++j) {
                        const int i = tid + j * kThreads;
                        if (i < G) cnt_sel[i] += cnt_pub[j];
                    }
                    __syncthreads();
                } else {
                    // counts path: every valid key (all_valid) or keys above T plus the lowest ties
                    T = S.prefix;
                    ties_need = S.all_valid ? 0u : S.need;
                    for (int i = tid; i < G; i += kThreads) {
                        const uint32_t a = __ldcg(&GS.cnt[si][i][0]);
                        cnt_sel[i] = a;
                        cands[i].x = __ldcg(&GS.cnt[si][i][1]);  // ties per CTA (cands reused as [G])
                    }
                    __syncthreads();
                    if (tid == 0) {
                        uint32_t tb = 0;
                        for (int i = 0; i < G; ++i) {
                            const uint32_t ti = cands[i].x;
                            const uint32_t q = (ties_need > tb) ? min(ties_need - tb, ti) : 0u;
                            M.bcast[4] = (i == g) ? q : M.bcast[4];
                            cnt_sel[i] += q;
                            tb += ti;
                        }
                    }
                    __syncthreads();
                }
                const uint32_t my_quota = (st == kPubCount) ? M.bcast[4] : 0u;
                const uint32_t my_count = cnt_sel[g];
                const uint32_t total = block_exclusive_scan(cnt_sel, G, M.scratch);
                const uint32_t my_off = cnt_sel[g];
                __syncthreads();
                // ---- write this CTA's winners in candidate order
                const uint32_t K = S.K;
                int32_t *out = (tg == 0 ? job.out_idx[r] : job.out_pool[r]) + (int64_t)b * K;
                const int span = (nk + kWarps - 1) / kWarps;
                const int r0 = min(nk, warp * span), r1 = min(nk, r0 + span);
                const int nbq = S.nb;
                const uint32_t pq = S.prefix;
                auto selected = [&](uint32_t key, int64_t idx, bool tie_ok) -> bool {
                    if (!key) return false;
                    if (st == kPubCount) return S.all_valid || key > T || (key == T && tie_ok);
                    const uint32_t pk = prefix_of(key, nbq);
                    if (pk != pq) return pk > pq;
                    return key > T || (key == T && idx <= cut);
                };
                uint32_t wa = 0, wt = 0;
                for (int c = r0; c < r1; c += 32) {
                    const int i = c + lane;
                    const uint32_t key = i < r1 ? rk[i] : 0u;
                    const bool is_tie = st == kPubCount && !S.all_valid && key == T && key;
                    wa += __popc(__ballot_sync(0xFFFFFFFFu, selected(key, c0 + i, false) && !is_tie));
                    wt += __popc(__ballot_sync(0xFFFFFFFFu, is_tie));
                }
                if (lane == 0) {
                    M.warp_a[warp] = wa;
                    M.warp_t[warp] = wt;
                }
                __syncthreads();
                uint32_t sel_before = my_off, tie_before = 0;
                for (int w = 0; w < warp; ++w) {
                    const uint32_t q = (my_quota > tie_before) ? min(my_quota - tie_before, M.warp_t[w]) : 0u;
                    sel_before += M.warp_a[w] + q;
                    tie_before += M.warp_t[w];
                }
                const uint32_t lt = (1u << lane) - 1u;
                uint32_t written = 0, ties_seen = tie_before;
                for (int c = r0; c < r1; c += 32) {
                    const int i = c + lane;
                    const uint32_t key = i < r1 ? rk[i] : 0u;
                    const bool is_tie = st == kPubCount && !S.all_valid && key == T && key;
                    const uint32_t tm = __ballot_sync(0xFFFFFFFFu, is_tie);
                    const uint32_t tie_rank = ties_seen + __popc(tm & lt);
                    const bool sel = is_tie ? (tie_rank < my_quota) : selected(key, c0 + i, false);
                    const uint32_t sm = __ballot_sync(0xFFFFFFFFu, sel);
                    if (sel) {
                        const uint32_t at = sel_before + written + __popc(sm & lt);
                        if (at < K) {
                            const int32_t pos = direct ? (int32_t)(c0 + i) : __ldcg(pool + c0 + i);
                            out[at] = pos;
                            if (tg == 0 && job.has_warm) warm_row(job.warm, b, pos);
                        }
                    }
                    written += __popc(sm);
                    ties_seen += __popc(tm);
                }
                (void)my_count;
                for (uint32_t i = total + (uint32_t)g * kThreads + tid; i < K; i += (uint32_t)G * kThreads) out[i] = -1;
                __syncthreads();
                if (tid == 0) M.sel[si].state = kDone;
                __syncthreads();
                continue;
            }
            // ---- kRefine: the histogram of the next digit is complete
            pending = true;
            {
                Sel S = M.sel[si];
                // digits: 11 bits (the scan's histogram), 11, then the last 10
                const uint32_t *gh = S.nb == 0 ? GS.hist1[r] : (S.nb <= 11 ? GS.hist2[si] : GS.hist3[si]);
                const int bits = S.nb == 0 ? kHistBits : min(11, 32 - S.nb);
                uint32_t *h = reinterpret_cast<uint32_t *>(ring);  // idle after the scan
                load_to_smem(h, gh, 1 << bits);
                __syncthreads();
                const Thresh th = find_threshold(h, max(1 << bits, kThreads), S.need, M.scratch);
                if (tid == 0) {
                    Sel &W = M.sel[si];
                    if (th.bin < 0) {
                        // fewer valid candidates than wanted (only possible at the first digit)
                        W.all_valid = 1;
                        W.state = kPubCount;
                    } else {
                        W.above = S.above + th.above;
                        W.need = S.need - th.above;
                        W.at = th.at;
                        W.prefix = (S.prefix << bits) | (uint32_t)th.bin;
                        W.nb = S.nb + bits;
                        W.state = (th.at <= (uint32_t)cap) ? kPubCand : (W.nb >= 32 ? kPubCount : kRefine);
                    }
                }
                __syncthreads();
            }
            // publish what the next round reads
            const Sel S = M.sel[si];
            if (S.state == kPubCand) {
                // keys above the prefix are counted; keys at it go to the group's
                // candidate list, one global reservation per CTA
                uint32_t na = 0, nc = 0;
                for (int i = tid; i < nk; i += kThreads) {
                    const uint32_t key = rk[i];
                    if (!key) continue;
                    const uint32_t pk = prefix_of(key, S.nb);
                    na += pk > S.prefix;
                    nc += pk == S.prefix;
                }
                na = __reduce_add_sync(0xFFFFFFFFu, na);
                nc = __reduce_add_sync(0xFFFFFFFFu, nc);
                if (lane == 0) {
                    M.warp_a[warp] = na;
                    M.warp_t[warp] = nc;
                }
                __syncthreads();
                if (tid == 0) {
                    uint32_t sa = 0, sc = 0;
                    for (int w = 0; w < kWarps; ++w) {
                        sa += M.warp_a[w];
                        sc += M.warp_t[w];
                    }
                    GS.cnt[si][g][0] = sa;
                    M.bcast[0] = sc ? atomicAdd(&GS.hdr.cand_n[si], sc) : 0u;  // this CTA's first slot
                }
                __syncthreads();
                for (int i = tid; i < nk; i += kThreads) {
                    const uint32_t key = rk[i];
                    if (key && prefix_of(key, S.nb) == S.prefix) {
                        const uint32_t at = atomicAdd(&M.bcast[0], 1u);
                        if (at < (uint32_t)kCandCap) GS.cand[si][at] = make_uint2(key, (uint32_t)(c0 + i));
                    }
                }
            } else if (S.state == kPubCount) {
                uint32_t na = 0, nt = 0;
                for (int i = tid; i < nk; i += kThreads) {
                    const uint32_t key = rk[i];
                    if (!key) continue;
                    if (S.all_valid || key > S.prefix) ++na;
                    else if (key == S.prefix) ++nt;
                }
                na = __reduce_add_sync(0xFFFFFFFFu, na);
                nt = __reduce_add_sync(0xFFFFFFFFu, nt);
                if (lane == 0) {
                    M.warp_a[warp] = na;
                    M.warp_t[warp] = nt;
                }
                __syncthreads();
                if (tid == 0) {
                    uint32_t sa = 0, stt = 0;
                    for (int w = 0; w < kWarps; ++w) {
                        sa += M.warp_a[w];
                        stt += M.warp_t[w];
                    }
                    GS.cnt[si][g][0] = sa;
                    GS.cnt[si][g][1] = stt;
                }
            } else {
                // next digit's histogram of the keys at the prefix
                const int bits = min(11, 32 - S.nb);
                uint32_t *lh = reinterpret_cast<uint32_t *>(ring);
                for (int i = tid; i < 2048; i += kThreads) lh[i] = 0u;
                __syncthreads();
                const int shift = 32 - S.nb - bits;
                for (int i = tid; i < nk; i += kThreads) {
                    const uint32_t key = rk[i];
                    if (key && prefix_of(key, S.nb) == S.prefix) atomicAdd(&lh[(key >> shift) & ((1u << bits) - 1u)], 1u);
                }
                __syncthreads();
                uint32_t *gh = (S.nb <= 11) ? GS.hist2[si] : GS.hist3[si];
                for (int i = tid; i < (1 << bits); i += kThreads)
                    if (lh[i]) atomicAdd(gh + i, lh[i]);
            }
            __syncthreads();
        }
    }

    // ---- leave the group's state zero for the next launch
    // (every histogram was read before the last barrier)
    {
        const int per1 = (2 * kHistBins + G - 1) / G;
        for (int i = g * per1 + tid; i < min(2 * kHistBins, (g + 1) * per1); i += kThreads) (&GS.hist1[0][0])[i] = 0u;
        const int per2 = (kMaxSel * kHistBins + G - 1) / G;
        for (int i = g * per2 + tid; i < min(kMaxSel * kHistBins, (g + 1) * per2); i += kThreads)
            (&GS.hist2[0][0])[i] = 0u;
        const int per3 = (kMaxSel * 1024 + G - 1) / G;
        for (int i = g * per3 + tid; i < min(kMaxSel * 1024, (g + 1) * per3); i += kThreads) (&GS.hist3[0][0])[i] = 0u;
    }
    __syncthreads();
    if (tid == 0) {
        if (!M.ok) raise_flag(flags, kFlagTimeout);
        __threadfence();
        const uint32_t ticket = atomicAdd(&GS.hdr.exit, 1u);
        if (ticket == (uint32_t)G - 1) {
            // the last CTA out: nobody reads the counters any more
            __threadfence();
            for (int s = 0; s < kMaxSel; ++s) GS.hdr.cand_n[s] = 0u;
            GS.hdr.bar = 0u;
            GS.hdr.exit = 0u;
        }
    }
}

}  // namespace

// ---- host side ---------------------------------------------------------------------------

size_t fused_state_bytes(int n_groups) { return (size_t)n_groups * sizeof(GroupState); }

namespace {

size_t fused_smem(int ring_slots, int chunk)
{
    return (size_t)ring_slots * kBatchBytes + (size_t)2 * chunk * 4 + (size_t)2 * kHistBins * 4 + sizeof(Misc);
}

int g_first_wait_limit = -1;  // test hook: polls of the first tile wait, < 0 = the normal limit

}  // namespace

void fused_set_first_wait_limit(int polls) { g_first_wait_limit = polls; }

bool fused_plan(int n_jobs, int batch, int64_t max_cand, FusedPlan &fp, int reserve_sms)
{
    int dev = 0, n_sm = 148;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
    const int n_groups = n_jobs * batch;
    if (n_groups <= 0 || n_jobs > kMaxFusedJobs) return false;
    const int64_t cand = std::max<int64_t>(1, max_cand);
    // `reserve_sms` SMs are left to a kernel that still runs when this launch
    // starts (in a decode step, the previous layer's attention): every CTA of
    // the grid becomes resident at once and issues its tile copies before the
    // wait, instead of the last ones starting when that kernel ends
    int G = (int)std::max<int64_t>(
        1, std::min<int64_t>((cand + 63) / 64, std::max(1, n_sm - std::max(0, reserve_sms)) / n_groups));
    if (G < 1) G = 1;
    int64_t chunk = ((cand + G - 1) / G + 63) / 64 * 64;
    if (chunk > kMaxChunk) {
        log_plan("index: %lld candidates per CTA exceed %d: scan + select kernels", (long long)chunk, kMaxChunk);
        return false;
    }
    const int batches = (int)((chunk + kBatchKeys - 1) / kBatchKeys);
    // every batch of the CTA in flight at once, up to kMaxRing, as shared memory allows: the copies are
    // latency-bound, and a CTA of the phased launch (four groups) scans 3.5 batches
    int slots = batches > 1 ? 2 : 1;
    while (slots < std::min(batches, kMaxRing) && fused_smem(slots + 1, (int)chunk) <= kMaxSmem) ++slots;
    const size_t smem = fused_smem(slots, (int)chunk);
    static bool attr[64] = {};
    if (dev >= 0 && dev < 64 && !attr[dev]) {
        if (cudaFuncSetAttribute(index_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)kMaxSmem) != cudaSuccess)
            return false;
        attr[dev] = true;
    }
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, index_fused_kernel, kThreads, smem) != cudaSuccess ||
        per_sm < 1)
        return false;
    if ((int64_t)G * n_groups > (int64_t)per_sm * n_sm) {
        log_plan("index: %d groups x %d CTAs do not fit (%d per SM): scan + select kernels", n_groups, G, per_sm);
        return false;
    }
    fp.G = G;
    fp.chunk = (int)chunk;
    fp.ring_slots = slots;
    fp.smem = smem;
    fp.cap = (int)std::min<size_t>(kCandCap, (size_t)slots * kBatchBytes / 8 - kMaxG / 2);
    log_plan("index: %d groups x %d CTAs of %lld candidates (%d per SM fit), candidate capacity %d", n_groups, G,
             (long long)chunk, per_sm, fp.cap);
    return true;
}

cudaError_t launch_fused(const FusedLaunch &L, const FusedPlan &fp, int *flags, cudaStream_t stream)
{
    if (L.n_jobs <= 0 || L.n_jobs > kMaxFusedJobs) return cudaErrorInvalidValue;
    std::vector<uint8_t> buf(sizeof(FusedParams), 0);
    FusedParams &p = *reinterpret_cast<FusedParams *>(buf.data());
    for (int j = 0; j < L.n_jobs; ++j) {
        const FusedJobDesc &d = L.jobs[j];
        FusedJob &J = p.jobs[j];
        J.keys = d.keys;
        J.pool = d.pool;
        J.pool_len = d.pool_len;
        J.n_q = d.n_q;
        for (int q = 0; q < 2; ++q) {
            J.q_idx[q] = d.q_idx[q];
            J.w[q] = d.w[q];
            J.out_idx[q] = d.out_idx[q];
            J.out_pool[q] = d.out_pool[q];
            J.out_scores[q] = d.out_scores[q];
        }
        J.kv = d.kv;
        J.new_kv = d.new_kv;
        J.new_key = d.new_key;
        J.warm = d.warm;
        J.has_warm = d.has_warm;
    }
    p.seq_lens = L.seq_lens;
    p.state = L.state;
    p.scores_stride = L.scores_stride;
    p.batch = L.batch;
    p.topk = L.topk;
    p.pool_out = L.pool_out;
    p.max_len = L.max_len;
    p.keys_ready = L.keys_ready;
    p.G = fp.G;
    p.chunk = fp.chunk;
    p.cap = fp.cap;
    p.ring_slots = fp.ring_slots;
    p.spin_limit = 1u << 22;
    p.first_wait_limit = g_first_wait_limit >= 0 ? (uint32_t)g_first_wait_limit : tc::kWaitLimit;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)fp.G, (unsigned)L.batch, (unsigned)L.n_jobs);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = fp.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    int dev = 0;
    cudaGetDevice(&dev);
    static int pdl_state[64] = {};  // 0 unknown, 1 accepted, -1 refused with the cooperative attribute
    const bool try_pdl = L.pdl && !(dev >= 0 && dev < 64 && pdl_state[dev] < 0);
    cfg.numAttrs = try_pdl ? 2 : 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, index_fused_kernel, p, flags);
    if (e != cudaSuccess && try_pdl && dev >= 0 && dev < 64 && pdl_state[dev] == 0) {
        (void)cudaGetLastError();
        pdl_state[dev] = -1;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, index_fused_kernel, p, flags);
    } else if (e == cudaSuccess && try_pdl && dev >= 0 && dev < 64) {
        pdl_state[dev] = 1;
    }
    count_launches(1);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

}  // namespace csa2
