// Step 2 of the CSA2 decode path: indexer scoring and deterministic Top-K.
//
// Helmcode "DeepSeek V4.1 Flash" explainer, "03 · CSA2": a Full layer scores
// every position, a Reindex layer rescores a Full layer's keys with its own
// query; Louis Bouchard's KV-cache report, "Share the cache and the search
// work": the decoder's first indexing layer keeps a candidate pool that later
// indexing layers search; 0x0moeen's note: layers share the indexer keys.
// The score form and its rounding points are this library's choice (see
// include/csa2.h) and make the result exact up to a fixed fp32 sequence, so
// the selected index sets are reproducible bit for bit.
//
// Kernels
//  scan    HBM-bound pass over the FP4 keys (36 B per position).  A CTA owns
//          1,024 candidates: for a full-context scan it pulls its 16 key
//          tiles (2,304 B each) into shared memory with bulk async copies
//          completing on one mbarrier, so every tile is in flight at once;
//          for a pool scan it gathers each key.  A thread scores whole keys
//          for up to two queries (a Full layer and the pool-free Reindex
//          layer that shares its keys): the E2M1 block dot products as exact
//          integer sums (dp4a over the doubled codes), then the key scales and
//          head weights in the fixed order.  It writes an order-preserving
//          uint32 key per candidate (0 = not a candidate) and adds its CTA's
//          2,048-bin histogram of the keys' top 11 bits into the row's global
//          histogram.  Used for problems too large for the fused launch.
//  select  one cluster of 8 CTAs per (row, target): an exact radix select
//          of the K-th largest key (11 + 11 + 10 bit digits) with the
//          histograms reduced across the cluster through distributed shared
//          memory, the ties at the threshold resolved to the lowest
//          positions by a prefix over the cluster's slices, and the winners
//          written as ascending positions (-1 padded).
#include <cooperative_groups.h>

#include "internal.h"
#include "scan.cuh"
#include "tc.cuh"

namespace cg = cooperative_groups;

namespace csa2 {
namespace {

constexpr int kScanWarps = 8;
constexpr int kScanKeys = 1024;                 // candidates per scan CTA
constexpr int kScanTiles = kScanKeys / kIdxTile;  // 16 key tiles
constexpr int kSelThreads = 512;

struct ScanBatch {
    ScanJob jobs[kMaxScanJobs];
    float *out_scores[kMaxScanJobs][2];
    int64_t scores_stride;
    int32_t n_jobs;
};

struct __align__(128) ScanSmem {
    uint8_t tiles[kScanTiles][kIdxTileBytes];  // 36,864 B
    uint32_t hist[2][kHistBins];
    scan::QuerySet qs;
    int32_t tile_ok[kScanTiles];
    float sk_lut[256];  // E4M3 code -> value
    uint64_t bar;
};

__global__ void __launch_bounds__(kScanWarps * 32, 4) scan_kernel(const __grid_constant__ ScanBatch sb,
                                                                 SelectBufs bufs, const int32_t *seq_lens,
                                                                 int batch, int max_len, int *flags)
{
    extern __shared__ __align__(128) uint8_t smem_raw[];
    ScanSmem &S = *reinterpret_cast<ScanSmem *>(smem_raw);
    const ScanJob &job = sb.jobs[blockIdx.z];
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    int L = __ldg(seq_lens + b);
    if (L < 0 || L > max_len) {
        if (tid == 0 && blockIdx.x == 0) raise_flag(flags, kFlagBounds);
        L = L < 0 ? 0 : max_len;
    }
    const int64_t n_cand = job.pool ? job.pool_len : L;
    const int64_t base = (int64_t)blockIdx.x * kScanKeys;
    if (base >= n_cand) return;
    const bool direct = job.pool == nullptr;

    // 1. issue the bulk copies of this CTA's key tiles (full-context scans)
    if (direct && tid == 0) {
        tc::mbar_init(&S.bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        uint32_t bytes = 0;
        const uint8_t *src[kScanTiles];
        for (int i = 0; i < kScanTiles; ++i) {
            src[i] = nullptr;
            const int64_t p0 = base + (int64_t)i * kIdxTile;
            int ok = 0;
            if (p0 < n_cand) {
                const int64_t slot = slot_of(job.keys, b, p0);
                // a 64-aligned position block maps to one whole tile (page and stride are multiples of 64)
                if (slot >= 0 && slot + kIdxTile <= job.keys.n_slots) {
                    src[i] = job.keys.data + (slot / kIdxTile) * kIdxTileBytes;
                    bytes += kIdxTileBytes;
                    ok = 1;
                } else {
                    raise_flag(flags, kFlagBounds);
                }
            }
            S.tile_ok[i] = ok;
        }
        tc::mbar_expect_tx(&S.bar, bytes);
        for (int i = 0; i < kScanTiles; ++i)
            if (src[i]) tc::bulk_g2s(S.tiles[i], src[i], kIdxTileBytes, &S.bar);
    }

    for (int i = tid; i < 2 * kHistBins; i += blockDim.x) (&S.hist[0][0])[i] = 0u;
    S.sk_lut[tid] = e4m3_value((uint32_t)tid);  // 256 threads
    scan::prep_query_set(tid, job.n_q, job.q_idx, job.w, b, S.qs);
    __syncthreads();
    const int32_t *pool = job.pool ? job.pool + (int64_t)b * job.pool_len : nullptr;

    // 2. wait for the tiles (bounded)
    bool have_tiles = true;
    if (direct) {
        have_tiles = tc::mbar_wait(&S.bar, 0);
        if (!have_tiles) {
            if (tid == 0) raise_flag(flags, kFlagTimeout);
            tc::mbar_wait(&S.bar, 0);  // give copies in flight a last chance to land
        }
    }

    // 3. one thread scores whole keys, for every query of the job
#pragma unroll 1
    for (int i = tid; i < kScanKeys; i += kScanWarps * 32) {
        const int64_t cc = base + i;
        bool ok = cc < n_cand;
        uint4 c0v = make_uint4(0u, 0u, 0u, 0u), c1v = c0v;
        uint32_t scw = 0u;
        if (ok && direct) {
            const int ti = i / kIdxTile, rr = i % kIdxTile;
            ok = have_tiles && S.tile_ok[ti];
            c0v = *reinterpret_cast<const uint4 *>(S.tiles[ti] + rr * 32);
            c1v = *reinterpret_cast<const uint4 *>(S.tiles[ti] + rr * 32 + 16);
            scw = *reinterpret_cast<const uint32_t *>(S.tiles[ti] + kIdxTile * 32 + rr * 4);
        } else if (ok) {
            const int64_t pos = (int64_t)__ldcg(pool + cc);
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
        uint32_t kw[16];
        float sk[4];
        scan::unpack_key(c0v, c1v, scw, S.sk_lut, kw, sk);
        for (int q = 0; q < job.n_q; ++q) {
            const float sc = scan::score_key_int(kw, sk, S.qs, q);
            const uint32_t key = ok ? score_key(sc) : 0u;
            if (cc < n_cand) {
                bufs.keys[((int64_t)job.row[q] * batch + b) * bufs.cand_cap + cc] = key;
                if (ok) {
                    atomicAdd(&S.hist[q][key >> (32 - kHistBits)], 1u);
                    float *so = sb.out_scores[blockIdx.z][q];
                    if (so) so[(int64_t)b * sb.scores_stride + cc] = sc;
                }
            }
        }
    }
    __syncthreads();
    for (int qi = 0; qi < job.n_q; ++qi) {
        uint32_t *gh = bufs.hist + ((int64_t)job.row[qi] * batch + b) * kHistBins;
        for (int i = tid; i < kHistBins; i += blockDim.x) {
            const uint32_t c = S.hist[qi][i];
            if (c) atomicAdd(gh + i, c);
        }
    }
}

// ---- threshold search over a histogram (block-wide) --------------------------
// Finds bin d with above(d) < need <= above(d) + h[d], where above(d) is the
// count in bins > d.  If the total is < need, returns bin = -1, above = total.
// Requires nbins % NT == 0.
struct Thresh {
    int bin;
    uint32_t above;
    uint32_t at;
};

template <int NT>
__device__ Thresh find_threshold(const uint32_t *h, int nbins, uint32_t need, uint32_t *scratch /*>= NT/32+3*/)
{
    const int tid = threadIdx.x;
    const int per = nbins / NT;
    const int hi = nbins - tid * per;  // this thread covers [hi - per, hi), descending from the top
    uint32_t local = 0;
    for (int i = 1; i <= per; ++i) local += h[hi - i];
    uint32_t incl = local;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = (lane < NT / 32) ? scratch[lane] : 0u;
        uint32_t s = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t u = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += u;
        }
        if (lane < NT / 32) scratch[lane] = s - v;      // exclusive warp offsets
        if (lane == NT / 32 - 1) scratch[NT / 32] = s;  // total
    }
    __syncthreads();
    const uint32_t excl = scratch[warp] + incl - local;
    const uint32_t total = scratch[NT / 32];
    __syncthreads();
    if (total < need) {
        if (tid == 0) {
            scratch[NT / 32 + 1] = 0xFFFFFFFFu;
            scratch[NT / 32 + 2] = total;
        }
    } else if (excl < need && need <= excl + local) {
        uint32_t above = excl;
        for (int i = 1; i <= per; ++i) {
            const uint32_t c = h[hi - i];
            if (need <= above + c) {
                scratch[NT / 32 + 1] = (uint32_t)(hi - i);
                scratch[NT / 32 + 2] = above;
                break;
            }
            above += c;
        }
    }
    __syncthreads();
    Thresh r;
    r.bin = (int)scratch[NT / 32 + 1];
    r.above = scratch[NT / 32 + 2];
    r.at = (r.bin >= 0) ? h[r.bin] : 0u;
    __syncthreads();
    return r;
}

__device__ __forceinline__ int row_len(const int32_t *seq_lens, int b, int max_len)
{
    int L = __ldg(seq_lens + b);
    return L < 0 ? 0 : (L > max_len ? max_len : L);
}

struct SelSmem {
    uint32_t h1[2048];   // local histogram of digit 2 (read by the cluster)
    uint32_t h2[1024];   // local histogram of digit 3 (read by the cluster)
    uint32_t red[2048];  // cluster-reduced histogram (this CTA's copy)
    uint32_t cnt[4];     // [0] keys above T in this CTA, [1] ties at T (read by the cluster)
    uint32_t wabove[kSelThreads / 32];
    uint32_t wties[kSelThreads / 32];
    uint32_t scratch[48];
};

constexpr int kSelWarps = kSelThreads / 32;
constexpr int kSelUnroll = 4;  // independent key loads in flight per lane

// Visits a warp's contiguous range [r0, r1) in order, 32 keys per step (lane
// = key), kSelUnroll steps of loads in flight: f(c, key, in_range) is called
// by every lane of the warp for every step (f may use warp collectives).
template <class F>
__device__ __forceinline__ void for_range(const uint32_t *src, int64_t base, int64_t r0, int64_t r1, F &&f)
{
    const int lane = threadIdx.x & 31;
    for (int64_t c0 = r0; c0 < r1; c0 += 32 * kSelUnroll) {
        uint32_t k[kSelUnroll];
#pragma unroll
        for (int j = 0; j < kSelUnroll; ++j) {
            const int64_t c = c0 + 32 * j + lane;
            k[j] = (c < r1) ? src[c - base] : 0u;
        }
#pragma unroll
        for (int j = 0; j < kSelUnroll; ++j) {
            const int64_t c = c0 + 32 * j + lane;
            f(c, k[j], c < r1);
        }
    }
}

// ---- select (one cluster of CS CTAs per row and target) -------------------------
// The row's candidates are split into CS contiguous slices (one per
// CTA) and each slice into kSelWarps contiguous warp ranges, so position
// order is (CTA rank, warp, lane).  Dynamic shared memory holds the CTA's
// slice of keys when it fits (staged); otherwise the passes read it from
// global memory (L2).
template <int CS>
__global__ void __launch_bounds__(kSelThreads)
    select_kernel(SelectPlan plan, int max_len, int64_t stage_cap, int *flags)
{
    __shared__ SelSmem S;
    __shared__ uint64_t stage_bar;
    extern __shared__ __align__(16) uint32_t staged_keys[];
    cg::cluster_group cluster = cg::this_cluster();
    const uint32_t rank = cluster.block_rank();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rb = blockIdx.y / plan.batch, b = blockIdx.y % plan.batch, tg = blockIdx.z;
    const SelectRow &R = plan.rows[rb];
    if (tg == 1 && !(R.out_pool && plan.pool_out_len > 0)) return;  // uniform across the cluster
    const int64_t row = (int64_t)rb * plan.batch + b;
    const int L = row_len(plan.seq_lens, b, max_len);
    const int64_t n_cand = R.pool ? R.pool_len : L;
    const uint32_t K = (uint32_t)(tg == 0 ? plan.topk : plan.pool_out_len);
    int32_t *out = (tg == 0 ? R.out_idx : R.out_pool) + (int64_t)b * K;
    const uint32_t *keys = plan.bufs.keys + row * plan.bufs.cand_cap;
    const int32_t *pool = R.pool ? R.pool + (int64_t)b * R.pool_len : nullptr;
    // slices of a multiple of 32 keys, so each starts 128-B aligned
    const int64_t chunk = ceil_div(ceil_div(n_cand, CS), 32) * 32;
    const int64_t s0 = min(n_cand, (int64_t)rank * chunk), s1 = min(n_cand, s0 + chunk);
    const int64_t span = ceil_div(s1 - s0, kSelWarps);
    const int64_t r0 = min(s1, s0 + warp * span), r1 = min(s1, r0 + span);
    const bool staged = (s1 - s0) <= stage_cap;
    const uint32_t *src = staged ? staged_keys : keys;
    const int64_t base = staged ? s0 : 0;

    // digit 1: the global histogram of the top 11 bits (built by the scan)
    for (int i = tid; i < 2048; i += kSelThreads) S.red[i] = plan.bufs.hist[row * kHistBins + i];
    for (int i = tid; i < 2048; i += kSelThreads) S.h1[i] = 0u;
    for (int i = tid; i < 1024; i += kSelThreads) S.h2[i] = 0u;
    // stage the slice with bulk async copies (16-B multiples; the row is padded to 64 keys)
    const uint32_t stage_bytes = staged ? (uint32_t)(ceil_div(s1 - s0, 4) * 16) : 0u;
    if (stage_bytes && tid == 0) {
        tc::mbar_init(&stage_bar, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        tc::mbar_expect_tx(&stage_bar, stage_bytes);
        for (uint32_t off = 0; off < stage_bytes; off += 16384u)
            tc::bulk_g2s(reinterpret_cast<uint8_t *>(staged_keys) + off,
                     reinterpret_cast<const uint8_t *>(keys + s0) + off, min(16384u, stage_bytes - off), &stage_bar);
    }
    __syncthreads();
    if (stage_bytes && !tc::mbar_wait(&stage_bar, 0)) {
        if (tid == 0) raise_flag(flags, kFlagTimeout);
        tc::mbar_wait(&stage_bar, 0);  // give copies in flight a last chance to land
    }
    const Thresh t0 = find_threshold<kSelThreads>(S.red, 2048, K, S.scratch);
    const bool all_valid = t0.bin < 0;  // fewer candidates than K: take every valid one
    uint32_t T = 0;                      // threshold key: select key > T, plus ties at T
    uint32_t ties_needed = 0;
    if (!all_valid) {
        // digit 2: histogram of the threshold bin's keys
        const uint32_t d0 = (uint32_t)t0.bin;
        for_range(src, base, r0, r1, [&](int64_t, uint32_t k, bool) {
            if (k != 0u && (k >> 21) == d0) atomicAdd(&S.h1[(k >> 10) & 2047u], 1u);
        });
        __syncthreads();
        cluster.sync();
        for (int i = tid; i < 2048; i += kSelThreads) {
            uint32_t v = 0;
#pragma unroll
            for (int r = 0; r < CS; ++r) v += cluster.map_shared_rank(S.h1, r)[i];
            S.red[i] = v;
        }
        __syncthreads();
        const Thresh t1 = find_threshold<kSelThreads>(S.red, 2048, K - t0.above, S.scratch);
        // digit 3
        const uint32_t p01 = (d0 << 11) | (uint32_t)t1.bin;
        for_range(src, base, r0, r1, [&](int64_t, uint32_t k, bool) {
            if (k != 0u && (k >> 10) == p01) atomicAdd(&S.h2[k & 1023u], 1u);
        });
        __syncthreads();
        cluster.sync();
        for (int i = tid; i < 1024; i += kSelThreads) {
            uint32_t v = 0;
#pragma unroll
            for (int r = 0; r < CS; ++r) v += cluster.map_shared_rank(S.h2, r)[i];
            S.red[i] = v;
        }
        __syncthreads();
        const Thresh t2 = find_threshold<kSelThreads>(S.red, 1024, K - t0.above - t1.above, S.scratch);
        T = (p01 << 10) | (uint32_t)t2.bin;
        ties_needed = K - t0.above - t1.above - t2.above;
    }
    // per-warp counts of keys above T and of ties at T, in position order
    uint32_t wa = 0, wt = 0;
    for_range(src, base, r0, r1, [&](int64_t, uint32_t k, bool) {
        const bool valid = k != 0u;
        wa += __popc(__ballot_sync(0xFFFFFFFFu, valid && (all_valid || k > T)));
        wt += __popc(__ballot_sync(0xFFFFFFFFu, valid && !all_valid && k == T));
    });
    if (lane == 0) {
        S.wabove[warp] = wa;
        S.wties[warp] = wt;
    }
    __syncthreads();
    if (tid == 0) {
        uint32_t a = 0, t = 0;
        for (int w = 0; w < kSelWarps; ++w) {
            a += S.wabove[w];
            t += S.wties[w];
        }
        S.cnt[0] = a;
        S.cnt[1] = t;
    }
    __syncthreads();
    cluster.sync();
    // CTA-level prefixes over the cluster (rank order = position order)
    uint32_t tie_before = 0, sel_before = 0, total = 0;
    {
        uint32_t tb = 0;
        for (int r = 0; r < CS; ++r) {
            const uint32_t *c = cluster.map_shared_rank(S.cnt, r);
            const uint32_t ab = c[0], ti = c[1];
            const uint32_t q = (ties_needed > tb) ? min(ties_needed - tb, ti) : 0u;
            if ((uint32_t)r < rank) {
                tie_before += ti;
                sel_before += ab + q;
            }
            total += ab + q;
            tb += ti;
        }
    }
    __syncthreads();
    cluster.sync();  // no remote shared-memory reads after this point
    // warp-level prefixes inside the CTA
    uint32_t wtie_before = tie_before, wsel_before = sel_before;
    for (int w = 0; w < warp; ++w) {
        const uint32_t ti = S.wties[w];
        const uint32_t q = (ties_needed > wtie_before) ? min(ties_needed - wtie_before, ti) : 0u;
        wsel_before += S.wabove[w] + q;
        wtie_before += ti;
    }
    const uint32_t quota = (ties_needed > wtie_before) ? min(ties_needed - wtie_before, wt) : 0u;

    // write this warp's winners in position order
    const uint32_t lt = (1u << lane) - 1u;
    uint32_t written = 0, ties_seen = 0;
    for_range(src, base, r0, r1, [&](int64_t c, uint32_t k, bool) {
        const bool valid = k != 0u;
        const bool is_tie = valid && !all_valid && k == T;
        const uint32_t tm = __ballot_sync(0xFFFFFFFFu, is_tie);
        const uint32_t tie_rank = ties_seen + __popc(tm & lt);
        const bool sel = valid && (all_valid || k > T || (is_tie && tie_rank < quota));
        const uint32_t sm = __ballot_sync(0xFFFFFFFFu, sel);
        if (sel) {
            const uint32_t at = wsel_before + written + __popc(sm & lt);
            if (at < K) out[at] = pool ? __ldg(pool + c) : (int32_t)c;
        }
        written += __popc(sm);
        ties_seen += __popc(tm);
    });
    for (uint32_t i = total + rank * kSelThreads + tid; i < K; i += CS * kSelThreads) out[i] = -1;
}

}  // namespace

// Key rows are padded to a multiple of 64 candidates (256 B) so every row and
// every select slice starts 16-B aligned for bulk copies.
static int64_t padded_cap(int64_t cand_cap) { return ceil_div(cand_cap, 64) * 64; }

size_t select_bytes(int n_rows, int64_t cand_cap, int max_seq_len)
{
    (void)max_seq_len;
    auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
    return r256((size_t)n_rows * kHistBins * 4) + r256((size_t)n_rows * padded_cap(cand_cap) * 4);
}

SelectBufs carve_select(uint8_t *base, int n_rows, int64_t cand_cap, int max_seq_len)
{
    (void)max_seq_len;
    SelectBufs s;
    s.cand_cap = padded_cap(cand_cap);
    s.hist = reinterpret_cast<uint32_t *>(base);
    s.keys = reinterpret_cast<uint32_t *>(base + (((size_t)n_rows * kHistBins * 4 + 255) & ~(size_t)255));
    return s;
}

size_t select_hist_bytes(int n_rows) { return (size_t)n_rows * kHistBins * 4; }

cudaError_t launch_scan(const ScanJob *jobs, int n_jobs, const SelectPlan &plan, int max_cand,
                        float *const (*scores)[2], int64_t scores_stride, int *flags, cudaStream_t stream)
{
    const size_t smem = sizeof(ScanSmem);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    for (int first = 0; first < n_jobs; first += kMaxScanJobs) {
        ScanBatch sb;
        sb.n_jobs = (n_jobs - first < kMaxScanJobs) ? n_jobs - first : kMaxScanJobs;
        sb.scores_stride = scores_stride;
        for (int j = 0; j < sb.n_jobs; ++j) {
            sb.jobs[j] = jobs[first + j];
            sb.out_scores[j][0] = scores ? scores[first + j][0] : nullptr;
            sb.out_scores[j][1] = scores ? scores[first + j][1] : nullptr;
        }
        dim3 grid((unsigned)ceil_div(max_cand > 0 ? max_cand : 1, kScanKeys), (unsigned)plan.batch,
                  (unsigned)sb.n_jobs);
        scan_kernel<<<grid, kScanWarps * 32, smem, stream>>>(sb, plan.bufs, plan.seq_lens, plan.batch,
                                                             plan.max_len, flags);
        count_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

// Launches select_kernel<CS> as clusters of CS CTAs along x.
template <int CS>
cudaError_t launch_select_cs(const SelectPlan &plan, int64_t cap, size_t smem, int *flags, cudaStream_t stream)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)CS, (unsigned)(plan.n_row_blocks * plan.batch), 2u);
    cfg.blockDim = dim3(kSelThreads, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CS;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, select_kernel<CS>, plan, plan.max_len, cap, flags);
}

// Stages up to 160 KB of keys per CTA.  Eight CTAs per row: 16-CTA clusters
// were measured slower (the cross-rank histogram sums grow with the cluster).
// When the rows' 8-CTA clusters would take two waves of the device but
// 4-CTA clusters fit in one (and still stage their slices), 4 are used.
cudaError_t launch_select(const SelectPlan &plan, int max_cand, int *flags, cudaStream_t stream,
                          cudaEvent_t mid_event)
{
    (void)mid_event;
    constexpr int64_t kStageMax = 40960;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int n_sms_of[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!n_sms_of[dev]) {
        e = cudaFuncSetAttribute(select_kernel<8>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kStageMax * 4));
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(select_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)(kStageMax * 4));
        int n = 0;
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        n_sms_of[dev] = n > 0 ? n : 1;
    }
    const int64_t rows = (int64_t)plan.n_row_blocks * plan.batch;
    auto slice_of = [&](int cs) { return ceil_div(ceil_div(max_cand > 0 ? max_cand : 1, cs), 32) * 32; };
    const bool four = rows * 8 > n_sms_of[dev] && rows * 4 <= n_sms_of[dev] && slice_of(4) <= kStageMax;
    const int64_t slice = slice_of(four ? 4 : 8);
    const int64_t cap = slice <= kStageMax ? slice : 0;
    e = four ? launch_select_cs<4>(plan, cap, (size_t)cap * 4, flags, stream)
             : launch_select_cs<8>(plan, cap, (size_t)cap * 4, flags, stream);
    count_launches(1);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace csa2
