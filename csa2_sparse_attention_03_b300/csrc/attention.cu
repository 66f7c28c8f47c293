// Step 3 of the CSA2 decode path: gather of the selected FP4 main-KV rows and
// the FP8 sliding-window rows, dequantisation, and one softmax attention over
// both (Louis Bouchard's KV-cache report, "Share the cache and the search
// work": the selected global entries beside a local 128-token window;
// Helmcode "DeepSeek V4.1 Flash" explainer, "04 · FP4": FP4 global KV, FP8
// window KV; "03 · CSA2": a Reuse layer attends with its own query over the
// selection of another layer).  16 query heads attend over one shared
// 512-channel row that is both key and value.
//
// Work decomposition.  A *unit* is up to NL layers that attend over the same
// selected rows (an indexing layer and Reuse layers that take its Top-K);
// its rows are read and dequantised once for all of them.  The unit's rows
// come in tiles of 128: the selected rows, then each layer's window rows.  One
// thread-block cluster of CS CTAs takes one (unit, sequence); CTA r takes
// tiles r, r + CS, ...  Per tile, with the rows as the M = 128 of every
// tensor-core product and the unit's queries as N:
//   S^T = K Q^T    M 128 rows, N 32 NL (every query twice: its fp16 value
//                  and the fp16 remainder q - fp16(q), so the logits carry
//                  the fp32 query to about 2^-22), K 512 channels;
//   softmax        fp32, per query over the tile's rows, with a running
//                  maximum that moves lazily (only when a tile's maximum
//                  exceeds it by more than 2, rescaling O^T in tensor
//                  memory), so every weight P = exp(z - m) <= e^2 as fp16;
//   O^T += V^T P   M 128 channels (four blocks), N 16 NL queries, K the rows.
// The CTAs of a cluster then merge their partials through distributed shared
// memory: each pushes its running (max, sum) per query into every peer,
// stages its O^T normalised by its own sum, and sends each CTA, by one bulk
// copy, its block of that CTA's slice of the channels; each CTA weighs and
// sums its slice over the cluster and writes it.  When one (unit,
// sequence) has more tiles than a cluster takes well, it is split over two
// clusters, the tiles dealt round-robin over all their CTAs: the second
// cluster's CTAs (satellites) skip the cluster merge and write their partial
// (max, sum, normalised output) to the workspace, then count themselves into
// a counter per owner of a channel slice of the first cluster; each owner
// waits for its counter (bounded, left zero again), and sums the satellites'
// share of its slice with the cluster's.  A split is only planned when every
// cluster of the launch fits on the device at once, so the satellites are
// resident while the owners wait.  With no workspace every (unit, sequence)
// is one cluster.
//
// Value precision: E2M1 x E4M3 values and E4M3 codes x 2^-8 are exact in
// fp16; an FP8 window row's fp32 scale (x 2^8) multiplies its logit in fp32
// and its softmax weight before the weight is rounded to fp16.
//
// The launch may overlap the previous kernel of the stream (programmatic
// dependent launch): barrier set-up and the tensor-memory allocation run
// first, every global read after the dependency wait.
#include <algorithm>
#include <cstring>
#include <vector>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kRows = 128;                       // rows per tile (M of every MMA)
constexpr int kThreads = 256;                    // 8 warps
constexpr int kMaxNL = 2;                        // layers per unit
constexpr int kMaxCS = 16;                       // CTAs per cluster
constexpr int kMaxUnits = 2 * kMaxAttnEntries;
constexpr float kRescaleGap = 2.0f;              // lazy rescale threshold (natural log): P <= e^2
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kTileBytes = kRows * kDim * 2;     // 131,072: one tile, fp16
constexpr int kQBytes = 32 * kDim * 2;           // 32,768 per layer: 16 heads x (value, remainder)
constexpr int kPBytes = kRows * 16 * 2;          // 4,096 per layer

constexpr int kSAcc = 1;                         // QK^T accumulators (partial sums over the channels)
constexpr int kChunks = 4;                       // channel chunks of a row (the layout of a thread's gathered bytes)

template <int NL>
struct Cols {
    static constexpr uint32_t S = 0;               // S^T: kSAcc partial sums of 32 NL columns each
    static constexpr uint32_t O = kSAcc * 32 * NL; // O^T: 4 blocks x 16 NL columns
    static constexpr uint32_t alloc = NL == 1 ? 256 : 512;
};
static_assert(Cols<2>::O + 64 * 2 <= Cols<2>::alloc && Cols<1>::O + 64 <= Cols<1>::alloc, "tensor memory plan");

struct UnitDev {
    CacheView kv;            // FP4_KV cache of the selected rows
    const int32_t *idx;      // [B][topk] or null
    int32_t n_layers;        // 1..kMaxNL
    int32_t entry[kMaxNL];
    int32_t row_tiles;       // ceil(topk / 128) when idx, else 0
    int32_t n_tiles;         // row tiles + n_layers * window tiles
};

struct EntryDev {
    CacheView swa;           // FP8_SWA ring (when the call has a window)
    const float *q;          // [B][16][512]
    const float *new_swa;    // optional [B][512]: quantised into the ring at position L-1 first
    float *out;              // [B][16][512]
    float *lse;              // [B][16] or null
};

struct AttnParams {
    UnitDev units[kMaxUnits];
    EntryDev entries[kMaxAttnEntries];
    int32_t n_units, batch, topk, window, win_tiles, cs;
    int32_t split;           // clusters per (unit, sequence): 1, or 2 (the second one's CTAs are satellites)
    int32_t inputs_ready;    // indices, caches, rings and lengths predate the previous kernel
    const int32_t *seq_lens;
    float *parts;            // split 2: satellite partials [unit][b][satellite rank < cs][kSatFloats]
    uint32_t *tickets;       // split 2: satellite counters per owner rank [unit][b][kMaxCS], zero at launch, left zero
};

// One satellite's partial in the workspace: its running maximum and sum per
// query, then its output normalised by that sum, [query][channel].
constexpr int kSatHdr = 2 * 16 * kMaxNL;
constexpr int kSatFloats = kSatHdr + 16 * kMaxNL * kDim;

struct Misc {
    uint32_t vmask[4];               // valid rows of the tile in the buffer
    float rowfac[kRows];             // per-row logit factor (window rows: fp32 scale x 256)
    float red[4][16 * kMaxNL];       // cross-warp reductions of the softmax warps
    float m_run[16 * kMaxNL];        // running maximum per query
    float l_run[16 * kMaxNL];        // running sum per query (relative to m_run)
    float2 mlall[kMaxCS][16 * kMaxNL];  // merge: every CTA's (m, l) per query, pushed by that CTA
    float wall[kMaxCS][16 * kMaxNL];    // merge: every CTA's (or part's) weight per query
    float cm[16 * kMaxNL], cl[16 * kMaxNL];  // merge: the cluster's (max, sum) per query
    float inv_l[16 * kMaxNL];        // merge: 1 / this CTA's sum per query (0 without rows)
    float2 mlsat[kMaxCS][16 * kMaxNL];  // merge: every satellite's (m, l) per query
    float wsat[kMaxCS][16 * kMaxNL];    // merge: every satellite's final weight per query
    float w0[16 * kMaxNL];              // merge: the final weight of the cluster's merged result
    float mu[16 * kMaxNL];           // the maximum a tile's weights are taken against
    float alpha[16 * kMaxNL];        // factor moving O^T to that maximum
    __align__(16) uint8_t app[kMaxNL][kDim];  // appended window row per layer slot (E4M3 codes)
    float app_scale[kMaxNL];
    float app_max[kMaxNL][4];        // per-warp maxima of an appended row
    uint64_t bar_qk, bar_pv, bar_rx;
    uint32_t tmem_slot;
    int32_t ok;
    int32_t any_resc;
};

template <int NL>
constexpr size_t smem_bytes()
{
    return (size_t)kTileBytes + (size_t)NL * (kQBytes + kPBytes) + sizeof(Misc);
}
static_assert(smem_bytes<2>() <= 232448, "attention shared memory over the 227 KB limit");
// the merge's staged and received blocks (cs x cpc <= 512 + 4 cs <= 576 channels)
// fit the tile and query buffers
static_assert(2 * 16 * kMaxNL * 576 * 4 <= kTileBytes + kMaxNL * kQBytes &&
                  2 * 16 * 1 * 576 * 4 <= kTileBytes + 1 * kQBytes,
              "merge blocks fit");

// Byte offset of fp16 element (row r, channel c) of a 512-channel operand in
// the no-swizzle core-matrix layout: 8-row groups 8,192 B apart, 8-channel
// groups 128 B apart.
__host__ __device__ __forceinline__ uint32_t cm_off(uint32_t r, uint32_t c)
{
    return (r >> 3) * 8192u + (c >> 3) * 128u + (r & 7u) * 16u + (c & 7u) * 2u;
}

__device__ __forceinline__ uint32_t pack_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// Reduces v[0..N) over the 32 lanes of a warp by halving exchanges: after
// the call v[0] holds the reduction of entry qlane(lane) = lane >> (5 -
// log2 N) over all lanes (N = 8, 16 or 32).
template <int N, bool MAX>
__device__ __forceinline__ void warp_transpose_reduce(float (&v)[N], int lane)
{
    static_assert(N == 8 || N == 16 || N == 32, "8, 16 or 32 entries");
    auto op = [](float a, float b) { return MAX ? fmaxf(a, b) : a + b; };
    constexpr int kStages = N == 8 ? 3 : (N == 16 ? 4 : 5);
#pragma unroll
    for (int half = N / 2, bit = 4; half >= 1; half >>= 1, --bit) {
        const bool up = (lane >> bit) & 1;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = up ? v[i] : v[i + half];
            const float keep = up ? v[i + half] : v[i];
            v[i] = op(keep, __shfl_xor_sync(0xFFFFFFFFu, send, 1 << bit));
        }
    }
    // the lanes that share an entry hold partials over the rest of the lane bits
#pragma unroll
    for (int bit = 4 - kStages; bit >= 0; --bit) v[0] = op(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], 1 << bit));
}

// A thread's share of a tile, in registers between its loads and its
// dequantisation.
//  - Row tile (FP4 main KV) by quarter rows, when a CTA takes more than one
//    tile: rows 16 w + i and 16 w + 8 + i (w = tid / 32, i = tid % 8), a
//    quarter of each: lane quarter q = (tid / 8) % 4 holds the row's code
//    bytes 64 q + 16 s (s = 0..3: channels 128 q + 32 s .. + 31) and its
//    block scales 8 q .. 8 q + 7.  One load of a warp so reads a 16-byte
//    piece of 8 rows, four lanes to a row (8 cache lines, not 32), and the
//    dequantised 16-byte stores of a warp fill four whole 128-byte
//    core-matrix rows.  The loads of the next tile then issue in about a
//    quarter of the time.
//  - Otherwise by half rows, like a window tile: row r = tid % 128, channels
//    128 k + 64 h .. + 63 of every chunk k (h = tid / 128); one position
//    load per row, the shortest chain for a CTA's only tile.
struct Raw {
    uint4 g[16];     // quarter rows: row g's piece s in g[4 g + s], its scales in words 2 g, 2 g + 1 of g[8];
                     // half rows, FP4: chunk k's codes in g[2 k], g[2 k + 1], its 4 scales in word k of g[8];
                     // window tile: chunk k in g[4 k .. 4 k + 3]
    float scale;     // window tile: the row's fp32 scale
    int32_t app;     // window tile: layer slot whose appended row this is, or -1
    bool valid;      // the thread's (first) row
    bool valid1;     // quarter rows: the thread's second row
};

struct Ctx {
    const AttnParams *P;
    const UnitDev *U;
    Misc *M;
    int *flags;
    int b, L, W;
    bool quarter;    // row tiles by quarter rows
};

__device__ __forceinline__ bool tile_is_window(const UnitDev &U, int tile) { return tile >= U.row_tiles; }

// Row g (0, 1) of thread tid in a row tile, and the thread's quarter of it.
__device__ __forceinline__ int quarter_row(int tid, int g) { return 16 * (tid >> 5) + 8 * g + (tid & 7); }
__device__ __forceinline__ int row_quarter(int tid) { return (tid >> 3) & 3; }

// Selected positions of a thread's rows of a row tile (-1: none, or a
// window tile): two rows by quarters, or row tid % 128 (and none) by halves.
// Loaded a tile ahead of the row gather so that the gather never waits on
// them.
struct RowPos {
    int32_t p[2];
};

__device__ __forceinline__ RowPos no_rows() { return RowPos{{-1, -1}}; }

__device__ __forceinline__ RowPos load_pos(const Ctx &c, int tile)
{
    const UnitDev &U = *c.U;
    RowPos rp = no_rows();
    if (tile_is_window(U, tile)) return rp;
    const int32_t *sel = U.idx + (int64_t)c.b * c.P->topk;
    if (!c.quarter) {
        const int v = tile * kRows + (threadIdx.x & (kRows - 1));
        if (v < c.P->topk) rp.p[0] = __ldcg(sel + v);
        return rp;
    }
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int v = tile * kRows + quarter_row(threadIdx.x, g);
        if (v < c.P->topk) rp.p[g] = __ldcg(sel + v);
    }
    return rp;
}

// The selected rows' places in the main-KV cache, found in two steps so that
// a paged cache's page-table loads are in flight while other work runs:
// row_issue() starts the loads of the physical pages, row_slot() forms a
// slot (the same slot as slot_of: -1 when the page is unmapped or out of
// range, or the position is not below the sequence length).
struct RowRef {
    int32_t pos[2];   // selected positions, -1 for none
    int32_t phys[2];  // paged cache: physical page of pos, -1 when unmapped or out of range
};

__device__ __forceinline__ RowRef row_issue(const Ctx &c, RowPos rp)
{
    const CacheView &kv = c.U->kv;
    RowRef ref;
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        ref.pos[g] = rp.p[g];
        ref.phys[g] = -1;
        if (kv.page_size != 0 && rp.p[g] >= 0 && rp.p[g] < c.L) {
            const int32_t pg = rp.p[g] / kv.page_size;  // p >= 0, page_size > 0
            if (pg < kv.max_pages) ref.phys[g] = __ldg(kv.page_table + (int64_t)c.b * kv.max_pages + pg);
        }
    }
    return ref;
}

__device__ __forceinline__ int64_t row_slot(const Ctx &c, int32_t pos, int32_t phys)
{
    const CacheView &kv = c.U->kv;
    if (pos < 0 || pos >= c.L) return -1;
    int64_t s;
    if (kv.page_size == 0) {
        s = (int64_t)c.b * kv.seq_stride + pos;
    } else {
        if (phys < 0) return -1;
        s = (int64_t)phys * kv.page_size + pos % kv.page_size;
    }
    return (s >= 0 && s < kv.n_slots) ? s : -1;
}

// Issues the loads of this thread's share of `tile` into registers (`ref`:
// row_issue of its rows' positions for a row tile).
__device__ __forceinline__ void gather(const Ctx &c, int tile, const RowRef &ref, int r, int h, Raw &raw)
{
    const UnitDev &U = *c.U;
    raw.valid = false;
    raw.valid1 = false;
    raw.scale = 0.0f;
    raw.app = -1;
    if (!tile_is_window(U, tile)) {
        const int q = row_quarter(threadIdx.x);
#pragma unroll
        for (int g = 0; g < 2; ++g) {
            if (g > 0 && !c.quarter) break;
            const uint8_t *ptr = nullptr;
            if (ref.pos[g] >= 0) {
                const int64_t slot = row_slot(c, ref.pos[g], ref.phys[g]);
                if (slot < 0) {
                    if ((c.quarter ? q : h) == 0) raise_flag(c.flags, kFlagBounds);
                } else {
                    ptr = U.kv.data + slot * kKvRow;
                }
            }
            if (g == 0) raw.valid = ptr != nullptr;
            else raw.valid1 = ptr != nullptr;
            if (!ptr) continue;
            if (c.quarter) {
#pragma unroll
                for (int p = 0; p < 4; ++p)
                    raw.g[4 * g + p] = __ldcg(reinterpret_cast<const uint4 *>(ptr + 64 * q + 16 * p));
                const uint2 sc = __ldcg(reinterpret_cast<const uint2 *>(ptr + kKvCodes + 8 * q));
                (&raw.g[8].x)[2 * g] = sc.x;
                (&raw.g[8].x)[2 * g + 1] = sc.y;
            } else {
#pragma unroll
                for (int k = 0; k < kChunks; ++k) {
                    const uint4 *codes = reinterpret_cast<const uint4 *>(ptr + 64 * k + 32 * h);
                    raw.g[2 * k] = __ldcg(codes);
                    raw.g[2 * k + 1] = __ldcg(codes + 1);
                    (&raw.g[8].x)[k] = __ldcg(reinterpret_cast<const uint32_t *>(ptr + kKvCodes + 8 * k + 4 * h));
                }
            }
        }
    } else {
        const int wt = tile - U.row_tiles;
        const int j = wt / c.P->win_tiles;
        const int k = wt % c.P->win_tiles;
        const int rowi = k * kRows + r;
        const int64_t pos = (int64_t)c.L - c.W + rowi;
        if (rowi < c.W && pos >= 0) {
            const EntryDev &E = c.P->entries[U.entry[j]];
            if (E.new_swa && pos == (int64_t)c.L - 1) {
                // the row this CTA appends itself: taken from shared memory at dequantisation
                raw.valid = true;
                raw.app = j;
            } else {
                const int64_t slot = slot_of(E.swa, c.b, pos);
                if (slot < 0) {
                    if (h == 0) raise_flag(c.flags, kFlagBounds);
                } else {
                    raw.valid = true;
#pragma unroll
                    for (int k = 0; k < kChunks; ++k) {
                        const uint4 *codes = reinterpret_cast<const uint4 *>(E.swa.data + slot * kDim + 128 * k + 64 * h);
#pragma unroll
                        for (int i = 0; i < 4; ++i) raw.g[4 * k + i] = __ldcg(codes + i);
                    }
                    raw.scale = __ldcg(reinterpret_cast<const float *>(E.swa.data + E.swa.n_slots * kDim) + slot);
                }
            }
        }
    }
}

// Dequantises this thread's part of channel chunk k of its window row into
// the tile buffer (exact fp16): channels 128 k + 64 h .. + 63.
__device__ __forceinline__ void dequant_window_chunk(const Ctx &c, int r, int h, int k, const Raw &raw, uint8_t *T)
{
    const int ch0 = 128 * k + 64 * h;
    if (!raw.valid) {
#pragma unroll
        for (int g = 0; g < 8; ++g) *reinterpret_cast<uint4 *>(T + cm_off(r, ch0 + 8 * g)) = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const __half2 k2m8 = __half2half2(__float2half_rn(0.00390625f));  // 2^-8
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint4 cw = raw.g[4 * k + i];
        if (raw.app >= 0) cw = *reinterpret_cast<const uint4 *>(&c.M->app[raw.app][ch0 + 16 * i]);
        const int ch = ch0 + 16 * i;
        *reinterpret_cast<uint4 *>(T + cm_off(r, ch)) =
            make_uint4(pack_h2(__hmul2(e4m3x2_half2(cw.x & 0xFFFFu), k2m8)),
                       pack_h2(__hmul2(e4m3x2_half2(cw.x >> 16), k2m8)),
                       pack_h2(__hmul2(e4m3x2_half2(cw.y & 0xFFFFu), k2m8)),
                       pack_h2(__hmul2(e4m3x2_half2(cw.y >> 16), k2m8)));
        *reinterpret_cast<uint4 *>(T + cm_off(r, ch + 8)) =
            make_uint4(pack_h2(__hmul2(e4m3x2_half2(cw.z & 0xFFFFu), k2m8)),
                       pack_h2(__hmul2(e4m3x2_half2(cw.z >> 16), k2m8)),
                       pack_h2(__hmul2(e4m3x2_half2(cw.w & 0xFFFFu), k2m8)),
                       pack_h2(__hmul2(e4m3x2_half2(cw.w >> 16), k2m8)));
    }
}

// Dequantises this thread's quarters of its two rows of a row tile into the
// tile buffer (exact fp16: an E2M1 value times an E4M3 scale).  Piece s of
// quarter q is channels 128 q + 32 s .. + 31, two 16-channel blocks whose
// scales are bytes 2 s, 2 s + 1 of the quarter's eight.
__device__ __forceinline__ void dequant_rows(const Raw &raw, uint8_t *T)
{
    const int tid = threadIdx.x, q = row_quarter(tid);
#pragma unroll
    for (int g = 0; g < 2; ++g) {
        const int R = quarter_row(tid, g);
        const bool ok = g == 0 ? raw.valid : raw.valid1;
#pragma unroll
        for (int p = 0; p < 4; ++p) {
            const int ch = 128 * q + 32 * p;
            if (!ok) {
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    *reinterpret_cast<uint4 *>(T + cm_off(R, ch + 8 * j)) = make_uint4(0u, 0u, 0u, 0u);
                continue;
            }
            const uint32_t sw = (&raw.g[8].x)[2 * g + (p >> 1)];
            const __half2 sp = e4m3x2_half2((p & 1) ? (sw >> 16) : (sw & 0xFFFFu));  // the piece's two block scales
            const uint4 cw = raw.g[4 * g + p];  // 32 codes, channel 2 b in the low nibble of byte b
#pragma unroll
            for (int blk = 0; blk < 2; ++blk) {
                const __half2 s2 = blk ? __high2half2(sp) : __low2half2(sp);
                const uint32_t w0 = blk ? cw.z : cw.x, w1 = blk ? cw.w : cw.y;  // 16 codes
                uint32_t hv[8];
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const uint32_t bits = e2m1x2_half2_bits(((i < 4 ? w0 : w1) >> (8 * (i & 3))) & 0xFFu);
                    hv[i] = pack_h2(__hmul2(*reinterpret_cast<const __half2 *>(&bits), s2));
                }
                *reinterpret_cast<uint4 *>(T + cm_off(R, ch + 16 * blk)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
                *reinterpret_cast<uint4 *>(T + cm_off(R, ch + 16 * blk + 8)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
            }
        }
    }
}

// Dequantises this thread's half of channel chunk k of its row of a row tile
// (half rows; exact fp16): channels 128 k + 64 h .. + 63, four 16-channel
// blocks whose scales are byte blk of word k.
__device__ __forceinline__ void dequant_half_chunk(int r, int h, int k, const Raw &raw, uint8_t *T)
{
    const int ch0 = 128 * k + 64 * h;
    if (!raw.valid) {
#pragma unroll
        for (int g = 0; g < 8; ++g) *reinterpret_cast<uint4 *>(T + cm_off(r, ch0 + 8 * g)) = make_uint4(0u, 0u, 0u, 0u);
        return;
    }
    const uint32_t sw = (&raw.g[8].x)[k];  // the four blocks' scales, block 0 in the low byte
    const __half2 s01 = e4m3x2_half2(sw & 0xFFFFu), s23 = e4m3x2_half2(sw >> 16);
#pragma unroll
    for (int blk = 0; blk < 4; ++blk) {
        const __half2 sp = blk < 2 ? s01 : s23;
        const __half2 s2 = (blk & 1) ? __high2half2(sp) : __low2half2(sp);
        const uint4 cw = raw.g[2 * k + (blk >> 1)];
        const uint32_t w0 = (blk & 1) ? cw.z : cw.x, w1 = (blk & 1) ? cw.w : cw.y;  // 16 codes
        uint32_t hv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const uint32_t bits = e2m1x2_half2_bits(((i < 4 ? w0 : w1) >> (8 * (i & 3))) & 0xFFu);
            hv[i] = pack_h2(__hmul2(*reinterpret_cast<const __half2 *>(&bits), s2));
        }
        *reinterpret_cast<uint4 *>(T + cm_off(r, ch0 + 16 * blk)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(T + cm_off(r, ch0 + 16 * blk + 8)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
    }
}

// Dequantises this thread's whole share of the tile.
__device__ __forceinline__ void dequant(const Ctx &c, bool window, int r, int h, const Raw &raw, uint8_t *T)
{
    if (!window && c.quarter) {
        dequant_rows(raw, T);
        return;
    }
#pragma unroll
    for (int k = 0; k < kChunks; ++k) {
        if (window) dequant_window_chunk(c, r, h, k, raw, T);
        else dequant_half_chunk(r, h, k, raw, T);
    }
}

// Quantises a layer's appended window row into its ring slot at position
// L-1 (FP8, scale = absmax / 448) and keeps the codes in shared memory for
// this CTA's own window tile.  128 threads (four warps, named barrier 1 + j);
// thread t: channels 4t .. 4t+3.  With `patch`, also writes the row's fp16
// values into row r_app of the (already dequantised) tile buffer.
__device__ __forceinline__ void append_window_row(const Ctx &c, const EntryDev &E, int j, int t, bool patch, int r_app,
                                                  uint8_t *T)
{
    Misc &M = *c.M;
    const float4 v = __ldcg(reinterpret_cast<const float4 *>(E.new_swa + (int64_t)c.b * kDim) + t);
    float amax = fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w)));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
    if ((t & 31) == 0) M.app_max[j][t >> 5] = amax;
    if (j == 0)
        asm volatile("bar.sync 1, 128;\n" ::: "memory");
    else
        asm volatile("bar.sync 2, 128;\n" ::: "memory");
    amax = fmaxf(fmaxf(M.app_max[j][0], M.app_max[j][1]), fmaxf(M.app_max[j][2], M.app_max[j][3]));
    const float s = __fdiv_rn(amax, 448.0f);
    uint32_t w = 0u;
    if (s != 0.0f)
        w = e4m3_code(__fdiv_rn(v.x, s)) | (e4m3_code(__fdiv_rn(v.y, s)) << 8) | (e4m3_code(__fdiv_rn(v.z, s)) << 16) |
            (e4m3_code(__fdiv_rn(v.w, s)) << 24);
    reinterpret_cast<uint32_t *>(M.app[j])[t] = w;
    const int64_t slot = slot_of(E.swa, c.b, (int64_t)c.L - 1);
    if (slot < 0) {
        if (t == 0) raise_flag(c.flags, kFlagBounds);
    } else {
        reinterpret_cast<uint32_t *>(E.swa.data + slot * kDim)[t] = w;
        if (t == 0) reinterpret_cast<float *>(E.swa.data + E.swa.n_slots * kDim)[slot] = s;
    }
    if (t == 0) M.app_scale[j] = s;
    if (patch) {
        // the row in the tile buffer: codes x 2^-8 (exact in fp16), its row factor
        const __half2 k2m8 = __half2half2(__float2half_rn(0.00390625f));
        *reinterpret_cast<uint2 *>(T + cm_off(r_app, 4 * t)) =
            make_uint2(pack_h2(__hmul2(e4m3x2_half2(w & 0xFFFFu), k2m8)), pack_h2(__hmul2(e4m3x2_half2(w >> 16), k2m8)));
        if (t == 0) M.rowfac[r_app] = s * 256.0f;
    }
}

// Softmax of one tile, all eight warps: thread (row r = TMEM lane, query half
// qh = warp / 4) takes half of the queries of its row.  Writes P as fp16 into
// the PV operand, updates the running (m, l) and rescales O^T in tensor
// memory when a query's maximum moves.
template <int NL>
__device__ __forceinline__ void softmax_tile(const Ctx &c, uint32_t tmem, uint8_t *Ps, int tile, bool first)
{
    constexpr int NQ = 16 * NL, NH = NQ / 2;
    Misc &M = *c.M;
    const UnitDev &U = *c.U;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, quad = warp & 3, qh = warp >> 2;
    const int r = tid & (kRows - 1);
    const bool window = tile_is_window(U, tile);
    const int owner = window ? (tile - U.row_tiles) / c.P->win_tiles : -1;
    const int ql = lane >> (NH == 8 ? 2 : 1);  // this lane's entry after a transpose reduction
    // S^T: this half's value columns qh NH.. and remainder columns NQ + qh NH..
    float s[NH], v[NH];
    {
        float hv[NH], lv[NH];
        tc::tmem_ld<NH>(tc::taddr(tmem, 32u * quad, Cols<NL>::S + (uint32_t)(qh * NH)), hv);
        tc::tmem_ld<NH>(tc::taddr(tmem, 32u * quad, Cols<NL>::S + (uint32_t)(NQ + qh * NH)), lv);
#pragma unroll
        for (int i = 0; i < NH; ++i) s[i] = hv[i] + lv[i];
    }
    const bool valid = (M.vmask[r >> 5] >> (r & 31)) & 1u;
    const float fac = M.rowfac[r];
    // logits times the row factor
#pragma unroll
    for (int i = 0; i < NH; ++i) {
        const int q = qh * NH + i, j = q >> 4;
        const bool own = window ? (j == owner) : (j < U.n_layers);
        s[i] = (valid && own) ? fac * s[i] : -INFINITY;
        v[i] = s[i];
    }
    warp_transpose_reduce<NH, true>(v, lane);
    M.red[quad][qh * NH + ql] = v[0];
    __syncthreads();
    // one thread per query: the tile maximum, the lazy move of the running maximum
    if (tid < NQ) {
        const int q = tid;
        const float mt = fmaxf(fmaxf(M.red[0][q], M.red[1][q]), fmaxf(M.red[2][q], M.red[3][q]));
        const float mo = M.m_run[q];
        const float mn = fmaxf(mo, mt);
        const bool resc = mn > mo + kRescaleGap || (mo == -INFINITY && mn != -INFINITY);
        const float al = resc ? (mo == -INFINITY ? 0.0f : __expf(mo - mn)) : 1.0f;
        M.mu[q] = resc ? mn : mo;
        M.alpha[q] = al;
        const uint32_t any = __ballot_sync(NQ == 32 ? 0xFFFFFFFFu : 0xFFFFu, resc && al != 0.0f);
        if (q == 0) M.any_resc = any != 0u;
    }
    __syncthreads();
#pragma unroll
    for (int i = 0; i < NH; ++i) {
        s[i] = (s[i] == -INFINITY) ? 0.0f : tc::exp2_fast((s[i] - M.mu[qh * NH + i]) * kLog2e);
        v[i] = s[i];
    }
    // P (weights times the row factor) as fp16: core matrices 8 rows x 8 queries,
    // query groups 128 B apart, row groups 256 NL B apart
    uint8_t *prow = Ps + (r >> 3) * (256 * NL) + (r & 7) * 16;
#pragma unroll
    for (int g = 0; g < NH / 8; ++g) {
        uint32_t hv[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            hv[i] = pack_h2(__floats2half2_rn(s[8 * g + 2 * i] * fac, s[8 * g + 2 * i + 1] * fac));
        *reinterpret_cast<uint4 *>(prow + (qh * (NH / 8) + g) * 128) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
    }
    warp_transpose_reduce<NH, false>(v, lane);
    M.red[quad][qh * NH + ql] = v[0];  // the maxima in red[][] were read before the last barrier
    __syncthreads();
    if (tid < NQ) {
        const int q = tid;
        const float lt = (M.red[0][q] + M.red[1][q]) + (M.red[2][q] + M.red[3][q]);
        M.l_run[q] = M.l_run[q] * M.alpha[q] + lt;
        M.m_run[q] = M.mu[q];
    }
    // O^T holds earlier tiles' PV: scale it where a query's maximum moved
    // (thread: channel lane 32 quad + lane, columns of its half)
    if (!first && M.any_resc) {
        float o[32];
#pragma unroll
        for (int c0 = qh * 32 * NL; c0 < (qh + 1) * 32 * NL; c0 += 32) {
            tc::tmem_ld32(tc::taddr(tmem, 32u * quad, Cols<NL>::O + c0), o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= M.alpha[(c0 + i) % NQ];
            tc::tmem_st32(tc::taddr(tmem, 32u * quad, Cols<NL>::O + c0), o);
        }
    }
    tc::fence_async_smem();
    tc::fence_before_sync();
}

// From the (max, sum) table M.mlall[0..ns) of each query: the merged maximum
// and sum (M.cm, M.cl) and each source's weight l_s exp(m_s - max) / sum
// (M.wall).  All 256 threads: sixteen lanes per query, lane = source.
template <int NQ>
__device__ __forceinline__ void merge_weights(Misc &M, int ns)
{
    static_assert((NQ * 16) % kThreads == 0, "whole warps per pass");
#pragma unroll 1
    for (int i = threadIdx.x; i < NQ * 16; i += kThreads) {
        const int q = i >> 4, src = i & 15, lead = threadIdx.x & 16;  // lane of source 0 of this query
        const float2 ml = src < ns ? M.mlall[src][q] : make_float2(-INFINITY, 0.0f);
        float mx = ml.y > 0.0f ? ml.x : -INFINITY;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xFFFFFFFFu, mx, o));
        const float e = ml.y > 0.0f ? ml.y * __expf(ml.x - mx) : 0.0f;
        float lsum = e;
#pragma unroll
        for (int o = 8; o > 0; o >>= 1) lsum += __shfl_xor_sync(0xFFFFFFFFu, lsum, o);
        lsum = __shfl_sync(0xFFFFFFFFu, lsum, lead);  // one sum for every source of the query
        const float inv = lsum > 0.0f ? 1.0f / lsum : 0.0f;
        if (src < ns) M.wall[src][q] = e * inv;
        if (src == 0) {
            M.cm[q] = mx;
            M.cl[q] = lsum;
        }
    }
}

// Weighted sums for this thread's items of one channel slice: item = (query
// q, four channels), n4 items per query.  For each item, the cluster's
// sources in order, sum_k wall[k][q] x load(k, q, ch); with satellites, that
// sum times w0[q] plus sum_s wsat[s][q] x load_sat(s, q, ch) in order.  Every
// load is in flight before the first is used (the satellites' global loads
// first).  (The launch shapes the host picks give a thread one or two items.)
template <int NQ, typename Load, typename LoadSat, typename Store>
__device__ __forceinline__ void slice_reduce(int ns, int n_sat, int n4, int c_lo, int n_layers, const Misc &M,
                                             Load load, LoadSat load_sat, Store store)
{
    const int total = NQ * n4;
#pragma unroll 1
    for (int item = threadIdx.x; item < total; item += kThreads) {
        const int q = item / n4, ch = c_lo + 4 * (item % n4);
        if ((q >> 4) >= n_layers) continue;
        float4 u[kMaxCS], v[kMaxCS];
#pragma unroll
        for (int k = 0; k < kMaxCS; ++k)
            if (k < n_sat) u[k] = load_sat(k, q, ch);
#pragma unroll
        for (int k = 0; k < kMaxCS; ++k)
            if (k < ns) v[k] = load(k, q, ch);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int k = 0; k < kMaxCS; ++k)
            if (k < ns) {
                const float w = M.wall[k][q];
                acc.x += w * v[k].x;
                acc.y += w * v[k].y;
                acc.z += w * v[k].z;
                acc.w += w * v[k].w;
            }
        if (n_sat > 0) {
            const float w0 = M.w0[q];
            acc = make_float4(w0 * acc.x, w0 * acc.y, w0 * acc.z, w0 * acc.w);
#pragma unroll
            for (int k = 0; k < kMaxCS; ++k)
                if (k < n_sat) {
                    const float w = M.wsat[k][q];
                    acc.x += w * u[k].x;
                    acc.y += w * u[k].y;
                    acc.z += w * u[k].z;
                    acc.w += w * u[k].w;
                }
        }
        store(q, ch, acc);
    }
}

template <int NL, bool QR>
__global__ void __launch_bounds__(kThreads, 1) attn_kernel(const __grid_constant__ AttnParams P, int *flags)
{
    constexpr int NQ = 16 * NL;
    extern __shared__ __align__(1024) uint8_t smem[];
    uint8_t *T = smem;
    uint8_t *Qs = smem + kTileBytes;
    uint8_t *Ps = Qs + NL * kQBytes;
    Misc &M = *reinterpret_cast<Misc *>(Ps + NL * kPBytes);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int cs = P.cs;
    const int rank = (int)tc::cluster_rank();
    const int cluster = (int)blockIdx.x / cs;
    const int unit = cluster / P.split, part = cluster % P.split;
    const UnitDev &U = P.units[unit];

    // ---- prologue: nothing here reads memory another kernel writes
    if (tid == 0) {
        tc::mbar_init(&M.bar_qk, 1);
        tc::mbar_init(&M.bar_pv, 1);
        tc::mbar_init(&M.bar_rx, 1);
        tc::mbar_init_fence();
        M.ok = 1;
    }
    if (tid < NQ) {
        M.m_run[tid] = -INFINITY;
        M.l_run[tid] = 0.0f;
    }
    if (warp == 0) tc::tmem_alloc(&M.tmem_slot, Cols<NL>::alloc);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = M.tmem_slot;
    tc::cluster_arrive_relaxed();  // waited for before the first access to a peer's shared memory

    Ctx c;
    c.P = &P;
    c.U = &U;
    c.M = &M;
    c.flags = flags;
    c.b = blockIdx.y;
    c.L = 0;
    c.W = P.window;
    c.quarter = QR;  // a constant: every branch on it is resolved at compile time
    // this CTA's tiles: every (split cs)-th of the unit's, from its index in
    // the (unit, sequence): the first cluster's CTAs, then the satellites'
    const int gc = part * cs + rank, stride = P.split * cs;
    const int t0 = gc, t_end = U.n_tiles;
    const int n_my = t_end > t0 ? (t_end - 1 - t0) / stride + 1 : 0;
    const int r = tid & (kRows - 1), h = tid >> 7;

    Raw raw;
    RowPos pos_next = no_rows();
    auto first_gather = [&]() {
        // the length and the positions are independent loads: both in flight at once
        const int32_t Lraw = __ldcg(P.seq_lens + c.b);
        const RowPos pos0 = n_my > 0 ? load_pos(c, t0) : no_rows();
        if (n_my > 1) pos_next = load_pos(c, t0 + stride);
        c.L = max(0, Lraw);
        if (n_my > 0) gather(c, t0, row_issue(c, pos0), r, h, raw);
    };
    auto row_masks = [&](bool window) {
        if (window || !c.quarter) {
            if (h == 0) {
                const uint32_t m = __ballot_sync(0xFFFFFFFFu, raw.valid);
                if (lane == 0) M.vmask[warp] = m;
                M.rowfac[r] = window ? (raw.app >= 0 ? M.app_scale[raw.app] : raw.scale) * 256.0f : 1.0f;
            }
        } else {
            // rows 16 warp + lane and 16 warp + 8 + lane (lanes 0..7) in one 16-bit half of a mask word
            const uint32_t m0 = __ballot_sync(0xFFFFFFFFu, raw.valid), m1 = __ballot_sync(0xFFFFFFFFu, raw.valid1);
            if (lane == 0) reinterpret_cast<uint16_t *>(M.vmask)[warp] = (uint16_t)((m0 & 0xFFu) | ((m1 & 0xFFu) << 8));
            if (lane < 8) {
                M.rowfac[16 * warp + lane] = 1.0f;
                M.rowfac[16 * warp + 8 + lane] = 1.0f;
            }
        }
    };
    // the queries' and appended window rows' lines into L2 while the previous kernel runs
    for (int i = tid; i < U.n_layers * (kHeads * kDim * 4 / 128); i += kThreads) {
        const int j = i / (kHeads * kDim * 4 / 128), line = i % (kHeads * kDim * 4 / 128);
        tc::prefetch_l2(reinterpret_cast<const uint8_t *>(P.entries[U.entry[j]].q + (int64_t)c.b * kHeads * kDim) +
                        128 * line);
    }
    if (warp < U.n_layers && P.entries[U.entry[warp]].new_swa && lane < kDim * 4 / 128)
        tc::prefetch_l2(reinterpret_cast<const uint8_t *>(P.entries[U.entry[warp]].new_swa + (int64_t)c.b * kDim) +
                        128 * lane);
    const bool pre = P.inputs_ready && n_my > 0;
    if (pre) {
        // nothing the previous kernel writes is read here: the first tile is
        // gathered and dequantised while that kernel runs (an appended window
        // row, written after the wait, is patched in below)
        first_gather();
        dequant(c, tile_is_window(U, t0), r, h, raw, T);
        row_masks(tile_is_window(U, t0));
        if (n_my > 1) {
            gather(c, t0 + stride, row_issue(c, pos_next), r, h, raw);
            pos_next = n_my > 2 ? load_pos(c, t0 + 2 * stride) : no_rows();
        }
    }
    tc::pdl_wait();
    tc::pdl_launch_dependents();

    // queries: every load in flight at once (before the first tile's dependent
    // position and row loads), then the fp16 value and fp16 remainder into
    // K-major core matrices (query rows n, 8,192 B per 8 rows; remainders at
    // n + 16 NL)
    float4 qv[4 * NL][2];
#pragma unroll
    for (int k = 0; k < 4 * NL; ++k) {
        const int item = tid + kThreads * k;
        const int qi = (item & 7) | ((item >> 9) << 3);
        const int cg = (item >> 3) & 63;
        if ((qi >> 4) < U.n_layers) {
            const float4 *src = reinterpret_cast<const float4 *>(P.entries[U.entry[qi >> 4]].q +
                                                                 ((int64_t)c.b * kHeads + (qi & 15)) * kDim + 8 * cg);
            qv[k][0] = __ldcg(src);
            qv[k][1] = __ldcg(src + 1);
        } else {
            qv[k][0] = qv[k][1] = make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    if (!pre) first_gather();

    // appended window rows of this CTA's window tiles (position L-1 of each
    // layer): layer slot j by threads 128 j .. 128 j + 127
    if (P.window > 0 && c.L > 0 && (tid >> 7) < U.n_layers) {
        const int j = tid >> 7;
        const EntryDev &E = P.entries[U.entry[j]];
        const int t_app = U.row_tiles + j * P.win_tiles + (P.window - 1) / kRows;
        if (E.new_swa && t_app >= t0 && t_app < t_end && (t_app - t0) % stride == 0)
            append_window_row(c, E, j, tid & 127, pre && t_app == t0, (P.window - 1) % kRows, T);
    }

#pragma unroll
    for (int k = 0; k < 4 * NL; ++k) {
        const int item = tid + kThreads * k;
        const int qi = (item & 7) | ((item >> 9) << 3);
        const int cg = (item >> 3) & 63;
        const float x[8] = {qv[k][0].x, qv[k][0].y, qv[k][0].z, qv[k][0].w,
                            qv[k][1].x, qv[k][1].y, qv[k][1].z, qv[k][1].w};
        uint32_t hi[4], lo[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hv = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
            const float2 hf = __half22float2(hv);
            hi[i] = pack_h2(hv);
            lo[i] = pack_h2(__floats2half2_rn(x[2 * i] - hf.x, x[2 * i + 1] - hf.y));
        }
        *reinterpret_cast<uint4 *>(Qs + cm_off(qi, 8 * cg)) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(Qs + cm_off(NQ + qi, 8 * cg)) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
    __syncthreads();  // queries and appended rows in shared memory before any dequantisation

    constexpr uint32_t kIdescQK = tc::idesc_f16(128, 2 * NQ, false, false);
    constexpr uint32_t kIdescPV = tc::idesc_f16(128, NQ, true, true);
    for (int it = 0; it < n_my; ++it) {
        const int tile = t0 + it * stride;
        const bool window = tile_is_window(U, tile);
        if (it > 0 || !pre) {
            // the next tile's page-table loads (its positions arrived during the
            // previous tile) in flight across the wait and this tile's dequantisation
            const RowRef ref_next = row_issue(c, pos_next);
            if (it > 0 && tid == 0 && !tc::mbar_wait(&M.bar_pv, (it - 1) & 1)) M.ok = 0;  // tile and P buffers free
            __syncthreads();
            tc::fence_after_sync();
            dequant(c, window, r, h, raw, T);
            row_masks(window);
            if (it + 1 < n_my) {  // in flight during this tile
                gather(c, tile + stride, ref_next, r, h, raw);
                pos_next = it + 2 < n_my ? load_pos(c, tile + 2 * stride) : no_rows();
            }
        }
        tc::fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint64_t a0 = tc::sdesc(tc::smem_u32(T), 128, 8192);
            const uint64_t b0 = tc::sdesc(tc::smem_u32(Qs), 128, 8192);
            // rolled: the issue rate of the tensor core, not the loop, bounds these
#pragma unroll 1
            for (int ks = 0; ks < kDim / 16; ++ks)
                tc::mma_f16(tmem + Cols<NL>::S, a0 + 16 * ks, b0 + 16 * ks, kIdescQK, ks > 0 ? 1u : 0u);
            tc::mma_commit(&M.bar_qk);
        }
        if (!tc::mbar_wait(&M.bar_qk, it & 1) && tid == 0) M.ok = 0;
        tc::fence_after_sync();
        softmax_tile<NL>(c, tmem, Ps, tile, it == 0);
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            // the four channel blocks are independent accumulators: interleaved
#pragma unroll 1
            for (int ks = 0; ks < kRows / 16; ++ks)
#pragma unroll
                for (int cb = 0; cb < 4; ++cb)
                    tc::mma_f16(tmem + Cols<NL>::O + cb * NQ,
                                tc::sdesc(tc::smem_u32(T) + 2048u * cb + 16384u * ks, 8192, 128),
                                tc::sdesc(tc::smem_u32(Ps) + (uint32_t)(2 * 256 * NL * ks), 256 * NL, 128), kIdescPV,
                                (it > 0 || ks > 0) ? 1u : 0u);
            tc::mma_commit(&M.bar_pv);
        }
    }
    if (n_my > 0 && tid == 0 && !tc::mbar_wait(&M.bar_pv, (n_my - 1) & 1)) {
        M.ok = 0;
        tc::mbar_wait(&M.bar_pv, (n_my - 1) & 1);  // a last chance for MMAs in flight
    }
    __syncthreads();
    tc::fence_after_sync();
    if (tid == 0 && !M.ok) raise_flag(flags, kFlagTimeout);
    if (tid < NQ) M.inv_l[tid] = M.l_run[tid] > 0.0f ? 1.0f / M.l_run[tid] : 0.0f;
    __syncthreads();

    // ---- a satellite (a CTA of the second cluster of a split (unit,
    // sequence)) hands its partial to the first cluster through the
    // workspace: its running (max, sum) per query and O^T normalised by that
    // sum, then one counter increment per owner of a channel slice
    if (part > 0) {
        if (n_my > 0) {
            float *rec = P.parts + (((int64_t)unit * P.batch + c.b) * cs + rank) * (int64_t)kSatFloats;
            if (tid < NQ) {
                rec[tid] = M.m_run[tid];
                rec[16 * kMaxNL + tid] = M.l_run[tid];
            }
            const int quad = warp & 3, half = warp >> 2;  // TMEM lanes 32 quad.., column half
            const int ch_in = 32 * quad + lane;
#pragma unroll 1
            for (int c0 = half * 32 * NL; c0 < (half + 1) * 32 * NL; c0 += 32) {
                float o[32];
                tc::tmem_ld32(tc::taddr(tmem, 32u * quad, Cols<NL>::O + c0), o);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int col = c0 + i, q = col % NQ;
                    rec[kSatHdr + q * kDim + 128 * (col / NQ) + ch_in] = o[i] * M.inv_l[q];
                }
            }
            tc::fence_before_sync();
            __syncthreads();  // the record is written
            if (tid < cs) {
                __threadfence();
                atomicAdd(P.tickets + ((int64_t)unit * P.batch + c.b) * kMaxCS + tid, 1u);
            }
        }
        if (warp == 0) {
            tc::fence_after_sync();
            tc::tmem_dealloc(tmem, Cols<NL>::alloc);
        }
        tc::cluster_wait();  // pairs with the prologue's arrival
        return;
    }

    // ---- merge across the cluster: every CTA stages its output normalised by its
    // own sum, with its (max, sum); one cluster barrier; each CTA then weighs
    // and sums one slice of the channels over the cluster (and over the
    // satellites' partials of that slice, when the (unit, sequence) is split)
    // channel slices: CTA r owns channels [r cpc, min(512, (r + 1) cpc))
    const int cpc = ((kDim + cs - 1) / cs + 3) & ~3;
    const int c_lo = rank * cpc, c_hi = min(kDim, c_lo + cpc);
    const int n4 = max(0, (c_hi - c_lo) / 4);
    const uint32_t blk_bytes = (uint32_t)(NQ * cpc * 4);  // one owner's block: [query][cpc] fp32
    // staged output, [owner][query][channel of the owner's slice], in the idle
    // tile buffer; the blocks this CTA receives follow it (into the query
    // buffer, idle too, for two layers)
    float *stage = reinterpret_cast<float *>(T);
    float *recv = reinterpret_cast<float *>(T + ((cs * blk_bytes + 127u) & ~127u));
    // this CTA's (m, l) of every query into every CTA's table (remote stores,
    // visible after the cluster barrier; every peer has started by now)
    tc::cluster_wait();
    for (int i = tid; i < NQ * cs; i += kThreads) {
        const int q = i % NQ, dst = i / NQ;
        tc::st_cluster_f2(tc::mapa(tc::smem_u32(&M.mlall[rank][q]), (uint32_t)dst), M.m_run[q], M.l_run[q]);
    }
    if (tid == 0) tc::mbar_expect_tx(&M.bar_rx, (uint32_t)cs * blk_bytes);  // every peer's block for this slice
    {
        const int quad = warp & 3, half = warp >> 2;  // TMEM lanes 32 quad.., column half
        const int ch_in = 32 * quad + lane;
#pragma unroll 1
        for (int c0 = half * 32 * NL; c0 < (half + 1) * 32 * NL; c0 += 32) {
            float o[32];
            if (n_my > 0) {
                tc::tmem_ld32(tc::taddr(tmem, 32u * quad, Cols<NL>::O + c0), o);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) {
                const int col = c0 + i, cb = col / NQ, q = col % NQ;
                const int ch = 128 * cb + ch_in, own = ch / cpc;
                stage[(own * NQ + q) * cpc + (ch - own * cpc)] = o[i] * M.inv_l[q];
            }
        }
    }
    tc::fence_async_smem();  // the staged blocks are read by bulk copies
    tc::fence_before_sync();
    tc::cluster_sync();
    if (warp == 0) {  // O^T is staged: tensor memory is done
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, Cols<NL>::alloc);
    }
    // one bulk copy per owner: this CTA's block of its slice, into the owner's
    // receive area at this CTA's rank, completing on the owner's barrier
    if (tid < cs) {
        const uint32_t dst = tc::mapa(tc::smem_u32(recv) + (uint32_t)rank * blk_bytes, (uint32_t)tid);
        tc::bulk_s2peer(dst, reinterpret_cast<const uint8_t *>(stage) + (size_t)tid * blk_bytes, blk_bytes,
                        tc::mapa(tc::smem_u32(&M.bar_rx), (uint32_t)tid));
    }
    merge_weights<NQ>(M, cs);
    // the satellites with a tile wrote their partials while this cluster was
    // still computing: wait (bounded) for this slice's counter
    const int n_sat = P.split > 1 ? max(0, min(cs, U.n_tiles - cs)) : 0;
    const float *sat = n_sat > 0 ? P.parts + ((int64_t)unit * P.batch + c.b) * cs * (int64_t)kSatFloats : nullptr;
    if (n_sat > 0 && tid == 0) {
        uint32_t *cnt = P.tickets + ((int64_t)unit * P.batch + c.b) * kMaxCS + rank;
        bool got = false;
        for (uint32_t i = 0; i < tc::kWaitLimit && !got; ++i) got = tc::ld_acquire_gpu(cnt) >= (uint32_t)n_sat;
        if (got) {
            *cnt = 0u;  // only this CTA reads it: left zero for the next launch
        } else {
            M.ok = 0;
        }
    }
    if (!tc::mbar_wait(&M.bar_rx, 0)) {
        M.ok = 0;
        tc::mbar_wait(&M.bar_rx, 0);  // a last chance for the copies in flight
    }
    __syncthreads();
    // every block for this CTA has landed, so its peers' copies out of their
    // shared memory are done: arrive now, wait only before leaving
    tc::cluster_arrive();
    if (tid == 0 && !M.ok) raise_flag(flags, kFlagTimeout);
    if (n_sat > 0) {
        // every satellite's (m, l); the cluster's merged (max, sum) is one more
        // source: the final weights of the cluster's CTAs are their cluster
        // weights times w0, a satellite's its own
        for (int i = tid; i < n_sat * NQ; i += kThreads) {
            const int sidx = i / NQ, q = i % NQ;
            const float *rec = sat + (int64_t)sidx * kSatFloats;
            M.mlsat[sidx][q] = make_float2(__ldcg(rec + q), __ldcg(rec + 16 * kMaxNL + q));
        }
        __syncthreads();
        if (tid < NQ) {
            const int q = tid;
            float mx = M.cl[q] > 0.0f ? M.cm[q] : -INFINITY;
            for (int k = 0; k < n_sat; ++k)
                if (M.mlsat[k][q].y > 0.0f) mx = fmaxf(mx, M.mlsat[k][q].x);
            const float w0 = M.cl[q] > 0.0f ? M.cl[q] * __expf(M.cm[q] - mx) : 0.0f;
            float tot = w0;
            for (int k = 0; k < n_sat; ++k) {
                const float2 ml = M.mlsat[k][q];
                const float e = ml.y > 0.0f ? ml.y * __expf(ml.x - mx) : 0.0f;
                M.wsat[k][q] = e;
                tot += e;
            }
            const float inv = tot > 0.0f ? 1.0f / tot : 0.0f;
            for (int k = 0; k < n_sat; ++k) M.wsat[k][q] *= inv;
            M.w0[q] = w0 * inv;
            M.cm[q] = mx;
            M.cl[q] = tot;
        }
        __syncthreads();
    }
    slice_reduce<NQ>(
        cs, n_sat, n4, c_lo, U.n_layers, M,
        [&](int src, int q, int ch) {
            return *reinterpret_cast<const float4 *>(recv + (src * NQ + q) * cpc + (ch - c_lo));
        },
        [&](int sidx, int q, int ch) {
            return __ldcg(reinterpret_cast<const float4 *>(sat + (int64_t)sidx * kSatFloats + kSatHdr + q * kDim + ch));
        },
        [&](int q, int ch, float4 acc) {
            *reinterpret_cast<float4 *>(P.entries[U.entry[q >> 4]].out + ((int64_t)c.b * kHeads + (q & 15)) * kDim +
                                        ch) = acc;
        });
    if (tid < NQ && rank == 0) {
        const int q = tid, j = q >> 4;
        if (j < U.n_layers && P.entries[U.entry[j]].lse) {
            P.entries[U.entry[j]].lse[(int64_t)c.b * kHeads + (q & 15)] =
                M.cl[q] > 0.0f ? M.cm[q] + logf(M.cl[q]) : -INFINITY;
        }
    }
    tc::cluster_wait();  // no CTA leaves while a copy out of its shared memory may be in flight
}

}  // namespace

// ---- host planning ---------------------------------------------------------------------
namespace {

struct UnitPlan {
    std::vector<std::vector<int>> units;  // entry ids per unit (<= max_group each)
    std::vector<int> has_idx;
};

// Units: entries that read the same index list over the same cache, in groups
// of at most `max_group`; an entry without an index list is a unit alone.
UnitPlan group_units(const AttnEntry *entries, int n_entries, int max_group)
{
    UnitPlan up;
    std::vector<std::pair<const void *, const void *>> keys;
    std::vector<std::vector<int>> groups;
    for (int e = 0; e < n_entries; ++e) {
        const AttnEntry &en = entries[e];
        if (en.has_kv && en.idx) {
            const std::pair<const void *, const void *> k(en.idx, en.kv.data);
            size_t g = 0;
            while (g < keys.size() && keys[g] != k) ++g;
            if (g == keys.size()) {
                keys.push_back(k);
                groups.emplace_back();
            }
            groups[g].push_back(e);
        } else {
            up.units.push_back({e});
            up.has_idx.push_back(0);
        }
    }
    for (auto &g : groups)
        for (size_t i = 0; i < g.size(); i += (size_t)max_group) {
            up.units.emplace_back(g.begin() + i, g.begin() + std::min(g.size(), i + (size_t)max_group));
            up.has_idx.push_back(1);
        }
    return up;
}

template <int NL>
cudaError_t prepare_kernel(int dev)
{
    static bool done[64] = {};
    if (dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
    cudaError_t e = cudaSuccess;
    for (auto *k : {attn_kernel<NL, false>, attn_kernel<NL, true>}) {
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_bytes<NL>());
        if (e == cudaSuccess) e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    }
    if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
    return e;
}

// Clusters of `cs` CTAs of attn_kernel<NL, *> that fit on the device at once (both gathers take the same
// threads and shared memory, one CTA per SM).
template <int NL>
int active_clusters(int dev, int cs)
{
    static int cache[64][kMaxCS + 1] = {};
    if (dev >= 0 && dev < 64 && cache[dev][cs]) return cache[dev][cs];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)cs, 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<NL>();
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveClusters(&n, attn_kernel<NL, false>, &cfg);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        log_plan("attention NL=%d: cluster size %d not available (%s)", NL, cs, cudaGetErrorString(e));
        n = 0;
    }
    if (dev >= 0 && dev < 64) cache[dev][cs] = n > 0 ? n : -1;
    return n;
}

struct Shape {
    int split = 1, cs = 1;
    size_t ws = 0;
};

// Workspace of a launch that splits each (unit, sequence) over two clusters
// of `cs`: a partial per satellite and a counter per owner rank.
size_t split_bytes(int n_units, int batch, int split, int cs)
{
    if (split <= 1) return 0;
    auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
    const size_t groups = (size_t)n_units * batch;
    return r256(groups * cs * kSatFloats * sizeof(float)) + r256(groups * kMaxCS * sizeof(uint32_t));
}

// Launch shape: the (split, cluster size) with the lowest modelled time whose
// workspace fits `budget`.  A cluster costs a fixed part (queries in, merge),
// its busiest CTA's tiles and a little per CTA; clusters run `active` at a
// time.  A split (two clusters per (unit, sequence), the second one's CTAs
// handing their partials to the first through the workspace) adds the
// satellites' reads to the merge; the first cluster waits for the second, so
// a split is only planned when every cluster of the launch fits on the
// device at once.  Costs are in microseconds, from global-timer stamps of the
// L = 131,072 step on B300: a tile's tensor-core work alone is 64 MMAs at
// about 46 cycles each, so a CTA's second tile costs about 4 us of
// dequantisation, products and softmax.
template <int NL>
Shape choose_shape(int dev, int max_tiles, int n_groups, size_t budget)
{
    constexpr double kFixed = 6.0, kPerTile = 4.0, kPerCta = 0.05, kSat = 1.0;
    Shape best;
    double best_cost = 1e300;
    for (int split = 1; split <= 2; ++split) {
        if (split > 1 && split > max_tiles) break;
        const int tiles = (max_tiles + split - 1) / split;
        for (int cs = 1; cs <= kMaxCS; ++cs) {
            if (cs > 1 && cs > tiles) break;
            const size_t ws = split_bytes(1, n_groups, split, cs);
            if (ws > budget) continue;
            const int act = active_clusters<NL>(dev, cs);
            if (act <= 0) continue;
            if (split > 1 && (int64_t)n_groups * split > act) continue;  // one wave: the satellites are resident
            const int per = (max_tiles + split * cs - 1) / (split * cs);
            const double waves = std::ceil((double)n_groups * split / act);
            const double cost = waves * (kFixed + kPerTile * per + kPerCta * cs) + (split > 1 ? kSat : 0.0);
            if (cost < best_cost - 1e-9) {
                best_cost = cost;
                best.split = split;
                best.cs = cs;
                best.ws = ws;
            }
        }
    }
    return best;
}

template <int NL>
cudaError_t launch_nl(AttnParams &p, int max_tiles, const AttnPlan &plan, int *flags, cudaStream_t stream)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if ((e = prepare_kernel<NL>(dev)) != cudaSuccess) return e;
    const Shape sh = choose_shape<NL>(dev, std::max(1, max_tiles), p.n_units * plan.batch,
                                      plan.workspace ? plan.workspace_bytes : 0);
    p.cs = sh.cs;
    p.split = sh.split;
    // quarter-row gathers when some CTA takes more than one tile
    const bool quarter = (std::max(1, max_tiles) + sh.split * sh.cs - 1) / (sh.split * sh.cs) > 1;
    if (sh.split > 1) {
        uint8_t *ws = static_cast<uint8_t *>(plan.workspace);
        const size_t groups = (size_t)p.n_units * plan.batch;
        p.parts = reinterpret_cast<float *>(ws);
        p.tickets = reinterpret_cast<uint32_t *>(ws + (((groups * sh.cs * kSatFloats * sizeof(float)) + 255) &
                                                      ~(size_t)255));
    }
    log_plan("attention NL=%d: %d units x %d sequences, %d tiles at most, %d cluster(s) of %d each (%d fit at once)",
             NL, p.n_units, plan.batch, max_tiles, sh.split, sh.cs, active_clusters<NL>(dev, sh.cs));
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.n_units * sh.split * sh.cs), (unsigned)plan.batch, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = smem_bytes<NL>();
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)sh.cs;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = plan.pdl ? 2 : 1;
    e = quarter ? cudaLaunchKernelEx(&cfg, attn_kernel<NL, true>, p, flags)
                : cudaLaunchKernelEx(&cfg, attn_kernel<NL, false>, p, flags);
    count_launches(1);
    return e == cudaSuccess ? cudaGetLastError() : e;
}

// Units and tile counts of a plan; returns the largest layer count of a unit.
int fill_params(const AttnPlan &plan, AttnParams &p, int &max_tiles)
{
    const int max_group = std::max(1, std::min(kMaxNL, plan.max_group));
    const UnitPlan up = group_units(plan.entries, plan.n_entries, max_group);
    if ((int)up.units.size() > kMaxUnits) return -1;
    p.batch = plan.batch;
    p.topk = plan.topk;
    p.window = plan.window;
    p.win_tiles = plan.window > 0 ? (plan.window + kRows - 1) / kRows : 0;
    p.seq_lens = plan.seq_lens;
    p.split = 1;
    p.inputs_ready = plan.inputs_ready && plan.pdl;
    for (int e = 0; e < plan.n_entries; ++e) {
        const AttnEntry &en = plan.entries[e];
        EntryDev &E = p.entries[e];
        E.swa = en.swa;
        E.q = en.q;
        E.new_swa = (en.has_swa && plan.window > 0) ? en.new_swa : nullptr;
        E.out = en.out;
        E.lse = en.lse;
    }
    int nl_used = 1;
    max_tiles = 0;
    for (size_t u = 0; u < up.units.size(); ++u) {
        UnitDev &U = p.units[u];
        const std::vector<int> &g = up.units[u];
        const AttnEntry &e0 = plan.entries[g[0]];
        U.kv = e0.kv;
        U.idx = up.has_idx[u] ? e0.idx : nullptr;
        U.n_layers = (int)g.size();
        for (size_t j = 0; j < g.size(); ++j) U.entry[j] = g[j];
        U.row_tiles = (U.idx && plan.topk > 0) ? (plan.topk + kRows - 1) / kRows : 0;
        U.n_tiles = U.row_tiles + U.n_layers * p.win_tiles;
        max_tiles = std::max(max_tiles, U.n_tiles);
        nl_used = std::max(nl_used, U.n_layers);
    }
    p.n_units = (int)up.units.size();
    return nl_used;
}

}  // namespace

size_t attn_workspace_bytes(const AttnPlan &plan, size_t budget)
{
    if (plan.n_entries <= 0 || plan.n_entries > kMaxAttnEntries || plan.batch <= 0) return 0;
    std::vector<uint8_t> pbuf(sizeof(AttnParams), 0);
    AttnParams &p = *reinterpret_cast<AttnParams *>(pbuf.data());
    int max_tiles = 0;
    const int nl = fill_params(plan, p, max_tiles);
    if (nl < 0) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if ((nl == 1 ? prepare_kernel<1>(dev) : prepare_kernel<2>(dev)) != cudaSuccess) return 0;
    const Shape sh = nl == 1 ? choose_shape<1>(dev, std::max(1, max_tiles), p.n_units * plan.batch, budget)
                             : choose_shape<2>(dev, std::max(1, max_tiles), p.n_units * plan.batch, budget);
    return split_bytes(p.n_units, plan.batch, sh.split, sh.cs);
}

cudaError_t launch_attention(const AttnPlan &plan, int *flags, cudaStream_t stream, cudaEvent_t mid_event)
{
    (void)mid_event;
    if (plan.n_entries <= 0 || plan.n_entries > kMaxAttnEntries || plan.batch <= 0) return cudaErrorInvalidValue;
    std::vector<uint8_t> pbuf(sizeof(AttnParams), 0);
    AttnParams &p = *reinterpret_cast<AttnParams *>(pbuf.data());
    int max_tiles = 0;
    const int nl = fill_params(plan, p, max_tiles);
    if (nl < 0) return cudaErrorInvalidValue;
    if (nl == 1) return launch_nl<1>(p, max_tiles, plan, flags, stream);
    return launch_nl<2>(p, max_tiles, plan, flags, stream);
}

}  // namespace csa2
