// Step 3 of the CSA2 decode path: gather of the selected FP4 main-KV rows and
// the FP8 sliding-window rows, dequantisation, and one softmax attention over
// both (Louis Bouchard's KV-cache report, "Share the cache and the search
// work": the selected global entries beside a local 128-token window;
// Helmcode "DeepSeek V4.1 Flash" explainer, "04 · FP4": FP4 global KV, FP8
// window KV; "03 · CSA2": a Reuse layer attends with its own query over the
// selection of another layer).  16 query heads attend over one shared
// 512-channel row that is both key and value.
//
// Work decomposition.  Layers that attend over the same selected rows (an
// indexing layer and the Reuse layers that take its Top-K) form a *row unit*
// of up to 8 layers: their 8 x 16 = 128 query rows share every gathered row,
// so a row is read and dequantised once for all of them and QK^T and PV are
// 128-row tensor-core products.  Each layer's own window rows form a *window
// unit*.  A *CTA pair* (a cluster of two) takes one (unit, chunk of rows,
// sequence) and splits the work by stage, not by data:
//   rank 0 (scores)  S = Q K^T over all 512 channels (queries in tensor
//                    memory, the A operand), fp32 online softmax, and P as
//                    fp16 -- the PV operand's own precision -- sent to rank 1
//                    with one bulk shared-memory copy per 64-row tile,
//                    together with each row's rescale factor;
//   rank 1 (output)  applies the rescale factors to O, then O += P V over all
//                    512 channels (O is the whole of its tensor memory).
// The hand-off runs one way, so the copy overlaps the next tile's scores; the
// PV commit is multicast to both CTAs' barriers, which tells rank 0 that its
// P buffer is free again.  Each pair leaves a partial (running max and sum
// from rank 0, unnormalised output from rank 1) per consumer layer; a second
// kernel merges each layer's partials.
//
// One CTA, 17 warps:
//   warps 8-15  producers (both ranks): per 64-row tile each thread owns one
//               row and a quarter of its 512 channels, dequantises (E2M1 x
//               E4M3 and E4M3 are exact in fp16) into the core-matrix layout;
//   warp 16     tcgen05.mma issue: rank 0 QK^T (M 128, N 64, K 512), rank 1
//               PV (M 128, N 2 x 256, K 64);
//   warps 0-7   rank 0 softmax: warp w serves query rows 32(w%4)..+31 (its
//               tensor-memory lanes) and keys 32(w/4)..+31 of each tile;
//   warps 0-3   rank 1: O rescale when rank 0 asks for it, and the final
//               read-out of O.
// Tiles, S and P are double-buffered.  Every hand-off is an mbarrier with a
// bounded wait (a wait that gives up raises the timeout flag and the CTA
// drains); both CTAs of a pair meet at a cluster barrier before either exits,
// so neither touches the shared memory of a CTA that has finished.
#include <algorithm>
#include <cstring>
#include <queue>
#include <utility>
#include <vector>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kTile = 64;                  // rows per tile
constexpr int kSoftThreads = 256;          // rank 0 warps 0-7
constexpr int kWorkers = 128;              // rank 1 warps 0-3
constexpr int kProdWarp0 = 8;
constexpr int kProducers = 256;            // warps 8-15
constexpr int kMmaWarp = 16;
constexpr int kThreads = 544;              // 17 warps
constexpr int kMaxChunkRows = 2048;        // rows per chunk of a row unit
constexpr int kTileBytes = kTile * kDim * 2;   // 65,536: one 64-row tile, all channels, fp16
constexpr int kPBytes = 128 * kTile * 2;       // 16,384: P of one tile, fp16
constexpr int kMsgBytes = kPBytes + 128 * 4 + 16;  // P, per-row rescale factor, header
constexpr int kOffTiles = 0;
constexpr int kOffMsg = kOffTiles + 2 * kTileBytes;
constexpr int kOffMisc = kOffMsg + 2 * kMsgBytes;
constexpr int kPartFloats = 64 + kHeads * kDim;  // m[2][16], l[2][16], O[16][512]
constexpr int kMaxUnits = 2 * kMaxAttnEntries;
constexpr int kMaxParts = 64;              // partials per layer: at most 63 row chunks and the window
constexpr float kRescaleGap = 8.0f;        // lazy O rescale threshold (natural log)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;              // rank 0: 256 columns, query rows as fp16 pairs
constexpr uint32_t kColS = 256;            // rank 0: 2 x 64 columns
constexpr uint32_t kColO = 0;              // rank 1: 512 columns
// Instruction descriptors: QK^T (A from tensor memory, B K-major), PV (A K-major, B = V read MN-major).
constexpr uint32_t kIdescQK = tc::idesc_f16(128, kTile, false, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(128, 256, false, true);
// named barriers: 1 producers, 2 rank-0 softmax
constexpr uint32_t kBarProd = 1, kBarSoft = 2;
static_assert(kMsgBytes % 16 == 0, "bulk copies move multiples of 16 bytes");
constexpr int kStageRow = 256 * 4 + 16;    // rank 1 read-out: one row-half of O, padded
static_assert(128 * kStageRow <= kOffMisc, "the read-out stage fits in the tile and message buffers");

// The P message of one tile (rank 0 Pout / rank 1 Pin).
struct PMsg {
    uint8_t p[kPBytes];       // K-major core-matrix layout: 8 groups of 8 keys, 1,024 B per 8-row group
    float alpha[128];         // per query row: factor to apply to O before this tile's PV
    uint32_t rescale;         // nonzero: some alpha differs from 1
    uint32_t pad[3];
};
static_assert(sizeof(PMsg) == kMsgBytes, "P message layout");

struct AttnMisc {
    float mscale[2][kTile];   // per tile buffer: per-row scale (FP8 window rows)
    uint32_t vmask[2][2];     // per tile buffer: valid rows (bit j of word j/32)
    float xmax[2][2][128];    // per tile parity and key half: tile max of each query row
    float lpart[128];         // running sum of the second key half, for the final combine
    uint64_t q_bar;           // rank 0: queries in tensor memory
    uint64_t full_t[2];       // tile dequantised
    uint64_t s_full[2];       // rank 0: QK^T committed
    uint64_t s_free[2];       // rank 0: S loaded by the softmax (QK^T of that tile had finished)
    uint64_t sm_done[2];      // rank 0: the softmax of that tile is complete
    uint64_t p_full[2];       // rank 1: a P message landed (bulk copy)
    uint64_t o_ready[2];      // rank 1: O holds the rescale that tile asks for
    uint64_t pv_evt[2];       // both: PV of that tile finished (multicast commit)
    uint32_t tmem_slot;
};
static_assert(kOffMisc + (int)sizeof(AttnMisc) <= 232448, "attention shared memory over the 227 KB limit");

struct UnitDev {
    CacheView cache;        // FP4_KV cache (row unit) or FP8_SWA ring (window unit)
    const int32_t *idx;     // row unit: [B][topk]
    int32_t is_window;
    int32_t n_layers;       // consumer layers (1..8)
    int32_t entry[8];
    int32_t cta_begin;      // first flat CTA (x) index of this unit (even)
};

struct EntryDev {
    const float *q;         // [B][16][512]
    float *out;             // [B][16][512]
    float *lse;             // [B][16] or null
    int32_t n_parts;        // partials of this layer: row chunks + window
    int32_t part_win;       // part id of the window partial (or -1); row chunk c has part id c
};

struct AttnParams {
    UnitDev units[kMaxUnits];
    EntryDev entries[kMaxAttnEntries];
    int32_t n_units;
    int32_t batch, topk, window, rows_per_chunk, max_parts;
    const int32_t *seq_lens;
    const uint8_t *q16;     // [entry][B][16][512] fp16 query rows
    float *partials;        // [entry][B][max_parts][kPartFloats]
};

// Byte offset of fp16 element (row r, channel c) of a 512-channel operand in
// the no-swizzle core-matrix layout: 8-row groups 8,192 B apart, 8-channel
// groups 128 B apart.
__host__ __device__ __forceinline__ uint32_t cm_off512(uint32_t r, uint32_t c)
{
    return (r >> 3) * 8192u + (c >> 3) * 128u + (r & 7u) * 16u + (c & 7u) * 2u;
}

__device__ __forceinline__ uint32_t pack_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// OR-reduction of a predicate over the `count` threads of named barrier `id`
// (also a barrier); every participant gets the same result.
__device__ __forceinline__ bool bar_any(uint32_t id, uint32_t count, bool p)
{
    uint32_t r;
    asm volatile(
        "{\n .reg .pred a, o;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred o, %2, %3, a;\n selp.u32 %0, 1, 0, o;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Everything one CTA needs to know about its work item.
struct Ctx {
    const AttnParams *P;
    const UnitDev *U;
    AttnMisc *M;
    uint8_t *T;         // 2 tiles
    PMsg *Msg;          // 2 P messages (rank 0: outgoing, rank 1: incoming)
    int *flags;
    uint32_t tmem;
    int b, L, W, row0, n_rows, n_tiles, chunk, rank;
};

// ---- rank 0, warps 0-15: the queries into tensor memory ---------------------------------
// Thread (row r = 32(w%4) + lane, part w/4) moves channels 128 part..+127 of
// its row (fp16, packed by the step's first kernel; one round of 16-byte
// loads) into tensor-memory columns 64 part..+63 as fp16 pairs.  The packed
// layout of one (layer, sequence) is [part 4][granule 16][head 16][8 channels],
// so the 16 heads of a layer read one contiguous 256-B run per load.
__device__ __forceinline__ void load_q(const Ctx &c)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int quad = warp & 3, part = warp >> 2;
    const int r = 32 * quad + lane, slot_layer = r >> 4, head = r & 15;
    const UnitDev &U = *c.U;
    uint4 v[16];
    if (slot_layer < U.n_layers) {
        const uint4 *src = reinterpret_cast<const uint4 *>(
                               c.P->q16 + ((int64_t)U.entry[slot_layer] * c.P->batch + c.b) * (kHeads * kDim * 2)) +
                           (part * 16) * kHeads + head;
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __ldg(src + i * kHeads);
    } else {
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = make_uint4(0u, 0u, 0u, 0u);
    }
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
        float h[32];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            h[4 * i] = __uint_as_float(v[8 * cc + i].x);
            h[4 * i + 1] = __uint_as_float(v[8 * cc + i].y);
            h[4 * i + 2] = __uint_as_float(v[8 * cc + i].z);
            h[4 * i + 3] = __uint_as_float(v[8 * cc + i].w);
        }
        tc::tmem_st32(tc::taddr(c.tmem, (uint32_t)(32 * quad), kColQ + 64 * part + 32 * cc), h);
    }
    tc::fence_before_sync();
    tc::mbar_arrive(&c.M->q_bar);
}

// ---- producers (warps 8-15, both ranks): gather + dequantise 64-row tiles ------------
// Thread ptid owns row j = ptid % 64 of every tile and the quarter w = ptid / 64
// of its channels, 128w..128w+127 (FP4 rows: four 16-byte granules of 32
// channels and eight E4M3 scales; FP8 rows: eight granules of 16 channels).
template <bool FP8>
struct RowRegs {
    uint4 g[FP8 ? 8 : 4];
    uint32_t s[FP8 ? 1 : 2];  // FP4: the eight E4M3 scales; FP8: the row's fp32 scale bits
    bool valid;
};

// Position of row j of tile t of the chunk (row units; -1 past the chunk's end).
__device__ __forceinline__ int32_t row_pos(const Ctx &c, int t, int j)
{
    const int v = t * kTile + j;
    return v < c.n_rows ? __ldg(c.U->idx + (int64_t)c.b * c.P->topk + c.row0 + v) : -1;
}

template <bool FP8>
__device__ __forceinline__ void load_row(const Ctx &c, int t, int j, int w, int32_t pos_fp4, RowRegs<FP8> &r)
{
    const UnitDev &U = *c.U;
    const int v = t * kTile + j;  // row within this chunk
    const uint8_t *ptr = nullptr;
    uint32_t sc = 0u;
    if (v < c.n_rows) {
        if (!FP8) {
            const int32_t pos = pos_fp4;
            if (pos >= 0) {
                const int64_t slot = pos < c.L ? slot_of(U.cache, c.b, pos) : -1;
                if (slot < 0) {
                    if (w == 0) raise_flag(c.flags, kFlagBounds);
                } else {
                    ptr = U.cache.data + slot * kKvRow;
                }
            }
        } else {
            const int64_t pos = (int64_t)c.L - c.W + c.row0 + v;
            if (pos >= 0) {
                const int64_t slot = slot_of(U.cache, c.b, pos);
                if (slot < 0) {
                    if (w == 0) raise_flag(c.flags, kFlagBounds);
                } else {
                    ptr = U.cache.data + slot * kDim;
                    sc = __ldg(reinterpret_cast<const uint32_t *>(U.cache.data + U.cache.n_slots * kDim) + slot);
                }
            }
        }
    }
    r.valid = ptr != nullptr;
    if (FP8) {
        r.s[0] = sc;
        const uint8_t *base = ptr ? ptr + 128 * w : nullptr;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            r.g[i] = base ? __ldg(reinterpret_cast<const uint4 *>(base + 16 * i)) : make_uint4(0u, 0u, 0u, 0u);
    } else {
        const uint8_t *base = ptr ? ptr + 64 * w : nullptr;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            r.g[i] = base ? __ldg(reinterpret_cast<const uint4 *>(base + 16 * i)) : make_uint4(0u, 0u, 0u, 0u);
        const uint2 sc2 = ptr ? __ldg(reinterpret_cast<const uint2 *>(ptr + kKvCodes + 8 * w)) : make_uint2(0u, 0u);
        r.s[0] = sc2.x;
        r.s[1] = sc2.y;
    }
}

template <bool FP8>
__device__ __forceinline__ void store_row(uint8_t *V, int j, int w, const RowRegs<FP8> &r)
{
    if (FP8) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int ch = 128 * w + 16 * i;  // channels ch..ch+15
            const uint4 cw = r.g[i];
            *reinterpret_cast<uint4 *>(V + cm_off512(j, ch)) =
                make_uint4(pack_h2(e4m3x2_half2(cw.x & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.x >> 16)),
                           pack_h2(e4m3x2_half2(cw.y & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.y >> 16)));
            *reinterpret_cast<uint4 *>(V + cm_off512(j, ch + 8)) =
                make_uint4(pack_h2(e4m3x2_half2(cw.z & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.z >> 16)),
                           pack_h2(e4m3x2_half2(cw.w & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.w >> 16)));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int ch = 128 * w + 32 * i;  // channels ch..ch+31; scales of its two 16-channel blocks
            const uint32_t sw = r.s[i >> 1] >> (16 * (i & 1));
            const __half2 s0 = __half2half2(__float2half_rn(e4m3_value(sw & 0xFFu)));
            const __half2 s1 = __half2half2(__float2half_rn(e4m3_value((sw >> 8) & 0xFFu)));
            const uint32_t wd[4] = {r.g[i].x, r.g[i].y, r.g[i].z, r.g[i].w};
            uint32_t h[16];
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const uint32_t bits = e2m1x2_half2_bits((wd[k >> 2] >> (8 * (k & 3))) & 0xFFu);
                const __half2 x = *reinterpret_cast<const __half2 *>(&bits);
                h[k] = pack_h2(__hmul2(x, k < 8 ? s0 : s1));
            }
#pragma unroll
            for (int k = 0; k < 4; ++k)
                *reinterpret_cast<uint4 *>(V + cm_off512(j, ch + 8 * k)) =
                    make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
        }
    }
}

// Tile buffer b is free for tile t >= 2 once, on rank 0, the softmax has
// loaded S(t-2) (so QK^T(t-2) is done; FP8 tiles also need the softmax of
// t-2 complete, for the row scales) and, on rank 1, PV(t-2) has finished.
template <bool FP8>
__device__ __forceinline__ bool wait_tile_free(const Ctx &c, int t)
{
    AttnMisc &M = *c.M;
    const int b = t & 1;
    const uint32_t par = ((t - 2) >> 1) & 1;
    if (c.rank == 0) return tc::mbar_wait(FP8 ? &M.sm_done[b] : &M.s_free[b], par);
    return tc::mbar_wait(&M.pv_evt[b], par);
}

template <bool FP8>
__device__ __forceinline__ void produce(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const int ptid = threadIdx.x - kProdWarp0 * 32;
    const int j = ptid & (kTile - 1), w = ptid >> 6;
    if (c.rank == 0) load_q(c);
    // FP4: row positions run two tiles ahead and row bytes one tile ahead;
    // FP8 window tiles (few) load in place
    int32_t pos_next = FP8 ? -1 : row_pos(c, 1, j);
    RowRegs<FP8> cur, nxt;
    if (!FP8 && c.n_tiles > 0) load_row<FP8>(c, 0, j, w, row_pos(c, 0, j), cur);
    for (int t = 0; t < c.n_tiles; ++t) {
        const int b = t & 1;
        if (FP8) {
            load_row<FP8>(c, t, j, w, -1, cur);
        } else {
            if (t + 1 < c.n_tiles) load_row<FP8>(c, t + 1, j, w, pos_next, nxt);  // in flight during this tile
            pos_next = row_pos(c, t + 2, j);
        }
        const bool bad = (t >= 2) && !wait_tile_free<FP8>(c, t);
        if (bar_any(kBarProd, kProducers, bad)) {
            if (ptid == 0) raise_flag(c.flags, kFlagTimeout);
            break;
        }
        store_row<FP8>(c.T + b * kTileBytes, j, w, cur);
        if (w == 0) {
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, cur.valid);
            if ((j & 31) == 0) M.vmask[b][j >> 5] = mask;
            M.mscale[b][j] = FP8 ? __uint_as_float(cur.s[0]) : 1.0f;
        }
        tc::fence_async_smem();
        tc::mbar_arrive(&M.full_t[b]);
        if (!FP8) cur = nxt;
    }
}

// ---- rank 0: QK^T issue (one thread) --------------------------------------------------
// S(t) = Q K(t)^T: 32 MMAs of K 16 (A: queries in tensor memory, 8 columns per
// K step; B: the tile, K-major, 256 B per K step).
__device__ __forceinline__ void issue_qk(const Ctx &c)
{
    AttnMisc &M = *c.M;
    bool ok = tc::mbar_wait(&M.q_bar, 0);
    const uint64_t kd0 = tc::sdesc(tc::smem_u32(c.T), 128, 8192);
    const uint64_t kd1 = tc::sdesc(tc::smem_u32(c.T + kTileBytes), 128, 8192);
    uint64_t *last_bar = nullptr;
    uint32_t last_par = 0;
    for (int t = 0; t < c.n_tiles && ok; ++t) {
        const int b = t & 1;
        ok = tc::mbar_wait(&M.full_t[b], (t >> 1) & 1) && (t < 2 || tc::mbar_wait(&M.s_free[b], ((t - 2) >> 1) & 1));
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t d = c.tmem + kColS + kTile * b;
        const uint64_t kd = b ? kd1 : kd0;
#pragma unroll
        for (int ks = 0; ks < kDim / 16; ++ks)
            tc::mma_f16_ta(d, c.tmem + kColQ + 8 * ks, kd + 16 * ks, kIdescQK, ks > 0 ? 1u : 0u);
        tc::mma_commit(&M.s_full[b]);
        last_bar = &M.s_full[b];
        last_par = (t >> 1) & 1;
    }
    if (!ok) raise_flag(c.flags, kFlagTimeout);
    if (last_bar) tc::mbar_wait(last_bar, last_par);  // every MMA done before tensor memory is released
}

// ---- rank 0: softmax (warps 0-7) ------------------------------------------------------
// Thread (row r = 32(w%4) + lane, key half kh = w/4) holds the row's scores of
// keys 32kh..32kh+31 of each tile.  Per tile: S from tensor memory, mask and
// scale, the row's tile max (both key halves), the lazy rescale decision (a
// row moves its reference max only when the tile max exceeds it by more than
// e^8; the factor for O travels to rank 1), then P = exp(S - m) as fp16 into
// the outgoing message, which thread 0 copies to rank 1.  A failed wait clears
// `ok`; the loop leaves only at a reduction over all 256 threads, so every
// softmax thread meets every named barrier the same number of times.
template <bool FP8>
__device__ __forceinline__ void softmax_rows(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const UnitDev &U = *c.U;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int quad = warp & 3, kh = warp >> 2;
    const int r = 32 * quad + lane;
    const int slot_layer = r >> 4, head = r & 15;
    const bool active = slot_layer < U.n_layers;
    const uint32_t lane_base = (uint32_t)(32 * quad);
    const uint32_t pin_peer = tc::mapa(tc::smem_u32(c.Msg), 1);
    const uint32_t pfull_peer = tc::mapa(tc::smem_u32(&M.p_full[0]), 1);

    load_q(c);

    float m_used = -INFINITY, l_half = 0.0f;
    bool ok = true;
    for (int t = 0; t < c.n_tiles; ++t) {
        const int b = t & 1;
        ok = ok && tc::mbar_wait(&M.full_t[b], (t >> 1) & 1) && tc::mbar_wait(&M.s_full[b], (t >> 1) & 1);
        tc::fence_after_sync();
        float s[32];
        tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColS + kTile * b + 32 * kh), s);
        const uint32_t vm = M.vmask[b][kh];  // read before S is released: the tile buffer may refill after
        tc::fence_before_sync();
        tc::mbar_arrive(&M.s_free[b]);
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            const float z = FP8 ? s[j] * M.mscale[b][32 * kh + j] : s[j];
            s[j] = ((vm >> j) & 1u) ? z : -INFINITY;
            mx[j & 3] = fmaxf(mx[j & 3], s[j]);
        }
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        M.xmax[b][kh][r] = mt;
        if (bar_any(kBarSoft, kSoftThreads, !ok)) break;  // also: both key halves' maxima are written
        const float m_tile = fmaxf(mt, M.xmax[b][kh ^ 1][r]);
        const float m_new = active ? fmaxf(m_used, m_tile) : m_used;
        const bool resc = active && m_new > m_used + kRescaleGap;
        const float alpha = resc ? (m_used == -INFINITY ? 0.0f : __expf(m_used - m_new)) : 1.0f;
        if (resc) {
            l_half *= alpha;
            m_used = m_new;
        }
        // the outgoing message of this parity is free once rank 1 finished PV(t-2)
        ok = ok && (t < 2 || tc::mbar_wait_cluster(&M.pv_evt[b], ((t - 2) >> 1) & 1));
        PMsg &msg = c.Msg[b];
        // P = exp(S - m) as fp16; window rows hold raw E4M3 codes, so their scale joins the weight
        const float mb = m_used * kLog2e;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            s[j] = (active && s[j] != -INFINITY) ? tc::exp2_fast(fmaf(s[j], kLog2e, -mb)) : 0.0f;
            ls[j & 3] += s[j];
        }
        l_half += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        uint8_t *Pb = msg.p + (r >> 3) * 1024 + (r & 7) * 16;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t ph[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 8 * g + 2 * i;
                const float a = FP8 ? s[j] * M.mscale[b][32 * kh + j] : s[j];
                const float d = FP8 ? s[j + 1] * M.mscale[b][32 * kh + j + 1] : s[j + 1];
                ph[i] = pack_h2(__floats2half2_rn(a, d));
            }
            *reinterpret_cast<uint4 *>(Pb + (4 * kh + g) * 128) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        }
        if (kh == 0) msg.alpha[r] = alpha;
        tc::fence_async_smem();
        const bool any_resc = bar_any(kBarSoft, kSoftThreads, resc);  // also: the whole message is written
        tc::mbar_arrive(&M.sm_done[b]);
        if (tid == 0) {
            msg.rescale = any_resc ? 1u : 0u;
            tc::fence_async_smem();
            tc::bulk_s2peer(pin_peer + b * kMsgBytes, &msg, kMsgBytes, pfull_peer + b * 8);
        }
    }
    if (c.n_tiles > 0) {
        // rank 1 has consumed the last message (and its multicast arrival has landed here)
        const int last = c.n_tiles - 1;
        ok = ok && tc::mbar_wait_cluster(&M.pv_evt[last & 1], (last >> 1) & 1);
    }
    if (!ok) raise_flag(c.flags, kFlagTimeout);
    // both key halves' sums; the partial's (m, l), the same for both channel halves
    if (kh == 1) M.lpart[r] = l_half;
    const bool have = !bar_any(kBarSoft, kSoftThreads, !ok) && c.n_tiles > 0;
    if (active && kh == 0) {
        const int e = U.entry[slot_layer];
        const EntryDev &E = c.P->entries[e];
        const int part = U.is_window ? E.part_win : c.chunk;
        float *rec = c.P->partials + (((int64_t)e * c.P->batch + c.b) * c.P->max_parts + part) * kPartFloats;
        const float l_sum = l_half + M.lpart[r];
        const bool any = have && l_sum > 0.0f;
        rec[head] = rec[16 + head] = any ? m_used : -INFINITY;
        rec[32 + head] = rec[48 + head] = any ? l_sum : 0.0f;
    }
}

// ---- rank 1: PV issue (one thread) ----------------------------------------------------
// O += P(t) V(t): 4 K steps of 16 keys x 2 channel halves of N 256 (A: P from
// the landed message, K-major, 256 B per K step; B: the tile read MN-major,
// 16,384 B per K step, channel half n at +4,096 B).  The commit is multicast
// to both CTAs' pv_evt: here it frees the tile buffer and (with o_ready) lets
// the workers rescale O; on rank 0 it frees the outgoing message.
__device__ __forceinline__ void issue_pv(const Ctx &c)
{
    AttnMisc &M = *c.M;
    bool ok = true;
    bool issued = false;
    int last = -1;
    for (int t = 0; t < c.n_tiles; ++t) {
        const int b = t & 1;
        const uint32_t par = (t >> 1) & 1;
        ok = tc::mbar_wait(&M.full_t[b], par) && tc::mbar_wait_cluster(&M.p_full[b], par) &&
             tc::mbar_wait(&M.o_ready[b], par);
        if (!ok) break;
        tc::fence_after_sync();
        const uint32_t va = tc::smem_u32(c.T + b * kTileBytes);
        const uint64_t pd = tc::sdesc(tc::smem_u32(c.Msg[b].p), 128, 1024);
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
#pragma unroll
            for (int n = 0; n < 2; ++n)
                tc::mma_f16(c.tmem + kColO + 256 * n, pd + 16 * k, tc::sdesc(va + 4096 * n + 16384 * k, 8192, 128),
                            kIdescPV, (t > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit_multicast(&M.pv_evt[b], 0x3);
        issued = true;
        last = t;
    }
    if (!ok) raise_flag(c.flags, kFlagTimeout);
    if (issued) tc::mbar_wait(&M.pv_evt[last & 1], (last >> 1) & 1);  // every MMA done before tensor memory is released
}

// ---- rank 1: O rescale and read-out (warps 0-3, thread = tensor-memory lane = query row) ----
__device__ __forceinline__ void o_workers(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const UnitDev &U = *c.U;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int r = tid, slot_layer = r >> 4, head = r & 15;
    const bool active = slot_layer < U.n_layers;
    const uint32_t lane_base = (uint32_t)(32 * warp);
    bool ok = true;
    for (int t = 0; t < c.n_tiles; ++t) {
        const int b = t & 1;
        const bool landed = tc::mbar_wait_cluster(&M.p_full[b], (t >> 1) & 1);
        if (tid == 0 && landed && t + 2 < c.n_tiles) tc::mbar_expect_tx(&M.p_full[b], kMsgBytes);  // tile t+2
        ok = __all_sync(0xFFFFFFFFu, landed);
        if (!ok) break;
        const PMsg &msg = c.Msg[b];
        if (msg.rescale && t >= 1) {
            // O must hold PV(t-1) before it is scaled
            ok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&M.pv_evt[(t - 1) & 1], ((t - 1) >> 1) & 1));
            if (!ok) break;
            tc::fence_after_sync();
            const float a = msg.alpha[r];
            if (__any_sync(0xFFFFFFFFu, a != 1.0f)) {
#pragma unroll 1
                for (int c0 = 0; c0 < kDim; c0 += 32) {
                    float o[32];
                    tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= a;
                    tc::tmem_st32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
                }
            }
            tc::fence_before_sync();
        }
        tc::mbar_arrive(&M.o_ready[b]);
    }
    if (ok && c.n_tiles > 0) {
        const int last = c.n_tiles - 1;
        ok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&M.pv_evt[last & 1], (last >> 1) & 1));
    }
    if (!ok && (tid & 31) == 0) raise_flag(c.flags, kFlagTimeout);
    tc::fence_after_sync();
    // this chunk's unnormalised output, all 512 channels, in two channel halves:
    // each thread puts its row-half in shared memory (the tile buffers are idle
    // now; rows 1,040 B apart, so a quarter-warp's 16-byte stores of 8
    // consecutive rows fall in distinct banks) and sends it with one bulk copy
    const bool have = ok && c.n_tiles > 0;
    float *orow = nullptr;
    if (active) {
        const int e = U.entry[slot_layer];
        const EntryDev &E = c.P->entries[e];
        const int part = U.is_window ? E.part_win : c.chunk;
        orow = c.P->partials + (((int64_t)e * c.P->batch + c.b) * c.P->max_parts + part) * kPartFloats + 64 +
               head * kDim;
    }
    float *srow = reinterpret_cast<float *>(c.T + r * kStageRow);
#pragma unroll 1
    for (int hh = 0; hh < 2; ++hh) {
        if (hh == 1 && active) tc::bulk_wait_read0();  // the first copy has read this row
#pragma unroll 1
        for (int c0 = 0; c0 < 256; c0 += 32) {
            float o[32];
            if (have) {
                tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + 256 * hh + c0), o);
            } else {
#pragma unroll
                for (int i = 0; i < 32; ++i) o[i] = 0.0f;
            }
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(srow + c0 + i) = make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]);
        }
        if (active) {
            tc::fence_async_smem();
            tc::bulk_s2g(orow + 256 * hh, srow, 1024);
            tc::bulk_commit();
        }
    }
    if (active) tc::bulk_wait0();
    tc::fence_before_sync();
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnParams P, int *flags)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx c;
    c.P = &P;
    c.M = reinterpret_cast<AttnMisc *>(smem + kOffMisc);
    c.T = smem + kOffTiles;
    c.Msg = reinterpret_cast<PMsg *>(smem + kOffMsg);
    c.flags = flags;
    c.b = blockIdx.y;
    int u = 0;
    while (u + 1 < P.n_units && (int)blockIdx.x >= P.units[u + 1].cta_begin) ++u;
    c.U = &P.units[u];
    const int local = (int)blockIdx.x - c.U->cta_begin;
    c.chunk = local >> 1;
    c.rank = (int)tc::cluster_rank();  // = local & 1: a pair is one cluster
    c.L = max(0, __ldg(P.seq_lens + c.b));
    c.W = P.window;
    const bool fp8 = c.U->is_window != 0;
    if (fp8) {
        c.row0 = 0;
        c.n_rows = c.W;
    } else {
        c.row0 = c.chunk * P.rows_per_chunk;
        c.n_rows = max(0, min(P.rows_per_chunk, P.topk - c.row0));
    }
    c.n_tiles = (c.n_rows + kTile - 1) / kTile;
    AttnMisc &M = *c.M;

    if (tid == 0) {
        tc::mbar_init(&M.q_bar, kSoftThreads + kProducers);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&M.full_t[i], kProducers);
            tc::mbar_init(&M.s_full[i], 1);
            tc::mbar_init(&M.s_free[i], kSoftThreads);
            tc::mbar_init(&M.sm_done[i], kSoftThreads);
            tc::mbar_init(&M.p_full[i], 1);
            tc::mbar_init(&M.o_ready[i], kWorkers);
            tc::mbar_init(&M.pv_evt[i], 1);
        }
        tc::mbar_init_fence();
        if (c.rank == 1)  // armed for the first two tiles' messages
            for (int i = 0; i < 2 && i < c.n_tiles; ++i) tc::mbar_expect_tx(&M.p_full[i], kMsgBytes);
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&M.tmem_slot, kTmemCols);
    tc::fence_before_sync();
    tc::cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc::fence_after_sync();
    c.tmem = M.tmem_slot;

    if (warp >= kProdWarp0 && warp < kMmaWarp) {
        if (fp8) produce<true>(c);
        else produce<false>(c);
    } else if (warp == kMmaWarp) {
        if (lane == 0) {
            if (c.rank == 0) issue_qk(c);
            else issue_pv(c);
        }
        __syncwarp();
    } else if (c.rank == 0) {
        if (fp8) softmax_rows<true>(c);
        else softmax_rows<false>(c);
    } else if (warp < 4) {
        o_workers(c);
    }
    tc::fence_before_sync();
    tc::cluster_sync();  // no remote shared-memory access after this point
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(c.tmem, kTmemCols);
    }
}

// ---- merge: the partials of one (layer, sequence) -> out, lse -------------------------
// Grid (layer, sequence, eighth of the channels); 256 threads, thread = (head
// tid/16, 4 channels).  The (m, l) of every part are staged in shared memory
// in one round of independent loads; 16 threads turn them into per-part
// weights exp(m_p - max); every thread then sums one float4 per part.  A
// layer with no parts writes zeros.
struct MergeParams {
    EntryDev entries[kMaxAttnEntries];
    int32_t batch, max_parts;
    const float *partials;  // [entry][B][max_parts][kPartFloats]
};

__global__ void __launch_bounds__(256) attn_merge_kernel(const __grid_constant__ MergeParams P)
{
    __shared__ float m_sh[kMaxParts][kHeads], l_sh[kMaxParts][kHeads];
    __shared__ float inv_sh[kHeads];
    const int e = blockIdx.x, b = blockIdx.y, tid = threadIdx.x;
    const int c_base = blockIdx.z * (kDim / 8), half = c_base / 256;
    const EntryDev &E = P.entries[e];
    const int np = min(E.n_parts, kMaxParts);
    const float *recs = P.partials + ((int64_t)e * P.batch + b) * P.max_parts * kPartFloats;
    for (int i = tid; i < np * kHeads; i += 256) {
        const float *rp = recs + (int64_t)(i / kHeads) * kPartFloats;
        m_sh[i / kHeads][i % kHeads] = __ldcg(rp + half * 16 + i % kHeads);
        l_sh[i / kHeads][i % kHeads] = __ldcg(rp + 32 + half * 16 + i % kHeads);
    }
    __syncthreads();
    if (tid < kHeads) {
        float mx = -INFINITY;
        for (int p = 0; p < np; ++p)
            if (l_sh[p][tid] > 0.0f) mx = fmaxf(mx, m_sh[p][tid]);
        float ls = 0.0f;
        for (int p = 0; p < np; ++p) {
            const float wp = l_sh[p][tid] > 0.0f ? __expf(m_sh[p][tid] - mx) : 0.0f;
            ls += wp * l_sh[p][tid];
            m_sh[p][tid] = wp;  // m becomes the part's weight
        }
        inv_sh[tid] = ls > 0.0f ? 1.0f / ls : 0.0f;
        if (blockIdx.z == 0 && E.lse) E.lse[(int64_t)b * kHeads + tid] = ls > 0.0f ? mx + logf(ls) : -INFINITY;
    }
    __syncthreads();
    const int h = tid >> 4, c0 = c_base + (tid & 15) * 4;
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int p = 0; p < np; ++p) {
        const float wp = m_sh[p][h];
        const float4 v = __ldcg(reinterpret_cast<const float4 *>(recs + (int64_t)p * kPartFloats + 64 + h * kDim + c0));
        acc.x += wp * v.x;
        acc.y += wp * v.y;
        acc.z += wp * v.z;
        acc.w += wp * v.w;
    }
    const float inv = inv_sh[h];
    *reinterpret_cast<float4 *>(E.out + ((int64_t)b * kHeads + h) * kDim + c0) =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

}  // namespace

// ---- host planning ---------------------------------------------------------------------
namespace {

struct UnitPlan {
    std::vector<std::vector<int>> row_units;  // entry ids per row unit (<= 8 each)
    std::vector<int> window_units;            // entry id per window unit
};

// Row units: entries that read the same index list over the same cache, in
// groups of at most 8; window units: one per entry with a window.
UnitPlan group_units(const AttnEntry *entries, int n_entries, int window)
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
        }
        if (en.has_swa && window > 0) up.window_units.push_back(e);
    }
    for (auto &g : groups)
        for (size_t i = 0; i < g.size(); i += 8)
            up.row_units.emplace_back(g.begin() + i, g.begin() + std::min(g.size(), i + 8));
    return up;
}

struct WsLayout {
    size_t q16 = 0, partials = 0, total = 0;
    int rpc = kMaxChunkRows, chunks = 0, max_parts = 1;
};

// Workspace layout of a launch that splits row units into chunks of `rpc` rows.
WsLayout layout_for(const UnitPlan &up, int n_entries, int batch, int topk, int window, int rpc)
{
    WsLayout w;
    w.rpc = rpc;
    w.chunks = (topk > 0 && !up.row_units.empty()) ? (topk + w.rpc - 1) / w.rpc : 0;
    w.max_parts = std::max(1, w.chunks + (window > 0 ? 1 : 0));
    auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
    w.q16 = r256((size_t)n_entries * batch * kHeads * kDim * 2);
    w.partials = r256((size_t)n_entries * batch * w.max_parts * kPartFloats * 4);
    w.total = w.q16 + w.partials;
    return w;
}

// Rows per chunk of a row unit: a multiple of the 64-row tile, at most 2,048
// and at most 63 chunks.  Candidates (the smallest tile multiple giving 1..8
// chunks, and the powers of two) are scored by dispatching the pairs in launch
// order onto 74 pair slots (148 SMs, one CTA per SM), a pair costing, in tile
// units, its tiles plus a fixed set-up and a quarter tile per consumer layer
// (its queries in, its partial out), plus the merge, which reads one partial
// per chunk; the lowest score wins, ties going to longer chunks.
int rows_per_chunk(const UnitPlan &up, int n_entries, int batch, int topk, int window, size_t budget)
{
    if (up.row_units.empty() || topk <= 0) return kMaxChunkRows;
    constexpr int kPairSlots = 74;
    constexpr double kPairSetup = 3.0, kPerLayer = 0.25, kMergePerPart = 0.02;
    const int rmax = std::min(kMaxChunkRows, (topk + kTile - 1) / kTile * kTile);
    const int win_tiles = (window + kTile - 1) / kTile;
    size_t max_layers = 1;
    for (const auto &g : up.row_units) max_layers = std::max(max_layers, g.size());
    // candidates: the smallest tile multiple giving 1..8 chunks, and the powers of two
    std::vector<int> cand;
    for (int n = 1; n <= 8; ++n) cand.push_back(std::min(rmax, ((topk + n - 1) / n + kTile - 1) / kTile * kTile));
    for (int r = kTile; r < rmax; r *= 2) cand.push_back(r);
    std::sort(cand.begin(), cand.end());
    cand.erase(std::unique(cand.begin(), cand.end()), cand.end());
    int best = -1, smallest = rmax;
    double best_score = 1e300;
    for (const int r : cand) {
        const int chunks = (topk + r - 1) / r;
        if (chunks > kMaxParts - 1) continue;
        if (layout_for(up, n_entries, batch, topk, window, r).total > budget) continue;
        std::priority_queue<double, std::vector<double>, std::greater<double>> slots;
        for (int i = 0; i < kPairSlots; ++i) slots.push(0.0);
        double span = 0.0;
        auto dispatch = [&](double cost) {
            const double t0 = slots.top();
            slots.pop();
            slots.push(t0 + cost);
            span = std::max(span, t0 + cost);
        };
        for (int b = 0; b < batch; ++b) {
            for (const auto &g : up.row_units)
                for (int ch = 0; ch < chunks; ++ch)
                    dispatch(kPairSetup + kPerLayer * (double)g.size() + (std::min(r, topk - ch * r) + kTile - 1) / kTile);
            for (size_t u = 0; u < up.window_units.size(); ++u) dispatch(kPairSetup + kPerLayer + win_tiles);
        }
        const double score = span + kMergePerPart * (double)(chunks + 1) * (double)max_layers;
        if (score < best_score - 1e-9 || (score <= best_score + 1e-9 && r > best)) {
            best_score = score;
            best = r;
        }
    }
    return best > 0 ? best : smallest;  // nothing fits the budget: the smallest workspace
}

// The launch's layout: the fastest chunking whose workspace fits `budget`.
WsLayout ws_layout(const UnitPlan &up, int n_entries, int batch, int topk, int window, size_t budget)
{
    return layout_for(up, n_entries, batch, topk, window, rows_per_chunk(up, n_entries, batch, topk, window, budget));
}

}  // namespace

int attn_pack_jobs(const AttnPlan &plan, QuantJob *jobs, int cap)
{
    int n = 0;
    uint8_t *q16 = static_cast<uint8_t *>(plan.workspace);
    for (int e = 0; e < plan.n_entries && n < cap; ++e) {
        QuantJob j;
        std::memset(&j, 0, sizeof(j));
        j.src = plan.entries[e].q;
        j.dst.format = kFmtPackF16;
        j.dst.data = q16 + (size_t)e * plan.batch * kHeads * kDim * 2;
        j.rows_per_seq = kHeads;
        j.n_seqs = plan.batch;
        jobs[n++] = j;
    }
    return n;
}

size_t attn_workspace_bytes(const AttnEntry *entries, int n_entries, int batch, int topk, int window, size_t budget)
{
    const UnitPlan up = group_units(entries, n_entries, window);
    return ws_layout(up, n_entries, batch, topk, window, budget).total;
}

cudaError_t launch_attention(const AttnPlan &plan, int *flags, cudaStream_t stream, cudaEvent_t mid_event)
{
    if (plan.n_entries <= 0 || plan.n_entries > kMaxAttnEntries) return cudaErrorInvalidValue;
    const UnitPlan up = group_units(plan.entries, plan.n_entries, plan.window);
    const WsLayout wl = ws_layout(up, plan.n_entries, plan.batch, plan.topk, plan.window, plan.workspace_bytes);
    if (plan.workspace_bytes < wl.total || (int)(up.row_units.size() + up.window_units.size()) > kMaxUnits)
        return cudaErrorInvalidValue;
    uint8_t *ws = static_cast<uint8_t *>(plan.workspace);

    std::vector<uint8_t> pbuf(sizeof(AttnParams), 0);
    AttnParams &p = *reinterpret_cast<AttnParams *>(pbuf.data());
    p.batch = plan.batch;
    p.topk = plan.topk;
    p.window = plan.window;
    p.rows_per_chunk = wl.rpc;
    p.max_parts = wl.max_parts;
    p.seq_lens = plan.seq_lens;
    p.q16 = ws;
    p.partials = reinterpret_cast<float *>(ws + wl.q16);
    for (int e = 0; e < plan.n_entries; ++e) {
        p.entries[e].q = plan.entries[e].q;
        p.entries[e].out = plan.entries[e].out;
        p.entries[e].lse = plan.entries[e].lse;
        p.entries[e].n_parts = 0;
        p.entries[e].part_win = -1;
    }
    int cta = 0, nu = 0;
    for (const auto &g : up.row_units) {
        UnitDev &U = p.units[nu++];
        U.cache = plan.entries[g[0]].kv;
        U.idx = plan.entries[g[0]].idx;
        U.is_window = 0;
        U.n_layers = (int)g.size();
        for (size_t j = 0; j < g.size(); ++j) {
            U.entry[j] = g[j];
            p.entries[g[j]].n_parts = wl.chunks;  // row chunk c is part c
        }
        U.cta_begin = cta;
        cta += 2 * wl.chunks;
    }
    for (int e : up.window_units) {
        UnitDev &U = p.units[nu++];
        U.cache = plan.entries[e].swa;
        U.idx = nullptr;
        U.is_window = 1;
        U.n_layers = 1;
        U.entry[0] = e;
        U.cta_begin = cta;
        cta += 2;
        p.entries[e].part_win = p.entries[e].n_parts;
        p.entries[e].n_parts += 1;
    }
    p.n_units = nu;

    cudaError_t err = cudaSuccess;
    if (cta > 0 && !plan.q_packed) {
        std::vector<QuantJob> jobs((size_t)plan.n_entries);
        const int n = attn_pack_jobs(plan, jobs.data(), plan.n_entries);
        err = launch_quantize(jobs.data(), n, flags, stream);
    }
    if (err == cudaSuccess && cta > 0) {
        const size_t smem = kOffMisc + sizeof(AttnMisc);
        int dev = 0;
        err = cudaGetDevice(&dev);
        static bool attr_set[64] = {};
        if (err == cudaSuccess && (dev < 0 || dev >= 64 || !attr_set[dev])) {
            err = cudaFuncSetAttribute(attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
            if (err == cudaSuccess && dev >= 0 && dev < 64) attr_set[dev] = true;
        }
        if (err == cudaSuccess) {
            attn_tc_kernel<<<dim3((unsigned)cta, (unsigned)plan.batch), kThreads, smem, stream>>>(p, flags);
            count_launches(1);
            err = cudaGetLastError();
        }
    }
    if (err == cudaSuccess && mid_event) err = record_event(mid_event, stream);
    // merge (a layer with neither selected rows nor a window gets zeros)
    if (err == cudaSuccess) {
        MergeParams mp;
        std::memset(&mp, 0, sizeof(mp));
        std::memcpy(mp.entries, p.entries, sizeof(mp.entries));
        mp.batch = plan.batch;
        mp.max_parts = wl.max_parts;
        mp.partials = p.partials;
        attn_merge_kernel<<<dim3((unsigned)plan.n_entries, (unsigned)plan.batch, 8u), 256, 0, stream>>>(mp);
        count_launches(1);
        err = cudaGetLastError();
    }
    return err;
}

}  // namespace csa2
