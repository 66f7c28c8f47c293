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
// sequence); CTA h of the pair owns channels 256h..256h+255 of the queries,
// of every gathered row and of the output.  QK^T is split along channels:
// each CTA forms the partial scores of its half, the two swap partials with
// one bulk shared-memory copy each way and both add them (fp32 addition
// commutes, so both hold bit-identical scores and run the identical softmax).
// PV then touches only the CTA's own channels.  Each CTA leaves a partial
// (running max, sum, unnormalised output of its half) per consumer layer; a
// second kernel merges each (layer, sequence, half)'s partials in parallel.
//
// Tensor memory (512 columns): the 128 query rows of the CTA's half as fp16
// pairs (128 columns, the A operand of QK^T), S double-buffered (2 x 64), and
// O (256 columns).
//
// One CTA, 13 warps:
//   warps 0-7  softmax: warp w serves query rows 32(w%4)..+31 (its tensor-
//              memory lanes) and keys 32(w/4)..+31 of each 64-row tile; it
//              first writes its rows' queries into tensor memory;
//   warps 8-11 producers: per 64-row tile each thread owns one row and half
//              of the CTA's channels; it loads the next tile's bytes into
//              registers while it dequantises the current one (E2M1 x E4M3
//              and E4M3 are exact in fp16) into the core-matrix layout;
//   warp 12    tensor-memory allocation and tcgen05.mma issue: S[b] = Q_h V_h^T
//              (M 128, N 64, K 256; A from tensor memory), then O_h += P V_h
//              (M 128, N 256, K 64), O_h resident in tensor memory.
// V, S and P are double-buffered, so the softmax of tile t+1 does not wait
// for PV(t) unless O must be rescaled (lazy: only when a row's running max
// grows by more than e^8).  Every hand-off is an mbarrier with a bounded wait
// (a wait that gives up raises the timeout flag and the CTA drains); both
// CTAs of a pair meet at a cluster barrier before either exits, so neither
// touches the shared memory of a CTA that has finished.
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
constexpr int kHalf = 256;                 // channels per CTA of a pair
constexpr int kSoftThreads = 256;          // warps 0-7
constexpr int kProducers = 128;            // warps 8-11
constexpr int kMmaWarp = 12;
constexpr int kThreads = 416;              // 13 warps
constexpr int kMaxChunkRows = 2048;        // rows per chunk of a row unit
constexpr int kVBytes = kTile * kHalf * 2; // 32,768 per buffer
constexpr int kPBytes = 128 * kTile * 2;   // 16,384 per buffer
constexpr int kXBytes = 128 * kTile * 4;   // 32,768: partial scores of one tile
constexpr int kOffV = 0;
constexpr int kOffP = kOffV + 2 * kVBytes;
constexpr int kOffXin = kOffP + 2 * kPBytes;   // the peer's partial lands here
constexpr int kOffXout = kOffXin + kXBytes;    // ours, staged for the copy to the peer
constexpr int kOffMisc = kOffXout + kXBytes;
constexpr int kPartFloats = 64 + kHeads * kDim;  // m[2][16], l[2][16], O[16][512]
constexpr int kMaxUnits = 2 * kMaxAttnEntries;
constexpr int kMaxParts = 64;              // partials per layer: at most 63 row chunks and the window
constexpr float kRescaleGap = 8.0f;        // lazy O rescale threshold (natural log)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColQ = 0;              // 128 columns: query rows, fp16 pairs
constexpr uint32_t kColS = 128;            // 2 x 64 columns
constexpr uint32_t kColO = 256;            // 256 columns
// Instruction descriptors: QK^T (A from tensor memory, B K-major), PV (A K-major, B = V read MN-major).
constexpr uint32_t kIdescQK = tc::idesc_f16(128, kTile, false, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(128, kHalf, false, true);
// named barriers: 1 producers, 2 softmax (all 256)
constexpr uint32_t kBarProd = 1, kBarSoft = 2;

struct AttnMisc {
    float mscale[2][kTile];   // per V buffer: per-row scale (FP8 window rows)
    uint32_t vmask[2][2];     // per V buffer: valid rows (bit j of word j/32)
    float xmax[2][2][128];    // per tile parity and key half: tile max of each query row
    float lpart[128];         // running sum of the second key half, for the final combine
    uint64_t q_bar, full_v[2], s_full[2], s_free[2], p_full[2], pv_done[2];
    uint64_t x_full;          // the peer's partial scores have landed in Xin (bulk copy)
    uint64_t x_free;          // the peer has consumed the partial this CTA sent it
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
    float *partials;        // [entry][B][max_parts][kPartFloats]
};

// Byte offset of fp16 element (row r, channel c) of an operand with 256-channel
// rows in the no-swizzle core-matrix layout: 8-row groups 4,096 B apart,
// 8-channel groups 128 B apart.
__host__ __device__ __forceinline__ uint32_t cm_off256(uint32_t r, uint32_t c)
{
    return (r >> 3) * 4096u + (c >> 3) * 128u + (r & 7u) * 16u + (c & 7u) * 2u;
}

// Partial scores of one tile: row r holds 16 float4 (64 keys), chunk k at
// position k ^ (r & 7), so a quarter-warp's 16-byte accesses (8 consecutive
// rows, same k) fall in distinct banks.
__host__ __device__ __forceinline__ uint32_t x_off(uint32_t r, uint32_t k)
{
    return r * (kTile * 4) + ((k ^ (r & 7u)) * 16u);
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
    uint8_t *Vs, *Ps, *Xin, *Xout;
    int *flags;
    uint32_t tmem;
    int b, L, W, row0, n_rows, n_tiles, chunk, half;
};

// ---- producers (warps 8-11): gather + dequantise 64-row tiles -------------------------
// Thread ptid owns row j = ptid % 64 of every tile and the half w = ptid / 64
// of the CTA's 256 channels: channels 256h + 128w .. +127 (FP4 rows: four
// 16-byte granules of 32 channels and eight E4M3 scales; FP8 rows: eight
// granules of 16).
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
        const uint8_t *base = ptr ? ptr + c.half * 256 + 128 * w : nullptr;
#pragma unroll
        for (int i = 0; i < 8; ++i)
            r.g[i] = base ? __ldg(reinterpret_cast<const uint4 *>(base + 16 * i)) : make_uint4(0u, 0u, 0u, 0u);
    } else {
        const uint8_t *base = ptr ? ptr + c.half * 128 + 64 * w : nullptr;
#pragma unroll
        for (int i = 0; i < 4; ++i)
            r.g[i] = base ? __ldg(reinterpret_cast<const uint4 *>(base + 16 * i)) : make_uint4(0u, 0u, 0u, 0u);
        const uint2 sc2 = ptr ? __ldg(reinterpret_cast<const uint2 *>(ptr + kKvCodes + c.half * 16 + 8 * w))
                              : make_uint2(0u, 0u);
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
            const int ch = 128 * w + 16 * i;  // channels ch..ch+15 of the half
            const uint4 cw = r.g[i];
            *reinterpret_cast<uint4 *>(V + cm_off256(j, ch)) =
                make_uint4(pack_h2(e4m3x2_half2(cw.x & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.x >> 16)),
                           pack_h2(e4m3x2_half2(cw.y & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.y >> 16)));
            *reinterpret_cast<uint4 *>(V + cm_off256(j, ch + 8)) =
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
                *reinterpret_cast<uint4 *>(V + cm_off256(j, ch + 8 * k)) =
                    make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
        }
    }
}

template <bool FP8>
__device__ __forceinline__ void produce(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const int ptid = threadIdx.x - kSoftThreads;
    const int j = ptid & (kTile - 1), w = ptid >> 6;
    // row positions run two tiles ahead of the row bytes, so no load waits on another
    int32_t pos_next = FP8 ? -1 : row_pos(c, 1, j);
    RowRegs<FP8> cur, nxt;
    if (c.n_tiles > 0) load_row<FP8>(c, 0, j, w, FP8 ? -1 : row_pos(c, 0, j), cur);
    for (int t = 0; t < c.n_tiles; ++t) {
        const int vb = t & 1;
        if (t + 1 < c.n_tiles) load_row<FP8>(c, t + 1, j, w, pos_next, nxt);  // in flight during this tile's work
        if (!FP8) pos_next = row_pos(c, t + 2, j);
        // V[vb] and its row metadata are free once PV(t-2) has finished
        const bool bad = (t >= 2) && !tc::mbar_wait(&M.pv_done[vb], ((t - 2) >> 1) & 1);
        if (bar_any(kBarProd, kProducers, bad)) {
            if (ptid == 0) raise_flag(c.flags, kFlagTimeout);
            break;
        }
        store_row<FP8>(c.Vs + vb * kVBytes, j, w, cur);
        if (w == 0) {
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, cur.valid);
            if ((j & 31) == 0) M.vmask[vb][j >> 5] = mask;
            M.mscale[vb][j] = FP8 ? __uint_as_float(cur.s[0]) : 1.0f;
        }
        tc::fence_async_smem();
        tc::mbar_arrive(&M.full_v[vb]);
        cur = nxt;
    }
}

// ---- MMA issuer (one thread) ---------------------------------------------------------
// QK^T of tile t is issued in two groups of 8 MMAs; between groups (and while
// waiting for the next tile) the issuer polls for a finished P and issues its
// PV at once, so PV never queues behind a whole QK^T.
__device__ __forceinline__ void issue_mmas(const Ctx &c)
{
    AttnMisc &M = *c.M;
    bool ok = tc::mbar_wait(&M.q_bar, 0);  // the queries are in tensor memory
    // descriptors; a K step of 16 adds 8 columns to the tensor-memory A operand,
    // 256 B (16 in the 16-byte address field) to K-major smem operands and
    // 8,192 B (512) to V read MN-major
    const uint32_t va0 = tc::smem_u32(c.Vs), va1 = tc::smem_u32(c.Vs + kVBytes);
    const uint64_t vd0 = tc::sdesc(va0, 128, 4096), vd1 = tc::sdesc(va1, 128, 4096);
    const uint64_t vm0 = tc::sdesc(va0, 4096, 128), vm1 = tc::sdesc(va1, 4096, 128);
    const uint64_t pd0 = tc::sdesc(tc::smem_u32(c.Ps), 128, 1024);
    const uint64_t pd1 = tc::sdesc(tc::smem_u32(c.Ps + kPBytes), 128, 1024);
    const uint32_t qa = c.tmem + kColQ;
    int qk_done = 0;  // tiles whose QK^T has been issued
    int pv_next = 0;  // next tile whose PV is due
    uint64_t *last_bar = nullptr;
    uint32_t last_par = 0;
    auto issue_pv = [&](int t) {
        const int pb = t & 1;
        tc::fence_after_sync();
        const uint64_t pdb = pb ? pd1 : pd0, vmb = pb ? vm1 : vm0;
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k)
            tc::mma_f16(c.tmem + kColO, pdb + 16 * k, vmb + 512 * k, kIdescPV, (t > 0 || k > 0) ? 1u : 0u);
        tc::mma_commit(&M.pv_done[pb]);
        last_bar = &M.pv_done[pb];
        last_par = (t >> 1) & 1;
    };
    // issue every PV whose P is ready (non-blocking)
    auto poll_pv = [&]() {
        while (pv_next < qk_done && tc::mbar_try_wait(&M.p_full[pv_next & 1], (pv_next >> 1) & 1)) {
            issue_pv(pv_next);
            ++pv_next;
        }
    };
    // bounded wait on (bar, parity) that keeps issuing ready PVs meanwhile
    auto wait_polling = [&](uint64_t *bar, uint32_t par) {
        for (uint32_t i = 0; i < tc::kWaitLimit; ++i) {
            if (tc::mbar_try_wait(bar, par)) return true;
            poll_pv();
        }
        return false;
    };
    for (int t = 0; t < c.n_tiles && ok; ++t) {
        const int vb = t & 1;
        if (!wait_polling(&M.full_v[vb], (t >> 1) & 1) ||
            (t >= 2 && !wait_polling(&M.s_free[vb], ((t - 2) >> 1) & 1))) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        const uint32_t d = c.tmem + kColS + kTile * vb;
        const uint64_t vdb = vb ? vd1 : vd0;
#pragma unroll
        for (int g = 0; g < 2; ++g) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ks = 8 * g + k;
                tc::mma_f16_ta(d, qa + 8 * ks, vdb + 16 * ks, kIdescQK, ks > 0 ? 1u : 0u);
            }
            if (g == 1) {
                tc::mma_commit(&M.s_full[vb]);
                last_bar = &M.s_full[vb];
                last_par = (t >> 1) & 1;
                qk_done = t + 1;
            }
            poll_pv();
        }
    }
    // the remaining PVs, in order
    while (ok && pv_next < qk_done) {
        if (!tc::mbar_wait(&M.p_full[pv_next & 1], (pv_next >> 1) & 1)) {
            ok = false;
            break;
        }
        issue_pv(pv_next);
        ++pv_next;
    }
    if (!ok) raise_flag(c.flags, kFlagTimeout);
    // every issued MMA must have finished before the tensor memory is released
    if (last_bar) tc::mbar_wait(last_bar, last_par);
}

// ---- softmax (warps 0-7) --------------------------------------------------------------
// Thread (row r = 32(w%4) + lane, key half kh = w/4) holds the row's scores of
// keys 32kh..32kh+31 of each tile and O columns 128kh..128kh+127.  A failed
// wait clears `ok`; the loop leaves only at a reduction over all 256 threads,
// so every softmax thread meets every named barrier the same number of times.
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
    const uint32_t peer = (uint32_t)(c.half ^ 1);
    const uint32_t xin_peer = tc::mapa(tc::smem_u32(c.Xin), peer);
    const uint32_t xfull_peer = tc::mapa(tc::smem_u32(&M.x_full), peer);
    const uint32_t xfree_peer = tc::mapa(tc::smem_u32(&M.x_free), peer);

    // this row's queries (channels 128kh..+127 of the half) into tensor memory as fp16 pairs
    {
        const float *q = active ? c.P->entries[U.entry[slot_layer]].q + ((int64_t)c.b * kHeads + head) * kDim +
                                      c.half * kHalf + 128 * kh
                                : nullptr;
#pragma unroll 1
        for (int cc = 0; cc < 2; ++cc) {
            float h[32];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float4 a = q ? __ldg(reinterpret_cast<const float4 *>(q + 64 * cc + 4 * i))
                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                h[2 * i] = __uint_as_float(pack_h2(__floats2half2_rn(a.x, a.y)));
                h[2 * i + 1] = __uint_as_float(pack_h2(__floats2half2_rn(a.z, a.w)));
            }
            tc::tmem_st32(tc::taddr(c.tmem, lane_base, kColQ + 64 * kh + 32 * cc), h);
        }
        tc::fence_before_sync();
        tc::mbar_arrive(&M.q_bar);
    }

    float m_used = -INFINITY, l_half = 0.0f;
    bool ok = true;
    for (int t = 0; t < c.n_tiles; ++t) {
        const int vb = t & 1;
        ok = ok && tc::mbar_wait(&M.full_v[vb], (t >> 1) & 1) && tc::mbar_wait(&M.s_full[vb], (t >> 1) & 1);
        tc::fence_after_sync();
        float s[32];
        tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColS + kTile * vb + 32 * kh), s);
        tc::fence_before_sync();
        tc::mbar_arrive(&M.s_free[vb]);
        // our partial scores to the peer, once it has consumed the previous ones
        ok = ok && (t < 1 || tc::mbar_wait_cluster(&M.x_free, (t - 1) & 1));
#pragma unroll
        for (int k = 0; k < 8; ++k)
            *reinterpret_cast<float4 *>(c.Xout + x_off(r, 8 * kh + k)) =
                make_float4(s[4 * k], s[4 * k + 1], s[4 * k + 2], s[4 * k + 3]);
        tc::fence_async_smem();
        if (bar_any(kBarSoft, kSoftThreads, !ok)) break;
        if (tid == 0) tc::bulk_s2peer(xin_peer, c.Xout, kXBytes, xfull_peer);
        // full scores = ours + the peer's, masked and scaled; this key half's tile max
        ok = tc::mbar_wait_cluster(&M.x_full, t & 1);
        if (tid == 0 && ok && t + 1 < c.n_tiles) tc::mbar_expect_tx(&M.x_full, kXBytes);  // arm the next tile
        const uint32_t vm = M.vmask[vb][kh];
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const float4 v = *reinterpret_cast<const float4 *>(c.Xin + x_off(r, 8 * kh + k));
            const float pv[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 4 * k + i;
                const float z = s[j] + pv[i];
                const float zs = FP8 ? z * M.mscale[vb][32 * kh + j] : z;
                s[j] = ((vm >> j) & 1u) ? zs : -INFINITY;
                mx[i] = fmaxf(mx[i], s[j]);
            }
        }
        const float mt = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        M.xmax[vb][kh][r] = mt;
        if (bar_any(kBarSoft, kSoftThreads, !ok)) break;  // also: every Xin read and xmax write is done
        if (tid == 32) tc::mbar_arrive_cluster(xfree_peer);  // not the copy issuer: its release would wait on the copy
        const float m_tile = fmaxf(mt, M.xmax[vb][kh ^ 1][r]);
        const float m_new = active ? fmaxf(m_used, m_tile) : m_used;
        // lazy rescale of this warp's O columns, warp-uniform (both key halves decide alike)
        if (__any_sync(0xFFFFFFFFu, active && m_new > m_used + kRescaleGap)) {
            if (t >= 1) {
                ok = ok && tc::mbar_wait(&M.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1);  // O is current
                tc::fence_after_sync();
                const float alpha = (active && m_used != -INFINITY) ? __expf(m_used - m_new) : (active ? 0.0f : 1.0f);
#pragma unroll 1
                for (int c0 = 0; c0 < 128; c0 += 32) {
                    float o[32];
                    tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + 128 * kh + c0), o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tc::tmem_st32(tc::taddr(c.tmem, lane_base, kColO + 128 * kh + c0), o);
                }
                if (active) l_half *= alpha;
            }
            if (active) m_used = m_new;
        }
        // P[vb] is free once PV(t-2) has finished
        ok = ok && (t < 2 || tc::mbar_wait(&M.pv_done[vb], ((t - 2) >> 1) & 1));
        // P = exp(S - m) as fp16, K-major core-matrix layout (8 groups of 8 keys, 1,024 B
        // per 8-row group); window rows hold raw E4M3 codes, so their scale joins the weight
        const float mb = m_used * kLog2e;
        float ls[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int j = 0; j < 32; ++j) {
            s[j] = (active && s[j] != -INFINITY) ? exp2f(fmaf(s[j], kLog2e, -mb)) : 0.0f;
            ls[j & 3] += s[j];
        }
        l_half += (ls[0] + ls[1]) + (ls[2] + ls[3]);
        uint8_t *Pb = c.Ps + vb * kPBytes + (r >> 3) * 1024 + (r & 7) * 16;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
            uint32_t ph[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int j = 8 * g + 2 * i;
                const float a = FP8 ? s[j] * M.mscale[vb][32 * kh + j] : s[j];
                const float d = FP8 ? s[j + 1] * M.mscale[vb][32 * kh + j + 1] : s[j + 1];
                ph[i] = pack_h2(__floats2half2_rn(a, d));
            }
            *reinterpret_cast<uint4 *>(Pb + (4 * kh + g) * 128) = make_uint4(ph[0], ph[1], ph[2], ph[3]);
        }
        tc::fence_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(&M.p_full[vb]);
    }
    if (c.n_tiles > 0) {
        const int last = c.n_tiles - 1;
        ok = ok && tc::mbar_wait(&M.pv_done[last & 1], (last >> 1) & 1);
    }
    if (!ok) raise_flag(c.flags, kFlagTimeout);
    // both key halves' sums, then this chunk's partial for the channel half: (m, l, unnormalised O)
    if (kh == 1) M.lpart[r] = l_half;
    const bool have = !bar_any(kBarSoft, kSoftThreads, !ok) && c.n_tiles > 0;
    tc::fence_after_sync();
    float *orow = nullptr;
    if (active) {
        const int e = U.entry[slot_layer];
        const EntryDev &E = c.P->entries[e];
        const int part = U.is_window ? E.part_win : c.chunk;
        float *rec = c.P->partials + (((int64_t)e * c.P->batch + c.b) * c.P->max_parts + part) * kPartFloats;
        if (kh == 0) {
            const float l_sum = l_half + M.lpart[r];
            const bool any = have && l_sum > 0.0f;
            rec[c.half * 16 + head] = any ? m_used : -INFINITY;
            rec[32 + c.half * 16 + head] = any ? l_sum : 0.0f;
        }
        orow = rec + 64 + head * kDim + c.half * kHalf + 128 * kh;
    }
    for (int c0 = 0; c0 < 128; c0 += 32) {
        float o[32];
        if (have) tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + 128 * kh + c0), o);
        if (active) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(orow + c0 + i) =
                    have ? make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    tc::fence_before_sync();
}

// ---- merge: one CTA per (layer, sequence, channel half) combines the partials ----------
// 256 threads.  The (m, l) of every part are staged in shared memory in one
// round of independent loads; 16 threads then turn them into per-part weights
// exp(m_p - max) (one head each), and every thread accumulates 16 output
// channels of one head over the parts.  A layer with no parts writes zeros.
struct MergeParams {
    EntryDev entries[kMaxAttnEntries];
    int32_t batch, max_parts;
    const float *partials;  // [entry][B][max_parts][kPartFloats]
};

__global__ void __launch_bounds__(256) attn_merge_kernel(const __grid_constant__ MergeParams P)
{
    __shared__ float m_sh[kMaxParts][kHeads], l_sh[kMaxParts][kHeads];
    __shared__ float inv_sh[kHeads];
    const int e = blockIdx.x, b = blockIdx.y, half = blockIdx.z, tid = threadIdx.x;
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
        if (half == 0 && E.lse) E.lse[(int64_t)b * kHeads + tid] = ls > 0.0f ? mx + logf(ls) : -INFINITY;
    }
    __syncthreads();
    const int h = tid >> 4, c0 = half * kHalf + (tid & 15) * 16;
    float acc[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll 4
    for (int p = 0; p < np; ++p) {
        const float wp = m_sh[p][h];
        const float4 *op = reinterpret_cast<const float4 *>(recs + (int64_t)p * kPartFloats + 64 + h * kDim + c0);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 v = __ldcg(op + i);
            acc[4 * i] += wp * v.x;
            acc[4 * i + 1] += wp * v.y;
            acc[4 * i + 2] += wp * v.z;
            acc[4 * i + 3] += wp * v.w;
        }
    }
    const float inv = inv_sh[h];
    float4 *out = reinterpret_cast<float4 *>(E.out + ((int64_t)b * kHeads + h) * kDim + c0);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        out[i] = make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kThreads, 1)
    attn_tc_kernel(const __grid_constant__ AttnParams P, int *flags)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx c;
    c.P = &P;
    c.M = reinterpret_cast<AttnMisc *>(smem + kOffMisc);
    c.Vs = smem + kOffV;
    c.Ps = smem + kOffP;
    c.Xin = smem + kOffXin;
    c.Xout = smem + kOffXout;
    c.flags = flags;
    c.b = blockIdx.y;
    int u = 0;
    while (u + 1 < P.n_units && (int)blockIdx.x >= P.units[u + 1].cta_begin) ++u;
    c.U = &P.units[u];
    const int local = (int)blockIdx.x - c.U->cta_begin;
    c.chunk = local >> 1;
    c.half = (int)tc::cluster_rank();  // = local & 1: a pair is one cluster
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
        tc::mbar_init(&M.q_bar, kSoftThreads);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&M.full_v[i], kProducers);
            tc::mbar_init(&M.s_full[i], 1);
            tc::mbar_init(&M.s_free[i], kSoftThreads);
            tc::mbar_init(&M.pv_done[i], 1);
            tc::mbar_init(&M.p_full[i], kSoftThreads);
        }
        tc::mbar_init(&M.x_full, 1);
        tc::mbar_init(&M.x_free, 1);
        tc::mbar_init_fence();
        if (c.n_tiles > 0) tc::mbar_expect_tx(&M.x_full, kXBytes);  // armed for the first tile's partial
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&M.tmem_slot, kTmemCols);
    tc::fence_before_sync();
    tc::cluster_sync();  // both CTAs' barriers exist before either signals the other
    tc::fence_after_sync();
    c.tmem = M.tmem_slot;

    if (warp < 8) {
        if (fp8) softmax_rows<true>(c);
        else softmax_rows<false>(c);
    } else if (warp < kMmaWarp) {
        if (fp8) produce<true>(c);
        else produce<false>(c);
    } else {
        if (lane == 0) issue_mmas(c);
        __syncwarp();
    }
    tc::fence_before_sync();
    tc::cluster_sync();  // no remote shared-memory access after this point
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(c.tmem, kTmemCols);
    }
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

// Rows per chunk of a row unit (a multiple of the 64-row tile, at most the
// 2,048 rows whose positions a CTA stages).  Each candidate is scored by
// dispatching the pairs in launch order onto 74 pair slots (148 SMs, one CTA
// per SM), a pair costing, in tile units, its tiles plus a fixed set-up and
// half a tile per consumer layer (its queries in, its partial out), and by the
// merge tail, which reads one partial per chunk; the lowest score wins, ties
// going to longer chunks.
int rows_per_chunk(const UnitPlan &up, int batch, int topk, int window)
{
    if (up.row_units.empty() || topk <= 0) return kMaxChunkRows;
    constexpr int kPairSlots = 74;
    constexpr double kPairSetup = 1.0, kPerLayer = 0.5, kMergePerPart = 0.02;
    const int rmax = std::min(kMaxChunkRows, (topk + kTile - 1) / kTile * kTile);
    int rmin = kTile;  // at most kMaxParts - 1 chunks
    while (rmin < rmax && (topk + rmin - 1) / rmin > kMaxParts - 1) rmin *= 2;
    const int win_tiles = (window + kTile - 1) / kTile;
    size_t max_layers = 1;
    for (const auto &g : up.row_units) max_layers = std::max(max_layers, g.size());
    int best = rmax;
    double best_score = 1e300;
    for (int r = rmin; r <= rmax; r *= 2) {
        std::priority_queue<double, std::vector<double>, std::greater<double>> slots;
        for (int i = 0; i < kPairSlots; ++i) slots.push(0.0);
        double span = 0.0;
        auto dispatch = [&](double cost) {
            const double t0 = slots.top();
            slots.pop();
            slots.push(t0 + cost);
            span = std::max(span, t0 + cost);
        };
        const int chunks = (topk + r - 1) / r;
        for (int b = 0; b < batch; ++b) {
            for (const auto &g : up.row_units)
                for (int ch = 0; ch < chunks; ++ch)
                    dispatch(kPairSetup + kPerLayer * (double)g.size() + (std::min(r, topk - ch * r) + kTile - 1) / kTile);
            for (size_t u = 0; u < up.window_units.size(); ++u) dispatch(kPairSetup + kPerLayer + win_tiles);
        }
        const double score = span + kMergePerPart * (double)(chunks + 1) * (double)max_layers;
        if (score <= best_score) {
            best_score = score;
            best = r;
        }
        if (r >= rmax) break;
    }
    return best;
}

struct WsLayout {
    size_t partials = 0, total = 0;
    int rpc = kMaxChunkRows, chunks = 0, max_parts = 1;
};

WsLayout ws_layout(const UnitPlan &up, int n_entries, int batch, int topk, int window)
{
    WsLayout w;
    w.rpc = rows_per_chunk(up, batch, topk, window);
    w.chunks = (topk > 0 && !up.row_units.empty()) ? (topk + w.rpc - 1) / w.rpc : 0;
    w.max_parts = std::max(1, w.chunks + (window > 0 ? 1 : 0));
    auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
    w.partials = r256((size_t)n_entries * batch * w.max_parts * kPartFloats * 4);
    w.total = w.partials;
    return w;
}

}  // namespace

size_t attn_workspace_bytes(const AttnEntry *entries, int n_entries, int batch, int topk, int window)
{
    const UnitPlan up = group_units(entries, n_entries, window);
    return ws_layout(up, n_entries, batch, topk, window).total;
}

cudaError_t launch_attention(const AttnPlan &plan, int *flags, cudaStream_t stream, cudaEvent_t mid_event)
{
    if (plan.n_entries <= 0 || plan.n_entries > kMaxAttnEntries) return cudaErrorInvalidValue;
    const UnitPlan up = group_units(plan.entries, plan.n_entries, plan.window);
    const WsLayout wl = ws_layout(up, plan.n_entries, plan.batch, plan.topk, plan.window);
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
    p.partials = reinterpret_cast<float *>(ws);
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
    if (cta > 0) {
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
        attn_merge_kernel<<<dim3((unsigned)plan.n_entries, (unsigned)plan.batch, 2u), 256, 0, stream>>>(mp);
        count_launches(1);
        err = cudaGetLastError();
    }
    return err;
}

}  // namespace csa2
