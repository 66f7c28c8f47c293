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
// unit*.  A CTA takes one (unit, chunk of rows, half of the output channels,
// sequence) and produces a partial (running max, sum, unnormalised output);
// the last CTA to finish a (layer, sequence, half) merges its partials.
//
// One CTA, 9 warps:
//   warps 4-7  producers: each thread owns one row of a 32-row tile and a
//              quarter of its bytes; it loads the next tile's bytes into
//              registers while it dequantises the current one (E2M1 x E4M3
//              and E4M3 are exact in fp16) into the core-matrix layout;
//   warp 8     tensor-memory allocation and tcgen05.mma issue, descriptors
//              precomputed: S[b] = Q V^T (M 128, N 32, K 512) into tensor
//              memory, then O += P V (M 128, N 256, K 32), O resident in
//              tensor memory;
//   warps 0-3  one thread per query row: S from tensor memory, fp32 online
//              softmax with lazy rescaling of O (only when the running max
//              grows by more than e^8), P to shared memory as fp16.
// V, S and P are double-buffered, so the softmax of tile t+1 does not wait
// for PV(t) unless O must be rescaled.  Every hand-off is an mbarrier with a
// bounded wait (a wait that gives up raises the timeout flag and the CTA
// drains and exits).
#include <algorithm>
#include <cstring>
#include <utility>
#include <vector>

#include "internal.h"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kTile = 32;                  // rows per tile
constexpr int kProducers = 256;            // producer threads (warps 4-11)
constexpr int kMmaWarp = 12;
constexpr int kThreads = 416;              // 13 warps
constexpr int kMaxChunkRows = 2048;        // rows per chunk of a row unit (indices staged in smem)
constexpr int kQRowsBytes = kHeads * kDim * 2;  // 16 KB: one layer's 16 query rows in fp16
constexpr int kQBytes = 8 * kQRowsBytes;   // 131,072: 128 query rows
constexpr int kVBytes = kTile * kDim * 2;  // 32,768 per buffer
constexpr int kPBytes = 128 * kTile * 2;   // 8,192 per buffer
constexpr int kOffV = kQBytes;
constexpr int kOffP = kOffV + 2 * kVBytes;
constexpr int kOffIdx = kOffP + 2 * kPBytes;
constexpr int kOffMisc = kOffIdx + kMaxChunkRows * 4;
constexpr int kPartFloats = 64 + kHeads * kDim;  // m[2][16], l[2][16], O[16][512]
constexpr int kMaxUnits = 2 * kMaxAttnEntries;
constexpr float kRescaleGap = 8.0f;        // lazy O rescale threshold (natural log)
constexpr float kLog2e = 1.4426950408889634f;
constexpr uint32_t kTmemCols = 512;        // S[0] cols 0-31, S[1] cols 32-63, O cols 256-511
constexpr uint32_t kColO = 256;
// Instruction descriptors: QK^T (both operands K-major), PV (B = V read MN-major).
constexpr uint32_t kIdescQK = tc::idesc_f16(128, kTile, false, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(128, 256, false, true);

struct AttnMisc {
    float mscale[2][kTile];   // per V buffer: per-row scale (FP8 window rows)
    uint32_t vmask[2];        // per V buffer: valid rows
    uint64_t q_bar, full_v[2], s_full[2], s_free[2], p_full[2], pv_done[2];
    uint32_t tmem_slot;
    int32_t last[8];
};
static_assert(kOffMisc + (int)sizeof(AttnMisc) <= 232448, "attention shared memory over the 227 KB limit");

struct UnitDev {
    CacheView cache;        // FP4_KV cache (row unit) or FP8_SWA ring (window unit)
    const int32_t *idx;     // row unit: [B][topk]
    int32_t is_window;
    int32_t n_layers;       // consumer layers (1..8)
    int32_t entry[8];
    int32_t cta_begin;      // first flat CTA (x) index of this unit
};

struct EntryDev {
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
    const uint8_t *q16;     // [entry][B][16 KB] fp16 query rows in core-matrix layout
    float *partials;        // [entry][B][max_parts][kPartFloats]
    uint32_t *counters;     // [entry][B][2]
};

struct QList {
    const float *q[kMaxAttnEntries];
};

// Byte offset of fp16 element (row r, channel c) of an operand with 512-channel
// rows in the no-swizzle core-matrix layout: 8-row groups 8,192 B apart,
// 8-channel groups 128 B apart.
__host__ __device__ __forceinline__ uint32_t cm_off512(uint32_t r, uint32_t c)
{
    return (r >> 3) * 8192u + (c >> 3) * 128u + (r & 7u) * 16u + (c & 7u) * 2u;
}

__device__ __forceinline__ uint32_t pack_h2(__half2 v) { return *reinterpret_cast<uint32_t *>(&v); }

// q (fp32 [B][16][512]) -> fp16 core-matrix rows, 16 KB per layer and sequence.
__global__ void __launch_bounds__(256) pack_q_kernel(const __grid_constant__ QList qs, uint8_t *q16, int batch)
{
    const int e = blockIdx.x, b = blockIdx.y;
    const float *q = qs.q[e] + (int64_t)b * kHeads * kDim;
    uint8_t *dst = q16 + ((int64_t)e * batch + b) * kQRowsBytes;
    for (int it = threadIdx.x; it < kHeads * kDim / 8; it += blockDim.x) {
        const int r = it / (kDim / 8), c = (it % (kDim / 8)) * 8;
        const float4 a = __ldg(reinterpret_cast<const float4 *>(q + r * kDim + c));
        const float4 d = __ldg(reinterpret_cast<const float4 *>(q + r * kDim + c + 4));
        *reinterpret_cast<uint4 *>(dst + cm_off512(r, c)) =
            make_uint4(pack_h2(__floats2half2_rn(a.x, a.y)), pack_h2(__floats2half2_rn(a.z, a.w)),
                       pack_h2(__floats2half2_rn(d.x, d.y)), pack_h2(__floats2half2_rn(d.z, d.w)));
    }
}

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
    uint8_t *Qs, *Vs, *Ps;
    int32_t *sidx;      // the chunk's row positions (row units)
    int *flags;
    uint32_t tmem;
    int b, L, W, row0, n_rows, n_tiles, chunk, half;
    bool fp8;
};

// ---- producers (warps 4-11): gather + dequantise 32-row tiles ------------------------
// Thread ptid owns row j = ptid % 32 of every tile and the eighth w = ptid / 32
// of its 16-byte granules (FP4 rows: 16 granules of 32 channels, g = w, w + 8;
// FP8 rows: 32 granules of 16 channels, g = w + 8i).
constexpr int kPW = kProducers / 32;  // producer warps
template <bool FP8>
struct RowRegs {
    uint4 g[FP8 ? 32 / kPW : 16 / kPW];
    uint32_t s[FP8 ? 1 : 16 / kPW];  // FP4: two E4M3 scales per granule; FP8: the row's fp32 scale bits
    bool valid;
};

template <bool FP8>
__device__ __forceinline__ void load_row(const Ctx &c, int t, int j, int w, RowRegs<FP8> &r)
{
    const UnitDev &U = *c.U;
    const int v = t * kTile + j;  // row within this chunk
    const uint8_t *ptr = nullptr;
    uint32_t sc = 0u;
    if (v < c.n_rows) {
        if (!FP8) {
            const int32_t pos = c.sidx[v];
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
#pragma unroll
        for (int i = 0; i < 32 / kPW; ++i)
            r.g[i] = ptr ? __ldg(reinterpret_cast<const uint4 *>(ptr + 16 * (w + kPW * i))) : make_uint4(0u, 0u, 0u, 0u);
    } else {
#pragma unroll
        for (int i = 0; i < 16 / kPW; ++i) {
            r.g[i] = ptr ? __ldg(reinterpret_cast<const uint4 *>(ptr + 16 * (w + kPW * i))) : make_uint4(0u, 0u, 0u, 0u);
            r.s[i] = ptr ? (uint32_t)__ldg(reinterpret_cast<const unsigned short *>(ptr + kKvCodes + 2 * (w + kPW * i)))
                         : 0u;
        }
    }
}

template <bool FP8>
__device__ __forceinline__ void store_row(uint8_t *V, int j, int w, const RowRegs<FP8> &r)
{
    if (FP8) {
#pragma unroll
        for (int i = 0; i < 32 / kPW; ++i) {
            const int g = w + kPW * i;  // channels 16g..16g+15
            const uint4 cw = r.g[i];
            *reinterpret_cast<uint4 *>(V + cm_off512(j, 16 * g)) =
                make_uint4(pack_h2(e4m3x2_half2(cw.x & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.x >> 16)),
                           pack_h2(e4m3x2_half2(cw.y & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.y >> 16)));
            *reinterpret_cast<uint4 *>(V + cm_off512(j, 16 * g + 8)) =
                make_uint4(pack_h2(e4m3x2_half2(cw.z & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.z >> 16)),
                           pack_h2(e4m3x2_half2(cw.w & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.w >> 16)));
        }
    } else {
#pragma unroll
        for (int i = 0; i < 16 / kPW; ++i) {
            const int g = w + kPW * i;  // channels 32g..32g+31, scales 2g (first 16) and 2g+1
            const __half2 s0 = __half2half2(__float2half_rn(e4m3_value(r.s[i] & 0xFFu)));
            const __half2 s1 = __half2half2(__float2half_rn(e4m3_value((r.s[i] >> 8) & 0xFFu)));
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
                *reinterpret_cast<uint4 *>(V + cm_off512(j, 32 * g + 8 * k)) =
                    make_uint4(h[4 * k], h[4 * k + 1], h[4 * k + 2], h[4 * k + 3]);
        }
    }
}

template <bool FP8>
__device__ __forceinline__ void produce(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const int ptid = threadIdx.x - 128;
    const int j = ptid & (kTile - 1), w = ptid >> 5;
    if (!FP8) {
        for (int i = ptid; i < c.n_rows; i += kProducers)
            c.sidx[i] = __ldg(c.U->idx + (int64_t)c.b * c.P->topk + c.row0 + i);
        tc::named_sync(1, kProducers);
    }
    RowRegs<FP8> cur, nxt;
    if (c.n_tiles > 0) load_row<FP8>(c, 0, j, w, cur);
    for (int t = 0; t < c.n_tiles; ++t) {
        const int vb = t & 1;
        if (t + 1 < c.n_tiles) load_row<FP8>(c, t + 1, j, w, nxt);  // in flight during this tile's work
        // V[vb] and its row metadata are free once PV(t-2) has finished
        const bool bad = (t >= 2) && !tc::mbar_wait(&M.pv_done[vb], ((t - 2) >> 1) & 1);
        if (bar_any(1, kProducers, bad)) {
            if (ptid == 0) raise_flag(c.flags, kFlagTimeout);
            break;
        }
        store_row<FP8>(c.Vs + vb * kVBytes, j, w, cur);
        if (w == 0) {
            const uint32_t mask = __ballot_sync(0xFFFFFFFFu, cur.valid);
            if (j == 0) M.vmask[vb] = mask;
            M.mscale[vb][j] = FP8 ? __uint_as_float(cur.s[0]) : 1.0f;
        }
        tc::fence_async_smem();
        tc::mbar_arrive(&M.full_v[vb]);
        cur = nxt;
    }
}

// ---- MMA issuer (one thread) ---------------------------------------------------------
// QK^T of tile t is issued in groups of 8 MMAs; between groups (and while
// waiting for the next tile) the issuer polls for a finished P and issues its
// PV at once, so PV never queues behind a whole QK^T.
__device__ __forceinline__ void issue_mmas(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const UnitDev &U = *c.U;
    // query rows of the consumer layers: layer slot j -> rows 16j..16j+15 (16 KB each)
    tc::mbar_expect_tx(&M.q_bar, (uint32_t)U.n_layers * kQRowsBytes);
    for (int j = 0; j < U.n_layers; ++j)
        tc::bulk_g2s(c.Qs + j * kQRowsBytes, c.P->q16 + ((int64_t)U.entry[j] * c.P->batch + c.b) * kQRowsBytes,
                     kQRowsBytes, &M.q_bar);
    bool ok = tc::mbar_wait(&M.q_bar, 0);
    if (!ok) tc::mbar_wait(&M.q_bar, 0);  // let copies in flight land before giving up
    // descriptors; a K step of 16 adds 256 B (16 in the 16-byte address field) to the
    // K-major operands and 16,384 B (1,024) to V read MN-major
    const uint64_t qd = tc::sdesc(tc::smem_u32(c.Qs), 128, 8192);
    const uint32_t va0 = tc::smem_u32(c.Vs), va1 = tc::smem_u32(c.Vs + kVBytes);
    const uint64_t vd0 = tc::sdesc(va0, 128, 8192), vd1 = tc::sdesc(va1, 128, 8192);
    const uint64_t vm0 = tc::sdesc(va0 + c.half * (256 / 8) * 128, 8192, 128);
    const uint64_t vm1 = tc::sdesc(va1 + c.half * (256 / 8) * 128, 8192, 128);
    const uint64_t pd0 = tc::sdesc(tc::smem_u32(c.Ps), 128, 512);
    const uint64_t pd1 = tc::sdesc(tc::smem_u32(c.Ps + kPBytes), 128, 512);
    int qk_done = 0;  // tiles whose QK^T has been issued
    int pv_next = 0;  // next tile whose PV is due
    uint64_t *last_bar = nullptr;
    uint32_t last_par = 0;
    auto issue_pv = [&](int t) {
        const int pb = t & 1;
        tc::fence_after_sync();
        const uint64_t pdb = pb ? pd1 : pd0, vmb = pb ? vm1 : vm0;
        tc::mma_f16(c.tmem + kColO, pdb, vmb, kIdescPV, t > 0 ? 1u : 0u);
        tc::mma_f16(c.tmem + kColO, pdb + 16, vmb + 1024, kIdescPV, 1u);
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
        const uint32_t d = c.tmem + 32 * vb;
        const uint64_t vdb = vb ? vd1 : vd0;
#pragma unroll
        for (int g = 0; g < 4; ++g) {
#pragma unroll
            for (int k = 0; k < 8; ++k) {
                const int ks = 8 * g + k;
                tc::mma_f16(d, qd + 16 * ks, vdb + 16 * ks, kIdescQK, ks > 0 ? 1u : 0u);
            }
            if (g == 3) {
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

// ---- softmax rows (warps 0-3, thread = tensor-memory lane = query row) ----------------
template <bool FP8>
__device__ __forceinline__ void softmax_rows(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const UnitDev &U = *c.U;
    const int tid = threadIdx.x, warp = tid >> 5;
    const int slot_layer = tid >> 4, head = tid & 15;
    const bool active = slot_layer < U.n_layers;
    const uint32_t lane_base = (uint32_t)(32 * warp);
    float m_used = -INFINITY, l_sum = 0.0f;
    bool ok = true;
    for (int t = 0; t < c.n_tiles; ++t) {
        const int vb = t & 1;
        bool w_ok = tc::mbar_wait(&M.full_v[vb], (t >> 1) & 1) && tc::mbar_wait(&M.s_full[vb], (t >> 1) & 1);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        float s[kTile];
        tc::tmem_ld32(tc::taddr(c.tmem, lane_base, 32 * vb), s);
        tc::fence_before_sync();
        tc::mbar_arrive(&M.s_free[vb]);
        const uint32_t vmask = M.vmask[vb];
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTile; ++j) {
            const float z = FP8 ? s[j] * M.mscale[vb][j] : s[j];
            s[j] = ((vmask >> j) & 1u) ? z : -INFINITY;
            mt = fmaxf(mt, s[j]);
        }
        const float m_new = active ? fmaxf(m_used, mt) : m_used;
        // lazy rescale, warp-uniform: every lane of the warp joins the tensor-memory traffic
        if (__any_sync(0xFFFFFFFFu, active && m_new > m_used + kRescaleGap)) {
            if (t >= 1) {
                w_ok = tc::mbar_wait(&M.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1);  // O is current
                if (!__all_sync(0xFFFFFFFFu, w_ok)) {
                    ok = false;
                    break;
                }
                tc::fence_after_sync();
                const float alpha = (active && m_used != -INFINITY) ? __expf(m_used - m_new) : (active ? 0.0f : 1.0f);
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    float o[32];
                    tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tc::tmem_st32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
                }
                if (active) l_sum *= alpha;
            }
            if (active) m_used = m_new;
        }
        // P[vb] is free once PV(t-2) has finished
        w_ok = (t < 2) || tc::mbar_wait(&M.pv_done[vb], ((t - 2) >> 1) & 1);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
            ok = false;
            break;
        }
        const float mb = m_used * kLog2e;
        float p[kTile];
        float ls = 0.0f;
#pragma unroll
        for (int j = 0; j < kTile; ++j) {
            p[j] = (active && s[j] != -INFINITY) ? exp2f(fmaf(s[j], kLog2e, -mb)) : 0.0f;
            ls += p[j];
        }
        l_sum += ls;
        uint32_t ph[kTile / 2];
#pragma unroll
        for (int j = 0; j < kTile; j += 2) {
            const float a = FP8 ? p[j] * M.mscale[vb][j] : p[j];      // window rows hold raw E4M3 codes:
            const float d = FP8 ? p[j + 1] * M.mscale[vb][j + 1] : p[j + 1];  // their scale joins the weight
            ph[j >> 1] = pack_h2(__floats2half2_rn(a, d));
        }
        // P row into its K-major core-matrix layout: 4 groups of 8 keys, 512 B per 8-row group
        uint8_t *Pb = c.Ps + vb * kPBytes;
#pragma unroll
        for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4 *>(Pb + (tid >> 3) * 512 + g * 128 + (tid & 7) * 16) =
                make_uint4(ph[4 * g], ph[4 * g + 1], ph[4 * g + 2], ph[4 * g + 3]);
        tc::fence_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(&M.p_full[vb]);
    }
    if (ok && c.n_tiles > 0) {
        const int last = c.n_tiles - 1;
        ok = __all_sync(0xFFFFFFFFu, tc::mbar_wait(&M.pv_done[last & 1], (last >> 1) & 1));
    }
    if (!ok && (tid & 31) == 0) raise_flag(c.flags, kFlagTimeout);
    tc::fence_after_sync();
    // this chunk's partial for its channel half: (m, l, unnormalised O)
    const bool have = ok && c.n_tiles > 0;
    float *orow = nullptr;
    if (active) {
        const int e = U.entry[slot_layer];
        const EntryDev &E = c.P->entries[e];
        const int part = U.is_window ? E.part_win : c.chunk;
        float *rec = c.P->partials + (((int64_t)e * c.P->batch + c.b) * c.P->max_parts + part) * kPartFloats;
        const bool any = have && l_sum > 0.0f;
        rec[c.half * 16 + head] = any ? m_used : -INFINITY;
        rec[32 + c.half * 16 + head] = any ? l_sum : 0.0f;
        orow = rec + 64 + head * kDim + c.half * 256;
    }
    for (int c0 = 0; c0 < 256; c0 += 32) {
        float o[32];
        if (have) tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
        if (active) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                *reinterpret_cast<float4 *>(orow + c0 + i) =
                    have ? make_float4(o[i], o[i + 1], o[i + 2], o[i + 3]) : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    }
    tc::fence_before_sync();
}

// ---- merge: the last CTA to finish a (layer, sequence, half) combines its partials ----
__device__ __forceinline__ void merge_if_last(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const UnitDev &U = *c.U;
    const AttnParams &P = *c.P;
    const int tid = threadIdx.x;
    tc::named_sync(2, 128);  // every row of this CTA has written its partial
    if (tid < U.n_layers) {
        const int e = U.entry[tid];
        __threadfence();
        const uint32_t old = atomicAdd(P.counters + ((int64_t)e * P.batch + c.b) * 2 + c.half, 1u);
        M.last[tid] = (old + 1 == (uint32_t)P.entries[e].n_parts) ? 1 : 0;
    }
    tc::named_sync(2, 128);
    for (int j = 0; j < U.n_layers; ++j) {
        if (!M.last[j]) continue;
        __threadfence();
        const int e = U.entry[j];
        const EntryDev &E = P.entries[e];
        const float *recs = P.partials + ((int64_t)e * P.batch + c.b) * P.max_parts * kPartFloats;
        const int h = tid >> 3, c0 = c.half * 256 + (tid & 7) * 32;  // head, 32 output channels
        float mx = -INFINITY;
        for (int p = 0; p < E.n_parts; ++p) {
            const float *rp = recs + (int64_t)p * kPartFloats;
            if (__ldcg(rp + 32 + c.half * 16 + h) > 0.0f) mx = fmaxf(mx, __ldcg(rp + c.half * 16 + h));
        }
        float acc[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) acc[i] = 0.0f;
        float ls = 0.0f;
        for (int p = 0; p < E.n_parts; ++p) {
            const float *rp = recs + (int64_t)p * kPartFloats;
            const float lp = __ldcg(rp + 32 + c.half * 16 + h);
            if (!(lp > 0.0f)) continue;
            const float wp = __expf(__ldcg(rp + c.half * 16 + h) - mx);
            ls += wp * lp;
            const float4 *op = reinterpret_cast<const float4 *>(rp + 64 + h * kDim + c0);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const float4 v = __ldcg(op + i);
                acc[4 * i] += wp * v.x;
                acc[4 * i + 1] += wp * v.y;
                acc[4 * i + 2] += wp * v.z;
                acc[4 * i + 3] += wp * v.w;
            }
        }
        const float inv = ls > 0.0f ? 1.0f / ls : 0.0f;
        float4 *out = reinterpret_cast<float4 *>(E.out + ((int64_t)c.b * kHeads + h) * kDim + c0);
#pragma unroll
        for (int i = 0; i < 8; ++i)
            out[i] = make_float4(acc[4 * i] * inv, acc[4 * i + 1] * inv, acc[4 * i + 2] * inv, acc[4 * i + 3] * inv);
        if (c.half == 0 && E.lse && (tid & 7) == 0)
            E.lse[(int64_t)c.b * kHeads + h] = ls > 0.0f ? mx + logf(ls) : -INFINITY;
    }
}

__global__ void __launch_bounds__(kThreads, 1) attn_tc_kernel(const __grid_constant__ AttnParams P, int *flags)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    Ctx c;
    c.P = &P;
    c.M = reinterpret_cast<AttnMisc *>(smem + kOffMisc);
    c.Qs = smem;
    c.Vs = smem + kOffV;
    c.Ps = smem + kOffP;
    c.sidx = reinterpret_cast<int32_t *>(smem + kOffIdx);
    c.flags = flags;
    c.b = blockIdx.y;
    int u = 0;
    while (u + 1 < P.n_units && (int)blockIdx.x >= P.units[u + 1].cta_begin) ++u;
    c.U = &P.units[u];
    const int local = (int)blockIdx.x - c.U->cta_begin;
    c.chunk = local >> 1;
    c.half = local & 1;
    c.L = max(0, __ldg(P.seq_lens + c.b));
    c.W = P.window;
    c.fp8 = c.U->is_window != 0;
    if (c.fp8) {
        c.row0 = 0;
        c.n_rows = c.W;
    } else {
        c.row0 = c.chunk * P.rows_per_chunk;
        c.n_rows = max(0, min(P.rows_per_chunk, P.topk - c.row0));
    }
    c.n_tiles = (c.n_rows + kTile - 1) / kTile;
    AttnMisc &M = *c.M;

    if (tid == 0) {
        tc::mbar_init(&M.q_bar, 1);
        for (int i = 0; i < 2; ++i) {
            tc::mbar_init(&M.full_v[i], kProducers);
            tc::mbar_init(&M.s_full[i], 1);
            tc::mbar_init(&M.s_free[i], 128);
            tc::mbar_init(&M.pv_done[i], 1);
            tc::mbar_init(&M.p_full[i], 128);
        }
        tc::mbar_init_fence();
    }
    if (warp == kMmaWarp) tc::tmem_alloc(&M.tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    c.tmem = M.tmem_slot;

    if (warp >= 4 && warp < kMmaWarp) {
        if (c.fp8) produce<true>(c);
        else produce<false>(c);
    } else if (warp == kMmaWarp) {
        if (lane == 0) issue_mmas(c);
        __syncwarp();
    } else {
        if (c.fp8) softmax_rows<true>(c);
        else softmax_rows<false>(c);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == kMmaWarp) {
        tc::fence_after_sync();
        tc::tmem_dealloc(c.tmem, kTmemCols);
    }
    if (warp < 4) merge_if_last(c);
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

// Rows per chunk of a row unit: 256 (8 tiles), doubled (up to the 2,048 rows
// whose positions a CTA stages) while the grid would exceed 8 waves of one
// CTA per SM (large batches need no split).
int rows_per_chunk(int n_row_units, int n_window_units, int batch, int topk)
{
    int rpc = 256;
    auto ctas = [&](int r) {
        return (int64_t)batch * 2 * ((int64_t)n_row_units * ((topk + r - 1) / r) + n_window_units);
    };
    while (rpc < topk && rpc < kMaxChunkRows && ctas(rpc) > 8 * 148) rpc *= 2;
    return rpc;
}

struct WsLayout {
    size_t counters = 0, q16 = 0, partials = 0, total = 0;
    int rpc = 256, chunks = 0, max_parts = 1;
};

WsLayout ws_layout(const UnitPlan &up, int n_entries, int batch, int topk, int window)
{
    WsLayout w;
    w.rpc = rows_per_chunk((int)up.row_units.size(), (int)up.window_units.size(), batch, topk);
    w.chunks = (topk > 0 && !up.row_units.empty()) ? (topk + w.rpc - 1) / w.rpc : 0;
    w.max_parts = std::max(1, w.chunks + (window > 0 ? 1 : 0));
    auto r256 = [](size_t n) { return (n + 255) & ~(size_t)255; };
    w.counters = r256((size_t)n_entries * batch * 2 * 4);
    w.q16 = r256((size_t)n_entries * batch * kQRowsBytes);
    w.partials = r256((size_t)n_entries * batch * w.max_parts * kPartFloats * 4);
    w.total = w.counters + w.q16 + w.partials;
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
    p.counters = reinterpret_cast<uint32_t *>(ws);
    p.q16 = ws + wl.counters;
    p.partials = reinterpret_cast<float *>(ws + wl.counters + wl.q16);
    for (int e = 0; e < plan.n_entries; ++e) {
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
    // a layer with neither selected rows nor a window attends over nothing
    for (int e = 0; e < plan.n_entries && err == cudaSuccess; ++e)
        if (p.entries[e].n_parts == 0)
            err = cudaMemsetAsync(plan.entries[e].out, 0, (size_t)plan.batch * kHeads * kDim * 4, stream);
    if (err == cudaSuccess) err = cudaMemsetAsync(ws, 0, wl.counters, stream);
    if (err == cudaSuccess && cta > 0) {
        QList qs;
        std::memset(&qs, 0, sizeof(qs));
        for (int e = 0; e < plan.n_entries; ++e) qs.q[e] = plan.entries[e].q;
        pack_q_kernel<<<dim3((unsigned)plan.n_entries, (unsigned)plan.batch), 256, 0, stream>>>(
            qs, const_cast<uint8_t *>(p.q16), plan.batch);
        count_launches(1);
        err = cudaGetLastError();
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
    return err;
}

}  // namespace csa2
