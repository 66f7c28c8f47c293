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
//   warps 4-7  producers: cp.async gather of the raw rows of a 32-row tile,
//              exact dequantisation to fp16 (E2M1 x E4M3 and E4M3 are exact
//              in fp16) into the tile's core-matrix layout;
//   warp 8     tensor-memory allocation and tcgen05.mma issue:
//              S[b] = Q V^T (M 128, N 32, K 512) into tensor memory, then
//              O += P V (M 128, N 256, K 32) with O resident in tensor memory;
//   warps 0-3  one thread per query row: S from tensor memory, fp32 online
//              softmax with lazy rescaling of O (only when the running max
//              grows by more than e^8), P to shared memory as fp16.
// V and S are double-buffered, P single; every hand-off is an mbarrier with
// a bounded wait (a wait that gives up raises the timeout flag and the CTA
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
constexpr int kThreads = 288;              // 9 warps
constexpr int kQRowsBytes = kHeads * kDim * 2;  // 16 KB: one layer's 16 query rows in fp16
constexpr int kQBytes = 8 * kQRowsBytes;   // 131,072: 128 query rows
constexpr int kVBytes = kTile * kDim * 2;  // 32,768 per buffer
constexpr int kPBytes = 128 * kTile * 2;   // 8,192
constexpr int kRawHalf = 9216;             // one tile of 32 FP4 rows (288 B each)
constexpr int kRawBytes = 2 * kRawHalf;    // two FP4 tiles, or one tile of 32 FP8 rows (16 KB)
constexpr int kOffV = kQBytes;
constexpr int kOffP = kOffV + 2 * kVBytes;
constexpr int kOffRaw = kOffP + kPBytes;
constexpr int kOffMisc = kOffRaw + kRawBytes;
constexpr int kPartFloats = 64 + kHeads * kDim;  // m[2][16], l[2][16], O[16][512]
constexpr int kMaxUnits = 2 * kMaxAttnEntries;
constexpr float kRescaleGap = 8.0f;        // lazy O rescale threshold (natural log)
constexpr uint32_t kTmemCols = 512;        // S[0] cols 0-31, S[1] cols 32-63, O cols 256-511
constexpr uint32_t kColO = 256;
// Instruction descriptors: QK^T (both operands K-major), PV (B = V read MN-major).
constexpr uint32_t kIdescQK = tc::idesc_f16(128, kTile, false, false);
constexpr uint32_t kIdescPV = tc::idesc_f16(128, 256, false, true);

struct AttnMisc {
    const uint8_t *rowptr[2][kTile];  // per raw buffer
    float rscale[2][kTile];
    int32_t rvalid[2][kTile];
    float mscale[2][kTile];           // per V buffer (read by the softmax warps)
    int32_t mvalid[2][kTile];
    uint64_t q_bar, full_v[2], s_full[2], s_free[2], p_full, pv_done[2];
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
__device__ __forceinline__ uint32_t cm_off512(uint32_t r, uint32_t c)
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

// OR-reduction of a predicate over the 128 threads of named barrier `id`
// (also a barrier); every participant gets the same result.
__device__ __forceinline__ bool bar_any(uint32_t id, bool p)
{
    uint32_t r;
    asm volatile(
        "{\n .reg .pred a, o;\n setp.ne.u32 a, %1, 0;\n bar.red.or.pred o, %2, 128, a;\n selp.u32 %0, 1, 0, o;\n}\n"
        : "=r"(r)
        : "r"((uint32_t)p), "r"(id)
        : "memory");
    return r != 0;
}

// Everything one CTA needs to know about its work item.
struct Ctx {
    const AttnParams *P;
    const UnitDev *U;
    AttnMisc *M;
    uint8_t *Qs, *Vs, *Ps, *Raw;
    int *flags;
    uint32_t tmem;
    int b, L, W, row0, n_rows, n_tiles, chunk, half;
    bool fp8;
};

// ---- producers (warps 4-7): gather + dequantise 32-row tiles -------------------------
__device__ __forceinline__ void produce(const Ctx &c)
{
    AttnMisc &M = *c.M;
    const UnitDev &U = *c.U;
    const int ptid = threadIdx.x - 128;
    // row metadata of tile t into raw buffer rb, then cp.async of its bytes
    auto gather = [&](int t, int rb) {
        if (ptid < kTile) {
            const int v = c.row0 + t * kTile + ptid;
            const uint8_t *ptr = nullptr;
            float sc = 0.0f;
            if (v < c.row0 + c.n_rows) {
                if (!c.fp8) {
                    const int32_t pos = __ldg(U.idx + (int64_t)c.b * c.P->topk + v);
                    if (pos >= 0) {
                        const int64_t slot = pos < c.L ? slot_of(U.cache, c.b, pos) : -1;
                        if (slot < 0) {
                            raise_flag(c.flags, kFlagBounds);
                        } else {
                            ptr = U.cache.data + slot * kKvRow;
                            sc = 1.0f;
                        }
                    }
                } else {
                    const int64_t pos = (int64_t)c.L - c.W + v;
                    if (pos >= 0) {
                        const int64_t slot = slot_of(U.cache, c.b, pos);
                        if (slot < 0) {
                            raise_flag(c.flags, kFlagBounds);
                        } else {
                            ptr = U.cache.data + slot * kDim;
                            sc = __ldg(reinterpret_cast<const float *>(U.cache.data + U.cache.n_slots * kDim) + slot);
                        }
                    }
                }
            }
            M.rowptr[rb][ptid] = ptr;
            M.rscale[rb][ptid] = sc;
            M.rvalid[rb][ptid] = ptr != nullptr;
        }
        tc::named_sync(1, 128);
        if (!c.fp8) {
            uint8_t *raw = c.Raw + rb * kRawHalf;
            for (int k = ptid; k < kTile * (kKvRow / 16); k += 128) {
                const int j = k / (kKvRow / 16), g = k % (kKvRow / 16);
                const uint8_t *src = M.rowptr[rb][j];
                if (src) tc::cp_async16(raw + j * kKvRow + g * 16, src + g * 16);
            }
        } else {
            for (int k = ptid; k < kTile * (kDim / 16); k += 128) {
                const int j = k / (kDim / 16), g = k % (kDim / 16);
                const uint8_t *src = M.rowptr[0][j];
                if (src) tc::cp_async16(c.Raw + j * kDim + g * 16, src + g * 16);
            }
        }
        tc::cp_async_commit();
    };

    if (c.n_tiles > 0) gather(0, 0);
    for (int t = 0; t < c.n_tiles; ++t) {
        const int vb = t & 1;
        const int rb = c.fp8 ? 0 : (t & 1);
        if (!c.fp8) {
            if (t + 1 < c.n_tiles) gather(t + 1, (t + 1) & 1);
            else tc::cp_async_commit();  // keep one group per iteration
            tc::cp_async_wait_one();
        } else {
            if (t > 0) gather(t, 0);
            tc::cp_async_wait_all();
        }
        // V[vb] and its row metadata are free once PV(t-2) has finished
        const bool bad = (t >= 2) && !tc::mbar_wait(&M.pv_done[vb], ((t - 2) >> 1) & 1);
        if (bar_any(1, bad)) {  // also the barrier after every producer's rows have landed
            if (ptid == 0) raise_flag(c.flags, kFlagTimeout);
            break;
        }
        uint8_t *V = c.Vs + vb * kVBytes;
        if (!c.fp8) {
            const uint8_t *raw = c.Raw + rb * kRawHalf;
            for (int k = ptid; k < kTile * 16; k += 128) {
                const int j = k & (kTile - 1), g = k >> 5;  // row j, channels 32g..32g+31
                uint4 o[4];
                if (M.rvalid[rb][j]) {
                    const uint8_t *src = raw + j * kKvRow;
                    const uint4 cw = *reinterpret_cast<const uint4 *>(src + g * 16);
                    const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(src + kKvCodes + 2 * g);
                    const __half2 s0 = __half2half2(__float2half_rn(e4m3_value(sc2 & 0xFFu)));
                    const __half2 s1 = __half2half2(__float2half_rn(e4m3_value(sc2 >> 8)));
                    const uint32_t w[4] = {cw.x, cw.y, cw.z, cw.w};
                    uint32_t h[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const uint32_t bits = e2m1x2_half2_bits((w[i >> 2] >> (8 * (i & 3))) & 0xFFu);
                        const __half2 x = *reinterpret_cast<const __half2 *>(&bits);
                        h[i] = pack_h2(__hmul2(x, i < 8 ? s0 : s1));
                    }
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) o[i] = make_uint4(0u, 0u, 0u, 0u);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) *reinterpret_cast<uint4 *>(V + cm_off512(j, 32 * g + 8 * i)) = o[i];
            }
        } else {
            for (int k = ptid; k < kTile * 32; k += 128) {
                const int j = k & (kTile - 1), g = k >> 5;  // row j, channels 16g..16g+15
                uint4 o0 = make_uint4(0u, 0u, 0u, 0u), o1 = o0;
                if (M.rvalid[0][j]) {
                    const uint4 cw = *reinterpret_cast<const uint4 *>(c.Raw + j * kDim + g * 16);
                    o0 = make_uint4(pack_h2(e4m3x2_half2(cw.x & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.x >> 16)),
                                    pack_h2(e4m3x2_half2(cw.y & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.y >> 16)));
                    o1 = make_uint4(pack_h2(e4m3x2_half2(cw.z & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.z >> 16)),
                                    pack_h2(e4m3x2_half2(cw.w & 0xFFFFu)), pack_h2(e4m3x2_half2(cw.w >> 16)));
                }
                *reinterpret_cast<uint4 *>(V + cm_off512(j, 16 * g)) = o0;
                *reinterpret_cast<uint4 *>(V + cm_off512(j, 16 * g + 8)) = o1;
            }
        }
        if (ptid < kTile) {
            M.mvalid[vb][ptid] = M.rvalid[rb][ptid];
            M.mscale[vb][ptid] = M.rscale[rb][ptid];
        }
        tc::fence_async_smem();
        tc::mbar_arrive(&M.full_v[vb]);
        tc::named_sync(1, 128);  // raw[rb] may be refilled after this
    }
    tc::cp_async_wait_all();
}

// ---- MMA issuer (warp 8, lane 0) -----------------------------------------------------
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
    uint64_t *last_bar = nullptr;
    uint32_t last_par = 0;
    const uint32_t qa = tc::smem_u32(c.Qs), pa = tc::smem_u32(c.Ps);
    auto issue_pv = [&](int t) {
        if (!tc::mbar_wait(&M.p_full, t & 1)) {
            ok = false;
            return;
        }
        tc::fence_after_sync();
        // B = V[t&1] read MN-major: N = this CTA's 256 channels (8-channel groups 128 B apart),
        // K = 32 keys (8-key groups 8,192 B apart)
        const uint32_t vb = tc::smem_u32(c.Vs + (t & 1) * kVBytes) + c.half * (256 / 8) * 128;
        for (int ks = 0; ks < kTile / 16; ++ks)
            tc::mma_f16(c.tmem + kColO, tc::sdesc(pa + ks * 256, 128, 512), tc::sdesc(vb + ks * 2 * 8192, 8192, 128),
                        kIdescPV, (t > 0 || ks > 0) ? 1u : 0u);
        tc::mma_commit(&M.pv_done[t & 1]);
        last_bar = &M.pv_done[t & 1];
        last_par = (t >> 1) & 1;
    };
    for (int t = 0; t < c.n_tiles && ok; ++t) {
        const int vb = t & 1;
        if (!tc::mbar_wait(&M.full_v[vb], (t >> 1) & 1) ||
            (t >= 2 && !tc::mbar_wait(&M.s_free[vb], ((t - 2) >> 1) & 1))) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        const uint32_t va = tc::smem_u32(c.Vs + vb * kVBytes);
        for (int ks = 0; ks < kDim / 16; ++ks)
            tc::mma_f16(c.tmem + 32 * vb, tc::sdesc(qa + ks * 256, 128, 8192), tc::sdesc(va + ks * 256, 128, 8192),
                        kIdescQK, ks > 0 ? 1u : 0u);
        tc::mma_commit(&M.s_full[vb]);
        last_bar = &M.s_full[vb];
        last_par = (t >> 1) & 1;
        if (t >= 1) issue_pv(t - 1);
    }
    if (ok && c.n_tiles > 0) issue_pv(c.n_tiles - 1);
    if (!ok) raise_flag(c.flags, kFlagTimeout);
    // every issued MMA must have finished before the tensor memory is released
    if (last_bar) tc::mbar_wait(last_bar, last_par);
}

// ---- softmax rows (warps 0-3, thread = tensor-memory lane = query row) ----------------
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
        float mt = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTile; ++j) {
            s[j] = M.mvalid[vb][j] ? s[j] * M.mscale[vb][j] : -INFINITY;
            mt = fmaxf(mt, s[j]);
        }
        // PV(t-1) must be done: O is then current and the P buffer free
        w_ok = (t == 0) || tc::mbar_wait(&M.pv_done[(t - 1) & 1], ((t - 1) >> 1) & 1);
        if (!__all_sync(0xFFFFFFFFu, w_ok)) {
            ok = false;
            break;
        }
        tc::fence_after_sync();
        const float m_new = active ? fmaxf(m_used, mt) : m_used;
        // lazy rescale, warp-uniform: every lane of the warp joins the tensor-memory traffic
        if (__any_sync(0xFFFFFFFFu, active && m_new > m_used + kRescaleGap)) {
            const float alpha = (active && m_used != -INFINITY) ? __expf(m_used - m_new) : (active ? 0.0f : 1.0f);
            if (t >= 1) {
#pragma unroll 1
                for (int c0 = 0; c0 < 256; c0 += 32) {
                    float o[32];
                    tc::tmem_ld32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] *= alpha;
                    tc::tmem_st32(tc::taddr(c.tmem, lane_base, kColO + c0), o);
                }
            }
            if (active) {
                l_sum *= alpha;
                m_used = m_new;
            }
        }
        uint32_t ph[kTile / 2];
#pragma unroll
        for (int j = 0; j < kTile; j += 2) {
            float p0 = 0.0f, p1 = 0.0f;
            if (active) {
                p0 = (s[j] == -INFINITY) ? 0.0f : __expf(s[j] - m_used);
                p1 = (s[j + 1] == -INFINITY) ? 0.0f : __expf(s[j + 1] - m_used);
                l_sum += p0 + p1;
            }
            // window rows hold raw E4M3 codes: their per-token scale joins the weight
            ph[j >> 1] = pack_h2(__floats2half2_rn(p0 * M.mscale[vb][j], p1 * M.mscale[vb][j + 1]));
        }
        // P row into its K-major core-matrix layout: 4 groups of 8 keys, 512 B per 8-row group
#pragma unroll
        for (int g = 0; g < 4; ++g)
            *reinterpret_cast<uint4 *>(c.Ps + (tid >> 3) * 512 + g * 128 + (tid & 7) * 16) =
                make_uint4(ph[4 * g], ph[4 * g + 1], ph[4 * g + 2], ph[4 * g + 3]);
        tc::fence_async_smem();
        tc::fence_before_sync();
        tc::mbar_arrive(&M.p_full);
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
    c.Raw = smem + kOffRaw;
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
            tc::mbar_init(&M.full_v[i], 128);
            tc::mbar_init(&M.s_full[i], 1);
            tc::mbar_init(&M.s_free[i], 128);
            tc::mbar_init(&M.pv_done[i], 1);
        }
        tc::mbar_init(&M.p_full, 128);
        tc::mbar_init_fence();
    }
    if (warp == 8) tc::tmem_alloc(&M.tmem_slot, kTmemCols);
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    c.tmem = M.tmem_slot;

    if (warp >= 4 && warp < 8) {
        produce(c);
    } else if (warp == 8) {
        if (lane == 0) issue_mmas(c);
        __syncwarp();
    } else {
        softmax_rows(c);
    }
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 8) {
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

// Rows per chunk of a row unit: 256 (8 tiles), doubled while the grid would
// exceed 8 waves of one CTA per SM (large batches need no split).
int rows_per_chunk(int n_row_units, int n_window_units, int batch, int topk)
{
    int rpc = 256;
    auto ctas = [&](int r) {
        return (int64_t)batch * 2 * ((int64_t)n_row_units * ((topk + r - 1) / r) + n_window_units);
    };
    while (rpc < topk && ctas(rpc) > 8 * 148) rpc *= 2;
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
