// Multi-query indexer scoring on the tensor cores, and its Top-K.
//
// Several queries of one sequence score the same keys: the tokens of a
// speculative verification (Helmcode "DeepSeek V4.1 Flash" explainer,
// "10 · other changes": DSpark checks several drafted tokens in one pass) or
// a chunk of prefill (the same explainer, "03 · CSA2": the Reuse layers' path
// counts kernels "in prefill" as well as in decode).  With many queries per key
// the score is a real dense contraction, so it goes through tcgen05.mma
// instead of the decode scan's one-thread-per-key integer dot products.
//
// Score (the library's fixed form, include/csa2.h): per query, head h and
// 16-channel block j, t_hj = sq_hj * sk_j * (E2M1 dot product), exact;
// s_h = ((t_h0 + t_h1) + t_h2) + t_h3 in fp32; score = the fma chain of the
// head weights over max(s_h, +0).
//
// Exactness on the tensor cores.  An E2M1 value times an E4M3 scale has at
// most 6 significant bits and lies in [2^-10, 2688], so it is exact in fp16:
// the keys enter the MMA as sk_j * e_k and the queries as sq_hj * e_q.  A
// 16-channel block is one kind::f16 MMA step (K = 16); every partial sum of
// its 16 products is sq_hj sk_j / 4 times an integer of magnitude at most
// 2,304 (the doubled codes are integers up to 12), so the fp32 accumulator
// holds t_hj exactly whatever order the tensor core adds in.
// Each block gets its own accumulator columns and the epilogue adds the four
// blocks in the fixed order, so the scores equal the single-query scan's bit
// for bit.  (A block-scaled FP4 MMA with unit scale factors and a block-
// diagonal query operand, one column per (head, block), would be exact as
// well and would read the codes without the unpack; this kernel folds the
// scales into exact fp16 operands of kind::f16 instead.)
//
// Shape: a CTA takes one sequence, a group of up to 32 queries and every
// gridDim.x-th tile of 128 keys.  Per tile: two 64-key tiles by bulk copy
// (a ring of 8 tiles in flight), unpacked to fp16 core matrices (A: 128 keys x 64
// channels), four MMAs (M = 128 keys, N = 4 heads x 32 queries, K = 16) into
// 512 tensor-memory columns, then the epilogue: thread = key x 8 queries.  The
// epilogue writes each query row's order-preserving keys (0 = not a
// candidate) and adds them to a shared 2,048-bin histogram of 16-bit counts,
// added into the row's global histogram at the end; the cluster radix select
// of the decode path then picks each row's Top-K.
#include <algorithm>
#include <cstring>

#include "internal.h"
#include "scan.cuh"
#include "tc.cuh"

namespace csa2 {
namespace {

constexpr int kMqThreads = 512;                       // 16 warps: the epilogue is latency-bound
constexpr int kMqKeys = 128;                          // keys per tile: the MMA's M
constexpr int kMqQueries = 32;                        // queries per CTA
constexpr int kMqN = kIdxHeads * kMqQueries;          // 128 B rows: (head, query)
constexpr int kMqBlocks = kIdxDim / 16;               // 4 channel blocks
constexpr uint32_t kMqCols = kMqBlocks * kMqN;        // 512 tensor-memory columns: (block, head, query)
constexpr int kMqStage = 2 * kIdxTileBytes;           // one tile of 128 keys as two 64-key tiles
constexpr int kMqRing = 8;                            // tiles in flight per CTA
constexpr int kMqMaxTilesPerCta = 511;                // < 65,536 keys: 16-bit histogram counts

struct MqParams {
    CacheView keys;
    const float *q_idx;       // [B][n_q][4][64]
    const float *w;           // [B][n_q][4]
    const int32_t *seq_lens;  // [B]
    SelectBufs bufs;          // rows b * n_q + i
    int32_t *row_lens;        // [B][n_q] candidates of each query row
    float *out_scores;        // optional [B][n_q][max_len]
    int32_t n_q;
    int32_t max_len;
    int32_t causal;
};

struct __align__(128) MqSmem {
    uint8_t a[kMqKeys * kIdxDim * 2];      // keys as fp16, K-major core matrices
    uint8_t bq[kMqN * kIdxDim * 2];        // queries as fp16, K-major core matrices
    uint8_t stage[kMqRing][kMqStage];      // raw key tiles, a ring
    uint32_t hist[kMqQueries][kHistBins / 2];  // two 16-bit counts per word (bin 2i low)
    float wq[kMqQueries][kIdxHeads];
    int32_t ncand[kMqQueries];
    int32_t tile_ok[kMqRing][2];
    uint64_t bar_ld[kMqRing];
    uint64_t bar_mma;
    uint32_t tmem_slot;
    int32_t ok;
};

static_assert(sizeof(MqSmem) <= 232448, "multi-query scoring shared memory over the 227 KB limit");

// Byte offset of element (row, k) in a K-major operand of 64 fp16 channels:
// core matrices of 8 rows x 8 channels, 128 B apart along K, 1,024 B apart
// along the rows.
__device__ __forceinline__ uint32_t cm64(int row, int k)
{
    return (uint32_t)((row >> 3) * 1024 + (k >> 3) * 128 + (row & 7) * 16 + (k & 7) * 2);
}

// Four loads of 8 consecutive columns of this thread's lane, one wait.
__device__ __forceinline__ void tmem_ld8x4(uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3, float (&v)[4][8])
{
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%32];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%33];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%34];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%24,%25,%26,%27,%28,%29,%30,%31}, [%35];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3)
        : "memory");
#pragma unroll
    for (int j = 0; j < 4; ++j)
#pragma unroll
        for (int i = 0; i < 8; ++i) v[j][i] = __uint_as_float(r[8 * j + i]);
}

__global__ void __launch_bounds__(kMqThreads, 1) mq_score_kernel(const __grid_constant__ MqParams P, int *flags)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    MqSmem &S = *reinterpret_cast<MqSmem *>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int b = blockIdx.y, g0 = blockIdx.z * kMqQueries;
    int L = __ldg(P.seq_lens + b);
    if (L < 0 || L > P.max_len) {
        if (tid == 0 && blockIdx.x == 0 && blockIdx.z == 0) raise_flag(flags, kFlagBounds);
        L = L < 0 ? 0 : P.max_len;
    }
    const int n_tiles = (L + kMqKeys - 1) / kMqKeys;

    if (tid == 0) {
        for (int i = 0; i < kMqRing; ++i) tc::mbar_init(&S.bar_ld[i], 1);
        tc::mbar_init(&S.bar_mma, 1);
        tc::mbar_init_fence();
        S.ok = 1;
    }
    if (tid < kMqQueries) {
        // candidates of query row g0 + tid: its causal prefix, or every position
        const int gq = g0 + tid;
        int nc = 0;
        if (gq < P.n_q) nc = P.causal ? max(0, min(L, L - P.n_q + gq + 1)) : L;
        S.ncand[tid] = nc;
        if (gq < P.n_q && blockIdx.x == 0) P.row_lens[(int64_t)b * P.n_q + gq] = nc;
    }
    if (warp == 0) tc::tmem_alloc(&S.tmem_slot, kMqCols);
    for (int i = tid; i < kMqQueries * kHistBins / 2; i += kMqThreads) (&S.hist[0][0])[i] = 0u;

    // queries: FP4 with an E4M3 scale per (head, block), entered as sq * e2m1
    // (exact in fp16); item = (query, head, block), row n = 32 h + query
    for (int item = tid; item < kMqQueries * kIdxHeads * kMqBlocks; item += kMqThreads) {
        const int qi = item >> 4, h = (item >> 2) & 3, j = item & 3;
        const int gq = g0 + qi;
        uint32_t hv[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
        if (gq < P.n_q) {
            const float4 *src =
                reinterpret_cast<const float4 *>(P.q_idx + (((int64_t)b * P.n_q + gq) * kIdxHeads + h) * kIdxDim + 16 * j);
            float x[16];
#pragma unroll
            for (int v = 0; v < 4; ++v) {
                const float4 f = __ldg(src + v);
                x[4 * v] = f.x;
                x[4 * v + 1] = f.y;
                x[4 * v + 2] = f.z;
                x[4 * v + 3] = f.w;
            }
            float amax = 0.0f;
#pragma unroll
            for (int c = 0; c < 16; ++c) amax = fmaxf(amax, fabsf(x[c]));
            const float sq = e4m3_value(e4m3_code(__fdiv_rn(amax, 6.0f)));
            if (sq != 0.0f) {
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const float lo = sq * scan::e2m1_value(e2m1_code(__fdiv_rn(x[2 * c], sq)));
                    const float hi = sq * scan::e2m1_value(e2m1_code(__fdiv_rn(x[2 * c + 1], sq)));
                    const __half2 h2 = __floats2half2_rn(lo, hi);
                    hv[c] = *reinterpret_cast<const uint32_t *>(&h2);
                }
            }
            if (j == 0) S.wq[qi][h] = __ldg(P.w + ((int64_t)b * P.n_q + gq) * kIdxHeads + h);
        } else if (j == 0) {
            S.wq[qi][h] = 0.0f;
        }
        const int n = h * kMqQueries + qi;
        *reinterpret_cast<uint4 *>(S.bq + cm64(n, 16 * j)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
        *reinterpret_cast<uint4 *>(S.bq + cm64(n, 16 * j + 8)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
    }

    // this CTA's tiles: blockIdx.x, + gridDim.x, ...
    const int my_first = blockIdx.x;
    const int n_my = my_first < n_tiles ? (n_tiles - 1 - my_first) / (int)gridDim.x + 1 : 0;
    auto issue = [&](int k) {  // thread 0: the two 64-key tiles of this CTA's k-th tile
        const int tile = my_first + k * (int)gridDim.x, s = k % kMqRing;
        uint32_t bytes = 0;
        const uint8_t *src[2] = {nullptr, nullptr};
        for (int hf = 0; hf < 2; ++hf) {
            const int64_t p0 = (int64_t)tile * kMqKeys + hf * kIdxTile;
            int ok = 0;
            if (p0 < L) {
                const int64_t slot = slot_of(P.keys, b, p0);
                if (slot >= 0 && slot + kIdxTile <= P.keys.n_slots) {
                    src[hf] = P.keys.data + (slot / kIdxTile) * kIdxTileBytes;
                    bytes += kIdxTileBytes;
                    ok = 1;
                } else {
                    raise_flag(flags, kFlagBounds);
                }
            }
            S.tile_ok[s][hf] = ok;
        }
        tc::mbar_expect_tx(&S.bar_ld[s], bytes);
        for (int hf = 0; hf < 2; ++hf)
            if (src[hf]) tc::bulk_g2s(S.stage[s] + hf * kIdxTileBytes, src[hf], kIdxTileBytes, &S.bar_ld[s]);
    };
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = S.tmem_slot;
    if (tid == 0)
        for (int k = 0; k < min(kMqRing, n_my); ++k) issue(k);

    constexpr uint32_t kIdesc = tc::idesc_f16(kMqKeys, kMqN, false, false);
    const int quad = warp & 3, qo = warp >> 2;  // lanes 32 quad.., queries 8 qo..
    const int r = 32 * quad + lane;             // this thread's key in the tile
    uint32_t ok = 1;
#pragma unroll 1
    for (int k = 0; k < n_my; ++k) {
        const int tile = my_first + k * (int)gridDim.x, s = k % kMqRing;
        // the stage of tile k - 1 was released at the end of the last iteration
        if (tid == 0 && k > 0 && k - 1 + kMqRing < n_my) issue(k - 1 + kMqRing);
        const uint32_t parity = (uint32_t)(k / kMqRing) & 1u;
        if (!tc::mbar_wait(&S.bar_ld[s], parity)) {
            ok = 0;
            tc::mbar_wait(&S.bar_ld[s], parity);  // a last chance for copies in flight
        }
        // keys -> fp16: item = (key, block), eight consecutive keys per block
        // in a quarter warp (conflict-free 16-B stores); sk * e2m1 is exact in fp16
        for (int item = tid; item < kMqKeys * kMqBlocks; item += kMqThreads) {
            const int kr = (item & 7) | ((item >> 5) << 3), j = (item >> 3) & 3, hf = kr >> 6, rr = kr & 63;
            uint32_t hv[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
            if (S.tile_ok[s][hf]) {
                const uint8_t *t = S.stage[s] + hf * kIdxTileBytes;
                const uint2 codes = *reinterpret_cast<const uint2 *>(t + rr * 32 + 8 * j);
                const uint32_t sc = t[kIdxTile * 32 + rr * 4 + j];
                const __half2 sk2 = e4m3x2_half2(sc | (sc << 8));
                const uint32_t cw[2] = {codes.x, codes.y};
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    const uint32_t bits = e2m1x2_half2_bits((cw[c >> 2] >> (8 * (c & 3))) & 0xFFu);
                    const __half2 v = __hmul2(*reinterpret_cast<const __half2 *>(&bits), sk2);
                    hv[c] = *reinterpret_cast<const uint32_t *>(&v);
                }
            }
            *reinterpret_cast<uint4 *>(S.a + cm64(kr, 16 * j)) = make_uint4(hv[0], hv[1], hv[2], hv[3]);
            *reinterpret_cast<uint4 *>(S.a + cm64(kr, 16 * j + 8)) = make_uint4(hv[4], hv[5], hv[6], hv[7]);
        }
        tc::fence_async_smem();
        __syncthreads();
        if (tid == 0) {
            tc::fence_after_sync();
            const uint64_t a0 = tc::sdesc(tc::smem_u32(S.a), 128, 1024);
            const uint64_t b0 = tc::sdesc(tc::smem_u32(S.bq), 128, 1024);
#pragma unroll
            for (int j = 0; j < kMqBlocks; ++j)  // block j: K = 16 channels, 256 B along K per block
                tc::mma_f16(tmem + (uint32_t)(j * kMqN), a0 + 16 * j, b0 + 16 * j, kIdesc, 0u);
            tc::mma_commit(&S.bar_mma);
        }
        if (!tc::mbar_wait(&S.bar_mma, (uint32_t)k & 1u)) {
            ok = 0;
            tc::mbar_wait(&S.bar_mma, (uint32_t)k & 1u);
        }
        tc::fence_after_sync();

        // epilogue: key r of the tile, queries 8 qo .. 8 qo + 7 (warps whose
        // eight query rows are all past n_q have nothing to do)
        if (g0 + 8 * qo < P.n_q) {
            const int64_t pos = (int64_t)tile * kMqKeys + r;
            const bool key_ok = pos < L && S.tile_ok[s][r >> 6];
            float sc[8];
#pragma unroll 1
            for (int h = 0; h < kIdxHeads; ++h) {
                float t[4][8];
                const uint32_t base = tc::taddr(tmem, 32u * quad, (uint32_t)(h * kMqQueries + 8 * qo));
                tmem_ld8x4(base, base + kMqN, base + 2 * kMqN, base + 3 * kMqN, t);
#pragma unroll
                for (int i = 0; i < 8; ++i) {
                    const float sh = __fadd_rn(__fadd_rn(__fadd_rn(t[0][i], t[1][i]), t[2][i]), t[3][i]);
                    const float rl = sh > 0.0f ? sh : 0.0f;
                    const float wh = S.wq[8 * qo + i][h];
                    sc[i] = h == 0 ? __fmul_rn(wh, rl) : __fmaf_rn(wh, rl, sc[i]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const int qi = 8 * qo + i, gq = g0 + qi;
                if (gq >= P.n_q || pos >= S.ncand[qi]) continue;
                const int64_t row = (int64_t)b * P.n_q + gq;
                const float score = sc[i] == 0.0f ? 0.0f : sc[i];
                const uint32_t key = key_ok ? score_key(score) : 0u;
                P.bufs.keys[row * P.bufs.cand_cap + pos] = key;
                if (key) {
                    const uint32_t bin = key >> (32 - kHistBits);
                    atomicAdd(&S.hist[qi][bin >> 1], (bin & 1u) ? 0x10000u : 1u);
                    if (P.out_scores) P.out_scores[row * (int64_t)P.max_len + pos] = score;
                }
            }
        }
        // tensor memory read and the stage consumed before the next tile's MMAs and copy
        tc::fence_before_sync();
        tc::fence_async_smem();
        __syncthreads();
    }
    if (!ok) S.ok = 0;
    tc::fence_before_sync();
    __syncthreads();
    if (warp == 0) {
        tc::fence_after_sync();
        tc::tmem_dealloc(tmem, kMqCols);
    }
    if (tid == 0 && !S.ok) raise_flag(flags, kFlagTimeout);
    // this CTA's counts into each query row's histogram
    for (int i = tid; i < kMqQueries * kHistBins / 2; i += kMqThreads) {
        const int qi = i / (kHistBins / 2), wd = i % (kHistBins / 2);
        const uint32_t c = S.hist[qi][wd];
        if (!c || g0 + qi >= P.n_q) continue;
        uint32_t *gh = P.bufs.hist + ((int64_t)b * P.n_q + g0 + qi) * kHistBins + 2 * wd;
        if (c & 0xFFFFu) atomicAdd(gh, c & 0xFFFFu);
        if (c >> 16) atomicAdd(gh + 1, c >> 16);
    }
}

}  // namespace

size_t index_multi_bytes(int batch, int n_q, int max_seq_len)
{
    const int rows = batch * n_q;
    return select_bytes(rows, max_seq_len, max_seq_len) + (((size_t)rows * 4 + 255) & ~(size_t)255);
}

cudaError_t run_index_multi(const CacheView &keys, const float *q_idx, const float *w, int batch, int n_q,
                            const int32_t *seq_lens, int max_seq_len, int causal, int topk, int32_t *out_idx,
                            float *out_scores, uint8_t *ws, int *flags, cudaStream_t stream)
{
    const int rows = batch * n_q;
    MqParams p;
    memset(&p, 0, sizeof(p));
    p.keys = keys;
    p.q_idx = q_idx;
    p.w = w;
    p.seq_lens = seq_lens;
    p.bufs = carve_select(ws, rows, max_seq_len, max_seq_len);
    p.row_lens = reinterpret_cast<int32_t *>(ws + select_bytes(rows, max_seq_len, max_seq_len));
    p.out_scores = out_scores;
    p.n_q = n_q;
    p.max_len = max_seq_len;
    p.causal = causal;

    cudaError_t e = cudaMemsetAsync(p.bufs.hist, 0, select_hist_bytes(rows), stream);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(MqSmem);
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static int n_sms_of[64] = {};
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!n_sms_of[dev]) {
        e = cudaFuncSetAttribute(mq_score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        n_sms_of[dev] = n > 0 ? n : 1;
    }
    const int n_sms = n_sms_of[dev];
    // one CTA per SM (shared memory and the 512 tensor-memory columns); the
    // tiles of a (sequence, query group) spread over enough CTAs to fill the
    // device, and over at least enough to keep 16-bit histogram counts
    const int n_tiles = (int)ceil_div(max_seq_len, kMqKeys);
    const int groups = (int)ceil_div(n_q, kMqQueries);
    const int64_t units = (int64_t)batch * groups;
    int gx = (int)std::min<int64_t>(n_tiles, std::max<int64_t>(1, ceil_div(n_sms, units)));
    gx = std::max(gx, (int)ceil_div(n_tiles, kMqMaxTilesPerCta));
    log_plan("[csa2] multi-query index: %d x %d x %d CTAs (tiles of 128 keys x 32 queries), %d tiles per sequence",
             gx, batch, groups, n_tiles);
    mq_score_kernel<<<dim3((unsigned)gx, (unsigned)batch, (unsigned)groups), kMqThreads, smem, stream>>>(p, flags);
    count_launches(1);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    if (!out_idx) return cudaSuccess;

    SelectPlan plan;
    memset(&plan, 0, sizeof(plan));
    plan.bufs = p.bufs;
    plan.rows[0].out_idx = out_idx;
    plan.n_row_blocks = 1;
    plan.batch = rows;
    plan.topk = topk;
    plan.pool_out_len = 0;
    plan.max_len = max_seq_len;
    plan.seq_lens = p.row_lens;
    return launch_select(plan, max_seq_len, flags, stream, nullptr);
}

}  // namespace csa2
