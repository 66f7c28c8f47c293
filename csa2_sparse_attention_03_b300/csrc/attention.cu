// Step 3 of the CSA2 decode path: gather of the selected FP4 main-KV rows and
// the FP8 sliding-window rows, dequantisation, and one softmax attention over
// both (Louis Bouchard's KV-cache report, "Share the cache and the search
// work": the selected global entries beside a local 128-token window;
// Helmcode "DeepSeek V4.1 Flash" explainer, "04 · FP4": FP4 global KV, FP8
// window KV).  16 query heads attend over one shared 512-channel row that is
// both key and value.
//
// Work item = (layer entry, sequence, chunk of the row list).  A CTA streams
// its chunk in 64-row tiles:
//   gather   cp.async 16-B copies of the raw rows into a double-buffered
//            staging area (288 B per FP4 row, 512 B per FP8 row), so the next
//            tile's HBM reads overlap this tile's math;
//   dequant  E2M1 x E4M3 -> fp16 and E4M3 -> fp16 are exact (<= 6 and 4
//            significant bits); the FP8 per-token scale is applied to the
//            logits and folded into the softmax weights instead;
//   QK, PV   m16n8k16 fp16 MMAs with fp32 accumulation; fp32 online softmax.
// Chunks of one (entry, sequence) are merged by log-sum-exp in a second kernel.
#include "internal.h"

namespace csa2 {
namespace {

constexpr int kAttnThreads = 128;  // 4 warps
constexpr int kTileRows = 64;
constexpr int kVStride = kDim + 8;    // halves per dequantised row (1,040 B: ldmatrix conflict-free)
constexpr int kPStride = kTileRows + 8;
constexpr int kStageRow = 512;        // staging bytes per row (FP4 rows use 288)
constexpr int kPartFloats = kHeads * kDim + 2 * kHeads;

struct AttnBatch {
    AttnEntry e[kMaxAttnEntries];
};

struct __align__(16) AttnSmem {
    __half V[kTileRows * kVStride];
    __half Q[kHeads * kVStride];
    __half P[kHeads * kPStride];
    uint8_t stage[2][kTileRows * kStageRow];
    const uint8_t *rowptr[2][kTileRows];
    float rowscale[2][kTileRows];
    int32_t rowtype[2][kTileRows];  // 0 invalid, 1 FP4 main row, 2 FP8 window row
    float red[2][4][kHeads];
};

__device__ __forceinline__ void mma_acc(float d[4], const uint32_t a[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};\n"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ void ldsm_x4(uint32_t r[4], const void *p)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t r[4], const void *p)
{
    const uint32_t a = (uint32_t)__cvta_generic_to_shared(p);
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
                 : "r"(a));
}

__device__ __forceinline__ void cp_async16(void *smem, const void *gmem)
{
    const uint32_t s = (uint32_t)__cvta_generic_to_shared(smem);
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;\n" ::"r"(s), "l"(gmem));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;\n" ::); }

// Row list of one (entry, sequence): [0, nsel) selected FP4 rows, then the window.
struct RowList {
    const AttnEntry *e;
    const int32_t *idx;
    int b, L, nsel, window;
};

__device__ __forceinline__ void row_meta(const RowList &rl, int64_t v, const uint8_t *&ptr, int &type,
                                         float &rs, int *flags)
{
    ptr = nullptr;
    type = 0;
    rs = 0.0f;
    if (v < rl.nsel) {
        const int32_t pos = __ldg(rl.idx + v);
        if (pos < 0) return;
        if (pos >= rl.L) {
            raise_flag(flags, kFlagBounds);
            return;
        }
        const int64_t slot = slot_of(rl.e->kv, rl.b, pos);
        if (slot < 0) {
            raise_flag(flags, kFlagBounds);
            return;
        }
        ptr = rl.e->kv.data + slot * kKvRow;
        type = 1;
        rs = 1.0f;
    } else if (v < (int64_t)rl.nsel + rl.window) {
        const int64_t pos = (int64_t)rl.L - rl.window + (v - rl.nsel);
        if (pos < 0) return;
        const int64_t slot = slot_of(rl.e->swa, rl.b, pos);
        if (slot < 0) {
            raise_flag(flags, kFlagBounds);
            return;
        }
        ptr = rl.e->swa.data + slot * kDim;
        type = 2;
        rs = __ldg(reinterpret_cast<const float *>(rl.e->swa.data + rl.e->swa.n_slots * kDim) + slot);
    }
}

__global__ void __launch_bounds__(kAttnThreads) attn_kernel(const __grid_constant__ AttnBatch ab, AttnPlan plan,
                                                             int *flags)
{
    extern __shared__ __align__(16) uint8_t smem_raw[];
    AttnSmem &S = *reinterpret_cast<AttnSmem *>(smem_raw);
    const int chunk = blockIdx.x, b = blockIdx.y, ei = blockIdx.z;
    const AttnEntry &E = ab.e[ei];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;

    RowList rl;
    rl.e = &E;
    rl.b = b;
    rl.L = __ldg(plan.seq_lens + b);
    if (rl.L < 0) rl.L = 0;
    rl.nsel = (E.has_kv && E.idx) ? plan.topk : 0;
    rl.idx = E.idx ? E.idx + (int64_t)b * plan.topk : nullptr;
    rl.window = E.has_swa ? plan.window : 0;
    const int total_rows = rl.nsel + rl.window;
    const int tiles = (total_rows + kTileRows - 1) / kTileRows;
    const int per = (tiles + plan.n_chunks - 1) / plan.n_chunks;
    const int t0 = chunk * per;
    const int t1 = min(tiles, t0 + per);

    // query -> fp16 in shared memory
    const float *q = E.q + (int64_t)b * kHeads * kDim;
    for (int i = tid; i < kHeads * kDim / 4; i += kAttnThreads) {
        const float4 v = __ldg(reinterpret_cast<const float4 *>(q) + i);
        const int h = (4 * i) / kDim, c = (4 * i) % kDim;
        __half2 *dst = reinterpret_cast<__half2 *>(&S.Q[h * kVStride + c]);
        dst[0] = __floats2half2_rn(v.x, v.y);
        dst[1] = __floats2half2_rn(v.z, v.w);
    }

    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.0f, 0.0f};
    float o[16][4];
#pragma unroll
    for (int i = 0; i < 16; ++i) o[i][0] = o[i][1] = o[i][2] = o[i][3] = 0.0f;

    auto issue = [&](int tile, int buf) {
        if (tid < kTileRows) {
            const uint8_t *p;
            int ty;
            float rs;
            row_meta(rl, (int64_t)tile * kTileRows + tid, p, ty, rs, flags);
            S.rowptr[buf][tid] = p;
            S.rowtype[buf][tid] = ty;
            S.rowscale[buf][tid] = rs;
        }
        __syncthreads();
        for (int k = tid; k < kTileRows * 32; k += kAttnThreads) {
            const int j = k >> 5, c = k & 31;
            const int ty = S.rowtype[buf][j];
            if (ty == 0 || (ty == 1 && c >= kKvRow / 16)) continue;
            cp_async16(&S.stage[buf][j * kStageRow + c * 16], S.rowptr[buf][j] + c * 16);
        }
        cp_async_commit();
    };

    if (t0 < t1) issue(t0, 0);
    for (int tile = t0; tile < t1; ++tile) {
        const int cb = (tile - t0) & 1;
        if (tile + 1 < t1) {
            issue(tile + 1, cb ^ 1);
        } else {
            cp_async_commit();  // empty group keeps the wait count uniform
        }
        cp_async_wait1();
        __syncthreads();

        // dequantise the staged tile into V (fp16); invalid rows become zeros
        for (int k = tid; k < kTileRows * 16; k += kAttnThreads) {
            const int j = k >> 4, grp = k & 15;  // 32 channels per task
            const int ty = S.rowtype[cb][j];
            uint4 *dst = reinterpret_cast<uint4 *>(&S.V[j * kVStride + grp * 32]);
            const uint8_t *src = &S.stage[cb][j * kStageRow];
            if (ty == 1) {
                const uint4 raw = *reinterpret_cast<const uint4 *>(src + grp * 16);
                const uint32_t sc2 = *reinterpret_cast<const uint16_t *>(src + kKvCodes + 2 * grp);
                const __half2 s0 = __half2half2(__ushort_as_half(__half_as_ushort(__float2half_rn(e4m3_value(sc2 & 0xFFu)))));
                const __half2 s1 = __half2half2(__ushort_as_half(__half_as_ushort(__float2half_rn(e4m3_value(sc2 >> 8)))));
                const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
                uint32_t h[16];
#pragma unroll
                for (int wd = 0; wd < 4; ++wd) {
#pragma unroll
                    for (int by = 0; by < 4; ++by) {
                        const uint32_t bits = e2m1x2_half2_bits((words[wd] >> (8 * by)) & 0xFFu);
                        __half2 v = *reinterpret_cast<const __half2 *>(&bits);
                        v = __hmul2(v, wd < 2 ? s0 : s1);
                        h[wd * 4 + by] = *reinterpret_cast<uint32_t *>(&v);
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
            } else if (ty == 2) {
                const uint4 r0 = *reinterpret_cast<const uint4 *>(src + grp * 32);
                const uint4 r1 = *reinterpret_cast<const uint4 *>(src + grp * 32 + 16);
                const uint32_t words[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
                uint32_t h[16];
#pragma unroll
                for (int wd = 0; wd < 8; ++wd) {
                    __half2 lo = e4m3x2_half2(words[wd] & 0xFFFFu);
                    __half2 hi = e4m3x2_half2(words[wd] >> 16);
                    h[2 * wd] = *reinterpret_cast<uint32_t *>(&lo);
                    h[2 * wd + 1] = *reinterpret_cast<uint32_t *>(&hi);
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
            } else {
#pragma unroll
                for (int i = 0; i < 4; ++i) dst[i] = make_uint4(0u, 0u, 0u, 0u);
            }
        }
        __syncthreads();

        // S = Q K^T for keys 16w .. 16w+15
        float s[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
#pragma unroll 8
        for (int ks = 0; ks < kDim / 16; ++ks) {
            uint32_t a[4], bq[4];
            ldsm_x4(a, &S.Q[(lane & 15) * kVStride + ks * 16 + 8 * (lane >> 4)]);
            ldsm_x4(bq, &S.V[(16 * warp + (lane & 7) + 8 * (lane >> 4)) * kVStride + ks * 16 + 8 * ((lane >> 3) & 1)]);
            mma_acc(s[0], a, bq[0], bq[1]);
            mma_acc(s[1], a, bq[2], bq[3]);
        }
        // logits: per-row scale (FP8 rows), masking of invalid rows
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 2; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int key = 16 * warp + 8 * nt + 2 * t + (e & 1);
                const float v = S.rowtype[cb][key] ? s[nt][e] * S.rowscale[cb][key] : -INFINITY;
                s[nt][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xFFFFFFFFu, mx[r], 2));
        }
        if (t == 0) {
            S.red[0][warp][g] = mx[0];
            S.red[0][warp][g + 8] = mx[1];
        }
        __syncthreads();
        float alpha[2], mnew[2], sum[2] = {0.0f, 0.0f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = g + 8 * r;
            float tm = fmaxf(fmaxf(S.red[0][0][row], S.red[0][1][row]), fmaxf(S.red[0][2][row], S.red[0][3][row]));
            mnew[r] = fmaxf(m_run[r], tm);
            alpha[r] = (mnew[r] == -INFINITY) ? 1.0f : __expf(m_run[r] - mnew[r]);
        }
#pragma unroll
        for (int nt = 0; nt < 2; ++nt) {
            float pv[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = e >> 1;
                const float p = (s[nt][e] == -INFINITY) ? 0.0f : __expf(s[nt][e] - mnew[r]);
                sum[r] += p;
                const int key = 16 * warp + 8 * nt + 2 * t + (e & 1);
                pv[e] = p * S.rowscale[cb][key];
            }
            *reinterpret_cast<__half2 *>(&S.P[g * kPStride + 16 * warp + 8 * nt + 2 * t]) = __floats2half2_rn(pv[0], pv[1]);
            *reinterpret_cast<__half2 *>(&S.P[(g + 8) * kPStride + 16 * warp + 8 * nt + 2 * t]) = __floats2half2_rn(pv[2], pv[3]);
        }
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            sum[r] += __shfl_xor_sync(0xFFFFFFFFu, sum[r], 1);
            sum[r] += __shfl_xor_sync(0xFFFFFFFFu, sum[r], 2);
        }
        if (t == 0) {
            S.red[1][warp][g] = sum[0];
            S.red[1][warp][g + 8] = sum[1];
        }
        __syncthreads();
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            const int row = g + 8 * r;
            const float ts = (S.red[1][0][row] + S.red[1][1][row]) + (S.red[1][2][row] + S.red[1][3][row]);
            l_run[r] = l_run[r] * alpha[r] + ts;
            m_run[r] = mnew[r];
        }
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            o[nt][0] *= alpha[0];
            o[nt][1] *= alpha[0];
            o[nt][2] *= alpha[1];
            o[nt][3] *= alpha[1];
        }
        // O += P V for channels 128w .. 128w+127
#pragma unroll
        for (int kk = 0; kk < kTileRows / 16; ++kk) {
            uint32_t a[4];
            ldsm_x4(a, &S.P[(lane & 15) * kPStride + kk * 16 + 8 * (lane >> 4)]);
#pragma unroll
            for (int np = 0; np < 8; ++np) {
                uint32_t bv[4];
                ldsm_x4_t(bv, &S.V[(kk * 16 + (lane & 7) + 8 * ((lane >> 3) & 1)) * kVStride + 128 * warp + 16 * np + 8 * (lane >> 4)]);
                mma_acc(o[2 * np], a, bv[0], bv[1]);
                mma_acc(o[2 * np + 1], a, bv[2], bv[3]);
            }
        }
        __syncthreads();
    }

    // epilogue
    if (plan.n_chunks == 1) {
        float *out = E.out + (int64_t)b * kHeads * kDim;
        const float inv0 = l_run[0] > 0.0f ? 1.0f / l_run[0] : 0.0f;
        const float inv1 = l_run[1] > 0.0f ? 1.0f / l_run[1] : 0.0f;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = 128 * warp + 8 * nt + 2 * t;
            *reinterpret_cast<float2 *>(out + g * kDim + c) = make_float2(o[nt][0] * inv0, o[nt][1] * inv0);
            *reinterpret_cast<float2 *>(out + (g + 8) * kDim + c) = make_float2(o[nt][2] * inv1, o[nt][3] * inv1);
        }
        if (E.lse && warp == 0 && t == 0) {
            E.lse[(int64_t)b * kHeads + g] = l_run[0] > 0.0f ? m_run[0] + logf(l_run[0]) : -INFINITY;
            E.lse[(int64_t)b * kHeads + g + 8] = l_run[1] > 0.0f ? m_run[1] + logf(l_run[1]) : -INFINITY;
        }
    } else {
        float *part = plan.partials + (((int64_t)ei * plan.batch + b) * plan.n_chunks + chunk) * kPartFloats;
#pragma unroll
        for (int nt = 0; nt < 16; ++nt) {
            const int c = 128 * warp + 8 * nt + 2 * t;
            *reinterpret_cast<float2 *>(part + g * kDim + c) = make_float2(o[nt][0], o[nt][1]);
            *reinterpret_cast<float2 *>(part + (g + 8) * kDim + c) = make_float2(o[nt][2], o[nt][3]);
        }
        if (warp == 0 && t == 0) {
            part[kHeads * kDim + g] = m_run[0];
            part[kHeads * kDim + g + 8] = m_run[1];
            part[kHeads * kDim + kHeads + g] = l_run[0];
            part[kHeads * kDim + kHeads + g + 8] = l_run[1];
        }
    }
}

// Log-sum-exp merge of the chunk partials of one (entry, sequence).
__global__ void __launch_bounds__(256) merge_kernel(const __grid_constant__ AttnBatch ab, AttnPlan plan)
{
    const int ei = blockIdx.x, b = blockIdx.y;
    const AttnEntry &E = ab.e[ei];
    const float *part = plan.partials + ((int64_t)ei * plan.batch + b) * plan.n_chunks * kPartFloats;
    __shared__ float wsm[64][kHeads];
    __shared__ float inv_l[kHeads];
    const int tid = threadIdx.x;
    if (tid < kHeads) {
        float M = -INFINITY;
        for (int c = 0; c < plan.n_chunks; ++c) M = fmaxf(M, part[c * kPartFloats + kHeads * kDim + tid]);
        float l = 0.0f;
        for (int c = 0; c < plan.n_chunks; ++c) {
            const float mc = part[c * kPartFloats + kHeads * kDim + tid];
            const float wc = (mc == -INFINITY) ? 0.0f : __expf(mc - M);
            wsm[c][tid] = wc;
            l += wc * part[c * kPartFloats + kHeads * kDim + kHeads + tid];
        }
        inv_l[tid] = l > 0.0f ? 1.0f / l : 0.0f;
        if (E.lse) E.lse[(int64_t)b * kHeads + tid] = l > 0.0f ? M + logf(l) : -INFINITY;
    }
    __syncthreads();
    float *out = E.out + (int64_t)b * kHeads * kDim;
    for (int i = tid; i < kHeads * kDim / 4; i += blockDim.x) {
        const int h = (4 * i) / kDim;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int c = 0; c < plan.n_chunks; ++c) {
            const float wc = wsm[c][h];
            if (wc == 0.0f) continue;
            const float4 v = reinterpret_cast<const float4 *>(part + c * kPartFloats)[i];
            acc.x += wc * v.x;
            acc.y += wc * v.y;
            acc.z += wc * v.z;
            acc.w += wc * v.w;
        }
        const float il = inv_l[h];
        reinterpret_cast<float4 *>(out)[i] = make_float4(acc.x * il, acc.y * il, acc.z * il, acc.w * il);
    }
}

}  // namespace

int attn_chunks(int n_entries, int batch, int topk, int window)
{
    const int rows = topk + window;
    const int tiles = (rows + kTileRows - 1) / kTileRows;
    const int items = n_entries * batch;
    // aim for about two waves of 148 SMs, at least 4 tiles per chunk, at most 64 chunks
    int chunks = (2 * 148 + items - 1) / items;
    const int max_by_tiles = tiles / 4 > 0 ? tiles / 4 : 1;
    if (chunks > max_by_tiles) chunks = max_by_tiles;
    if (chunks > 64) chunks = 64;
    if (chunks < 1) chunks = 1;
    return chunks;
}

size_t attn_partial_bytes(int n_entries, int batch, int n_chunks)
{
    if (n_chunks <= 1) return 0;
    return (size_t)n_entries * batch * n_chunks * kPartFloats * sizeof(float);
}

cudaError_t launch_attention(const AttnPlan &plan, int *flags, cudaStream_t stream, cudaEvent_t mid_event)
{
    const size_t smem = sizeof(AttnSmem);
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(attn_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    for (int first = 0; first < plan.n_entries; first += kMaxAttnEntries) {
        AttnBatch ab;
        const int n = (plan.n_entries - first < kMaxAttnEntries) ? plan.n_entries - first : kMaxAttnEntries;
        for (int i = 0; i < n; ++i) ab.e[i] = plan.entries[first + i];
        AttnPlan p = plan;
        p.n_entries = n;
        if (plan.partials)
            p.partials = plan.partials + (size_t)first * plan.batch * plan.n_chunks * kPartFloats;
        dim3 grid((unsigned)plan.n_chunks, (unsigned)plan.batch, (unsigned)n);
        attn_kernel<<<grid, kAttnThreads, smem, stream>>>(ab, p, flags);
        count_launches(1);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        if (mid_event && first + n >= plan.n_entries) {
            e = record_event(mid_event, stream);
            if (e != cudaSuccess) return e;
        }
        if (plan.n_chunks > 1) {
            merge_kernel<<<dim3((unsigned)n, (unsigned)plan.batch), 256, 0, stream>>>(ab, p);
            count_launches(1);
            e = cudaGetLastError();
            if (e != cudaSuccess) return e;
        }
    }
    return cudaSuccess;
}

}  // namespace csa2
