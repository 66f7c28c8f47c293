// Indexer scoring shared by the scan kernels (the Helmcode "DeepSeek V4.1
// Flash" explainer, "03 · CSA2": Full and Reindex layers score positions with
// their own indexer query; Louis Bouchard's KV-cache report, "What actually
// changed over V4 Flash": FP4 indexer keys).  Score form and rounding points
// are this library's stated choice (include/csa2.h):
//   q quantised by the FP4 rule; per head h and 16-channel block j
//   t_hj = sq_hj * sk_j * P_hj (the E2M1 block dot product, exact);
//   s_h = ((t_h0 + t_h1) + t_h2) + t_h3 in fp32;  r_h = max(s_h, +0);
//   score = fma(w3, r3, fma(w2, r2, fma(w1, r1, w0 * r0))); 0 -> +0.
// A warp scores 16 keys per MMA group: the block dot products of up to two
// queries x 4 heads (the 8 columns of an m16n8k16 fp16 MMA) are exact --
// E2M1 codes and the block-scaled query (scale x code, <= 6 significant
// bits) are exact in fp16 and every partial sum is a small multiple of the
// block's quantum -- and the epilogue applies the key scales and head weights
// in the fixed order on the CUDA cores.
#pragma once

#include "common.cuh"

namespace csa2 {
namespace scan {

__device__ __forceinline__ void mma16816(float d[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                         uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%10,%11,%12,%13};\n"
        : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(0.0f), "f"(0.0f), "f"(0.0f),
          "f"(0.0f));
}

// E2M1 value of a 4-bit code (sign bit 3).
__device__ __forceinline__ float e2m1_value(uint32_t code)
{
    const uint32_t m = code & 7u;
    const float mag = (m < 2u) ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * (1.0f + 0.5f * (float)(m & 1u));
    return (code & 8u) ? -mag : mag;
}

// Codes (the 4 words this thread needs) and the 4 block scales of one key.
struct KeyLoad {
    uint32_t w[4];
    uint32_t sc;
    bool ok;
};

// thread t of a quad uses bytes 8j+2t, 8j+2t+1 of block j: word 2j + t/2, half t%2
__device__ __forceinline__ KeyLoad key_from_tile(const uint8_t *tile, int rr, int t)
{
    KeyLoad k;
    const uint32_t *codes = reinterpret_cast<const uint32_t *>(tile + rr * 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) k.w[j] = codes[2 * j + (t >> 1)];
    k.sc = *reinterpret_cast<const uint32_t *>(tile + kIdxTile * 32 + rr * 4);
    k.ok = true;
    return k;
}

__device__ __forceinline__ KeyLoad key_from_global(const CacheView &keys, int b, int64_t pos, int t, int *flags)
{
    KeyLoad k;
    k.ok = false;
    k.sc = 0;
    k.w[0] = k.w[1] = k.w[2] = k.w[3] = 0;
    if (pos < 0) return k;
    const int64_t slot = slot_of(keys, b, pos);
    if (slot < 0) {
        raise_flag(flags, kFlagBounds);
        return k;
    }
    const uint8_t *tile = keys.data + (slot / kIdxTile) * kIdxTileBytes;
    const int rr = (int)(slot % kIdxTile);
    const uint32_t *codes = reinterpret_cast<const uint32_t *>(tile + rr * 32);
#pragma unroll
    for (int j = 0; j < 4; ++j) k.w[j] = __ldcg(codes + 2 * j + (t >> 1));
    k.sc = __ldcg(reinterpret_cast<const uint32_t *>(tile + kIdxTile * 32 + rr * 4));
    k.ok = true;
    return k;
}


// Query preparation by 256 threads (8 per 16-channel block of 2 queries x 4
// heads): the FP4 rule's block scale and codes, pre-scaled (scale x E2M1
// value, exact in fp16) into qpre[query][head][channel], and the head
// weights into wq[query][head].  Queries qi >= n_q get zeros.
__device__ __forceinline__ void prep_queries(int tid, int n_q, const float *const q_idx[2], const float *const w[2],
                                             int b, __half (*qpre)[kIdxHeads][kIdxDim], float (*wq)[kIdxHeads])
{
    const int bi = tid >> 3, pr = tid & 7;
    const int qi = bi >> 4, h = (bi >> 2) & 3, blk = bi & 3;
    const bool have = qi < n_q;
    float v0 = 0.0f, v1 = 0.0f;
    if (have) {
        const float *src = q_idx[qi] + ((int64_t)b * kIdxHeads + h) * kIdxDim + blk * 16 + 2 * pr;
        v0 = __ldcg(src);
        v1 = __ldcg(src + 1);
    }
    float amax = fmaxf(fabsf(v0), fabsf(v1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, 4));
    const float sq = have ? e4m3_value(e4m3_code(__fdiv_rn(amax, 6.0f))) : 0.0f;
    const float e0 = (sq != 0.0f) ? e2m1_value(e2m1_code(__fdiv_rn(v0, sq))) : 0.0f;
    const float e1 = (sq != 0.0f) ? e2m1_value(e2m1_code(__fdiv_rn(v1, sq))) : 0.0f;
    qpre[qi][h][blk * 16 + 2 * pr] = __float2half_rn(e0 * sq);
    qpre[qi][h][blk * 16 + 2 * pr + 1] = __float2half_rn(e1 * sq);
    if (blk == 0 && pr == 0) wq[qi][h] = have ? __ldcg(w[qi] + (int64_t)b * kIdxHeads + h) : 0.0f;
}

// B fragments of the m16n8k16 MMA for block j: column g = (query g/4, head
// g%4); k-slot 2t+e <-> channel 4t+e, k-slot 2t+8+e <-> channel 4t+2+e (a
// permutation of the block applied to both operands).
__device__ __forceinline__ void build_bfrag(const __half (*qpre)[kIdxHeads][kIdxDim], int g, int t,
                                            uint32_t bfrag[4][2])
{
    const int qi = g >> 2, h = g & 3;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const __half *q = &qpre[qi][h][j * 16 + 4 * t];
        bfrag[j][0] = (uint32_t)__half_as_ushort(q[0]) | ((uint32_t)__half_as_ushort(q[1]) << 16);
        bfrag[j][1] = (uint32_t)__half_as_ushort(q[2]) | ((uint32_t)__half_as_ushort(q[3]) << 16);
    }
}

// Scores of four keys (two 16-key groups: k[0], k[1] in group A rows g and
// g+8, k[2], k[3] in group B) for this thread's query (t >> 1); every thread
// of the quad gets the same four scores for its query.
__device__ __forceinline__ void score4(const KeyLoad k[4], const uint32_t bfrag[4][2], const float *sk_lut,
                                       float w0, float w1, float w2, float w3, int t, float sc[4])
{
    float d[2][4][4];
#pragma unroll
    for (int h2 = 0; h2 < 2; ++h2)
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t uA = (k[2 * h2].w[j] >> (16 * (t & 1))) & 0xFFFFu;
            const uint32_t uB = (k[2 * h2 + 1].w[j] >> (16 * (t & 1))) & 0xFFFFu;
            mma16816(d[h2][j], e2m1x2_half2_bits(uA & 0xFFu), e2m1x2_half2_bits(uB & 0xFFu),
                     e2m1x2_half2_bits(uA >> 8), e2m1x2_half2_bits(uB >> 8), bfrag[j][0], bfrag[j][1]);
        }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        // s = t0 + t1 + t2 + t3 in order; t_j = sk_j * (sq_j * P_j) is exact, so fma == add
        const float *dd = &d[i >> 1][0][0];
        const int e0 = 2 * (i & 1);  // accumulator pair of this key
        float s0 = sk_lut[k[i].sc & 0xFFu] * dd[e0];
        float s1 = sk_lut[k[i].sc & 0xFFu] * dd[e0 + 1];
#pragma unroll
        for (int j = 1; j < 4; ++j) {
            const float skj = sk_lut[(k[i].sc >> (8 * j)) & 0xFFu];
            s0 = __fmaf_rn(skj, dd[4 * j + e0], s0);
            s1 = __fmaf_rn(skj, dd[4 * j + e0 + 1], s1);
        }
        const float r0 = s0 > 0.0f ? s0 : 0.0f, r1 = s1 > 0.0f ? s1 : 0.0f;
        // heads 0,1 live on even t, heads 2,3 on odd t: chain w0*r0 -> +w1 r1 -> +w2 r2 -> +w3 r3
        float acc = __fmaf_rn(w1, r1, __fmul_rn(w0, r0));
        acc = __shfl_xor_sync(0xFFFFFFFFu, acc, 1);
        const float v = __fmaf_rn(w3, r1, __fmaf_rn(w2, r0, acc));
        sc[i] = (v == 0.0f) ? 0.0f : v;
    }
}

}  // namespace scan
}  // namespace csa2
