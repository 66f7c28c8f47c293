// Indexer scoring shared by the scan kernels (the Helmcode "DeepSeek V4.1
// Flash" explainer, "03 · CSA2": Full and Reindex layers score positions with
// their own indexer query; Louis Bouchard's KV-cache report, "What actually
// changed over V4 Flash": FP4 indexer keys).  Score form and rounding points
// are this library's stated choice (include/csa2.h):
//   q quantised by the FP4 rule; per head h and 16-channel block j
//   t_hj = sq_hj * sk_j * P_hj (the E2M1 block dot product, exact);
//   s_h = ((t_h0 + t_h1) + t_h2) + t_h3 in fp32;  r_h = max(s_h, +0);
//   score = fma(w3, r3, fma(w2, r2, fma(w1, r1, w0 * r0))); 0 -> +0.
// One thread scores a whole key for every query of its scan: the E2M1 codes
// doubled are small integers, so the block dot products are exact integer
// sums (dp4a), and the epilogue applies the scales and head weights in the
// fixed order on the CUDA cores.
#pragma once

#include "common.cuh"

namespace csa2 {
namespace scan {

// E2M1 value of a 4-bit code (sign bit 3).
__device__ __forceinline__ float e2m1_value(uint32_t code)
{
    const uint32_t m = code & 7u;
    const float mag = (m < 2u) ? 0.5f * (float)m : (float)(1u << ((m >> 1) - 1u)) * (1.0f + 0.5f * (float)(m & 1u));
    return (code & 8u) ? -mag : mag;
}

// ---- integer scoring: one thread scores whole keys ------------------------------
// Every E2M1 code doubled is an integer in [-12, 12], so each 16-channel block
// product P_hb = sum (2 e_q)(2 e_k) is an exact int32 from four dp4a steps;
// t_hb = (sq_hb * sk_b) * P_hb * 0.25 is exact in fp32 (at most 20
// significant bits), and the epilogue adds and weighs in the stated order.

// The queries of one scan in shared memory: doubled codes as int8 x 4
// (channels 4w..4w+3 in word w of a head), block scales, head weights.
struct __align__(16) QuerySet {
    uint32_t qi8[2][kIdxHeads][kIdxDim / 4];
    float sq[2][kIdxHeads][kIdxDim / 16];
    float w[2][kIdxHeads];
};

// 256 threads: thread = (query, head, block, pair of channels).
__device__ __forceinline__ void prep_query_set(int tid, int n_q, const float *const q_idx[2], const float *const w[2],
                                               int b, QuerySet &Q)
{
    const int qi = tid >> 7, h = (tid >> 5) & 3, blk = (tid >> 3) & 3, pr = tid & 7;
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
    const int d0 = (sq != 0.0f) ? (int)(2.0f * e2m1_value(e2m1_code(__fdiv_rn(v0, sq)))) : 0;
    const int d1 = (sq != 0.0f) ? (int)(2.0f * e2m1_value(e2m1_code(__fdiv_rn(v1, sq)))) : 0;
    // two channels per thread; the even thread of a pair assembles the word
    const uint32_t half = ((uint32_t)(d0 & 0xFF)) | ((uint32_t)(d1 & 0xFF) << 8);
    const uint32_t other = __shfl_down_sync(0xFFFFFFFFu, half, 1);
    if ((pr & 1) == 0) Q.qi8[qi][h][blk * 4 + (pr >> 1)] = half | (other << 16);
    if (pr == 0) Q.sq[qi][h][blk] = sq;
    if (blk == 0 && pr == 0) Q.w[qi][h] = have ? __ldcg(w[qi] + (int64_t)b * kIdxHeads + h) : 0.0f;
}

// Eight doubled E2M1 codes (one 32-bit word of nibbles) -> two int8 x 4 words.
__device__ __forceinline__ void e2m1_word_to_i8(uint32_t wd, uint32_t &lo4, uint32_t &hi4)
{
    // the 3-bit magnitude codes pick bytes from the tables of +v and -v,
    // v in {0,1,2,3,4,6,8,12}; the sign bit of each code picks the table
    constexpr uint32_t kPosLo = 0x03020100u, kPosHi = 0x0C080604u;
    constexpr uint32_t kNegLo = 0xFDFEFF00u, kNegHi = 0xF4F8FAFCu;
    const uint32_t sel0 = wd & 0x7777u, sel1 = (wd >> 16) & 0x7777u;
    const uint32_t s0 = __byte_perm(0x0000FF00u, 0u, (wd >> 3) & 0x1111u);  // 0xFF per negative code
    const uint32_t s1 = __byte_perm(0x0000FF00u, 0u, (wd >> 19) & 0x1111u);
    lo4 = (__byte_perm(kPosLo, kPosHi, sel0) & ~s0) | (__byte_perm(kNegLo, kNegHi, sel0) & s0);
    hi4 = (__byte_perm(kPosLo, kPosHi, sel1) & ~s1) | (__byte_perm(kNegLo, kNegHi, sel1) & s1);
}

// Score of one key (sixteen int8 x 4 words, four scale values) against one
// query's words qi8[h][w], block scales sq[h][j] and head weights w[h]; the
// arrays may live in shared memory or in registers.
template <typename QW, typename QS, typename QH>
__device__ __forceinline__ float score_words(const uint32_t (&kw)[16], const float (&sk)[4], const QW &qi8,
                                             const QS &sq, const QH &wt)
{
    float score = 0.0f;
#pragma unroll
    for (int h = 0; h < kIdxHeads; ++h) {
        float s = 0.0f;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            int P = 0;
#pragma unroll
            for (int w = 0; w < 4; ++w) P = __dp4a((int)kw[4 * blk + w], (int)qi8[h][4 * blk + w], P);
            const float t = __fmul_rn(__fmul_rn(__fmul_rn(sq[h][blk], sk[blk]), (float)P), 0.25f);
            s = blk == 0 ? t : __fadd_rn(s, t);
        }
        const float r = s > 0.0f ? s : 0.0f;
        score = h == 0 ? __fmul_rn(wt[0], r) : __fmaf_rn(wt[h], r, score);
    }
    return score == 0.0f ? 0.0f : score;
}

// Score of one key for query qi of a QuerySet in shared memory.
__device__ __forceinline__ float score_key_int(const uint32_t (&kw)[16], const float (&sk)[4], const QuerySet &Q,
                                               int qi)
{
    return score_words(kw, sk, Q.qi8[qi], Q.sq[qi], Q.w[qi]);
}

// Scores of two keys against query qi of a QuerySet in shared memory, with
// the same rounding points as score_words.  The heads run in a rolled loop
// and share their query loads between the two keys: the code stays small (a
// scan runs it once per launch, from a cold instruction cache) and the two
// keys' dependent chains interleave.
__device__ __forceinline__ void score_pair(const uint32_t (&ka)[16], const float (&sa)[4], const uint32_t (&kb)[16],
                                           const float (&sb)[4], const QuerySet &Q, int qi, float &out_a, float &out_b)
{
    float score_a = 0.0f, score_b = 0.0f;
#pragma unroll 1
    for (int h = 0; h < kIdxHeads; ++h) {
        const uint4 *qw = reinterpret_cast<const uint4 *>(Q.qi8[qi][h]);
        const float4 sq4 = *reinterpret_cast<const float4 *>(Q.sq[qi][h]);
        const float sq[4] = {sq4.x, sq4.y, sq4.z, sq4.w};
        float s_a = 0.0f, s_b = 0.0f;
#pragma unroll
        for (int blk = 0; blk < 4; ++blk) {
            const uint4 q4 = qw[blk];
            int pa = __dp4a((int)ka[4 * blk], (int)q4.x, 0), pb = __dp4a((int)kb[4 * blk], (int)q4.x, 0);
            pa = __dp4a((int)ka[4 * blk + 1], (int)q4.y, pa);
            pb = __dp4a((int)kb[4 * blk + 1], (int)q4.y, pb);
            pa = __dp4a((int)ka[4 * blk + 2], (int)q4.z, pa);
            pb = __dp4a((int)kb[4 * blk + 2], (int)q4.z, pb);
            pa = __dp4a((int)ka[4 * blk + 3], (int)q4.w, pa);
            pb = __dp4a((int)kb[4 * blk + 3], (int)q4.w, pb);
            const float ta = __fmul_rn(__fmul_rn(__fmul_rn(sq[blk], sa[blk]), (float)pa), 0.25f);
            const float tb = __fmul_rn(__fmul_rn(__fmul_rn(sq[blk], sb[blk]), (float)pb), 0.25f);
            s_a = blk == 0 ? ta : __fadd_rn(s_a, ta);
            s_b = blk == 0 ? tb : __fadd_rn(s_b, tb);
        }
        // fma(w, r, +0) rounds w r once, as the first head's product does
        const float wh = Q.w[qi][h];
        score_a = __fmaf_rn(wh, s_a > 0.0f ? s_a : 0.0f, score_a);
        score_b = __fmaf_rn(wh, s_b > 0.0f ? s_b : 0.0f, score_b);
    }
    out_a = score_a == 0.0f ? 0.0f : score_a;
    out_b = score_b == 0.0f ? 0.0f : score_b;
}

// The 64 channels of a key as int8 x 4 words, and its four block scales.
__device__ __forceinline__ void unpack_key(const uint4 c0, const uint4 c1, uint32_t scales, const float *sk_lut,
                                           uint32_t (&kw)[16], float (&sk)[4])
{
    const uint32_t wd[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
#pragma unroll
    for (int j = 0; j < 8; ++j) e2m1_word_to_i8(wd[j], kw[2 * j], kw[2 * j + 1]);
#pragma unroll
    for (int j = 0; j < 4; ++j) sk[j] = sk_lut[(scales >> (8 * j)) & 0xFFu];
}

}  // namespace scan
}  // namespace csa2
