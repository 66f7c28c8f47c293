// Internal definitions shared by the CSA2 CUDA kernels (sm_103a).
//
// Formats follow the Helmcode "DeepSeek V4.1 Flash" explainer, section
// "04 · FP4" (main KV: E2M1 values with one E4M3 scale per 16 channels, no
// extra global scale; SWA KV in FP8) and Louis Bouchard's KV-cache report,
// "What actually changed over V4 Flash" (FP4 indexer keys).  Byte layouts are
// this library's choice and are documented in include/csa2.h.
#pragma once

#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "csa2.h"

namespace csa2 {

constexpr int kHeads = 16;      // attention heads (MQA over one shared row)
constexpr int kDim = 512;       // main KV / query channels
constexpr int kIdxHeads = 4;    // indexer heads
constexpr int kIdxDim = 64;     // indexer channels
constexpr int kKvRow = 288;     // bytes per FP4 main-KV row
constexpr int kKvCodes = 256;   // code bytes in a main-KV row
constexpr int kIdxTile = 64;    // tokens per indexer-key tile
constexpr int kIdxTileBytes = 2304;
constexpr int kHistBits = 11;   // first Top-K radix digit: the key's top 11 bits
constexpr int kHistBins = 1 << kHistBits;

// Device flag bits, OR-ed into one word read by csa2_check_device().
constexpr int kFlagBounds = 1;    // an index / page / slot out of range was skipped
constexpr int kFlagTimeout = 2;   // a bounded wait gave up

struct CacheView {
    uint8_t *data;
    int32_t format;
    int32_t page_size;
    int64_t n_slots;
    int64_t seq_stride;
    const int32_t *page_table;
    int32_t max_pages;
};

inline CacheView view_of(const csa2_cache &c)
{
    CacheView v;
    v.data = static_cast<uint8_t *>(c.data);
    v.format = c.format;
    v.page_size = c.page_size;
    v.n_slots = c.n_slots;
    v.seq_stride = c.seq_stride;
    v.page_table = c.page_table;
    v.max_pages = c.max_pages;
    return v;
}

// Physical slot of logical (sequence b, position pos); -1 if unmapped or out
// of the cache.
__device__ __forceinline__ int64_t slot_of(const CacheView &c, int b, int64_t pos)
{
    int64_t s;
    if (c.page_size == 0) {
        s = (c.format == CSA2_FMT_FP8_SWA) ? (int64_t)b * c.seq_stride + pos % c.seq_stride
                                           : (int64_t)b * c.seq_stride + pos;
    } else {
        int64_t pg = pos / c.page_size;
        if (pg >= c.max_pages) return -1;
        int32_t phys = __ldg(c.page_table + (int64_t)b * c.max_pages + pg);
        if (phys < 0) return -1;
        s = (int64_t)phys * c.page_size + pos % c.page_size;
    }
    return (s >= 0 && s < c.n_slots) ? s : -1;
}

__device__ __forceinline__ void raise_flag(int *flags, int bit)
{
    if (flags) atomicOr(flags, bit);
}

// ---- codecs ---------------------------------------------------------------

// E2M1 code of v: nearest of {0,.5,1,1.5,2,3,4,6}, midpoints to the even
// code, saturating at 6; sign bit from v.  The thresholds are the grid's
// midpoints; ">" at a midpoint whose lower neighbour has the even code,
// ">=" where the upper neighbour has it.
__device__ __forceinline__ uint32_t e2m1_code(float v)
{
    float a = fabsf(v);
    uint32_t c = (uint32_t)(a > 0.25f) + (uint32_t)(a >= 0.75f) + (uint32_t)(a > 1.25f) +
                 (uint32_t)(a >= 1.75f) + (uint32_t)(a > 2.5f) + (uint32_t)(a >= 3.5f) +
                 (uint32_t)(a > 5.0f);
    return c | ((__float_as_uint(v) >> 28) & 8u);
}

// E4M3 code of v: the hardware's round-to-nearest-even, saturating
// conversion applied to |v|, with the sign bit taken from v.
__device__ __forceinline__ uint32_t e4m3_code(float v)
{
    uint32_t mag = (uint32_t)__nv_cvt_float_to_fp8(fabsf(v), __NV_SATFINITE, __NV_E4M3) & 0x7Fu;
    return mag | ((__float_as_uint(v) >> 24) & 0x80u);
}

__device__ __forceinline__ float e4m3_value(uint32_t code)
{
    __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(code & 0xFFu), __NV_E4M3);
    return __half2float(__half(h));
}

// Two E4M3 codes (low byte first) -> half2 (exact).
__device__ __forceinline__ __half2 e4m3x2_half2(uint32_t two_codes)
{
    __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(two_codes & 0xFFFFu), __NV_E4M3);
    return __half2(h);
}

// One byte of two E2M1 codes (channel 2i low nibble) -> half2 {low, high} (exact).
__device__ __forceinline__ uint32_t e2m1x2_half2_bits(uint32_t byte)
{
    __half2_raw h = __nv_cvt_fp4x2_to_halfraw2((__nv_fp4x2_storage_t)(byte & 0xFFu), __NV_E2M1);
    return (uint32_t)h.x | ((uint32_t)h.y << 16);
}

// Order-preserving map of an fp32 score to uint32 (larger score -> larger key).
__device__ __forceinline__ uint32_t score_key(float s)
{
    uint32_t u = __float_as_uint(s);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ float key_score(uint32_t k)
{
    uint32_t u = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(u);
}

// One 16-channel FP4 block: scale = E4M3(absmax / 6); code = E2M1(x / scale).
__device__ __forceinline__ void fp4_block16(const float x[16], uint2 &codes, uint32_t &scale)
{
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    scale = e4m3_code(__fdiv_rn(amax, 6.0f));
    float s = e4m3_value(scale);
    uint32_t w[2] = {0u, 0u};
    if (s != 0.0f) {
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            uint32_t lo = e2m1_code(__fdiv_rn(x[2 * i], s));
            uint32_t hi = e2m1_code(__fdiv_rn(x[2 * i + 1], s));
            w[i >> 2] |= (lo | (hi << 4)) << (8 * (i & 3));
        }
    }
    codes = make_uint2(w[0], w[1]);
}

__host__ __device__ inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace csa2
