// Step 1 of the CSA2 decode path: quantise-and-write of main-KV rows and
// indexer keys (FP4: E2M1 values, one E4M3 scale per 16 channels, no global
// scale -- Helmcode "DeepSeek V4.1 Flash" explainer, "04 · FP4"; 0x0moeen's
// KV-cache note) and SWA rows (FP8, same explainer section).
//
// HBM-bound: 4 B read per channel, 0.5625 B (FP4) or 1 B + 4/512 (FP8)
// written.  One warp per 512-channel row (lane = one 16-channel block) or per
// eight 64-channel keys; loads are 16-B vectors, stores are 8-B (codes) and
// byte (scales) writes that coalesce into whole sectors per warp.
#include "internal.h"

namespace csa2 {
namespace {

struct QuantBatch {
    QuantJob jobs[kMaxQuantJobs];
    int64_t unit_begin[kMaxQuantJobs + 1];
    int32_t n_jobs;
};

// The job whose unit range holds `unit` (binary search over the range starts).
__device__ __forceinline__ int find_job(const QuantBatch &qb, int64_t unit)
{
    int lo = 0, hi = qb.n_jobs - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (unit >= qb.unit_begin[mid]) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

// Logical position of row i of sequence b, or -1 if the row is skipped.
__device__ __forceinline__ int64_t row_position(const QuantJob &job, int b, int64_t i)
{
    if (job.append_last) {
        int32_t L = __ldg(job.seq_lens + b);
        return (L > 0) ? (int64_t)L - 1 : -1;
    }
    int64_t pos = (job.start_pos ? (int64_t)__ldg(job.start_pos + b) : 0) + i;
    if (job.seq_lens && pos >= __ldg(job.seq_lens + b)) return -1;
    return pos;
}

__device__ __forceinline__ void load16(const float *p, float x[16])
{
    const float4 *p4 = reinterpret_cast<const float4 *>(p);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
        float4 v = __ldcs(p4 + k);
        x[4 * k + 0] = v.x;
        x[4 * k + 1] = v.y;
        x[4 * k + 2] = v.z;
        x[4 * k + 3] = v.w;
    }
}

__global__ void __launch_bounds__(256) quantize_kernel(const __grid_constant__ QuantBatch qb, int *flags)
{
    const int lane = threadIdx.x & 31;
    const int64_t warps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t total = qb.unit_begin[qb.n_jobs];
    for (int64_t unit = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); unit < total;
         unit += warps) {
        const int j = find_job(qb, unit);
        const QuantJob &job = qb.jobs[j];
        const int64_t u = unit - qb.unit_begin[j];
        const int64_t n_rows = job.rows_per_seq * job.n_seqs;
        const int fmt = job.dst.format;
        if (fmt == kFmtPackF16) {
            // one 512-channel row (head h of sequence b), lane = 16 channels: fp32 -> fp16
            // (round to nearest), stored as granules of 8 channels in the order
            // [b][part 4][granule 16][head 16] that the attention's tensor-memory load reads
            const int64_t r = u;
            const int64_t b = r / job.rows_per_seq, hd = r % job.rows_per_seq;
            float x[16];
            load16(job.src + r * kDim + lane * 16, x);
            uint32_t h[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const __half2 v = __floats2half2_rn(x[2 * i], x[2 * i + 1]);
                h[i] = *reinterpret_cast<const uint32_t *>(&v);
            }
            uint4 *d = reinterpret_cast<uint4 *>(job.dst.data) + b * job.rows_per_seq * (kDim / 8) + hd;
            d[(2 * lane) * job.rows_per_seq] = make_uint4(h[0], h[1], h[2], h[3]);
            d[(2 * lane + 1) * job.rows_per_seq] = make_uint4(h[4], h[5], h[6], h[7]);
        } else if (fmt == CSA2_FMT_FP4_KV) {
            const int64_t r = u;
            const int b = (int)(r / job.rows_per_seq);
            const int64_t pos = row_position(job, b, r % job.rows_per_seq);
            if (pos < 0) continue;
            const int64_t slot = slot_of(job.dst, b, pos);
            if (slot < 0) {
                if (lane == 0) raise_flag(flags, kFlagBounds);
                continue;
            }
            float x[16];
            load16(job.src + r * kDim + lane * 16, x);
            uint2 codes;
            uint32_t sc;
            fp4_block16(x, codes, sc);
            uint8_t *row = job.dst.data + slot * kKvRow;
            *reinterpret_cast<uint2 *>(row + lane * 8) = codes;
            row[kKvCodes + lane] = (uint8_t)sc;
        } else if (fmt == CSA2_FMT_FP4_IDX) {
            const int64_t r = u * 8 + (lane >> 2);
            const int blk = lane & 3;
            if (r >= n_rows) continue;
            const int b = (int)(r / job.rows_per_seq);
            const int64_t pos = row_position(job, b, r % job.rows_per_seq);
            if (pos < 0) continue;
            const int64_t slot = slot_of(job.dst, b, pos);
            if (slot < 0) {
                if (blk == 0) raise_flag(flags, kFlagBounds);
                continue;
            }
            float x[16];
            load16(job.src + r * kIdxDim + blk * 16, x);
            uint2 codes;
            uint32_t sc;
            fp4_block16(x, codes, sc);
            uint8_t *tile = job.dst.data + (slot / kIdxTile) * kIdxTileBytes;
            const int rr = (int)(slot % kIdxTile);
            *reinterpret_cast<uint2 *>(tile + rr * 32 + blk * 8) = codes;
            tile[kIdxTile * 32 + rr * 4 + blk] = (uint8_t)sc;
        } else {  // CSA2_FMT_FP8_SWA: per-token scale absmax / 448
            const int64_t r = u;
            const int b = (int)(r / job.rows_per_seq);
            const int64_t pos = row_position(job, b, r % job.rows_per_seq);
            if (pos < 0) continue;  // warp-uniform
            const int64_t slot = slot_of(job.dst, b, pos);
            if (slot < 0) {
                if (lane == 0) raise_flag(flags, kFlagBounds);
                continue;
            }
            float x[16];
            load16(job.src + r * kDim + lane * 16, x);
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, o));
            const float s = __fdiv_rn(amax, 448.0f);
            uint32_t w[4] = {0u, 0u, 0u, 0u};
            if (s != 0.0f) {
#pragma unroll
                for (int i = 0; i < 16; ++i) w[i >> 2] |= e4m3_code(__fdiv_rn(x[i], s)) << (8 * (i & 3));
            }
            *reinterpret_cast<uint4 *>(job.dst.data + slot * kDim + lane * 16) = make_uint4(w[0], w[1], w[2], w[3]);
            if (lane == 0)
                reinterpret_cast<float *>(job.dst.data + job.dst.n_slots * kDim)[slot] = s;
        }
    }
}

}  // namespace

cudaError_t launch_quantize(const QuantJob *jobs, int n_jobs, int *flags, cudaStream_t stream)
{
    for (int first = 0; first < n_jobs; first += kMaxQuantJobs) {
        QuantBatch qb;
        qb.n_jobs = (n_jobs - first < kMaxQuantJobs) ? n_jobs - first : kMaxQuantJobs;
        int64_t units = 0;
        for (int j = 0; j < qb.n_jobs; ++j) {
            qb.jobs[j] = jobs[first + j];
            qb.unit_begin[j] = units;
            const int64_t rows = qb.jobs[j].rows_per_seq * qb.jobs[j].n_seqs;
            units += (qb.jobs[j].dst.format == CSA2_FMT_FP4_IDX) ? ceil_div(rows, 8) : rows;
        }
        qb.unit_begin[qb.n_jobs] = units;
        if (units == 0) continue;
        int64_t blocks = ceil_div(units, 8);
        if (blocks > 148 * 32) blocks = 148 * 32;
        quantize_kernel<<<(unsigned)blocks, 256, 0, stream>>>(qb, flags);
        count_launches(1);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

}  // namespace csa2
