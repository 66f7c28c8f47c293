// Step 2 of the CSA2 decode path: indexer scoring and deterministic Top-K.
//
// Helmcode "DeepSeek V4.1 Flash" explainer, "03 · CSA2": a Full layer scores
// every position, a Reindex layer rescores a Full layer's keys with its own
// query; Louis Bouchard's KV-cache report, "Share the cache and the search
// work": the decoder's first indexing layer keeps a pool of up to 16,384
// candidates that later indexing layers search; 0x0moeen's note: layers
// share the indexer keys.  The score form and its rounding points are this
// library's choice (see include/csa2.h) and make the result exact up to a
// fixed fp32 sequence, so the selected index sets are reproducible bit for bit.
//
// Kernels
//  scan     one pass over FP4 keys (HBM-bound, 36 B per position).  A warp
//           scores 16 keys per step: the E2M1 block dot products of up to two
//           queries (a Full layer and the pool-free Reindex layer that shares
//           its keys) x 4 heads run as one m16n8k16 fp16 MMA per 16-channel
//           block -- exact, because the E2M1 codes and the block-scaled query
//           (scale x code, <= 6 significant bits) are exact in fp16 and every
//           partial sum is a small multiple of the block's quantum.  The
//           epilogue applies the key scales and head weights in the fixed
//           order on CUDA cores, writes an order-preserving uint32 key per
//           candidate and builds a 4096-bin histogram of the key's top bits.
//  collect  per row: the histogram's boundary bin; positions above it are
//           set in a bitmap, boundary-bin candidates are appended to a list.
//  finish   one CTA per row and target: radix select inside the boundary bin
//           over (key, ~position), then bitmap -> ascending positions.
#include "internal.h"

namespace csa2 {
namespace {

constexpr int kScanWarps = 8;
constexpr int kScanChunk = 2048;     // candidates per scan CTA
constexpr int kCollectChunk = 4096;  // candidates per collect CTA
constexpr int kFinishThreads = 1024;

struct ScanBatch {
    ScanJob jobs[kMaxScanJobs];
    float *out_scores[kMaxScanJobs][2];
    int64_t scores_stride;
    int32_t n_jobs;
};

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

__device__ __constant__ float kE2M1[16] = {0.0f,  0.5f,  1.0f,  1.5f,  2.0f,  3.0f,  4.0f,  6.0f,
                                           -0.0f, -0.5f, -1.0f, -1.5f, -2.0f, -3.0f, -4.0f, -6.0f};

// Key of one candidate: cached-code words this thread needs (see below) and
// the four block scales.
struct KeyLoad {
    uint32_t w[4];
    uint32_t sc;
    bool ok;
};

__device__ __forceinline__ KeyLoad load_key(const CacheView &keys, int b, int64_t pos, int t, int *flags)
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
    // thread t uses bytes 8j+2t, 8j+2t+1 of block j: word 2j + t/2, half t%2
#pragma unroll
    for (int j = 0; j < 4; ++j) k.w[j] = __ldg(codes + 2 * j + (t >> 1));
    k.sc = __ldg(reinterpret_cast<const uint32_t *>(tile + kIdxTile * 32 + rr * 4));
    k.ok = true;
    return k;
}

__global__ void __launch_bounds__(kScanWarps * 32) scan_kernel(const __grid_constant__ ScanBatch sb,
                                                                 SelectBufs bufs, const int32_t *seq_lens,
                                                                 int batch, int max_len, int *flags)
{
    __shared__ uint32_t hist[2][kHistBins];
    __shared__ __half qpre[2][kIdxHeads][kIdxDim];
    __shared__ float wq[2][kIdxHeads];

    const ScanJob &job = sb.jobs[blockIdx.z];
    const int b = blockIdx.y;
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int g = lane >> 2, t = lane & 3;
    int L = __ldg(seq_lens + b);
    if (L < 0 || L > max_len) {
        if (tid == 0) raise_flag(flags, kFlagBounds);
        L = L < 0 ? 0 : max_len;
    }
    const int64_t n_cand = job.pool ? job.pool_len : L;

    for (int i = tid; i < 2 * kHistBins; i += blockDim.x) (&hist[0][0])[i] = 0u;
    // zero this CTA's slice of the rows' bitmaps (both targets)
    {
        const int per = (int)ceil_div(bufs.bm_words, gridDim.x);
        const int w0 = blockIdx.x * per;
        const int w1 = min(bufs.bm_words, w0 + per);
        for (int qi = 0; qi < job.n_q; ++qi) {
            const int64_t row = (int64_t)job.row[qi] * batch + b;
            uint32_t *bm = bufs.bitmap + row * 2 * bufs.bm_words;
            for (int w = w0 + tid; w < w1; w += blockDim.x) {
                bm[w] = 0u;
                bm[bufs.bm_words + w] = 0u;
            }
        }
    }
    // quantise the queries (FP4 rule) and pre-scale: qpre = scale * E2M1(code), exact in fp16
    if (tid < 32) {
        const int qi = tid >> 4, h = (tid >> 2) & 3, blk = tid & 3;
        float v[16];
        if (qi < job.n_q) {
            const float *src = job.q_idx[qi] + ((int64_t)b * kIdxHeads + h) * kIdxDim + blk * 16;
            float amax = 0.0f;
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                v[i] = __ldg(src + i);
                amax = fmaxf(amax, fabsf(v[i]));
            }
            const float s = e4m3_value(e4m3_code(__fdiv_rn(amax, 6.0f)));
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                const float e = (s != 0.0f) ? kE2M1[e2m1_code(__fdiv_rn(v[i], s))] : 0.0f;
                qpre[qi][h][blk * 16 + i] = __float2half_rn(e * s);
            }
            if (blk == 0) wq[qi][h] = __ldg(job.w[qi] + (int64_t)b * kIdxHeads + h);
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) qpre[qi][h][blk * 16 + i] = __float2half_rn(0.0f);
            if (blk == 0) wq[qi][h] = 0.0f;
        }
    }
    __syncthreads();

    // B fragments, block j: column g = (query g/4, head g%4); k-slot 2t+e <-> channel 4t+e,
    // k-slot 2t+8+e <-> channel 4t+2+e (a permutation of the block applied to both operands)
    uint32_t bfrag[4][2];
    {
        const int qi = g >> 2, h = g & 3;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half *q = &qpre[qi][h][j * 16 + 4 * t];
            bfrag[j][0] = (uint32_t)__half_as_ushort(q[0]) | ((uint32_t)__half_as_ushort(q[1]) << 16);
            bfrag[j][1] = (uint32_t)__half_as_ushort(q[2]) | ((uint32_t)__half_as_ushort(q[3]) << 16);
        }
    }
    const int my_q = t >> 1;  // query of this thread's two columns
    const bool finisher = (t & 1) != 0;
    const float w0 = wq[my_q][0], w1 = wq[my_q][1], w2 = wq[my_q][2], w3 = wq[my_q][3];
    const int64_t my_row = (int64_t)job.row[my_q < job.n_q ? my_q : 0] * batch + b;
    uint32_t *key_out = bufs.keys + my_row * bufs.cand_cap;
    float *score_out = (my_q < job.n_q) ? sb.out_scores[blockIdx.z][my_q] : nullptr;
    if (score_out) score_out += (int64_t)b * sb.scores_stride;
    const int32_t *pool = job.pool ? job.pool + (int64_t)b * job.pool_len : nullptr;

    const int64_t base = (int64_t)blockIdx.x * kScanChunk;
    for (int grp = warp; grp < kScanChunk / 16; grp += kScanWarps) {
        const int64_t c0 = base + grp * 16;
        if (c0 >= n_cand) break;
        const int64_t cA = c0 + g, cB = c0 + g + 8;
        int64_t pA = -1, pB = -1;
        if (cA < n_cand) pA = pool ? (int64_t)__ldg(pool + cA) : cA;
        if (cB < n_cand) pB = pool ? (int64_t)__ldg(pool + cB) : cB;
        if (pA >= L) pA = -1;
        if (pB >= L) pB = -1;
        const KeyLoad kA = load_key(job.keys, b, pA, t, flags);
        const KeyLoad kB = load_key(job.keys, b, pB, t, flags);

        float d[4][4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const uint32_t uA = (kA.w[j] >> (16 * (t & 1))) & 0xFFFFu;
            const uint32_t uB = (kB.w[j] >> (16 * (t & 1))) & 0xFFFFu;
            mma16816(d[j], e2m1x2_half2_bits(uA & 0xFFu), e2m1x2_half2_bits(uB & 0xFFu),
                     e2m1x2_half2_bits(uA >> 8), e2m1x2_half2_bits(uB >> 8), bfrag[j][0], bfrag[j][1]);
        }
        // s = t0 + t1 + t2 + t3 in order; t_j = sk_j * (sq_j * P_j) is exact, so fma == add
        float sA0, sA1, sB0, sB1;
        {
            float sk = e4m3_value(kA.sc & 0xFFu);
            sA0 = sk * d[0][0];
            sA1 = sk * d[0][1];
            sk = e4m3_value(kB.sc & 0xFFu);
            sB0 = sk * d[0][2];
            sB1 = sk * d[0][3];
#pragma unroll
            for (int j = 1; j < 4; ++j) {
                sk = e4m3_value((kA.sc >> (8 * j)) & 0xFFu);
                sA0 = __fmaf_rn(sk, d[j][0], sA0);
                sA1 = __fmaf_rn(sk, d[j][1], sA1);
                sk = e4m3_value((kB.sc >> (8 * j)) & 0xFFu);
                sB0 = __fmaf_rn(sk, d[j][2], sB0);
                sB1 = __fmaf_rn(sk, d[j][3], sB1);
            }
        }
        const float rA0 = sA0 > 0.0f ? sA0 : 0.0f, rA1 = sA1 > 0.0f ? sA1 : 0.0f;
        const float rB0 = sB0 > 0.0f ? sB0 : 0.0f, rB1 = sB1 > 0.0f ? sB1 : 0.0f;
        // heads 0,1 live on even t, heads 2,3 on odd t: chain w0*r0 -> +w1 r1 -> +w2 r2 -> +w3 r3
        float accA = __fmaf_rn(w1, rA1, __fmul_rn(w0, rA0));
        float accB = __fmaf_rn(w1, rB1, __fmul_rn(w0, rB0));
        accA = __shfl_xor_sync(0xFFFFFFFFu, accA, 1);
        accB = __shfl_xor_sync(0xFFFFFFFFu, accB, 1);
        if (finisher && my_q < job.n_q) {
            float scA = __fmaf_rn(w3, rA1, __fmaf_rn(w2, rA0, accA));
            float scB = __fmaf_rn(w3, rB1, __fmaf_rn(w2, rB0, accB));
            if (scA == 0.0f) scA = 0.0f;
            if (scB == 0.0f) scB = 0.0f;
            if (cA < n_cand) {
                const uint32_t key = kA.ok ? score_key(scA) : 0u;
                key_out[cA] = key;
                if (kA.ok) {
                    atomicAdd(&hist[my_q][key >> 20], 1u);
                    if (score_out) score_out[cA] = scA;
                }
            }
            if (cB < n_cand) {
                const uint32_t key = kB.ok ? score_key(scB) : 0u;
                key_out[cB] = key;
                if (kB.ok) {
                    atomicAdd(&hist[my_q][key >> 20], 1u);
                    if (score_out) score_out[cB] = scB;
                }
            }
        }
    }
    __syncthreads();
    for (int qi = 0; qi < job.n_q; ++qi) {
        uint32_t *gh = bufs.hist + ((int64_t)job.row[qi] * batch + b) * kHistBins;
        for (int i = tid; i < kHistBins; i += blockDim.x) {
            const uint32_t c = hist[qi][i];
            if (c) atomicAdd(gh + i, c);
        }
    }
}

// ---- threshold search over a histogram (block-wide) --------------------------
// Finds bin d with above(d) < need <= above(d) + hist[d], where above(d) is the
// count in bins > d.  If the total is < need, returns d = -1, above = total.
// Requires blockDim.x * per == nbins.
struct Thresh {
    int bin;
    uint32_t above;
    uint32_t at;
};

template <int NT>
__device__ Thresh find_threshold(const uint32_t *h, int nbins, uint32_t need, uint32_t *scratch /*>= NT/32+3*/)
{
    const int tid = threadIdx.x;
    const int per = nbins / NT;
    const int hi = nbins - tid * per;  // this thread covers [hi - per, hi), descending from the top
    uint32_t local = 0;
    for (int i = 1; i <= per; ++i) local += h[hi - i];
    // inclusive scan over threads (thread 0 = top bins)
    uint32_t incl = local;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t v = (lane < NT / 32) ? scratch[lane] : 0u;
        uint32_t s = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            uint32_t u = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += u;
        }
        if (lane < NT / 32) scratch[lane] = s - v;  // exclusive warp offsets
        if (lane == NT / 32 - 1) scratch[NT / 32] = s;  // total
    }
    __syncthreads();
    const uint32_t excl = scratch[warp] + incl - local;
    const uint32_t total = scratch[NT / 32];
    __syncthreads();
    if (total < need) {
        if (tid == 0) {
            scratch[NT / 32 + 1] = 0xFFFFFFFFu;
            scratch[NT / 32 + 2] = total;
        }
    } else if (excl < need && need <= excl + local) {
        uint32_t above = excl;
        for (int i = 1; i <= per; ++i) {
            const uint32_t c = h[hi - i];
            if (need <= above + c) {
                scratch[NT / 32 + 1] = (uint32_t)(hi - i);
                scratch[NT / 32 + 2] = above;
                break;
            }
            above += c;
        }
    }
    __syncthreads();
    Thresh r;
    r.bin = (int)scratch[NT / 32 + 1];
    r.above = scratch[NT / 32 + 2];
    r.at = (r.bin >= 0) ? h[r.bin] : 0u;
    __syncthreads();
    return r;
}

__device__ __forceinline__ int row_len(const int32_t *seq_lens, int b, int max_len)
{
    int L = __ldg(seq_lens + b);
    return L < 0 ? 0 : (L > max_len ? max_len : L);
}

// ---- collect ------------------------------------------------------------------
__global__ void __launch_bounds__(256) collect_kernel(SelectPlan plan, int max_len, int *flags)
{
    __shared__ uint32_t hsm[kHistBins];
    __shared__ uint32_t scratch[16];
    const int b = blockIdx.y, rb = blockIdx.z;
    const SelectRow &R = plan.rows[rb];
    const int64_t row = (int64_t)rb * plan.batch + b;
    const int L = row_len(plan.seq_lens, b, max_len);
    const int64_t n_cand = R.pool ? R.pool_len : L;
    const int64_t base = (int64_t)blockIdx.x * kCollectChunk;
    if (base >= n_cand) return;

    for (int i = threadIdx.x; i < kHistBins; i += blockDim.x)
        hsm[i] = plan.bufs.hist[row * kHistBins + i];
    __syncthreads();
    const int n_targets = (R.out_pool && plan.pool_out_len > 0) ? 2 : 1;
    Thresh th[2];
    th[0] = find_threshold<256>(hsm, kHistBins, (uint32_t)plan.topk, scratch);
    th[1] = th[0];
    if (n_targets == 2) th[1] = find_threshold<256>(hsm, kHistBins, (uint32_t)plan.pool_out_len, scratch);

    const uint32_t *keys = plan.bufs.keys + row * plan.bufs.cand_cap;
    const int32_t *pool = R.pool ? R.pool + (int64_t)b * R.pool_len : nullptr;
    const int lane = threadIdx.x & 31;
    const int64_t end = min(n_cand, base + (int64_t)kCollectChunk);
    for (int64_t c0 = base + (threadIdx.x & ~31); c0 < end; c0 += blockDim.x) {
        const int64_t c = c0 + lane;
        uint32_t key = 0;
        int64_t pos = -1;
        if (c < end) {
            key = keys[c];
            pos = pool ? (int64_t)__ldg(pool + c) : c;
        }
        const bool valid = key != 0u && pos >= 0 && pos < L;
        const int bin = (int)(key >> 20);
        for (int tg = 0; tg < n_targets; ++tg) {
            uint32_t *bm = plan.bufs.bitmap + (row * 2 + tg) * plan.bufs.bm_words;
            const bool sel = valid && bin > th[tg].bin;
            const bool eq = valid && bin == th[tg].bin;
            if (!pool) {
                const uint32_t word = __ballot_sync(0xFFFFFFFFu, sel);
                if (lane == 0) bm[c0 >> 5] = word;
            } else if (sel) {
                atomicOr(bm + (pos >> 5), 1u << (pos & 31));
            }
            const uint32_t m = __ballot_sync(0xFFFFFFFFu, eq);
            if (m) {
                uint32_t *cnt = plan.bufs.cand_count + row * 2 + tg;
                uint32_t off = 0;
                if (lane == 0) off = atomicAdd(cnt, (uint32_t)__popc(m));
                off = __shfl_sync(0xFFFFFFFFu, off, 0);
                if (eq) {
                    const uint32_t at = off + __popc(m & ((1u << lane) - 1u));
                    if (at < (uint32_t)plan.bufs.cand_max)
                        plan.bufs.cand[(row * 2 + tg) * plan.bufs.cand_max + at] =
                            ((uint64_t)key << 32) | (uint32_t)pos;
                }
            }
        }
    }
}

// ---- finish -------------------------------------------------------------------
// Composite order inside the boundary bin: (low 20 key bits, then ~position),
// 52 bits, larger = earlier.  Unique per candidate.
__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t pos)
{
    return ((uint64_t)(key & 0xFFFFFu) << 32) | (uint64_t)(~pos);
}

__global__ void __launch_bounds__(kFinishThreads) finish_kernel(SelectPlan plan, int max_len, int *flags)
{
    extern __shared__ __align__(16) uint8_t smem[];
    uint64_t *elem = reinterpret_cast<uint64_t *>(smem);                                // cand_max
    uint32_t *hsm = reinterpret_cast<uint32_t *>(smem + 8 * (size_t)plan.bufs.cand_max);  // 4096
    __shared__ uint32_t scratch[48];
    __shared__ uint64_t s_prefix;
    __shared__ int s_nb;
    __shared__ uint32_t s_need;

    const int b = blockIdx.x, rb = blockIdx.y, tg = blockIdx.z;
    const SelectRow &R = plan.rows[rb];
    if (tg == 1 && !(R.out_pool && plan.pool_out_len > 0)) return;
    const int64_t row = (int64_t)rb * plan.batch + b;
    const int L = row_len(plan.seq_lens, b, max_len);
    const int64_t n_cand = R.pool ? R.pool_len : L;
    const int K = tg == 0 ? plan.topk : plan.pool_out_len;
    int32_t *out = (tg == 0 ? R.out_idx : R.out_pool) + (int64_t)b * K;
    uint32_t *bm = plan.bufs.bitmap + (row * 2 + tg) * plan.bufs.bm_words;
    const int tid = threadIdx.x;

    for (int i = tid; i < kHistBins; i += blockDim.x) hsm[i] = plan.bufs.hist[row * kHistBins + i];
    __syncthreads();
    const Thresh th = find_threshold<kFinishThreads>(hsm, kHistBins, (uint32_t)K, scratch);
    const uint32_t need0 = (th.bin >= 0) ? (uint32_t)K - th.above : 0u;

    if (need0 > 0) {
        const uint32_t count = plan.bufs.cand_count[row * 2 + tg];
        const bool in_smem = count <= (uint32_t)plan.bufs.cand_max;
        const uint64_t *gcand = plan.bufs.cand + (row * 2 + tg) * plan.bufs.cand_max;
        const uint32_t *keys = plan.bufs.keys + row * plan.bufs.cand_cap;
        const int32_t *pool = R.pool ? R.pool + (int64_t)b * R.pool_len : nullptr;
        if (in_smem) {
            for (uint32_t i = tid; i < count; i += blockDim.x) {
                const uint64_t v = gcand[i];
                elem[i] = composite((uint32_t)(v >> 32), (uint32_t)v);
            }
        } else if (tid == 0) {
            raise_flag(flags, kFlagOverflow);
        }
        // Visit every boundary-bin candidate's composite (smem list, or a rescan of the
        // row on the overflow path).
        auto for_each = [&](auto &&f) {
            if (in_smem) {
                for (uint32_t i = tid; i < count; i += blockDim.x) f(elem[i]);
            } else {
                for (int64_t c = tid; c < n_cand; c += blockDim.x) {
                    const uint32_t key = keys[c];
                    const int64_t pos = pool ? (int64_t)__ldg(pool + c) : c;
                    if (key != 0u && pos >= 0 && pos < L && (int)(key >> 20) == th.bin)
                        f(composite(key, (uint32_t)pos));
                }
            }
        };
        if (tid == 0) {
            s_prefix = 0;
            s_nb = 0;
            s_need = need0;
        }
        __syncthreads();
        // radix select of the need0-th largest composite, 11-bit digits from bit 51
        for (;;) {
            const int nb = s_nb;
            const uint64_t prefix = s_prefix;
            const uint32_t need = s_need;
            const int wbits = (52 - nb) < 11 ? (52 - nb) : 11;
            const int shift = 52 - nb - wbits;
            const int nbins = 1 << wbits;
            for (int i = tid; i < 2048; i += blockDim.x) hsm[i] = 0u;
            __syncthreads();
            for_each([&](uint64_t cp) {
                if ((cp >> (52 - nb)) == prefix || nb == 0)
                    atomicAdd(&hsm[(cp >> shift) & (uint64_t)(nbins - 1)], 1u);
            });
            __syncthreads();
            // bins above nbins are zero, so searching 2048 bins is equivalent
            const Thresh d = find_threshold<kFinishThreads>(hsm, 2048, need, scratch);
            if (tid == 0) {
                s_prefix = (prefix << wbits) | (uint64_t)(d.bin < 0 ? 0 : d.bin);
                s_nb = nb + wbits;
                s_need = need - d.above;
            }
            __syncthreads();
            if (d.bin < 0 || d.at == s_need || s_nb >= 52) break;
        }
        const uint64_t T = s_prefix << (52 - s_nb);
        for_each([&](uint64_t cp) {
            if (cp >= T) {
                const uint32_t pos = ~(uint32_t)cp;
                atomicOr(bm + (pos >> 5), 1u << (pos & 31));
            }
        });
    }
    __syncthreads();

    // bitmap -> ascending positions
    const int words = (int)ceil_div(L, 32);
    const int per = (int)ceil_div(words, kFinishThreads);
    const int w0 = tid * per, w1 = min(words, w0 + per);
    uint32_t local = 0;
    for (int w = w0; w < w1; ++w) {
        uint32_t v = bm[w];
        if (w == words - 1 && (L & 31)) v &= (1u << (L & 31)) - 1u;
        local += __popc(v);
    }
    uint32_t incl = local;
    const int lane = tid & 31, warp = tid >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t v = __shfl_up_sync(0xFFFFFFFFu, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        const uint32_t v = scratch[lane];
        uint32_t s = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t u = __shfl_up_sync(0xFFFFFFFFu, s, o);
            if (lane >= o) s += u;
        }
        scratch[lane] = s - v;
        if (lane == 31) scratch[32] = s;
    }
    __syncthreads();
    uint32_t at = scratch[warp] + incl - local;
    const uint32_t total = scratch[32];
    for (int w = w0; w < w1; ++w) {
        uint32_t v = bm[w];
        if (w == words - 1 && (L & 31)) v &= (1u << (L & 31)) - 1u;
        while (v) {
            const int bit = __ffs(v) - 1;
            v &= v - 1u;
            if (at < (uint32_t)K) out[at] = w * 32 + bit;
            ++at;
        }
    }
    for (int i = (int)total + tid; i < K; i += blockDim.x) out[i] = -1;
    if (tid == 0 && total > (uint32_t)K) raise_flag(flags, kFlagBounds);
}

}  // namespace

size_t select_bytes(int n_rows, int64_t cand_cap, int max_seq_len)
{
    const int64_t bm_words = ceil_div(max_seq_len, 32);
    const int64_t cand_max = 8192;
    size_t bytes = 0;
    auto add = [&](size_t n) { bytes += (n + 255) & ~(size_t)255; };
    add((size_t)n_rows * kHistBins * 4);        // hist
    add((size_t)n_rows * 2 * 4);                // cand_count
    add((size_t)n_rows * cand_cap * 4);         // keys
    add((size_t)n_rows * 2 * bm_words * 4);     // bitmaps
    add((size_t)n_rows * 2 * cand_max * 8);     // boundary candidates
    return bytes;
}

SelectBufs carve_select(uint8_t *base, int n_rows, int64_t cand_cap, int max_seq_len)
{
    SelectBufs s;
    s.cand_cap = cand_cap;
    s.bm_words = (int32_t)ceil_div(max_seq_len, 32);
    s.cand_max = 8192;
    size_t off = 0;
    auto take = [&](size_t n) {
        uint8_t *p = base + off;
        off += (n + 255) & ~(size_t)255;
        return p;
    };
    s.hist = reinterpret_cast<uint32_t *>(take((size_t)n_rows * kHistBins * 4));
    s.cand_count = reinterpret_cast<uint32_t *>(take((size_t)n_rows * 2 * 4));
    s.keys = reinterpret_cast<uint32_t *>(take((size_t)n_rows * cand_cap * 4));
    s.bitmap = reinterpret_cast<uint32_t *>(take((size_t)n_rows * 2 * s.bm_words * 4));
    s.cand = reinterpret_cast<uint64_t *>(take((size_t)n_rows * 2 * s.cand_max * 8));
    return s;
}

cudaError_t launch_scan(const ScanJob *jobs, int n_jobs, const SelectPlan &plan, int max_cand,
                        float *const (*scores)[2], int64_t scores_stride, int *flags, cudaStream_t stream)
{
    for (int first = 0; first < n_jobs; first += kMaxScanJobs) {
        ScanBatch sb;
        sb.n_jobs = (n_jobs - first < kMaxScanJobs) ? n_jobs - first : kMaxScanJobs;
        sb.scores_stride = scores_stride;
        for (int j = 0; j < sb.n_jobs; ++j) {
            sb.jobs[j] = jobs[first + j];
            sb.out_scores[j][0] = scores ? scores[first + j][0] : nullptr;
            sb.out_scores[j][1] = scores ? scores[first + j][1] : nullptr;
        }
        dim3 grid((unsigned)ceil_div(max_cand > 0 ? max_cand : 1, kScanChunk), (unsigned)plan.batch,
                  (unsigned)sb.n_jobs);
        scan_kernel<<<grid, kScanWarps * 32, 0, stream>>>(sb, plan.bufs, plan.seq_lens, plan.batch,
                                                         plan.max_len, flags);
        count_launches(1);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
}

cudaError_t launch_select(const SelectPlan &plan, int max_cand, int *flags, cudaStream_t stream,
                          cudaEvent_t mid_event)
{
    const int max_len = plan.max_len;
    dim3 cgrid((unsigned)ceil_div(max_cand > 0 ? max_cand : 1, kCollectChunk), (unsigned)plan.batch,
               (unsigned)plan.n_row_blocks);
    collect_kernel<<<cgrid, 256, 0, stream>>>(plan, max_len, flags);
    count_launches(1);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const size_t smem = 8 * (size_t)plan.bufs.cand_max + 4 * kHistBins;
    int dev = 0;
    e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    static bool attr_set[64] = {};
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(finish_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    dim3 fgrid((unsigned)plan.batch, (unsigned)plan.n_row_blocks, 2u);
    finish_kernel<<<fgrid, kFinishThreads, smem, stream>>>(plan, max_len, flags);
    count_launches(1);
    (void)mid_event;
    return cudaGetLastError();
}

}  // namespace csa2
