// C interface of the CSA2 decode hot path: argument checks, workspace
// planning and the enqueue order of one decode step over a static layer-mode
// schedule (Helmcode "DeepSeek V4.1 Flash" explainer, "03 · CSA2": Full,
// Reindex, Reuse and SWA-only layers; Louis Bouchard's KV-cache report,
// "Share the cache and the search work": pool-restricted Reindex).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <algorithm>
#include <array>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <set>
#include <string>
#include <utility>
#include <vector>

#include "internal.h"

using namespace csa2;

namespace csa2 {
static std::atomic<int64_t> g_launches{0};
void count_launches(int n) { g_launches.fetch_add(n, std::memory_order_relaxed); }
}  // namespace csa2

namespace {

thread_local std::string g_err;
thread_local int32_t g_last_flags = 0;

csa2_status fail(csa2_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

}  // namespace

void csa2::log_plan(const char *fmt, ...)
{
    static const bool on = [] {
        const char *v = getenv("CSA2_LOG");
        return v && v[0] && !(v[0] == '0' && v[1] == 0);
    }();
    if (!on) return;
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    static std::mutex mu;
    static std::set<std::string> seen;
    std::lock_guard<std::mutex> lock(mu);
    if (seen.insert(buf).second) fprintf(stderr, "[csa2] %s\n", buf);
}

csa2_status csa2::set_error(csa2_status s, const char *fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return s;
}

namespace {

csa2_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(CSA2_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

// One flag word per device; its address is looked up once per device.
__device__ int g_device_flags;

int *flags_ptr()
{
    static int *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    if (!cache[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_flags) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int *>(p);
    }
    return cache[dev];
}

void *g_events[8] = {};
int g_n_events = 0;

cudaError_t mark(int phase, cudaStream_t s)
{
    if (phase < g_n_events && g_events[phase])
        return record_event(static_cast<cudaEvent_t>(g_events[phase]), s);
    return cudaSuccess;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }


csa2_status check_cache(const csa2_cache *c, int fmt, int batch, int64_t span, const char *name)
{
    if (!c) return fail(CSA2_ERR_INVALID_ARG, "%s: cache descriptor is NULL", name);
    if (c->format != fmt) return fail(CSA2_ERR_INVALID_ARG, "%s: format %d, expected %d", name, c->format, fmt);
    if (!c->data || !aligned(c->data, 16))
        return fail(CSA2_ERR_INVALID_ARG, "%s: data NULL or not 16-byte aligned", name);
    if (c->n_slots <= 0) return fail(CSA2_ERR_INVALID_ARG, "%s: n_slots must be > 0", name);
    if (c->reserved != 0) return fail(CSA2_ERR_INVALID_ARG, "%s: reserved must be 0", name);
    if (fmt == CSA2_FMT_FP4_IDX && c->n_slots % kIdxTile)
        return fail(CSA2_ERR_INVALID_ARG, "%s: n_slots must be a multiple of 64", name);
    if (fmt == CSA2_FMT_FP8_SWA && c->n_slots % 4)
        return fail(CSA2_ERR_INVALID_ARG, "%s: n_slots must be a multiple of 4", name);
    if (c->page_size < 0) return fail(CSA2_ERR_INVALID_ARG, "%s: page_size < 0", name);
    if (c->page_size > 0) {
        if (c->page_size % 64) return fail(CSA2_ERR_INVALID_ARG, "%s: page_size must be a multiple of 64", name);
        if (!c->page_table || c->max_pages <= 0)
            return fail(CSA2_ERR_INVALID_ARG, "%s: paged cache needs page_table and max_pages", name);
        if (fmt != CSA2_FMT_FP8_SWA && (int64_t)c->max_pages * c->page_size < span)
            return fail(CSA2_ERR_INVALID_ARG, "%s: max_pages * page_size < max_seq_len", name);
    } else {
        if (c->seq_stride <= 0) return fail(CSA2_ERR_INVALID_ARG, "%s: seq_stride must be > 0", name);
        if (fmt == CSA2_FMT_FP4_IDX && c->seq_stride % kIdxTile)
            return fail(CSA2_ERR_INVALID_ARG, "%s: seq_stride must be a multiple of 64", name);
        if (fmt != CSA2_FMT_FP8_SWA && c->seq_stride < span)
            return fail(CSA2_ERR_INVALID_ARG, "%s: seq_stride %lld < max_seq_len %lld", name,
                        (long long)c->seq_stride, (long long)span);
        if (fmt == CSA2_FMT_FP8_SWA && c->seq_stride < span)
            return fail(CSA2_ERR_INVALID_ARG, "%s: ring capacity %lld < window %lld", name,
                        (long long)c->seq_stride, (long long)span);
        if ((int64_t)batch * c->seq_stride > c->n_slots)
            return fail(CSA2_ERR_INVALID_ARG, "%s: batch * seq_stride > n_slots", name);
    }
    return CSA2_OK;
}

csa2_status check_ws(void *ws, size_t have, size_t need)
{
    if (need == 0) return CSA2_OK;
    if (!ws) return fail(CSA2_ERR_WORKSPACE, "workspace is NULL (%zu bytes needed)", need);
    if (!aligned(ws, 256)) return fail(CSA2_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    if (have < need) return fail(CSA2_ERR_WORKSPACE, "workspace has %zu bytes, %zu needed", have, need);
    return CSA2_OK;
}

size_t round256(size_t n) { return (n + 255) & ~(size_t)255; }


}  // namespace

namespace csa2 {

size_t sparse_attn_workspace_within(int32_t batch, int32_t topk, int32_t swa_window, size_t budget)
{
    if (batch <= 0 || topk < 0 || swa_window < 0) return 0;
    static const int32_t any_index = 0;  // stands for "an index list is given"
    static const float any_q = 0.0f;
    AttnEntry en;
    memset(&en, 0, sizeof(en));
    en.has_kv = topk > 0 ? 1 : 0;
    en.idx = topk > 0 ? &any_index : nullptr;
    en.kv.data = reinterpret_cast<uint8_t *>(const_cast<int32_t *>(&any_index));
    en.has_swa = swa_window > 0 ? 1 : 0;
    en.q = &any_q;
    AttnPlan plan;
    memset(&plan, 0, sizeof(plan));
    plan.entries = &en;
    plan.n_entries = 1;
    plan.batch = batch;
    plan.topk = topk;
    plan.window = swa_window;
    plan.max_group = 1;
    return attn_workspace_bytes(plan, budget);
}

}  // namespace csa2

namespace {

// One indexing level: jobs over key caches, each scored by up to two query
// rows (a Full layer and the pool-free Reindex layer over the same keys share
// the pass).  Runs as one fused co-resident launch when it fits, otherwise as
// the scan + select kernels (with the appends as a quantise launch first).
struct IdxJob {
    const csa2_cache *keys;
    const int32_t *pool;     // [B][pool_len] or null
    int32_t pool_len;
    int32_t n_q;
    const float *q_idx[2], *w[2];
    int32_t *out_idx[2], *out_pool[2];
    float *out_scores[2];
    const csa2_cache *kv;    // appends of a Full layer
    const float *new_kv, *new_key;
    const csa2_cache *warm;  // main-KV cache the selected rows are gathered from next, or null
};

int64_t level_max_cand(const IdxJob *jobs, int n_jobs, int max_seq_len)
{
    int64_t m = 1;
    for (int j = 0; j < n_jobs; ++j) m = std::max<int64_t>(m, jobs[j].pool ? jobs[j].pool_len : max_seq_len);
    return m;
}

// Workspace of one level: the fused launch's group state, or the scan +
// select buffers.
struct LevelWs {
    bool fused = false;
    FusedPlan plan{};
    size_t fused_bytes = 0, old_bytes = 0;
};

LevelWs level_ws(const IdxJob *jobs, int n_jobs, int batch, int max_seq_len)
{
    LevelWs w;
    if (n_jobs <= 0) return w;
    const int64_t mc = level_max_cand(jobs, n_jobs, max_seq_len);
    int n_rows = 0;
    for (int j = 0; j < n_jobs; ++j) n_rows += jobs[j].n_q;
    if (n_jobs <= 8 && fused_plan(n_jobs, batch, mc, w.plan)) {
        w.fused = true;
        w.fused_bytes = round256(fused_state_bytes(n_jobs * batch));
    } else {
        w.old_bytes = round256(select_bytes(n_rows * batch, mc, max_seq_len));
    }
    return w;
}

cudaError_t run_level(const IdxJob *jobs, int n_jobs, const LevelWs &lw, int batch, const int32_t *seq_lens,
                      int max_seq_len, int topk, int pool_out_len, int64_t scores_stride, uint8_t *fused_ws,
                      uint8_t *old_ws, int *fp, cudaStream_t s, int keys_ready = 0)
{
    if (lw.fused) {
        std::vector<FusedJobDesc> d((size_t)n_jobs);
        for (int j = 0; j < n_jobs; ++j) {
            const IdxJob &J = jobs[j];
            FusedJobDesc &D = d[(size_t)j];
            memset(&D, 0, sizeof(D));
            D.keys = view_of(*J.keys);
            D.pool = J.pool;
            D.pool_len = J.pool ? J.pool_len : 0;
            D.n_q = J.n_q;
            for (int q = 0; q < 2; ++q) {
                D.q_idx[q] = J.q_idx[q];
                D.w[q] = J.w[q];
                D.out_idx[q] = J.out_idx[q];
                D.out_pool[q] = J.out_pool[q];
                D.out_scores[q] = J.out_scores[q];
            }
            if (J.kv && J.new_kv) {
                D.kv = view_of(*J.kv);
                D.new_kv = J.new_kv;
            }
            D.new_key = J.new_key;
            if (J.warm) {
                D.warm = view_of(*J.warm);
                D.has_warm = 1;
            }
        }
        // a layer of a decode step follows the previous layer's attention launch
        // (18 CTAs at batch 1), which still runs when this one starts: leave it
        // 20 SMs so that every CTA of this grid starts at once
        FusedPlan plan = lw.plan;
        if (keys_ready) {
            FusedPlan p2;
            if (fused_plan(n_jobs, batch, level_max_cand(jobs, n_jobs, max_seq_len), p2, 20)) plan = p2;
        }
        FusedLaunch L;
        L.jobs = d.data();
        L.n_jobs = n_jobs;
        L.seq_lens = seq_lens;
        L.state = fused_ws;
        L.scores_stride = scores_stride;
        L.batch = batch;
        L.topk = topk;
        L.pool_out = pool_out_len;
        L.max_len = max_seq_len;
        L.pdl = 1;
        L.keys_ready = keys_ready;
        return launch_fused(L, plan, fp, s);
    }
    // scan + select, the appends first
    std::vector<QuantJob> qjobs;
    for (int j = 0; j < n_jobs; ++j) {
        const IdxJob &J = jobs[j];
        const std::pair<const float *, const csa2_cache *> ap[2] = {{J.new_kv, J.kv}, {J.new_key, J.keys}};
        for (const auto &a : ap) {
            if (!a.first || !a.second) continue;
            QuantJob q;
            memset(&q, 0, sizeof(q));
            q.src = a.first;
            q.seq_lens = seq_lens;
            q.dst = view_of(*a.second);
            q.rows_per_seq = 1;
            q.n_seqs = batch;
            q.append_last = 1;
            qjobs.push_back(q);
        }
    }
    cudaError_t e = cudaSuccess;
    if (!qjobs.empty() && (e = launch_quantize(qjobs.data(), (int)qjobs.size(), fp, s)) != cudaSuccess) return e;
    int n_rows = 0;
    for (int j = 0; j < n_jobs; ++j) n_rows += jobs[j].n_q;
    if (n_rows > kMaxSelectRows) return cudaErrorInvalidValue;
    const int64_t mc = level_max_cand(jobs, n_jobs, max_seq_len);
    SelectPlan plan;
    memset(&plan, 0, sizeof(plan));
    plan.bufs = carve_select(old_ws, n_rows * batch, mc, max_seq_len);
    plan.n_row_blocks = n_rows;
    plan.batch = batch;
    plan.topk = topk;
    plan.pool_out_len = pool_out_len;
    plan.max_len = max_seq_len;
    plan.seq_lens = seq_lens;
    std::vector<ScanJob> sj((size_t)n_jobs);
    std::vector<std::array<float *, 2>> sc((size_t)n_jobs);
    int row = 0;
    for (int j = 0; j < n_jobs; ++j) {
        const IdxJob &J = jobs[j];
        ScanJob &S = sj[(size_t)j];
        memset(&S, 0, sizeof(S));
        S.keys = view_of(*J.keys);
        S.pool = J.pool;
        S.pool_len = J.pool ? J.pool_len : 0;
        S.n_q = J.n_q;
        for (int q = 0; q < J.n_q; ++q) {
            S.q_idx[q] = J.q_idx[q];
            S.w[q] = J.w[q];
            S.row[q] = row;
            SelectRow &R = plan.rows[row++];
            R.out_idx = J.out_idx[q];
            R.out_pool = J.out_pool[q];
            R.pool = J.pool;
            R.pool_len = J.pool ? J.pool_len : 0;
            sc[(size_t)j][(size_t)q] = J.out_scores[q];
        }
        if (J.n_q < 2) sc[(size_t)j][1] = nullptr;
    }
    if ((e = cudaMemsetAsync(old_ws, 0, select_hist_bytes(n_rows * batch), s)) != cudaSuccess) return e;
    e = launch_scan(sj.data(), n_jobs, plan, (int)mc, reinterpret_cast<float *const (*)[2]>(sc.data()),
                    scores_stride, fp, s);
    if (e != cudaSuccess) return e;
    return launch_select(plan, (int)mc, fp, s, nullptr);
}

}  // namespace

extern "C" {

int32_t csa2_version(void) { return 200; }

int64_t csa2_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

const char *csa2_last_error(void) { return g_err.c_str(); }

size_t csa2_cache_bytes(int32_t format, int64_t n_slots)
{
    if (n_slots <= 0) return 0;
    switch (format) {
    case CSA2_FMT_FP4_KV: return (size_t)n_slots * kKvRow;
    case CSA2_FMT_FP4_IDX: return (n_slots % kIdxTile) ? 0 : (size_t)(n_slots / kIdxTile) * kIdxTileBytes;
    case CSA2_FMT_FP8_SWA: return (n_slots % 4) ? 0 : (size_t)n_slots * (kDim + 4);
    default: return 0;
    }
}

csa2_status csa2_set_phase_events(void *const *events, int32_t n)
{
    if (n < 0 || n > 8 || (n > 0 && !events)) return fail(CSA2_ERR_INVALID_ARG, "phase events: n must be 0..8");
    for (int i = 0; i < 8; ++i) g_events[i] = (i < n) ? events[i] : nullptr;
    g_n_events = n;
    return CSA2_OK;
}

csa2_status csa2_check_device(void *stream)
{
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "device flag word unavailable");
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cudaStreamSynchronize");
    int flags = 0;
    e = cudaMemcpy(&flags, fp, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "read device flags");
    const int zero = 0;
    e = cudaMemcpy(fp, &zero, sizeof(int), cudaMemcpyHostToDevice);
    if (e != cudaSuccess) return cuda_fail(e, "clear device flags");
    g_last_flags = flags;
    if (flags & kFlagTimeout) return fail(CSA2_ERR_TIMEOUT, "a bounded device wait gave up");
    if (flags & kFlagBounds) return fail(CSA2_ERR_INVALID_ARG, "an index, page or slot was out of range and skipped");
    return CSA2_OK;
}

int32_t csa2_last_device_flags(void) { return g_last_flags; }

csa2_status csa2_quantize_kv(const float *src, int32_t n_seqs, int64_t rows_per_seq, const int32_t *start_pos,
                             const int32_t *seq_lens, const csa2_cache *dst, void *stream)
{
    if (!dst) return fail(CSA2_ERR_INVALID_ARG, "dst is NULL");
    if (n_seqs < 0 || rows_per_seq < 0) return fail(CSA2_ERR_INVALID_ARG, "negative size");
    if (n_seqs == 0 || rows_per_seq == 0) return CSA2_OK;
    if (!src || !aligned(src, 16)) return fail(CSA2_ERR_INVALID_ARG, "src NULL or not 16-byte aligned");
    const int fmt = dst->format;
    if (fmt != CSA2_FMT_FP4_KV && fmt != CSA2_FMT_FP4_IDX && fmt != CSA2_FMT_FP8_SWA)
        return fail(CSA2_ERR_INVALID_ARG, "dst: unknown format %d", fmt);
    csa2_status st = check_cache(dst, fmt, n_seqs, fmt == CSA2_FMT_FP8_SWA ? 1 : 0, "dst");
    if (st) return st;
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    QuantJob job;
    job.src = src;
    job.start_pos = start_pos;
    job.seq_lens = seq_lens;
    job.dst = view_of(*dst);
    job.rows_per_seq = rows_per_seq;
    job.n_seqs = n_seqs;
    job.append_last = 0;
    cudaError_t e = launch_quantize(&job, 1, fp, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "quantize launch");
}

size_t csa2_index_topk_workspace(int32_t batch, int32_t max_seq_len, int32_t pool_len, int32_t topk,
                                 int32_t pool_out_len)
{
    (void)topk;
    (void)pool_out_len;
    if (batch <= 0 || max_seq_len < 1) return 0;
    IdxJob j;
    memset(&j, 0, sizeof(j));
    j.n_q = 1;
    static const int32_t any_pool = 0;
    j.pool = pool_len > 0 ? &any_pool : nullptr;
    j.pool_len = pool_len;
    const LevelWs lw = level_ws(&j, 1, batch, max_seq_len);
    return lw.fused_bytes + lw.old_bytes;
}

csa2_status csa2_index_topk(int32_t mode, const csa2_cache *keys, const float *q_idx, const float *w,
                            int32_t batch, int32_t n_heads, int32_t head_dim, const int32_t *seq_lens,
                            int32_t max_seq_len, const int32_t *pool, int32_t pool_len, int32_t topk,
                            int32_t *out_idx, int32_t *out_pool, int32_t pool_out_len, float *out_scores,
                            void *workspace, size_t workspace_bytes, void *stream)
{
    if (mode != CSA2_MODE_FULL && mode != CSA2_MODE_REINDEX)
        return fail(CSA2_ERR_INVALID_ARG, "mode must be FULL or REINDEX");
    if (n_heads != kIdxHeads || head_dim != kIdxDim)
        return fail(CSA2_ERR_UNSUPPORTED, "indexer must be 4 heads x 64 channels (got %d x %d)", n_heads, head_dim);
    if (batch <= 0 || batch > 65535) return fail(CSA2_ERR_INVALID_ARG, "batch must be in [1, 65535]");
    if (max_seq_len < 1 || max_seq_len > (1 << 24)) return fail(CSA2_ERR_INVALID_ARG, "max_seq_len must be in [1, 2^24]");
    if (topk < 1 || topk > 65536) return fail(CSA2_ERR_INVALID_ARG, "topk must be in [1, 65536]");
    if (!q_idx || !w || !seq_lens || !out_idx) return fail(CSA2_ERR_INVALID_ARG, "q_idx, w, seq_lens, out_idx are required");
    if (pool && (pool_len < 1 || pool_len > (1 << 24))) return fail(CSA2_ERR_INVALID_ARG, "pool_len must be in [1, 2^24]");
    if (out_pool && (mode != CSA2_MODE_FULL || pool_out_len < 1 || pool_out_len > 65536))
        return fail(CSA2_ERR_INVALID_ARG, "out_pool needs mode FULL and pool_out_len in [1, 65536]");
    csa2_status st = check_cache(keys, CSA2_FMT_FP4_IDX, batch, max_seq_len, "keys");
    if (st) return st;
    IdxJob j;
    memset(&j, 0, sizeof(j));
    j.keys = keys;
    j.pool = pool;
    j.pool_len = pool ? pool_len : 0;
    j.n_q = 1;
    j.q_idx[0] = q_idx;
    j.w[0] = w;
    j.out_idx[0] = out_idx;
    j.out_pool[0] = out_pool;
    j.out_scores[0] = out_scores;
    const LevelWs lw = level_ws(&j, 1, batch, max_seq_len);
    st = check_ws(workspace, workspace_bytes, lw.fused_bytes + lw.old_bytes);
    if (st) return st;
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    const int64_t stride = pool ? pool_len : max_seq_len;
    cudaError_t e = run_level(&j, 1, lw, batch, seq_lens, max_seq_len, topk, out_pool ? pool_out_len : 0, stride, ws,
                              ws + lw.fused_bytes, fp, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "index launch");
}

size_t csa2_index_topk_multi_workspace(int32_t batch, int32_t n_q, int32_t max_seq_len)
{
    if (batch <= 0 || n_q <= 0 || max_seq_len < 1 || (int64_t)batch * n_q > 65535) return 0;
    return index_multi_bytes(batch, n_q, max_seq_len);
}

csa2_status csa2_index_topk_multi(const csa2_cache *keys, const float *q_idx, const float *w, int32_t batch,
                                  int32_t n_q, int32_t n_heads, int32_t head_dim, const int32_t *seq_lens,
                                  int32_t max_seq_len, int32_t causal, int32_t topk, int32_t *out_idx,
                                  float *out_scores, void *workspace, size_t workspace_bytes, void *stream)
{
    if (n_heads != kIdxHeads || head_dim != kIdxDim)
        return fail(CSA2_ERR_UNSUPPORTED, "indexer must be 4 heads x 64 channels (got %d x %d)", n_heads, head_dim);
    if (batch <= 0 || n_q <= 0 || n_q > 4096 || (int64_t)batch * n_q > 65535)
        return fail(CSA2_ERR_INVALID_ARG, "need batch >= 1, n_q in [1, 4096] and batch * n_q <= 65535");
    if (max_seq_len < 1 || max_seq_len > (1 << 24)) return fail(CSA2_ERR_INVALID_ARG, "max_seq_len must be in [1, 2^24]");
    if (causal != 0 && causal != 1) return fail(CSA2_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!q_idx || !w || !seq_lens) return fail(CSA2_ERR_INVALID_ARG, "q_idx, w, seq_lens are required");
    if (!out_idx && !out_scores) return fail(CSA2_ERR_INVALID_ARG, "nothing to compute: out_idx and out_scores are NULL");
    if (out_idx && (topk < 1 || topk > 65536)) return fail(CSA2_ERR_INVALID_ARG, "topk must be in [1, 65536]");
    if (!aligned(q_idx, 16)) return fail(CSA2_ERR_INVALID_ARG, "q_idx must be 16-byte aligned");
    csa2_status st = check_cache(keys, CSA2_FMT_FP4_IDX, batch, max_seq_len, "keys");
    if (st) return st;
    st = check_ws(workspace, workspace_bytes, index_multi_bytes(batch, n_q, max_seq_len));
    if (st) return st;
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    cudaError_t e = run_index_multi(view_of(*keys), q_idx, w, batch, n_q, seq_lens, max_seq_len, causal, topk, out_idx,
                                    out_scores, static_cast<uint8_t *>(workspace), fp,
                                    static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "multi-query index launch");
}

size_t csa2_sparse_attn_workspace(int32_t batch, int32_t topk, int32_t swa_window)
{
    return csa2::sparse_attn_workspace_within(batch, topk, swa_window, SIZE_MAX);
}

csa2_status csa2_sparse_attn(const csa2_cache *kv, const csa2_cache *swa, const float *q, int32_t batch,
                             int32_t n_heads, int32_t head_dim, const int32_t *seq_lens, int32_t max_seq_len,
                             const int32_t *idx, int32_t topk, int32_t swa_window, float *out, float *lse,
                             void *workspace, size_t workspace_bytes, void *stream)
{
    if (n_heads != kHeads || head_dim != kDim)
        return fail(CSA2_ERR_UNSUPPORTED, "attention must be 16 heads x 512 channels (got %d x %d)", n_heads, head_dim);
    if (batch <= 0 || batch > 65535) return fail(CSA2_ERR_INVALID_ARG, "batch must be in [1, 65535]");
    if (max_seq_len < 0 || max_seq_len > (1 << 24)) return fail(CSA2_ERR_INVALID_ARG, "max_seq_len must be in [0, 2^24]");
    if (!q || !out || !seq_lens) return fail(CSA2_ERR_INVALID_ARG, "q, out, seq_lens are required");
    if (!aligned(q, 16) || !aligned(out, 16)) return fail(CSA2_ERR_INVALID_ARG, "q and out must be 16-byte aligned");
    if (topk < 0 || topk > 65536) return fail(CSA2_ERR_INVALID_ARG, "topk must be in [0, 65536]");
    if (swa_window < 0 || swa_window > 65536) return fail(CSA2_ERR_INVALID_ARG, "swa_window must be in [0, 65536]");
    csa2_status st;
    if (idx) {
        st = check_cache(kv, CSA2_FMT_FP4_KV, batch, max_seq_len, "kv");
        if (st) return st;
    }
    if (swa_window > 0) {
        st = check_cache(swa, CSA2_FMT_FP8_SWA, batch, swa_window, "swa");
        if (st) return st;
    }
    if (workspace && !aligned(workspace, 256)) return fail(CSA2_ERR_WORKSPACE, "workspace must be 256-byte aligned");
    const int eff_topk = idx ? topk : 0;
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    AttnEntry en;
    memset(&en, 0, sizeof(en));
    if (idx) en.kv = view_of(*kv);
    if (swa_window > 0) en.swa = view_of(*swa);
    en.q = q;
    en.idx = idx;
    en.out = out;
    en.lse = lse;
    en.has_kv = idx ? 1 : 0;
    en.has_swa = swa_window > 0 ? 1 : 0;
    AttnPlan plan;
    memset(&plan, 0, sizeof(plan));  // inputs_ready 0: the caller's indices may come from the previous kernel
    plan.entries = &en;
    plan.n_entries = 1;
    plan.batch = batch;
    plan.topk = eff_topk;
    plan.window = swa_window;
    plan.seq_lens = seq_lens;
    plan.max_group = 1;
    plan.pdl = 1;
    plan.workspace = workspace;
    plan.workspace_bytes = workspace ? workspace_bytes : 0;
    cudaError_t e = launch_attention(plan, fp, static_cast<cudaStream_t>(stream), nullptr);
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "attention launch");
}

// ---- decode step ------------------------------------------------------------

namespace {

// Attention entries of a step, one per layer (sources already validated).
std::vector<AttnEntry> step_entries(const csa2_layer_desc *layers, int n_layers, int swa_window)
{
    std::vector<AttnEntry> entries(n_layers);
    for (int l = 0; l < n_layers; ++l) {
        const csa2_layer_desc &d = layers[l];
        AttnEntry &en = entries[l];
        memset(&en, 0, sizeof(en));
        en.q = d.q;
        en.out = d.out;
        en.lse = d.lse;
        en.has_swa = swa_window > 0 ? 1 : 0;
        if (swa_window > 0) {
            en.swa = view_of(*d.swa);
            en.new_swa = d.new_swa;
        }
        if (d.mode != CSA2_MODE_SWA_ONLY) {
            en.kv = view_of(*layers[d.kv_src].kv);
            en.has_kv = 1;
            en.idx = (d.mode == CSA2_MODE_REUSE) ? layers[d.idx_src].idx_out : d.idx_out;
        }
    }
    return entries;
}

// Checks layer l of a schedule and the sources it names.
csa2_status check_layer(const csa2_layer_desc *layers, int32_t l, int32_t batch, int32_t max_seq_len,
                        int32_t pool_len, int32_t swa_window)
{
    const csa2_layer_desc &d = layers[l];
    char name[32];
    snprintf(name, sizeof(name), "layer %d", l);
    if (!d.q || !d.out || !aligned(d.q, 16) || !aligned(d.out, 16))
        return fail(CSA2_ERR_INVALID_ARG, "%s: q/out NULL or not 16-byte aligned", name);
    if (swa_window > 0) {
        csa2_status st = check_cache(d.swa, CSA2_FMT_FP8_SWA, batch, swa_window, name);
        if (st) return st;
    }
    if (d.new_swa && (!d.swa || !aligned(d.new_swa, 16)))
        return fail(CSA2_ERR_INVALID_ARG, "%s: new_swa needs swa and 16-byte alignment", name);
    switch (d.mode) {
    case CSA2_MODE_FULL: {
        if (d.kv_src != l) return fail(CSA2_ERR_INVALID_ARG, "%s: FULL kv_src must be its own index", name);
        csa2_status st = check_cache(d.kv, CSA2_FMT_FP4_KV, batch, max_seq_len, name);
        if (st) return st;
        st = check_cache(d.idx_keys, CSA2_FMT_FP4_IDX, batch, max_seq_len, name);
        if (st) return st;
        if (!d.q_idx || !d.w || !d.idx_out) return fail(CSA2_ERR_INVALID_ARG, "%s: q_idx, w, idx_out required", name);
        if (pool_len > 0 && !d.pool_out) return fail(CSA2_ERR_INVALID_ARG, "%s: pool_out required when pool_len > 0", name);
        if ((d.new_kv && !aligned(d.new_kv, 16)) || (d.new_idx_key && !aligned(d.new_idx_key, 16)))
            return fail(CSA2_ERR_INVALID_ARG, "%s: new rows must be 16-byte aligned", name);
        break;
    }
    case CSA2_MODE_REINDEX:
    case CSA2_MODE_REUSE: {
        if (d.kv_src < 0 || d.kv_src >= l || layers[d.kv_src].mode != CSA2_MODE_FULL)
            return fail(CSA2_ERR_INVALID_ARG, "%s: kv_src must name an earlier FULL layer", name);
        if (d.mode == CSA2_MODE_REINDEX) {
            if (!d.q_idx || !d.w || !d.idx_out) return fail(CSA2_ERR_INVALID_ARG, "%s: q_idx, w, idx_out required", name);
            if (d.use_pool && pool_len <= 0) return fail(CSA2_ERR_INVALID_ARG, "%s: use_pool needs pool_len > 0", name);
        } else {
            if (d.idx_src < 0 || d.idx_src >= l ||
                (layers[d.idx_src].mode != CSA2_MODE_FULL && layers[d.idx_src].mode != CSA2_MODE_REINDEX))
                return fail(CSA2_ERR_INVALID_ARG, "%s: idx_src must name an earlier FULL/REINDEX layer", name);
            if (layers[d.idx_src].mode == CSA2_MODE_REINDEX && layers[d.idx_src].kv_src != d.kv_src)
                return fail(CSA2_ERR_INVALID_ARG, "%s: idx_src indexes a different KV cache", name);
            if (layers[d.idx_src].mode == CSA2_MODE_FULL && d.idx_src != d.kv_src)
                return fail(CSA2_ERR_INVALID_ARG, "%s: idx_src indexes a different KV cache", name);
        }
        break;
    }
    case CSA2_MODE_SWA_ONLY:
        if (swa_window <= 0) return fail(CSA2_ERR_INVALID_ARG, "%s: SWA_ONLY needs swa_window > 0", name);
        break;
    default: return fail(CSA2_ERR_INVALID_ARG, "%s: unknown mode %d", name, d.mode);
    }
    return CSA2_OK;
}

csa2_status check_sizes(int32_t batch, int32_t max_seq_len, int32_t topk, int32_t pool_len, int32_t swa_window)
{
    if (batch <= 0 || batch > 65535) return fail(CSA2_ERR_INVALID_ARG, "batch must be in [1, 65535]");
    if (max_seq_len < 1 || max_seq_len > (1 << 24)) return fail(CSA2_ERR_INVALID_ARG, "max_seq_len must be in [1, 2^24]");
    if (topk < 1 || topk > 65536) return fail(CSA2_ERR_INVALID_ARG, "topk must be in [1, 65536]");
    if (pool_len < 0 || pool_len > 65536) return fail(CSA2_ERR_INVALID_ARG, "pool_len must be in [0, 65536]");
    if (swa_window < 0 || swa_window > 65536) return fail(CSA2_ERR_INVALID_ARG, "swa_window must be in [0, 65536]");
    return CSA2_OK;
}

// The indexing job of layer l (FULL or REINDEX), alone or joined to `open`
// when it scores the same keys and candidates (at most two queries a job).
void add_index_job(const csa2_layer_desc *layers, int l, int32_t pool_len, std::vector<IdxJob> &jobs)
{
    const csa2_layer_desc &d = layers[l];
    const int f = d.kv_src;
    const bool use_pool = d.mode == CSA2_MODE_REINDEX && d.use_pool;
    const int32_t *pool = use_pool ? layers[f].pool_out : nullptr;
    for (IdxJob &j : jobs) {
        if (j.n_q == 1 && j.keys->data == layers[f].idx_keys->data && j.pool == pool) {
            j.q_idx[1] = d.q_idx;
            j.w[1] = d.w;
            j.out_idx[1] = d.idx_out;
            j.out_pool[1] = (d.mode == CSA2_MODE_FULL && pool_len > 0) ? d.pool_out : nullptr;
            j.n_q = 2;
            if (d.mode == CSA2_MODE_FULL) {
                j.kv = d.kv;
                j.new_kv = d.new_kv;
                j.new_key = d.new_idx_key;
            }
            return;
        }
    }
    IdxJob j;
    memset(&j, 0, sizeof(j));
    j.keys = layers[f].idx_keys;
    j.pool = pool;
    j.pool_len = pool ? pool_len : 0;
    j.n_q = 1;
    j.q_idx[0] = d.q_idx;
    j.w[0] = d.w;
    j.out_idx[0] = d.idx_out;
    j.out_pool[0] = (d.mode == CSA2_MODE_FULL && pool_len > 0) ? d.pool_out : nullptr;
    if (d.mode == CSA2_MODE_FULL) {
        j.kv = d.kv;
        j.new_kv = d.new_kv;
        j.new_key = d.new_idx_key;
    }
    j.warm = layers[f].kv;  // every query of the job gathers from the keys' Full layer
    jobs.push_back(j);
}

// The per-layer call's workspace: [indexing region][attention region].
size_t layer_attn_offset(size_t idx_bytes) { return round256(idx_bytes); }
size_t layer_attn_bytes(int32_t batch, int32_t topk, int32_t swa_window)
{
    return round256(std::max(sparse_attn_workspace_within(batch, topk, swa_window, SIZE_MAX),
                             sparse_attn_workspace_within(batch, 0, swa_window, SIZE_MAX)));
}

// One decode step in the phased order: level 0 (Full layers and pool-free
// Reindex layers), level 1 (pool-restricted Reindex layers), then the
// attention of every layer.
struct StepLayout {
    std::vector<IdxJob> level[2];
    LevelWs lw[2];
    size_t fused_bytes = 0, old_bytes = 0, attn_bytes = 0, total = 0;
};

AttnPlan step_attn_plan(const std::vector<AttnEntry> &entries, int32_t batch, const int32_t *seq_lens, int32_t topk,
                        int32_t swa_window, void *ws, size_t ws_bytes)
{
    AttnPlan ap;
    memset(&ap, 0, sizeof(ap));
    ap.entries = entries.data();
    ap.n_entries = (int)entries.size();
    ap.batch = batch;
    ap.topk = topk;
    ap.window = swa_window;
    ap.seq_lens = seq_lens;
    ap.max_group = 2;
    ap.pdl = 1;
    ap.workspace = ws;
    ap.workspace_bytes = ws_bytes;
    return ap;
}

csa2_status plan_step(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch, int32_t max_seq_len,
                      int32_t topk, int32_t pool_len, int32_t swa_window, StepLayout &P)
{
    if (!layers || n_layers <= 0) return fail(CSA2_ERR_INVALID_ARG, "no layers");
    csa2_status st = check_sizes(batch, max_seq_len, topk, pool_len, swa_window);
    if (st) return st;
    if (n_layers > kMaxAttnEntries) return fail(CSA2_ERR_UNSUPPORTED, "at most %d layers per step", kMaxAttnEntries);
    for (int l = 0; l < n_layers; ++l) {
        st = check_layer(layers, l, batch, max_seq_len, pool_len, swa_window);
        if (st) return st;
    }
    for (int l = 0; l < n_layers; ++l) {
        const csa2_layer_desc &d = layers[l];
        if (d.mode != CSA2_MODE_FULL && d.mode != CSA2_MODE_REINDEX) continue;
        const int level = (d.mode == CSA2_MODE_REINDEX && d.use_pool) ? 1 : 0;
        add_index_job(layers, l, pool_len, P.level[level]);
    }
    for (int lv = 0; lv < 2; ++lv) {
        int rows = 0;
        for (const IdxJob &j : P.level[lv]) rows += j.n_q;
        if (rows > kMaxSelectRows) return fail(CSA2_ERR_UNSUPPORTED, "at most %d indexing layers per level", kMaxSelectRows);
        P.lw[lv] = level_ws(P.level[lv].data(), (int)P.level[lv].size(), batch, max_seq_len);
        P.fused_bytes = std::max(P.fused_bytes, P.lw[lv].fused_bytes);
        P.old_bytes = std::max(P.old_bytes, P.lw[lv].old_bytes);
    }
    {
        const std::vector<AttnEntry> entries = step_entries(layers, n_layers, swa_window);
        P.attn_bytes = round256(attn_workspace_bytes(step_attn_plan(entries, batch, nullptr, topk, swa_window, nullptr, 0)));
    }
    P.total = P.fused_bytes + P.old_bytes + P.attn_bytes;
    return CSA2_OK;
}

}  // namespace

size_t csa2_decode_layers_workspace(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch,
                                    int32_t max_seq_len, int32_t topk, int32_t pool_len, int32_t swa_window)
{
    StepLayout P;
    if (plan_step(layers, n_layers, batch, max_seq_len, topk, pool_len, swa_window, P) != CSA2_OK) return 0;
    return std::max<size_t>(P.total, 256);
}

csa2_status csa2_decode_layers(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch,
                               const int32_t *seq_lens, int32_t max_seq_len, int32_t topk, int32_t pool_len,
                               int32_t swa_window, void *workspace, size_t workspace_bytes, void *stream)
{
    StepLayout P;
    csa2_status st = plan_step(layers, n_layers, batch, max_seq_len, topk, pool_len, swa_window, P);
    if (st) return st;
    if (!seq_lens) return fail(CSA2_ERR_INVALID_ARG, "seq_lens is required");
    st = check_ws(workspace, workspace_bytes, P.total);
    if (st) return st;
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    uint8_t *ws = static_cast<uint8_t *>(workspace);
    cudaError_t e;
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "event");
    for (int lv = 0; lv < 2; ++lv) {
        if (!P.level[lv].empty()) {
            e = run_level(P.level[lv].data(), (int)P.level[lv].size(), P.lw[lv], batch, seq_lens, max_seq_len, topk,
                          lv == 0 ? pool_len : 0, 0, ws, ws + P.fused_bytes, fp, s);
            if (e != cudaSuccess) return cuda_fail(e, "index launch");
        }
        if (lv == 0 && ((e = mark(1, s)) != cudaSuccess || (e = mark(2, s)) != cudaSuccess)) return cuda_fail(e, "event");
    }
    if ((e = mark(3, s)) != cudaSuccess) return cuda_fail(e, "event");
    std::vector<AttnEntry> entries = step_entries(layers, n_layers, swa_window);
    const AttnPlan ap = step_attn_plan(entries, batch, seq_lens, topk, swa_window,
                                       P.attn_bytes ? ws + P.fused_bytes + P.old_bytes : nullptr, P.attn_bytes);
    e = launch_attention(ap, fp, s, nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    if ((e = mark(4, s)) != cudaSuccess || (e = mark(5, s)) != cudaSuccess) return cuda_fail(e, "event");
    return CSA2_OK;
}

size_t csa2_decode_layer_workspace(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch,
                                   int32_t max_seq_len, int32_t topk, int32_t pool_len, int32_t swa_window)
{
    if (!layers || n_layers <= 0 || check_sizes(batch, max_seq_len, topk, pool_len, swa_window)) return 0;
    size_t idx_need = 0;
    for (int l = 0; l < n_layers; ++l) {
        if (check_layer(layers, l, batch, max_seq_len, pool_len, swa_window)) return 0;
        const csa2_layer_desc &d = layers[l];
        if (d.mode != CSA2_MODE_FULL && d.mode != CSA2_MODE_REINDEX) continue;
        std::vector<IdxJob> jobs;
        add_index_job(layers, l, pool_len, jobs);
        const LevelWs lw = level_ws(jobs.data(), 1, batch, max_seq_len);
        idx_need = std::max(idx_need, lw.fused_bytes + lw.old_bytes);
    }
    return std::max<size_t>(256, layer_attn_offset(idx_need) + layer_attn_bytes(batch, topk, swa_window));
}

csa2_status csa2_decode_layer(const csa2_layer_desc *layers, int32_t n_layers, int32_t layer, int32_t batch,
                              const int32_t *seq_lens, int32_t max_seq_len, int32_t topk, int32_t pool_len,
                              int32_t swa_window, void *workspace, size_t workspace_bytes, void *stream)
{
    if (!layers || n_layers <= 0 || layer < 0 || layer >= n_layers)
        return fail(CSA2_ERR_INVALID_ARG, "layer %d outside the schedule of %d layers", layer, n_layers);
    csa2_status st = check_sizes(batch, max_seq_len, topk, pool_len, swa_window);
    if (st) return st;
    st = check_layer(layers, layer, batch, max_seq_len, pool_len, swa_window);
    if (st) return st;
    if (!seq_lens) return fail(CSA2_ERR_INVALID_ARG, "seq_lens is required");
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const csa2_layer_desc &d = layers[layer];
    cudaError_t e;
    if (d.mode == CSA2_MODE_FULL || d.mode == CSA2_MODE_REINDEX) {
        std::vector<IdxJob> jobs;
        add_index_job(layers, layer, pool_len, jobs);
        const LevelWs lw = level_ws(jobs.data(), 1, batch, max_seq_len);
        st = check_ws(workspace, workspace_bytes, lw.fused_bytes + lw.old_bytes);
        if (st) return st;
        uint8_t *ws = static_cast<uint8_t *>(workspace);
        // the keys were written before the previous layer's attention (a Full
        // layer's own new key is patched in by the kernel): copies start early
        e = run_level(jobs.data(), 1, lw, batch, seq_lens, max_seq_len, topk, d.mode == CSA2_MODE_FULL ? pool_len : 0, 0,
                      ws, ws + lw.fused_bytes, fp, s, 1);
        if (e != cudaSuccess) return cuda_fail(e, "index launch");
    }
    AttnEntry en;
    memset(&en, 0, sizeof(en));
    en.q = d.q;
    en.out = d.out;
    en.lse = d.lse;
    en.has_swa = swa_window > 0 ? 1 : 0;
    if (swa_window > 0) {
        en.swa = view_of(*d.swa);
        en.new_swa = d.new_swa;
    }
    if (d.mode != CSA2_MODE_SWA_ONLY) {
        en.kv = view_of(*layers[d.kv_src].kv);
        en.has_kv = 1;
        en.idx = (d.mode == CSA2_MODE_REUSE) ? layers[d.idx_src].idx_out : d.idx_out;
    }
    // the attention's region follows the largest indexing region of the schedule
    size_t idx_need = 0;
    for (int l = 0; l < n_layers; ++l) {
        const csa2_layer_desc &dl = layers[l];
        if (dl.mode != CSA2_MODE_FULL && dl.mode != CSA2_MODE_REINDEX) continue;
        std::vector<IdxJob> jobs;
        add_index_job(layers, l, pool_len, jobs);
        const LevelWs lw = level_ws(jobs.data(), 1, batch, max_seq_len);
        idx_need = std::max(idx_need, lw.fused_bytes + lw.old_bytes);
    }
    const size_t a_off = layer_attn_offset(idx_need), a_bytes = layer_attn_bytes(batch, topk, swa_window);
    st = check_ws(workspace, workspace_bytes, a_off + a_bytes);
    if (st) return st;
    AttnPlan ap;
    memset(&ap, 0, sizeof(ap));
    ap.entries = &en;
    ap.n_entries = 1;
    ap.batch = batch;
    ap.topk = d.mode == CSA2_MODE_SWA_ONLY ? 0 : topk;
    ap.window = swa_window;
    ap.seq_lens = seq_lens;
    ap.max_group = 1;
    ap.pdl = 1;
    // a Reuse layer's indices come from an earlier layer's call and an SWA-only
    // layer has none; its caches and ring were written before the previous
    // layer's attention: the first tile is gathered before the wait for it
    ap.inputs_ready = (d.mode == CSA2_MODE_REUSE || d.mode == CSA2_MODE_SWA_ONLY) ? 1 : 0;
    ap.workspace = a_bytes ? static_cast<uint8_t *>(workspace) + a_off : nullptr;
    ap.workspace_bytes = a_bytes;
    e = launch_attention(ap, fp, s, nullptr);
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "attention launch");
}

csa2_status csa2_test_set_wait_limit(int32_t polls)
{
    fused_set_first_wait_limit(polls);
    return CSA2_OK;
}

}  // extern "C"
