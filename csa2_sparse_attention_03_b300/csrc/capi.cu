// C interface of the CSA2 decode hot path: argument checks, workspace
// planning and the enqueue order of one decode step over a static layer-mode
// schedule (Helmcode "DeepSeek V4.1 Flash" explainer, "03 · CSA2": Full,
// Reindex, Reuse and SWA-only layers; Louis Bouchard's KV-cache report,
// "Share the cache and the search work": pool-restricted Reindex).
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
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

// bytes at the head of a select region that are zeroed per call (the histograms)
size_t select_head_bytes(int n_rows) { return select_hist_bytes(n_rows); }

}  // namespace

namespace csa2 {

size_t sparse_attn_workspace_within(int32_t batch, int32_t topk, int32_t swa_window, size_t budget)
{
    if (batch <= 0 || topk < 0 || swa_window < 0) return 0;
    static const int32_t any_index = 0;  // stands for "an index list is given"
    AttnEntry en;
    memset(&en, 0, sizeof(en));
    en.has_kv = topk > 0 ? 1 : 0;
    en.idx = topk > 0 ? &any_index : nullptr;
    en.has_swa = swa_window > 0 ? 1 : 0;
    return attn_workspace_bytes(&en, 1, batch, topk, swa_window, budget);
}

}  // namespace csa2

extern "C" {

int32_t csa2_version(void) { return 100; }

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
    if (batch <= 0 || max_seq_len < 0) return 0;
    const int64_t cap = max_seq_len > pool_len ? max_seq_len : pool_len;
    return select_bytes(batch, cap > 0 ? cap : 1, max_seq_len > 0 ? max_seq_len : 1);
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
    const size_t need = csa2_index_topk_workspace(batch, max_seq_len, pool ? pool_len : 0, topk, pool_out_len);
    st = check_ws(workspace, workspace_bytes, need);
    if (st) return st;
    int *fp = flags_ptr();
    if (!fp) return fail(CSA2_ERR_CUDA, "no CUDA device");
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    const int64_t cap = max_seq_len > pool_len ? max_seq_len : (pool ? pool_len : max_seq_len);
    SelectPlan plan;
    memset(&plan, 0, sizeof(plan));
    plan.bufs = carve_select(static_cast<uint8_t *>(workspace), batch, cap, max_seq_len);
    plan.n_row_blocks = 1;
    plan.batch = batch;
    plan.topk = topk;
    plan.pool_out_len = out_pool ? pool_out_len : 0;
    plan.max_len = max_seq_len;
    plan.seq_lens = seq_lens;
    plan.rows[0].out_idx = out_idx;
    plan.rows[0].out_pool = out_pool;
    plan.rows[0].pool = pool;
    plan.rows[0].pool_len = pool ? pool_len : 0;

    ScanJob job;
    memset(&job, 0, sizeof(job));
    job.keys = view_of(*keys);
    job.q_idx[0] = q_idx;
    job.w[0] = w;
    job.pool = pool;
    job.pool_len = pool ? pool_len : 0;
    job.n_q = 1;
    job.row[0] = 0;
    float *scores[1][2] = {{out_scores, nullptr}};
    const int max_cand = pool ? pool_len : max_seq_len;

    cudaError_t e = cudaMemsetAsync(workspace, 0, select_head_bytes(batch), s);
    if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
    e = launch_scan(&job, 1, plan, max_cand, scores, max_cand, fp, s);
    if (e != cudaSuccess) return cuda_fail(e, "scan launch");
    e = launch_select(plan, max_cand, fp, s, nullptr);
    return e == cudaSuccess ? CSA2_OK : cuda_fail(e, "select launch");
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
    st = check_ws(workspace, workspace_bytes, attn_workspace_bytes(&en, 1, batch, eff_topk, swa_window, workspace_bytes));
    if (st) return st;
    AttnPlan plan;
    plan.entries = &en;
    plan.n_entries = 1;
    plan.batch = batch;
    plan.topk = eff_topk;
    plan.window = swa_window;
    plan.seq_lens = seq_lens;
    plan.workspace = workspace;
    plan.workspace_bytes = workspace_bytes;
    plan.q_packed = 0;
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
        if (swa_window > 0) en.swa = view_of(*d.swa);
        if (d.mode != CSA2_MODE_SWA_ONLY) {
            en.kv = view_of(*layers[d.kv_src].kv);
            en.has_kv = 1;
            en.idx = (d.mode == CSA2_MODE_REUSE) ? layers[d.idx_src].idx_out : d.idx_out;
        }
    }
    return entries;
}

struct StepLayout {
    int n_idx = 0;              // indexing layers (FULL + REINDEX)
    std::vector<int> row_block; // per layer: row block id or -1
    int n_level0 = 0, n_level1 = 0;
    int64_t cand_cap = 1;
    size_t select_off = 0, select_size = 0, part_off = 0, part_size = 0, total = 0;
};

csa2_status plan_step(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch, int32_t max_seq_len,
                      int32_t topk, int32_t pool_len, int32_t swa_window, StepLayout &P)
{
    if (!layers || n_layers <= 0) return fail(CSA2_ERR_INVALID_ARG, "no layers");
    if (batch <= 0 || batch > 65535) return fail(CSA2_ERR_INVALID_ARG, "batch must be in [1, 65535]");
    if (max_seq_len < 1 || max_seq_len > (1 << 24)) return fail(CSA2_ERR_INVALID_ARG, "max_seq_len must be in [1, 2^24]");
    if (topk < 1 || topk > 65536) return fail(CSA2_ERR_INVALID_ARG, "topk must be in [1, 65536]");
    if (pool_len < 0 || pool_len > 65536) return fail(CSA2_ERR_INVALID_ARG, "pool_len must be in [0, 65536]");
    if (swa_window < 0 || swa_window > 65536) return fail(CSA2_ERR_INVALID_ARG, "swa_window must be in [0, 65536]");
    P.row_block.assign(n_layers, -1);
    // level 0: FULL and pool-free REINDEX; level 1: pool-restricted REINDEX
    for (int pass = 0; pass < 2; ++pass)
        for (int l = 0; l < n_layers; ++l) {
            const csa2_layer_desc &d = layers[l];
            const bool lvl1 = d.mode == CSA2_MODE_REINDEX && d.use_pool;
            if ((d.mode == CSA2_MODE_FULL || d.mode == CSA2_MODE_REINDEX) && (lvl1 == (pass == 1))) {
                P.row_block[l] = P.n_idx++;
                (pass == 0 ? P.n_level0 : P.n_level1)++;
            }
        }
    if (P.n_level0 > kMaxSelectRows || P.n_level1 > kMaxSelectRows)
        return fail(CSA2_ERR_UNSUPPORTED, "at most %d indexing layers per level", kMaxSelectRows);
    for (int l = 0; l < n_layers; ++l) {
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
    }
    P.cand_cap = max_seq_len > pool_len ? max_seq_len : pool_len;
    P.select_off = 0;
    P.select_size = P.n_idx ? round256(select_bytes(P.n_idx * batch, P.cand_cap, max_seq_len)) : 0;
    P.part_off = P.select_size;
    if (n_layers > kMaxAttnEntries) return fail(CSA2_ERR_UNSUPPORTED, "at most %d layers per step", kMaxAttnEntries);
    {
        const std::vector<AttnEntry> entries = step_entries(layers, n_layers, swa_window);
        P.part_size = round256(attn_workspace_bytes(entries.data(), n_layers, batch, topk, swa_window));
    }
    P.total = P.part_off + P.part_size;
    return CSA2_OK;
}

}  // namespace

size_t csa2_decode_layers_workspace(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch,
                                    int32_t max_seq_len, int32_t topk, int32_t pool_len, int32_t swa_window)
{
    StepLayout P;
    if (plan_step(layers, n_layers, batch, max_seq_len, topk, pool_len, swa_window, P) != CSA2_OK) return 0;
    return P.total;
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

    // appends (quantise-and-write the new token of each Full layer and each SWA ring)
    std::vector<QuantJob> qjobs;
    auto add_append = [&](const float *src, const csa2_cache *c) {
        QuantJob j;
        j.src = src;
        j.start_pos = nullptr;
        j.seq_lens = seq_lens;
        j.dst = view_of(*c);
        j.rows_per_seq = 1;
        j.n_seqs = batch;
        j.append_last = 1;
        qjobs.push_back(j);
    };
    for (int l = 0; l < n_layers; ++l) {
        const csa2_layer_desc &d = layers[l];
        if (d.mode == CSA2_MODE_FULL && d.new_kv) add_append(d.new_kv, d.kv);
        if (d.mode == CSA2_MODE_FULL && d.new_idx_key) add_append(d.new_idx_key, d.idx_keys);
        if (d.new_swa && swa_window > 0) add_append(d.new_swa, d.swa);
    }
    // the attention's queries to fp16 ride in the same launch
    std::vector<AttnEntry> entries = step_entries(layers, n_layers, swa_window);
    AttnPlan ap;
    ap.entries = entries.data();
    ap.n_entries = n_layers;
    ap.batch = batch;
    ap.topk = topk;
    ap.window = swa_window;
    ap.seq_lens = seq_lens;
    ap.workspace = ws + P.part_off;
    ap.workspace_bytes = P.part_size;
    ap.q_packed = 1;
    {
        const size_t n0 = qjobs.size();
        qjobs.resize(n0 + (size_t)n_layers);
        qjobs.resize(n0 + (size_t)attn_pack_jobs(ap, qjobs.data() + n0, n_layers));
    }
    if (P.n_idx) {
        e = cudaMemsetAsync(ws + P.select_off, 0, select_head_bytes(P.n_idx * batch), s);
        if (e != cudaSuccess) return cuda_fail(e, "workspace clear");
    }
    if (!qjobs.empty()) {
        e = launch_quantize(qjobs.data(), (int)qjobs.size(), fp, s);
        if (e != cudaSuccess) return cuda_fail(e, "append launch");
    }
    if ((e = mark(0, s)) != cudaSuccess) return cuda_fail(e, "event");

    SelectBufs bufs;
    if (P.n_idx) bufs = carve_select(ws + P.select_off, P.n_idx * batch, P.cand_cap, max_seq_len);
    for (int level = 0; level < 2; ++level) {
        const int n_rows = level == 0 ? P.n_level0 : P.n_level1;
        if (n_rows == 0) {
            if (level == 0) {
                if ((e = mark(1, s)) != cudaSuccess || (e = mark(2, s)) != cudaSuccess) return cuda_fail(e, "event");
            }
            continue;
        }
        const int rb0 = level == 0 ? 0 : P.n_level0;
        SelectPlan plan;
        memset(&plan, 0, sizeof(plan));
        plan.bufs = bufs;
        plan.n_row_blocks = n_rows;
        plan.batch = batch;
        plan.topk = topk;
        plan.pool_out_len = (level == 0) ? pool_len : 0;
        plan.max_len = max_seq_len;
        plan.seq_lens = seq_lens;
        // rebase buffers so that plan row block i is global row block rb0 + i
        const int64_t row_off = (int64_t)rb0 * batch;
        plan.bufs.keys += row_off * bufs.cand_cap;
        plan.bufs.hist += row_off * kHistBins;
        std::vector<ScanJob> jobs;
        int max_cand = 1;
        for (int l = 0; l < n_layers; ++l) {
            const int rb = P.row_block[l];
            if (rb < rb0 || rb >= rb0 + n_rows) continue;
            const csa2_layer_desc &d = layers[l];
            SelectRow &R = plan.rows[rb - rb0];
            R.out_idx = d.idx_out;
            R.out_pool = (d.mode == CSA2_MODE_FULL && pool_len > 0) ? d.pool_out : nullptr;
            R.pool = (level == 1) ? layers[d.kv_src].pool_out : nullptr;
            R.pool_len = (level == 1) ? pool_len : 0;
            R.out_scores = nullptr;
            // pair this query with an open job over the same keys and candidates
            const int f = d.kv_src;
            const int32_t *pool = R.pool;
            bool placed = false;
            for (auto &j : jobs) {
                if (j.n_q == 1 && j.keys.data == layers[f].idx_keys->data && j.pool == pool) {
                    j.q_idx[1] = d.q_idx;
                    j.w[1] = d.w;
                    j.row[1] = rb - rb0;
                    j.n_q = 2;
                    placed = true;
                    break;
                }
            }
            if (!placed) {
                ScanJob j;
                memset(&j, 0, sizeof(j));
                j.keys = view_of(*layers[f].idx_keys);
                j.q_idx[0] = d.q_idx;
                j.w[0] = d.w;
                j.pool = pool;
                j.pool_len = pool ? pool_len : 0;
                j.n_q = 1;
                j.row[0] = rb - rb0;
                jobs.push_back(j);
            }
            const int mc = pool ? pool_len : max_seq_len;
            if (mc > max_cand) max_cand = mc;
        }
        e = launch_scan(jobs.data(), (int)jobs.size(), plan, max_cand, nullptr, 0, fp, s);
        if (e != cudaSuccess) return cuda_fail(e, "scan launch");
        if (level == 0 && (e = mark(1, s)) != cudaSuccess) return cuda_fail(e, "event");
        e = launch_select(plan, max_cand, fp, s, nullptr);
        if (e != cudaSuccess) return cuda_fail(e, "select launch");
        if (level == 0 && (e = mark(2, s)) != cudaSuccess) return cuda_fail(e, "event");
    }
    if ((e = mark(3, s)) != cudaSuccess) return cuda_fail(e, "event");

    // attention of every layer
    cudaEvent_t mid = (g_n_events > 4) ? static_cast<cudaEvent_t>(g_events[4]) : nullptr;
    e = launch_attention(ap, fp, s, mid);
    if (e != cudaSuccess) return cuda_fail(e, "attention launch");
    if ((e = mark(5, s)) != cudaSuccess) return cuda_fail(e, "event");
    return CSA2_OK;
}

}  // extern "C"
