// Host-side launchers shared between the CSA2 translation units.
#pragma once

#include "common.cuh"

namespace csa2 {

// Records a profiling event on `s`.  Inside a stream capture the record
// becomes an external event node, so the event is re-recorded (with its
// timestamp) on every replay of the captured graph.
inline cudaError_t record_event(cudaEvent_t ev, cudaStream_t s)
{
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(ev, s, cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal
                                                                               : cudaEventRecordDefault);
}

// Kernels enqueued by this library since load (process-wide, relaxed).
void count_launches(int n);

// When the environment variable CSA2_LOG is set (non-empty, not "0"), writes
// the message to stderr, each distinct message once (launch plans: cluster
// sizes, co-resident grids, fallbacks).
void log_plan(const char *fmt, ...);

// Sets the calling thread's csa2_last_error() message; returns `s`.
csa2_status set_error(csa2_status s, const char *fmt, ...);

// ---- step 1: quantise-and-write ------------------------------------------
struct QuantJob {
    const float *src;         // [n_seqs][rows_per_seq][C]
    const int32_t *start_pos; // [n_seqs] or null
    const int32_t *seq_lens;  // [n_seqs] or null
    CacheView dst;
    int64_t rows_per_seq;
    int32_t n_seqs;
    int32_t append_last;      // 1: position = seq_lens[b] - 1 (decode append)
};
constexpr int kMaxQuantJobs = 128;
// Internal job format (not a cache format): rows of 512 fp32 channels to fp16,
// dst.data = [n_seqs][rows_per_seq][512] fp16 (the attention's query rows).
constexpr int32_t kFmtPackF16 = 0x7F;
// Enqueue quantisation of every job (one launch per call).
cudaError_t launch_quantize(const QuantJob *jobs, int n_jobs, int *flags, cudaStream_t stream);

// ---- step 2: indexer scan + Top-K ----------------------------------------
// One scan job: one indexer-key cache scored by up to two indexing layers
// (a Full layer and a pool-free Reindex layer over the same keys share one
// pass over the keys).
struct ScanJob {
    CacheView keys;
    const float *q_idx[2];    // [B][4][64]
    const float *w[2];        // [B][4]
    const int32_t *pool;      // [B][pool_len] candidate positions or null (= all)
    int32_t pool_len;
    int32_t n_q;              // 1 or 2
    int32_t row[2];           // selection-row block of each query (row id = block*B + b)
};
constexpr int kMaxScanJobs = 16;

// Per-row selection buffers inside the workspace.
struct SelectBufs {
    uint32_t *hist;       // [n_rows][kHistBins] histogram of the keys' top bits (zeroed per call)
    uint32_t *keys;       // [n_rows][cand_cap]  order-preserving score keys, 0 = not a candidate
    int64_t cand_cap;     // candidates per row (max_seq_len or pool_len)
};

// A selection row: which targets (topk, pool) it produces.
struct SelectRow {
    int32_t *out_idx;     // [B][topk]
    int32_t *out_pool;    // [B][pool_out_len] or null
    const int32_t *pool;  // candidate positions when scanning a pool, else null
    int32_t pool_len;
    float *out_scores;    // optional [B][cand_cap]
};
constexpr int kMaxSelectRows = 16;

struct SelectPlan {
    SelectBufs bufs;
    SelectRow rows[kMaxSelectRows];  // per row block
    int32_t n_row_blocks;
    int32_t batch;
    int32_t topk;
    int32_t pool_out_len;            // 0 = no pool target in this plan
    int32_t max_len;                 // max_seq_len of the call
    const int32_t *seq_lens;
};

// scores: optional per job and query fp32 outputs (row stride scores_stride).
cudaError_t launch_scan(const ScanJob *jobs, int n_jobs, const SelectPlan &plan, int max_cand,
                        float *const (*scores)[2], int64_t scores_stride, int *flags,
                        cudaStream_t stream);
cudaError_t launch_select(const SelectPlan &plan, int max_cand, int *flags, cudaStream_t stream,
                          cudaEvent_t mid_event);
size_t select_bytes(int n_rows, int64_t cand_cap, int max_seq_len);
size_t select_hist_bytes(int n_rows);  // the leading part of the region to zero before a scan
SelectBufs carve_select(uint8_t *base, int n_rows, int64_t cand_cap, int max_seq_len);

// ---- step 2, many queries per sequence: tensor-core scoring + Top-K --------
// Workspace of run_index_multi: the selection rows (batch * n_q of them) and
// their candidate counts.
size_t index_multi_bytes(int batch, int n_q, int max_seq_len);
// Scores every query row against its candidates (its causal prefix when
// `causal`, else every position < seq_lens[b]) and, when out_idx is given,
// selects each row's Top-K (two launches, plus a memset of the histograms).
cudaError_t run_index_multi(const CacheView &keys, const float *q_idx, const float *w, int batch, int n_q,
                            const int32_t *seq_lens, int max_seq_len, int causal, int topk, int32_t *out_idx,
                            float *out_scores, uint8_t *ws, int *flags, cudaStream_t stream);

// ---- step 2, fused: scan + Top-K in one co-resident launch ------------------
struct FusedJobDesc {
    CacheView keys;
    const int32_t *pool;     // [B][pool_len] ascending positions or null (= every position < L)
    int32_t pool_len;
    int32_t n_q;             // selection rows (queries) over these keys: 1 or 2
    const float *q_idx[2];   // [B][4][64]
    const float *w[2];       // [B][4]
    int32_t *out_idx[2];     // [B][topk]
    int32_t *out_pool[2];    // [B][pool_out] or null
    float *out_scores[2];    // optional [B][scores_stride]
    CacheView kv;            // Full layer appends: main-KV cache written when new_kv
    const float *new_kv;     // [B][512] or null: quantised to position L-1 of kv
    const float *new_key;    // [B][64] or null: quantised to position L-1 of keys
    CacheView warm;          // main-KV cache the Top-K rows are gathered from next (has_warm)
    int32_t has_warm;        // 1: bring each selected row into L2 as its index is written
};

struct FusedLaunch {
    const FusedJobDesc *jobs;
    int n_jobs;
    const int32_t *seq_lens;
    uint8_t *state;          // fused_state_bytes(n_jobs * batch), zero at the first call, left zero
    int64_t scores_stride;
    int batch, topk, pool_out, max_len;
    int pdl;
    int keys_ready;          // 1: the key caches predate the stream's previous kernel (copies start before the wait)
};

struct FusedPlan {
    int G, chunk, ring_slots, cap;
    size_t smem;
};

// Whether the fused launch fits (every CTA co-resident); fills the plan.
bool fused_plan(int n_jobs, int batch, int64_t max_cand, FusedPlan &fp, int reserve_sms = 0);
size_t fused_state_bytes(int n_groups);
cudaError_t launch_fused(const FusedLaunch &L, const FusedPlan &fp, int *flags, cudaStream_t stream);
// Test hook: polls of each CTA's first tile wait (< 0: the normal limit).
void fused_set_first_wait_limit(int polls);

// ---- step 3: sparse attention --------------------------------------------
struct AttnEntry {
    CacheView kv;
    CacheView swa;
    const float *q;        // [B][16][512]
    const int32_t *idx;    // [B][topk] or null
    float *out;            // [B][16][512]
    float *lse;            // [B][16] or null
    const float *new_swa;  // optional [B][512]: window row appended at position L-1 first
    int32_t has_kv;
    int32_t has_swa;
};
constexpr int kMaxAttnEntries = 48;

struct AttnPlan {
    const AttnEntry *entries;
    int n_entries;
    int batch;
    int topk;              // rows per index list (0 when no entry has one)
    int window;
    const int32_t *seq_lens;
    int max_group;         // layers that may share one gather (1 or 2)
    int pdl;               // 1: the launch may overlap the stream's previous kernel
    int inputs_ready;      // 1: indices, caches, window rings and lengths were written before the
                           // stream's previous kernel started, so they are read before the wait for it
    void *workspace;       // optional: lets a (group, sequence) split over several clusters
    size_t workspace_bytes;
};

// Workspace of the fastest launch shape whose workspace is at most `budget`
// (0: every (layer group, sequence) is one cluster, merged in distributed
// shared memory).  Part of it is a ticket region that must be zero at the
// first call and is left zero.
size_t attn_workspace_bytes(const AttnPlan &plan, size_t budget = SIZE_MAX);
cudaError_t launch_attention(const AttnPlan &plan, int *flags, cudaStream_t stream,
                             cudaEvent_t mid_event);

}  // namespace csa2
