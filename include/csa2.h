/*
 * csa2.h -- C interface of the CSA2 (Compressed Sparse Attention 2) decode hot
 * path on NVIDIA B300 (sm_103a).
 *
 * Sources: web pages about DeepSeek V4.1 Flash --
 *   [HC] Helmcode, "DeepSeek V4.1 Flash" architecture explainer, sections
 *        "03 · CSA2" (Full / Reindex / Reuse modes, 4F+4R+30U+2 SWA-only)
 *        and "04 · FP4" (main KV in E2M1 with one E4M3 scale per 16 channels,
 *        no extra global scale; SWA KV stays in FP8);
 *   [LB] Louis Bouchard, "DeepSeek V4.1 Flash: KV cache and writing benchmark",
 *        section "Share the cache and the search work" (512 selected entries
 *        beside a 128-token window; a candidate pool of up to 16,384
 *        positions searched by later indexing layers) and "What actually
 *        changed over V4 Flash" (the indexer already used FP4);
 *   [MO] 0x0moeen, "DeepSeek V4.1 Flash KV cache", section "Then every layer
 *        stops asking the same question" (static per-layer modes; shared main
 *        KV and indexer keys; reused Top-K indices; hierarchical indexer).
 * The pages give no interface, widths or arithmetic beyond the format names;
 * everything else below is this library's stated choice.
 *
 * Conventions
 *  - Every data pointer is a DEVICE pointer owned by the caller unless stated.
 *    The library calls no allocator: scratch comes from a caller workspace of
 *    the size the matching *_workspace() function returns (256-B aligned),
 *    except for csa2_sparse_attn_noalloc, which uses a fixed 1 MiB device
 *    array the library declares statically (see there).
 *    A workspace must be zero-filled before its first use (cudaMemset once
 *    after allocating it): part of it holds barrier counters and histograms
 *    that every call leaves zero again.  After a call whose device check
 *    reports CSA2_ERR_TIMEOUT, zero it again before reusing it.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *    All work is enqueued asynchronously on it; no call synchronises, except
 *    csa2_check_device().  Calls may be captured in a CUDA graph.
 *  - Functions return a csa2_status and never throw.  On failure nothing was
 *    enqueued (argument errors) or a launch failed (CSA2_ERR_CUDA);
 *    csa2_last_error() returns a message for the calling thread.
 *  - Data-dependent faults (an index or page outside its cache) never fault
 *    the GPU: the kernel skips the access and records a flag read by
 *    csa2_check_device().  Waits on asynchronous copies are bounded: one that
 *    gives up records a flag instead of hanging.
 *  - Widths are fixed: attention 16 heads x 512 channels (MQA over one shared
 *    512-channel row that is both key and value); indexer 4 heads x 64.
 *  - Positions of sequence b are 0 .. seq_lens[b]-1; the current decode
 *    token is position seq_lens[b]-1.  The SWA window is the positions
 *    [max(0, seq_lens[b]-window), seq_lens[b]).
 */
#ifndef CSA2_H
#define CSA2_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status ----------------------------------------------------------- */
typedef int32_t csa2_status;
#define CSA2_OK               0
#define CSA2_ERR_INVALID_ARG  1  /* bad argument (host check) or device bounds flag */
#define CSA2_ERR_UNSUPPORTED  2  /* width / size outside what the kernels support */
#define CSA2_ERR_CUDA         3  /* a CUDA runtime call or launch failed */
#define CSA2_ERR_TIMEOUT      4  /* a bounded device-side wait gave up */
#define CSA2_ERR_WORKSPACE    5  /* workspace NULL, misaligned or too small */

/* ---- layer modes ([HC] "03 · CSA2"; [MO]) ----------------------------- */
#define CSA2_MODE_FULL      0  /* builds its own caches; scores every position */
#define CSA2_MODE_REINDEX   1  /* rescoring of a Full layer's keys with its own query */
#define CSA2_MODE_REUSE     2  /* reuses another layer's Top-K over a Full layer's KV */
#define CSA2_MODE_SWA_ONLY  3  /* local window attention only */

/* ---- cache formats ---------------------------------------------------- */
/* Main KV, 512 channels, [HC] "04 · FP4": per token 288 B = 256 B of E2M1
 * codes (channel 2i in the low nibble of byte i) then 32 B of E4M3 scales
 * (scale j covers channels 16j..16j+15).  Row of slot s at data + 288*s. */
#define CSA2_FMT_FP4_KV    0
/* Indexer keys, 64 channels, FP4 with E4M3/16 ([LB]): tiles of 64 slots,
 * 2,304 B each = 64 x 32 B codes then 64 x 4 B scales.  Slot s lives in tile
 * s/64, row s%64: codes at data + 2304*(s/64) + 32*(s%64), scales at
 * data + 2304*(s/64) + 2048 + 4*(s%64).  n_slots must be a multiple of 64. */
#define CSA2_FMT_FP4_IDX   1
/* SWA rows, 512 channels, FP8 E4M3 ([HC] "04 · FP4"), one fp32 scale per
 * token: a plane of n_slots x 512 B codes, then n_slots fp32 scales at
 * data + 512*n_slots. */
#define CSA2_FMT_FP8_SWA   2

/* Quantisation rules (the pages name the formats only; stated choices):
 *  FP4 block of 16: scale = E4M3(absmax / 6), code = E2M1(x / scale), with
 *  IEEE fp32 division, round-half-even onto each grid, saturation at the
 *  largest finite value (6, 448), the code's sign bit = the sign bit of
 *  x / scale; a zero scale gives all-zero codes.  FP8 row: scale = absmax/448
 *  (fp32), code = E4M3(x / scale), same rounding/sign rules. */

/* A cache: where logical (sequence b, position p) lives.
 *   page_size == 0 : slot = b * seq_stride + p
 *                    (FP8_SWA rings: slot = b * seq_stride + p % seq_stride)
 *   page_size  > 0 : slot = page_table[b * max_pages + p / page_size] * page_size
 *                           + p % page_size
 * Slots outside [0, n_slots) or page ids < 0 are skipped and flagged. */
typedef struct csa2_cache {
    void          *data;        /* device bytes, 256-B aligned, caller-owned */
    int32_t        format;      /* CSA2_FMT_* */
    int32_t        page_size;   /* 0, or tokens per page (multiple of 64) */
    int64_t        n_slots;     /* capacity in tokens */
    int64_t        seq_stride;  /* contiguous: slots per sequence (multiple of 64 for
                                   FP4_IDX); FP8_SWA: ring capacity per sequence */
    const int32_t *page_table;  /* paged: device [batch][max_pages] physical page ids */
    int32_t        max_pages;   /* paged: row length of page_table */
    int32_t        reserved;    /* must be 0 */
} csa2_cache;

/* Bytes a cache of this format and capacity occupies (0 if invalid). */
size_t csa2_cache_bytes(int32_t format, int64_t n_slots);

/* ---- step 1: quantise-and-write (build or append) --------------------- */
/* [HC] "04 · FP4" / [MO]: FP4 E2M1 + E4M3 per 16 channels (main KV, indexer
 * keys); FP8 for the SWA rows.
 *   src       device fp32 [n_seqs][rows_per_seq][C], C = 512 (FP4_KV, FP8_SWA)
 *             or 64 (FP4_IDX), rows contiguous
 *   start_pos device int32 [n_seqs] or NULL (= 0): row r of sequence b is
 *             written at logical position start_pos[b] + r of sequence b
 *   seq_lens  device int32 [n_seqs] or NULL: rows at positions >= seq_lens[b]
 *             are skipped (ragged builds)
 *   dst       destination cache (host struct; its data is device memory)
 * Appending one decode token: rows_per_seq = 1, start_pos = seq_lens - 1. */
csa2_status csa2_quantize_kv(const float *src, int32_t n_seqs, int64_t rows_per_seq,
                             const int32_t *start_pos, const int32_t *seq_lens,
                             const csa2_cache *dst, void *stream);

/* ---- step 2: indexer score + Top-K ------------------------------------ */
/* [HC] "03 · CSA2": Full scores every position, Reindex rescores with its own
 * query; [LB]: the hierarchical Reindex scores only a candidate pool.
 * Score (form chosen for this library, the pages give none):
 *   q_idx is quantised by the FP4 rule; per head h and 16-channel block j
 *   t_hj = sq_hj * sk_j * (E2M1 dot product), exact;
 *   s_h = ((t_h0 + t_h1) + t_h2) + t_h3 in fp32;  r_h = s_h > 0 ? s_h : +0;
 *   score = fma(w3,r3, fma(w2,r2, fma(w1,r1, w0*r0))) in fp32; 0 -> +0.
 * Top-K: order by (score desc, position asc); the first `topk` are written
 * to out_idx[b] as ASCENDING positions, padded with -1 when fewer candidates
 * exist.  out_pool (FULL only) receives the first pool_out_len of the same
 * order, ascending, -1 padded.
 *   mode        CSA2_MODE_FULL or CSA2_MODE_REINDEX (same arithmetic)
 *   keys        FP4_IDX cache holding positions 0..seq_lens[b]-1
 *   q_idx, w    device fp32 [batch][4][64], [batch][4]
 *   seq_lens    device int32 [batch], each in [0, max_seq_len]
 *   pool        device int32 [batch][pool_len] ascending candidate positions
 *               (-1 entries ignored) or NULL = every position < seq_lens[b]
 *   out_idx     device int32 [batch][topk]
 *   out_pool    device int32 [batch][pool_out_len] or NULL
 *   out_scores  optional device fp32 [batch][pool ? pool_len : max_seq_len]:
 *               the score of each candidate (unwritten past the candidates)
 * Limits: topk, pool_out_len in [1, 65536]; max_seq_len <= 2^24.
 * Execution: when every CTA fits on the device at once (batch x the
 * candidates per sequence small enough), scoring and selection are one
 * launch whose CTAs meet at bounded group barriers; otherwise a scan launch
 * and a cluster-select launch.  Either way the result is the same. */
size_t csa2_index_topk_workspace(int32_t batch, int32_t max_seq_len, int32_t pool_len,
                                 int32_t topk, int32_t pool_out_len);
csa2_status csa2_index_topk(int32_t mode, const csa2_cache *keys, const float *q_idx,
                            const float *w, int32_t batch, int32_t n_heads, int32_t head_dim,
                            const int32_t *seq_lens, int32_t max_seq_len,
                            const int32_t *pool, int32_t pool_len, int32_t topk,
                            int32_t *out_idx, int32_t *out_pool, int32_t pool_out_len,
                            float *out_scores, void *workspace, size_t workspace_bytes,
                            void *stream);

/* ---- step 2 with many queries per sequence ----------------------------- */
/* Several tokens of one sequence index at once: a speculative verification
 * ([HC] "10 · other changes": DSpark checks drafted tokens together) or a
 * chunk of prefill ([HC] "03 · CSA2": the Reuse layers' kernel path in
 * prefill).  Query row i of sequence b is scored exactly as
 * csa2_index_topk(CSA2_MODE_FULL) scores one query (same quantisation, same
 * fp32 rounding points, bit-identical scores and index sets) over its
 * candidates: with causal = 1 the positions 0 .. L_b - n_q + i (the n_q
 * queries are the sequence's last n_q tokens, L_b = seq_lens[b]; rows with
 * no position have no candidates), with causal = 0 every position < L_b.
 * The scores are a dense contraction here, computed on the tensor cores
 * (tcgen05 kind::f16, one MMA per 16-channel block with the E4M3 scales
 * folded exactly into the fp16 operands; the epilogue adds the blocks in the
 * fixed order).
 *   keys        FP4_IDX cache holding positions 0..seq_lens[b]-1
 *   q_idx, w    device fp32 [batch][n_q][4][64] (16-byte aligned), [batch][n_q][4]
 *   seq_lens    device int32 [batch], each in [0, max_seq_len]
 *   causal      1: row i sees its causal prefix; 0: every position
 *   out_idx     device int32 [batch][n_q][topk]: ascending positions of the
 *               row's Top-K (order: score desc, position asc), -1 padded; or
 *               NULL (scores only, topk ignored)
 *   out_scores  optional device fp32 [batch][n_q][max_seq_len], written at
 *               the row's candidate positions only
 * Limits: n_q in [1, 4096], batch * n_q <= 65535, topk in [1, 65536],
 * max_seq_len <= 2^24; at least one of out_idx, out_scores.
 * Workspace: csa2_index_topk_multi_workspace() bytes, 256-byte aligned
 * (batch * n_q * (max_seq_len rounded up to 64) * 4 B of selection keys plus
 * 8 KB of histogram per row); the call zeroes what it needs.
 * Launches: a memset, the scoring kernel, and (with out_idx) the cluster
 * select. */
size_t csa2_index_topk_multi_workspace(int32_t batch, int32_t n_q, int32_t max_seq_len);
csa2_status csa2_index_topk_multi(const csa2_cache *keys, const float *q_idx, const float *w,
                                  int32_t batch, int32_t n_q, int32_t n_heads, int32_t head_dim,
                                  const int32_t *seq_lens, int32_t max_seq_len, int32_t causal,
                                  int32_t topk, int32_t *out_idx, float *out_scores,
                                  void *workspace, size_t workspace_bytes, void *stream);

/* ---- step 3: gather + dequantise + sparse attention with the SWA branch - */
/* [LB] "Share the cache and the search work": the selected global entries
 * beside the local 128-token window; [HC] "04 · FP4": FP4 global rows, FP8
 * window rows.  One softmax over the multiset {selected rows} + {window rows},
 * logit = q_h . row (q carries its own scale), out_h = sum p_j row_j.
 *   kv          FP4_KV cache (may be NULL when idx is NULL)
 *   swa         FP8_SWA ring holding the window positions
 *   q           device fp32 [batch][16][512]
 *   idx         device int32 [batch][topk] positions (-1 = skip) or NULL
 *               (SWA-only layer)
 *   swa_window  window length in tokens (0 = no window branch)
 *   out         device fp32 [batch][16][512];  lse: optional [batch][16]
 * Numerics: the FP4 rows, and the FP8 window codes times 2^-8, are exact in
 * fp16; each query enters the tensor cores as two fp16 parts (its rounded
 * value and the rounded remainder), so logits keep the fp32 query to about
 * 2^-22; softmax and every accumulation are fp32; the softmax weights enter
 * the PV product as fp16 (at most e^2 each, times the window row's fp32
 * scale x 2^8 -- window rows with |x| above ~15,000 would overflow it).
 * Launch shape and workspace: each sequence is one thread-block cluster
 * (up to 16 CTAs, a tile of 128 rows each, merged through distributed
 * shared memory), or two clusters when that is faster: the second
 * cluster's CTAs each write a partial (running max, sum, normalised output)
 * to the workspace and the first cluster folds them into its merge (planned
 * only when every cluster of the launch fits on the device at once).  The plan is the
 * fastest whose scratch fits `workspace_bytes`; csa2_sparse_attn_workspace()
 * is the most any plan of these sizes asks for.  `workspace` may be NULL
 * (with any size): then every sequence is one cluster.  The split path's
 * counters must be zero before the first use (zero-fill the
 * workspace once) and every call leaves them zero.  Results are identical
 * for equal inputs and equal workspace sizes; a different split merges in a
 * different order, which changes the rounding only. */
size_t csa2_sparse_attn_workspace(int32_t batch, int32_t topk, int32_t swa_window);
csa2_status csa2_sparse_attn(const csa2_cache *kv, const csa2_cache *swa, const float *q,
                             int32_t batch, int32_t n_heads, int32_t head_dim,
                             const int32_t *seq_lens, int32_t max_seq_len,
                             const int32_t *idx, int32_t topk, int32_t swa_window,
                             float *out, float *lse, void *workspace, size_t workspace_bytes,
                             void *stream);

/* Attention without a workspace argument, for callers that cannot allocate
 * device memory: a serving process that reserved nearly all HBM for its
 * cache pool up front (cudaMalloc would fail there, and it synchronises the
 * device), or a plugin living inside another runtime's allocator.  The paper
 * has no counterpart; this is a deployment convenience of this library.
 * Arguments, layouts, numerics and error codes are those of
 * csa2_sparse_attn minus the workspace; the result is bit-identical to
 * csa2_sparse_attn given a 1 MiB workspace.  Scratch for split clusters
 * comes from a 1 MiB array the library declares as a static __device__
 * variable on each device (zero when the module loads; every call leaves
 * its counters zero again), planned to fit it; no allocator is called.
 * Its device address is looked up once per device with
 * cudaGetSymbolAddress (thread-safe) and kept for the life of the
 * process (a cudaDeviceReset invalidates it: reload the library after
 * one); make the first call on each device before capturing it in a CUDA
 * graph, because the lookup may load the module.  All calls on a device share the array: calls that overlap in
 * time (on different streams, or from several threads) race on it and give
 * wrong results.  A sequence that needs more than the array holds runs as
 * one cluster, which needs no scratch, so no size is rejected for want of
 * scratch.  Returns CSA2_ERR_CUDA if the address lookup fails. */
csa2_status csa2_sparse_attn_noalloc(const csa2_cache *kv, const csa2_cache *swa, const float *q,
                                     int32_t batch, int32_t n_heads, int32_t head_dim,
                                     const int32_t *seq_lens, int32_t max_seq_len,
                                     const int32_t *idx, int32_t topk, int32_t swa_window,
                                     float *out, float *lse, void *stream);

/* ---- step 4: one decode step over a static mode schedule --------------- */
/* [HC] "03 · CSA2": static per-layer modes; a Reuse layer consumes another
 * layer's Top-K over a Full layer's KV with its own query and SWA state;
 * [LB]/[MO]: Reindex layers may search only the Full layer's pool.
 * Descriptors are host memory; every pointer inside is device memory. */
typedef struct csa2_layer_desc {
    int32_t mode;       /* CSA2_MODE_* */
    int32_t kv_src;     /* FULL: its own index; REINDEX/REUSE: index of the FULL
                           layer whose kv / idx_keys (and pool) are read */
    int32_t idx_src;    /* REUSE: index of the FULL/REINDEX layer whose Top-K is
                           reused; otherwise ignored */
    int32_t use_pool;   /* REINDEX: 1 = score only layer kv_src's pool_out */
    const csa2_cache *kv;        /* FULL: FP4_KV cache */
    const csa2_cache *idx_keys;  /* FULL: FP4_IDX cache */
    const csa2_cache *swa;       /* every layer: its own FP8_SWA ring */
    const float *q;              /* [batch][16][512] */
    const float *q_idx;          /* FULL/REINDEX: [batch][4][64] */
    const float *w;              /* FULL/REINDEX: [batch][4] */
    const float *new_kv;         /* FULL, optional [batch][512]: appended at seq_lens[b]-1 */
    const float *new_idx_key;    /* FULL, optional [batch][64]:  appended at seq_lens[b]-1 */
    const float *new_swa;        /* optional [batch][512]: appended to swa at seq_lens[b]-1 */
    float   *out;                /* [batch][16][512] */
    float   *lse;                /* optional [batch][16] */
    int32_t *idx_out;            /* FULL/REINDEX: [batch][topk] */
    int32_t *pool_out;           /* FULL when pool_len > 0: [batch][pool_len] */
} csa2_layer_desc;

/* Layer sources must point backwards (kv_src/idx_src < own index) except a
 * FULL layer's kv_src (itself).
 *
 * csa2_decode_layers runs the whole step in the *phased* order, valid when
 * every layer's inputs exist when the call is made: all level-0 indexing
 * (Full + pool-free Reindex layers, a Full layer and its Reindex partner
 * sharing one key scan; the Full layers' appended main-KV rows and keys are
 * quantised there), level-1 indexing (pool-restricted Reindex), then the
 * attention of every layer (each appends its own window row first).  Up to
 * three launches. */
size_t csa2_decode_layers_workspace(const csa2_layer_desc *layers, int32_t n_layers,
                                    int32_t batch, int32_t max_seq_len, int32_t topk,
                                    int32_t pool_len, int32_t swa_window);
csa2_status csa2_decode_layers(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch,
                               const int32_t *seq_lens, int32_t max_seq_len, int32_t topk,
                               int32_t pool_len, int32_t swa_window, void *workspace,
                               size_t workspace_bytes, void *stream);

/* Layer `layer` of the same schedule alone, in the order a model runs it:
 * its appends, its indexing (FULL / REINDEX: one launch, or two when the
 * problem is too large to be co-resident) and its attention (one launch).
 * A model calls it for layer 0, 1, ... with its own work in between; the
 * layers a call reads (kv_src's caches and pool, idx_src's indices) must
 * have run before on the same stream.  Launches may overlap the tail of
 * the stream's previous kernel (programmatic dependent launch).  What that
 * kernel may write (this layer's queries, indexer query and weights, its
 * appended rows) is read only after it completes.  Read before that, so
 * that their loads overlap the previous kernel: a FULL or REINDEX layer's
 * indexer keys (contiguous caches; a FULL layer's own new key is patched
 * in) and sequence lengths, and a REUSE or SWA_ONLY layer's indices,
 * sequence lengths, kv_src's cache and window ring.  These must have been written before the stream's
 * previous kernel started, as they are when the layers run in order
 * through this call: do not rewrite them with a kernel launched right
 * before this call.  Workspace: the size of
 * csa2_decode_layer_workspace() (zero-filled before its first use, see
 * the conventions above), shared by every layer's call. */
size_t csa2_decode_layer_workspace(const csa2_layer_desc *layers, int32_t n_layers, int32_t batch,
                                   int32_t max_seq_len, int32_t topk, int32_t pool_len,
                                   int32_t swa_window);
csa2_status csa2_decode_layer(const csa2_layer_desc *layers, int32_t n_layers, int32_t layer,
                              int32_t batch, const int32_t *seq_lens, int32_t max_seq_len,
                              int32_t topk, int32_t pool_len, int32_t swa_window,
                              void *workspace, size_t workspace_bytes, void *stream);

/* ---- planning (host only, no GPU work) ---------------------------------- */
/* Footprint of one session for a schedule `modes` (CSA2_MODE_* per layer) at
 * a context of `context` tokens: [HC] launch post ("890 bytes go a long
 * way") and [LB] "Share the cache and the search work" quote the global KV
 * per token (890 B) and per million tokens (0.89 GB); the pages give neither
 * widths nor the token compression, so these are this library's layouts'
 * figures, not a reproduction of 890 B.
 *   global_bytes_per_token  (288 + 36) B per Full layer (main KV + indexer key)
 *   cache_bytes             the Full layers' caches (context rounded up to 64
 *                           tokens) + every layer's FP8 window ring (window
 *                           rounded up to 4 slots, 516 B each)
 *   step_bytes              per-step buffers: q, out, lse per layer, indices
 *                           per indexing layer, pools per Full layer
 *   sessions                floor(hbm_bytes / (cache_bytes + step_bytes)) */
typedef struct csa2_footprint {
    int64_t global_bytes_per_token;
    int64_t cache_bytes;
    int64_t step_bytes;
    int64_t sessions;
} csa2_footprint;
csa2_status csa2_plan_footprint(const int32_t *modes, int32_t n_layers, int64_t context, int32_t topk,
                                int32_t pool_len, int32_t window, int64_t hbm_bytes, csa2_footprint *out);

/* Compute and traffic of one decode token through the schedule at a context
 * of `context` tokens, [HC] "07 · compute, memory, bill" (decode work weighted
 * BF16 = 1, FP8 = 0.5, FP4 = 0.25, followed from 4K to 1M), restricted to this
 * path.  Reindex layers score the pool when pool_len > 0.
 *   index_flops       2 x 4 heads x 64 per position scored (Full, Reindex)
 *   attn_flops        4 x 16 heads x 512 per attended row (QK^T + PV):
 *                     min(topk, context) selected rows (not SWA-only layers)
 *                     + min(window, context) window rows, every layer
 *   weighted_flops    index x 0.25 (FP4 keys and query) + selected-row
 *                     attention x 0.25 (FP4 rows) + window attention x 0.5
 *                     (FP8 rows)
 *   bytes_sequential  algorithmic bytes in the layer-sequential order: 36 B
 *                     per position scored (40 B per pool entry), 288 B per
 *                     selected row, 516 B per window row, q/out/lse, indexer
 *                     inputs, indices written and read, appended rows */
typedef struct csa2_cost {
    double index_flops;
    double attn_flops;
    double weighted_flops;
    double bytes_sequential;
} csa2_cost;
csa2_status csa2_plan_cost(const int32_t *modes, int32_t n_layers, int64_t context, int32_t topk,
                           int32_t pool_len, int32_t window, csa2_cost *out);

/* ---- diagnostics ------------------------------------------------------ */
/* Message for the last failure on the calling thread ("" if none). */
const char *csa2_last_error(void);
/* Synchronises `stream`, reads and clears the device flag word of the current
 * device: CSA2_OK, CSA2_ERR_INVALID_ARG (an index, page or slot was out of
 * range and skipped) or CSA2_ERR_TIMEOUT. */
csa2_status csa2_check_device(void *stream);
/* Raw flag bits seen by the calling thread's last csa2_check_device():
 * 1 = out-of-range access skipped, 2 = a bounded wait gave up. */
int32_t csa2_last_device_flags(void);
/* Profiling hook: when n > 0, csa2_decode_layers records events[i] (cudaEvent_t
 * created by the caller) on its stream after phase i: 0 start, 1 and 2
 * level-0 scoring and selection (one mark when fused), 3 level-1
 * scoring+selection, 4 and 5 attention.  Pass n = 0 to disable.
 * Process-wide; not thread-safe. */
csa2_status csa2_set_phase_events(void *const *events, int32_t n);
/* Kernels this library has enqueued since it was loaded, all threads and
 * devices together (a stream capture counts its launches once; replays of
 * the captured graph add nothing). */
int64_t csa2_launch_count(void);
/* Test hook: every CTA of a fused indexing launch polls its first tile
 * copy at most `polls` times before it records a timeout (CSA2_ERR_TIMEOUT
 * at the next csa2_check_device()); it then still waits, with the normal
 * bound, for the copy to land, so no CTA leaves with a copy in flight and
 * the results stay correct.  polls < 0 restores the normal bound.
 * Process-wide; for tests of the timeout path only. */
csa2_status csa2_test_set_wait_limit(int32_t polls);
/* Library version: major * 10000 + minor * 100 + patch. */
int32_t csa2_version(void);

#ifdef __cplusplus
}
#endif
#endif /* CSA2_H */
