// Planning calculators for the CSA2 decode path (host only, no GPU work).
//
// Footprint: the packed caches a session keeps (Helmcode "DeepSeek V4.1 Flash"
// launch post, "890 bytes go a long way"; Louis Bouchard's KV-cache report,
// "Share the cache and the search work": global KV per token and 0.89 GB per
// million tokens) for this library's layouts: per Full layer 288 B of FP4
// main KV and 36 B of FP4 indexer key per token, per layer one FP8 window
// ring of 516 B per slot.  The pages' own 890 B is not reproducible from what
// they give (widths, token compression); these are this layout's figures.
//
// Cost: the precision-weighted compute of one decode token (Helmcode
// explainer, "07 · compute, memory, bill": work weighted BF16 = 1, FP8 = 0.5,
// FP4 = 0.25, "from 4K to 1M") restricted to this path -- the indexer's
// FP4 x FP4 dot products over every position a Full or Reindex layer scores
// (or its pool), and the attention's QK^T and PV over the FP4 selected rows and
// the FP8 window rows -- with the algorithmic bytes the path moves.
#include <cstring>

#include "internal.h"

using namespace csa2;

namespace {

constexpr int64_t kSwaRow = kDim + 4;  // 516

int64_t round_up(int64_t x, int64_t m) { return (x + m - 1) / m * m; }

bool valid_modes(const int32_t *modes, int32_t n_layers)
{
    if (!modes || n_layers <= 0) return false;
    for (int i = 0; i < n_layers; ++i)
        if (modes[i] < CSA2_MODE_FULL || modes[i] > CSA2_MODE_SWA_ONLY) return false;
    return true;
}

}  // namespace

extern "C" {

csa2_status csa2_plan_footprint(const int32_t *modes, int32_t n_layers, int64_t context, int32_t topk,
                                int32_t pool_len, int32_t window, int64_t hbm_bytes, csa2_footprint *out)
{
    if (!out || !valid_modes(modes, n_layers) || context < 0 || topk < 0 || pool_len < 0 || window < 0 ||
        hbm_bytes < 0)
        return set_error(CSA2_ERR_INVALID_ARG, "plan_footprint: bad argument");
    int64_t n_full = 0, n_index = 0;
    for (int i = 0; i < n_layers; ++i) {
        n_full += modes[i] == CSA2_MODE_FULL;
        n_index += modes[i] == CSA2_MODE_FULL || modes[i] == CSA2_MODE_REINDEX;
    }
    memset(out, 0, sizeof(*out));
    out->global_bytes_per_token = n_full * (kKvRow + kIdxTileBytes / kIdxTile);
    // caches: Full layers' rows in 64-token units (indexer tiles, pages); each
    // layer's window ring rounded to 4 slots
    const int64_t tokens = round_up(context, kIdxTile);
    out->cache_bytes = tokens * out->global_bytes_per_token + (int64_t)n_layers * round_up(window, 4) * kSwaRow;
    // per-step buffers: q, out (fp32 16 x 512), lse per layer; indices per
    // indexing layer; pools per Full layer when hierarchical
    out->step_bytes = (int64_t)n_layers * (2 * kHeads * kDim * 4 + kHeads * 4) + n_index * (int64_t)topk * 4 +
                      (pool_len > 0 ? n_full * (int64_t)pool_len * 4 : 0);
    const int64_t per = out->cache_bytes + out->step_bytes;
    out->sessions = per > 0 ? hbm_bytes / per : 0;
    return CSA2_OK;
}

csa2_status csa2_plan_cost(const int32_t *modes, int32_t n_layers, int64_t context, int32_t topk, int32_t pool_len,
                           int32_t window, csa2_cost *out)
{
    if (!out || !valid_modes(modes, n_layers) || context < 0 || topk < 0 || pool_len < 0 || window < 0)
        return set_error(CSA2_ERR_INVALID_ARG, "plan_cost: bad argument");
    memset(out, 0, sizeof(*out));
    const double L = (double)context;
    const double sel = (double)(topk < context ? topk : context);   // selected rows per attending layer
    const double win = (double)(window < context ? window : context);
    const double idx_flops_per_pos = 2.0 * kIdxHeads * kIdxDim;     // one multiply-add per channel and head
    const double attn_flops_per_row = 4.0 * kHeads * kDim;          // QK^T and PV
    bool seen_full = false;
    for (int i = 0; i < n_layers; ++i) {
        const int m = modes[i];
        double scored = 0.0;
        if (m == CSA2_MODE_FULL) {
            scored = L;
            seen_full = true;
        } else if (m == CSA2_MODE_REINDEX) {
            scored = (pool_len > 0 && seen_full) ? (double)(pool_len < context ? pool_len : context) : L;
        }
        const double rows = (m == CSA2_MODE_SWA_ONLY) ? 0.0 : sel;
        out->index_flops += scored * idx_flops_per_pos;
        out->attn_flops += (rows + win) * attn_flops_per_row;
        out->weighted_flops += 0.25 * scored * idx_flops_per_pos + 0.25 * rows * attn_flops_per_row +
                               0.5 * win * attn_flops_per_row;
        // algorithmic bytes, layer by layer (the layer-sequential order)
        double by = 0.0;
        if (m == CSA2_MODE_FULL || m == CSA2_MODE_REINDEX) {
            const bool pooled = m == CSA2_MODE_REINDEX && pool_len > 0 && seen_full;
            by += pooled ? scored * (double)(kIdxTileBytes / kIdxTile + 4) : scored * (double)(kIdxTileBytes / kIdxTile);
            by += (double)(kIdxHeads * kIdxDim * 4 + kIdxHeads * 4) + (double)topk * 4.0;
            if (m == CSA2_MODE_FULL && pool_len > 0) by += (double)pool_len * 4.0;
            if (m == CSA2_MODE_FULL) by += (double)(kDim * 4 + kKvRow + kIdxDim * 4 + kIdxTileBytes / kIdxTile);
        }
        if (m != CSA2_MODE_SWA_ONLY) by += rows * kKvRow + (double)topk * 4.0;
        by += win * kSwaRow + (double)(2 * kHeads * kDim * 4 + kHeads * 4) + (double)(kDim * 4 + kSwaRow);
        out->bytes_sequential += by;
    }
    return CSA2_OK;
}

}  // extern "C"
