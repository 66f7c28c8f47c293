"""Footprint and precision-weighted cost of the CSA2 decode path, written out
from the format definitions.  TEST INFRASTRUCTURE ONLY (see oracle/__init__).

Footprint: the Helmcode launch post ("890 bytes go a long way") and Louis
Bouchard's KV-cache report ("Share the cache and the search work") quote the
global KV per token (890 B) and per million tokens (0.89 GB).  For this
library's layouts a Full layer keeps, per token, a main-KV row of 512 E2M1
codes (4 bits each) and 512 / 16 E4M3 scales (8 bits each), and an indexer
key of 64 codes and 64 / 16 scales; every layer keeps a window ring of 512
E4M3 codes and one fp32 scale per slot.

Cost: the Helmcode explainer, "07 · compute, memory, bill", weighs decode work
by precision (BF16 1, FP8 0.5, FP4 0.25) from 4K to 1M tokens of context.
Here: the indexer's dot products (FP4 key x FP4 query, 4 heads x 64
channels, one multiply and one add per channel) over every position a Full
or Reindex layer scores; the attention's two products (QK^T, PV; 16 heads x
512 channels, a multiply and an add each) over the FP4 selected rows and the
FP8 window rows.
"""
FULL, REINDEX, REUSE, SWA_ONLY = 0, 1, 2, 3


def row_bytes():
    """(main KV, indexer key, window row) bytes per token, from the formats."""
    kv = 512 * 4 // 8 + (512 // 16) * 8 // 8
    key = 64 * 4 // 8 + (64 // 16) * 8 // 8
    swa = 512 * 8 // 8 + 32 // 8
    return kv, key, swa


def footprint(modes, context, topk, pool_len, window, hbm_bytes):
    kv, key, swa = row_bytes()
    n_full = sum(1 for m in modes if m == FULL)
    n_index = sum(1 for m in modes if m in (FULL, REINDEX))
    per_token = n_full * (kv + key)
    tokens = -(-context // 64) * 64                      # whole 64-token tiles / pages
    ring = -(-window // 4) * 4
    cache = tokens * per_token + len(modes) * ring * swa
    q = out = 16 * 512 * 4
    lse = 16 * 4
    step = len(modes) * (q + out + lse) + n_index * topk * 4 + (n_full * pool_len * 4 if pool_len > 0 else 0)
    per = cache + step
    return dict(global_bytes_per_token=per_token, cache_bytes=cache, step_bytes=step,
                sessions=hbm_bytes // per if per else 0)


def cost(modes, context, topk, pool_len, window):
    kv, key, swa = row_bytes()
    sel = min(topk, context)
    win = min(window, context)
    idx_fl = 2 * 4 * 64
    att_fl = 2 * 2 * 16 * 512
    res = dict(index_flops=0.0, attn_flops=0.0, weighted_flops=0.0, bytes_sequential=0.0)
    seen_full = False
    for m in modes:
        if m == FULL:
            seen_full = True
        pooled = m == REINDEX and pool_len > 0 and seen_full
        scored = 0 if m in (REUSE, SWA_ONLY) else (min(pool_len, context) if pooled else context)
        rows = 0 if m == SWA_ONLY else sel
        res["index_flops"] += scored * idx_fl
        res["attn_flops"] += (rows + win) * att_fl
        res["weighted_flops"] += 0.25 * scored * idx_fl + 0.25 * rows * att_fl + 0.5 * win * att_fl
        b = 0
        if m in (FULL, REINDEX):
            b += scored * (key + 4 if pooled else key)
            b += 4 * 64 * 4 + 4 * 4 + topk * 4               # indexer query, weights, indices written
            if m == FULL:
                b += (pool_len * 4 if pool_len > 0 else 0) + 512 * 4 + kv + 64 * 4 + key   # pool, appends
        if m != SWA_ONLY:
            b += rows * kv + topk * 4                        # gathered rows, indices read
        b += win * swa + 2 * 16 * 512 * 4 + 16 * 4 + 512 * 4 + swa   # window, q/out/lse, window append
        res["bytes_sequential"] += b
    return res
