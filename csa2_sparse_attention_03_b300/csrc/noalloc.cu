// csa2_sparse_attn_noalloc: the gather-attention entry point for callers that
// cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: a serving process that
// reserved nearly all HBM for its KV-cache pool at start-up (a cudaMalloc
// then fails, and it would synchronise the device anyway), or a plugin that
// runs inside another runtime's allocator and has no way to ask it for
// scratch.  The attention kernel keeps every intermediate (the split
// partials of a sequence are merged inside one thread-block cluster through
// distributed shared memory), so this entry point needs neither a workspace
// nor any library-owned device array: it is the workspace-free form of
// csa2_sparse_attn and allocates nothing.
#include "internal.h"

extern "C" csa2_status csa2_sparse_attn_noalloc(const csa2_cache *kv, const csa2_cache *swa, const float *q,
                                                int32_t batch, int32_t n_heads, int32_t head_dim,
                                                const int32_t *seq_lens, int32_t max_seq_len, const int32_t *idx,
                                                int32_t topk, int32_t swa_window, float *out, float *lse,
                                                void *stream)
{
    return csa2_sparse_attn(kv, swa, q, batch, n_heads, head_dim, seq_lens, max_seq_len, idx, topk, swa_window,
                            out, lse, nullptr, 0, stream);
}
