// csa2_sparse_attn_noalloc: the gather-attention entry point for callers that
// cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: a serving process that
// reserved nearly all HBM for its KV-cache pool at start-up (a cudaMalloc
// then fails, and it would synchronise the device anyway), or a plugin that
// runs inside another runtime's allocator and has no way to ask it for
// scratch.  The attention kernel needs scratch only to split one (layer
// group, sequence) over two clusters (the second cluster's per-CTA partials
// and a counter per owner in the first); this variant takes that
// scratch from a fixed array the library owns for the life of the process,
// planned to fit it, instead of from a caller workspace.
#include <atomic>

#include "internal.h"

namespace {

// 1 MiB of scratch on every device that loads the library, held until the
// process exits; zero at load.  Every call on a device shares it.
constexpr size_t kNoAllocScratchBytes = size_t(1) << 20;
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

// Device address of g_attn_scratch on the current device.  In host code the
// symbol names a host-side stand-in, not device memory, so it is looked up
// (with that device current) on the device's first call; concurrent first
// calls from several threads each look it up and store the same value.
cudaError_t scratch_address(void **out)
{
    static std::atomic<void *> cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    void *p = cache[dev].load(std::memory_order_acquire);
    if (!p) {
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        cache[dev].store(p, std::memory_order_release);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" csa2_status csa2_sparse_attn_noalloc(const csa2_cache *kv, const csa2_cache *swa, const float *q,
                                                int32_t batch, int32_t n_heads, int32_t head_dim,
                                                const int32_t *seq_lens, int32_t max_seq_len, const int32_t *idx,
                                                int32_t topk, int32_t swa_window, float *out, float *lse,
                                                void *stream)
{
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return csa2::set_error(CSA2_ERR_CUDA, "csa2_sparse_attn_noalloc: scratch address lookup: %s",
                               cudaGetErrorString(e));
    // the fastest launch shape whose scratch fits the array (one cluster per
    // sequence, no scratch at all, always fits)
    return csa2_sparse_attn(kv, swa, q, batch, n_heads, head_dim, seq_lens, max_seq_len, idx, topk, swa_window,
                            out, lse, scratch, kNoAllocScratchBytes, stream);
}
