// csa2_sparse_attn_noalloc: the gather-attention entry point for callers that
// cannot allocate device memory.
//
// Some callers cannot hand this library a workspace: a serving process that
// reserved nearly all HBM for its KV-cache pool at start-up (a cudaMalloc
// then fails, and it would synchronise the device anyway), or a plugin that
// runs inside another runtime's allocator and has no way to ask it for
// scratch.  This variant runs the same attention kernels as
// csa2_sparse_attn, with the split partials placed in a fixed array that the
// library owns for the life of the process instead of in a caller workspace.
#include "internal.h"

namespace {

// Scratch for the split partials: 4 MiB, held on every device that loads the
// library until the process exits.  Shared by every call on a device.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_attn_scratch[kNoAllocScratchBytes];

// Device address of g_attn_scratch on the current device, looked up once per
// device (with that device current) on its first use.  Host code must not
// use the symbol itself: on the host it names a stand-in, not device memory.
cudaError_t scratch_address(void **out)
{
    static void *cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!cache[dev]) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_attn_scratch);
        if (e != cudaSuccess) return e;
        cache[dev] = p;
    }
    *out = cache[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" csa2_status csa2_sparse_attn_noalloc(const csa2_cache *kv, const csa2_cache *swa, const float *q,
                                                int32_t batch, int32_t n_heads, int32_t head_dim,
                                                const int32_t *seq_lens, int32_t max_seq_len, const int32_t *idx,
                                                int32_t topk, int32_t swa_window, float *out, float *lse,
                                                void *stream)
{
    const size_t need = csa2::sparse_attn_workspace_within(batch, idx ? topk : 0, swa_window, kNoAllocScratchBytes);
    if (need > kNoAllocScratchBytes)
        return csa2::set_error(CSA2_ERR_UNSUPPORTED,
                               "csa2_sparse_attn_noalloc: this call needs %zu bytes of scratch, more than the "
                               "%zu-byte static maximum; use csa2_sparse_attn with a workspace",
                               need, kNoAllocScratchBytes);
    void *scratch = nullptr;
    const cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return csa2::set_error(CSA2_ERR_CUDA, "csa2_sparse_attn_noalloc: scratch address lookup: %s",
                               cudaGetErrorString(e));
    return csa2_sparse_attn(kv, swa, q, batch, n_heads, head_dim, seq_lens, max_seq_len, idx, topk, swa_window,
                            out, lse, scratch, kNoAllocScratchBytes, stream);
}
