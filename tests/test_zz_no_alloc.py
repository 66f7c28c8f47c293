"""csa2_sparse_attn_noalloc: attention for callers that cannot allocate.

Some callers of this library cannot give it a workspace: a serving process
that reserved nearly all device memory for its cache pool when it started (a
cudaMalloc would fail, and would synchronise the device), or a plugin that
runs under another runtime's allocator.  The entry point takes the scratch
that a sequence split over several clusters needs from a 1 MiB array the
library owns, and plans its launch to fit it.  This file checks it through
the C interface against the oracle, against csa2_sparse_attn given a 1 MiB
workspace (the same plan, so bit-identical) and against csa2_sparse_attn with
its full workspace (within tolerance), on two calls in a row with different
inputs, at batch 2 and batch 32.  The second call finds the array as the
first left it, so it also checks that the split merge's tickets reset
themselves.  It is named to run last and builds its own inputs, so it passes
alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth
from helpers import within_tol

pytestmark = pytest.mark.gpu


def _inputs(cuda, orc, lens, K, window, seed):
    B, Lmax = len(lens), max(lens)
    stride = (Lmax + 63) // 64 * 64
    kv = cuda.Cache.contiguous(cuda.FMT_FP4_KV, B, stride)
    src = np.zeros((B, Lmax, 512), np.float32)
    for b, L in enumerate(lens):
        src[b, :L] = synth.normal_rows(seed, "na_kv", (b,), 0, L, 512)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(src).cuda(), kv, seq_lens=seq)
    ring = cuda.Cache.contiguous(cuda.FMT_FP8_SWA, B, (window + 3) // 4 * 4)
    sw = np.zeros((B, window, 512), np.float32)
    sref = []
    for b, L in enumerate(lens):
        n = min(window, L)
        v = synth.normal_rows(seed, "na_sw", (b,), 0, n, 512)
        sw[b, :n] = v
        sref.append(orc.quant_fp8(v))
    start = torch.tensor([L - min(window, L) for L in lens], dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(sw).cuda(), ring, start_pos=start, seq_lens=seq)
    rs = np.random.default_rng(seed)
    idx = np.full((B, K), -1, np.int32)
    for b, L in enumerate(lens):
        n = min(K, L)
        idx[b, :n] = np.sort(rs.choice(L, n, replace=False))
    q = np.stack([synth.normal_rows(seed, "na_q", (b,), 0, 16, 512, scale=1 / np.sqrt(512)) for b in range(B)])
    kref = [orc.quant_fp4(src[b, :L]) for b, L in enumerate(lens)]
    return kv, ring, seq, idx, q, kref, sref


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _noalloc(cuda, kv, ring, q, seq, Lmax, idx, K, window):
    """Calls the entry point through the C interface (ctypes), as a plugin would."""
    lib = cuda.load()
    B = q.shape[0]
    out = torch.empty_like(q)
    lse = torch.empty((B, 16), dtype=torch.float32, device=q.device)
    st = lib.csa2_sparse_attn_noalloc(kv.ref, ring.ref, _ptr(q), B, 16, 512, _ptr(seq), Lmax, _ptr(idx), K,
                                      window, _ptr(out), _ptr(lse),
                                      ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == cuda.OK, lib.csa2_last_error().decode()
    return out, lse


def _with_workspace(cuda, kv, ring, q, seq, Lmax, idx, K, window, nbytes):
    """csa2_sparse_attn through the C interface with a zeroed workspace of nbytes."""
    lib = cuda.load()
    B = q.shape[0]
    out = torch.empty_like(q)
    lse = torch.empty((B, 16), dtype=torch.float32, device=q.device)
    ws = torch.zeros(max(nbytes, 256), dtype=torch.uint8, device=q.device)
    st = lib.csa2_sparse_attn(kv.ref, ring.ref, _ptr(q), B, 16, 512, _ptr(seq), Lmax, _ptr(idx), K, window,
                              _ptr(out), _ptr(lse), _ptr(ws), ctypes.c_size_t(nbytes),
                              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == cuda.OK, lib.csa2_last_error().decode()
    return out, lse


@pytest.mark.parametrize("lens", [[9000, 2500], [3000 + 37 * b for b in range(32)]])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(cuda, orc, lens):
    K, window = 2048, 128
    for call, seed in enumerate((71, 72)):
        kv, ring, seq, idx, q, kref, sref = _inputs(cuda, orc, lens, K, window, seed)
        qd, idd = torch.from_numpy(q).cuda(), torch.from_numpy(idx).cuda()
        args = (cuda, kv, ring, qd, seq, max(lens), idd, K, window)
        same_out, same_lse = _with_workspace(*args, 1 << 20)
        full_out, full_lse = cuda.csa2_sparse_attn(kv, ring, qd, seq, max(lens), idd, K, window)
        out, lse = _noalloc(*args)
        torch.cuda.synchronize()
        out_h, lse_h = out.cpu().numpy(), lse.cpu().numpy()
        # the same kernels and the same plan: bit-identical to a 1 MiB workspace
        assert np.array_equal(out_h, same_out.cpu().numpy()), f"call {call}"
        assert np.array_equal(lse_h, same_lse.cpu().numpy()), f"call {call}"
        # a larger workspace may split differently: the merge order changes
        # the rounding, not the result beyond it
        ok, ex = within_tol(out_h, full_out.cpu().numpy())
        assert ok, f"call {call}: noalloc vs full workspace excess {ex:.3e}"
        assert np.allclose(lse_h, full_lse.cpu().numpy(), atol=1e-4, rtol=1e-6), f"call {call}"
        for b in (0, len(lens) // 2, len(lens) - 1):
            ro, rl = orc.sparse_attention(q[b], kref[b][0], kref[b][1], idx[b], *sref[b])
            ok, ex = within_tol(out_h[b], ro)
            assert ok, f"call {call}, sequence {b}: output excess {ex:.3e}"
            assert np.allclose(lse_h[b], rl, atol=2e-3, rtol=1e-5), f"call {call}, sequence {b}: lse"
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)
