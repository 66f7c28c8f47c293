"""csa2_sparse_attn_noalloc: attention for callers that cannot allocate.

Some callers of this library cannot give it a workspace: a serving process
that reserved nearly all device memory for its cache pool when it started (a
cudaMalloc would fail, and would synchronise the device), or a plugin that
runs under another runtime's allocator.  The no-allocation entry point keeps
its split partials in a fixed 4 MiB array owned by the library.  This file
checks it through the C interface against csa2_sparse_attn with a workspace,
on two calls in a row with different inputs (the second must not see the
first call's partials), and checks that a call too large for the array is
refused with a message.  It is named to run last and builds its own inputs,
so it passes alone or after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth
from helpers import within_tol

pytestmark = pytest.mark.gpu


def _inputs(cuda, lens, K, window, seed):
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
    for b, L in enumerate(lens):
        n = min(window, L)
        sw[b, :n] = synth.normal_rows(seed, "na_sw", (b,), 0, n, 512)
    start = torch.tensor([L - min(window, L) for L in lens], dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(sw).cuda(), ring, start_pos=start, seq_lens=seq)
    rs = np.random.default_rng(seed)
    idx = np.full((B, K), -1, np.int32)
    for b, L in enumerate(lens):
        n = min(K, L)
        idx[b, :n] = np.sort(rs.choice(L, n, replace=False))
    q = np.stack([synth.normal_rows(seed, "na_q", (b,), 0, 16, 512, scale=1 / np.sqrt(512)) for b in range(B)])
    return kv, ring, seq, torch.from_numpy(idx).cuda(), torch.from_numpy(q).cuda()


def test_noalloc_matches_workspace_entry_point_twice(cuda):
    lens, K, window = [9000, 2500], 2048, 128
    # the split partials are in use: more than one chunk per sequence
    assert cuda.load().csa2_sparse_attn_workspace(len(lens), K, window) > 0
    for call, seed in enumerate((71, 72)):
        kv, ring, seq, idx, q = _inputs(cuda, lens, K, window, seed)
        ref_out, ref_lse = cuda.csa2_sparse_attn(kv, ring, q, seq, max(lens), idx, K, window)
        out, lse = cuda.csa2_sparse_attn_noalloc(kv, ring, q, seq, max(lens), idx, K, window)
        torch.cuda.synchronize()
        ok, ex = within_tol(out.cpu().numpy(), ref_out.cpu().numpy().astype(np.float64))
        assert ok, f"call {call}: output excess {ex:.3e}"
        ok, ex = within_tol(lse.cpu().numpy(), ref_lse.cpu().numpy().astype(np.float64))
        assert ok, f"call {call}: lse excess {ex:.3e}"
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)


def test_noalloc_refuses_calls_beyond_its_scratch(cuda):
    lib = cuda.load()
    B, K, window = 64, 2048, 128
    assert lib.csa2_sparse_attn_workspace(B, K, window) > (4 << 20)
    kv, ring, seq, idx, q = _inputs(cuda, [300], K, window, 73)
    st = lib.csa2_sparse_attn_noalloc(kv.ref, ring.ref, ctypes.c_void_p(q.data_ptr()), B, 16, 512,
                                      ctypes.c_void_p(seq.data_ptr()), 300, ctypes.c_void_p(idx.data_ptr()), K,
                                      window, ctypes.c_void_p(q.data_ptr()), None, None)
    assert st == cuda.ERR_UNSUPPORTED
    assert "static maximum" in lib.csa2_last_error().decode()
