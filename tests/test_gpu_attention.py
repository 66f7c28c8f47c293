"""Step 3 parity: gather + dequantise + sparse attention with the FP8 window,
against the fp64 oracle (tolerance 2e-3 + 1e-2 * |ref|)."""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth
from helpers import within_tol

pytestmark = pytest.mark.gpu


def _setup(cuda, orc, lens, window=128, seed=21):
    B, Lmax = len(lens), max(lens)
    stride = (Lmax + 63) // 64 * 64
    kv = cuda.Cache.contiguous(cuda.FMT_FP4_KV, B, stride)
    xs = [synth.normal_rows(seed, "ak", (b,), 0, L, 512) for b, L in enumerate(lens)]
    src = np.zeros((B, Lmax, 512), np.float32)
    for b, x in enumerate(xs):
        src[b, :x.shape[0]] = x
    cuda.csa2_quantize_kv(torch.from_numpy(src).cuda(), kv,
                          seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    ring = cuda.Cache.contiguous(cuda.FMT_FP8_SWA, B, (max(window, 4) + 3) // 4 * 4)
    sw = np.zeros((B, max(window, 1), 512), np.float32)
    sref = []
    for b, L in enumerate(lens):
        n = min(window, L)
        v = synth.normal_rows(seed, "aw", (b,), 0, n, 512)
        sw[b, :n] = v
        sref.append(orc.quant_fp8(v))
    if window:
        start = torch.tensor([L - min(window, L) for L in lens], dtype=torch.int32, device="cuda")
        cuda.csa2_quantize_kv(torch.from_numpy(sw).cuda(), ring, start_pos=start,
                              seq_lens=torch.tensor(lens, dtype=torch.int32, device="cuda"))
    kref = [orc.quant_fp4(x) for x in xs]
    q = np.stack([synth.normal_rows(seed, "aq", (b,), 0, 16, 512, scale=1 / np.sqrt(512)) for b in range(B)])
    return kv, ring, kref, sref, q


def _idx(lens, K, seed):
    rs = np.random.default_rng(seed)
    out = np.full((len(lens), K), -1, np.int32)
    for b, L in enumerate(lens):
        n = min(K, L)
        out[b, :n] = np.sort(rs.choice(L, n, replace=False))
        # a few holes and repeats are legal inputs
        if n > 4:
            out[b, 1] = -1
            out[b, 3] = out[b, 2]
    return out


@pytest.mark.parametrize("lens,K,window", [([5000, 700, 90], 512, 128), ([3000], 2048, 128), ([257] * 40, 256, 128),
                                           ([1000, 2000], 512, 0), ([4000], 100, 17)])
def test_sparse_attention(cuda, orc, lens, K, window):
    kv, ring, kref, sref, q = _setup(cuda, orc, lens, window)
    idx = _idx(lens, K, 5)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, lse = cuda.csa2_sparse_attn(kv, ring if window else None, torch.from_numpy(q).cuda(), seq, max(lens),
                                     torch.from_numpy(idx).cuda(), K, window)
    st, flags = cuda.csa2_check_device()
    assert st == 0, flags
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(len(lens)):
        sc, ss = sref[b] if window else (None, None)
        ro, rl = orc.sparse_attention(q[b], kref[b][0], kref[b][1], idx[b], sc, ss)
        ok, ex = within_tol(out[b], ro)
        assert ok, (b, ex)
        assert np.allclose(lse[b], rl, atol=2e-3, rtol=1e-3), b


def test_swa_only(cuda, orc):
    lens = [300, 50]
    kv, ring, kref, sref, q = _setup(cuda, orc, lens, 128)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, lse = cuda.csa2_sparse_attn(None, ring, torch.from_numpy(q).cuda(), seq, max(lens), None, 0, 128)
    out = out.cpu().numpy()
    for b in range(2):
        ro, _ = orc.sparse_attention(q[b], kref[b][0], kref[b][1], np.zeros(0, np.int32), *sref[b])
        ok, ex = within_tol(out[b], ro)
        assert ok, (b, ex)


def test_out_of_range_index_is_flagged(cuda, orc):
    lens = [500]
    kv, ring, kref, sref, q = _setup(cuda, orc, lens, 128)
    idx = np.arange(64, dtype=np.int32)[None].copy()
    idx[0, 5] = 999  # >= seq_lens: skipped and flagged
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    out, _ = cuda.csa2_sparse_attn(kv, ring, torch.from_numpy(q).cuda(), seq, 500, torch.from_numpy(idx).cuda(), 64, 128)
    st, flags = cuda.csa2_check_device()
    assert st == cuda.ERR_INVALID_ARG and (flags & 1)
    idx[0, 5] = -1
    ro, _ = orc.sparse_attention(q[0], kref[0][0], kref[0][1], idx[0], *sref[0])
    ok, ex = within_tol(out[0].cpu().numpy(), ro)
    assert ok, ex
