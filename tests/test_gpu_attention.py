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


# ---- logits far from uniform: the running maximum moves, partials far apart ----------
# Unit-scale queries give logits of spread ~1, so a tile's maximum never leaves
# the running one and every CTA's partial has about the same maximum.  The
# cases below scale the queries (logits spanning tens of units) and arrange the
# rows so that the online softmax must move its maximum inside a CTA (a later
# tile larger by more than the lazy threshold) and the cluster merge must
# combine partials whose maxima differ by tens of units.  Without the O
# rescale the fp16 weights of such a tile would overflow (e^30 and more), so a
# result within tolerance shows that the rescale ran.

def _rows_growing(lens, seed, growth):
    return [synth.normal_rows(seed, "ak", (b,), 0, L, 512) * (1.0 + growth * np.arange(L, dtype=np.float32)[:, None] / L)
            for b, L in enumerate(lens)]


def _setup_rows(cuda, orc, xs, window, seed, wscale=1.0):
    lens = [x.shape[0] for x in xs]
    B, Lmax = len(lens), max(lens)
    stride = (Lmax + 63) // 64 * 64
    kv = cuda.Cache.contiguous(cuda.FMT_FP4_KV, B, stride)
    src = np.zeros((B, Lmax, 512), np.float32)
    for b, x in enumerate(xs):
        src[b, :x.shape[0]] = x
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(src).cuda(), kv, seq_lens=seq)
    ring = cuda.Cache.contiguous(cuda.FMT_FP8_SWA, B, max(4, (window + 3) // 4 * 4))
    sref = []
    if window:
        sw = np.zeros((B, window, 512), np.float32)
        for b, L in enumerate(lens):
            n = min(window, L)
            v = (synth.normal_rows(seed, "aw", (b,), 0, n, 512) * np.float32(wscale)).astype(np.float32)
            sw[b, :n] = v
            sref.append(orc.quant_fp8(v))
        start = torch.tensor([L - min(window, L) for L in lens], dtype=torch.int32, device="cuda")
        cuda.csa2_quantize_kv(torch.from_numpy(sw).cuda(), ring, start_pos=start, seq_lens=seq)
    kref = [orc.quant_fp4(x) for x in xs]
    return kv, ring, kref, sref, seq


def _check_against_oracle(cuda, orc, kv, ring, kref, sref, seq, q, idx, K, window):
    lens = seq.cpu().numpy().tolist()
    out, lse = cuda.csa2_sparse_attn(kv, ring if window else None, torch.from_numpy(q).cuda(), seq, max(lens),
                                     torch.from_numpy(idx).cuda() if idx is not None else None, K, window)
    st, flags = cuda.csa2_check_device()
    assert st == 0, flags
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for b in range(len(lens)):
        sc, ss = sref[b] if window else (None, None)
        ib = idx[b] if idx is not None else np.zeros(0, np.int32)
        ro, rl = orc.sparse_attention(q[b], kref[b][0], kref[b][1], ib, sc, ss)
        ok, ex = within_tol(out[b], ro)
        assert ok, (b, ex)
        assert np.allclose(lse[b], rl, atol=2e-3, rtol=1e-5), (b, np.abs(lse[b] - rl).max())


@pytest.mark.parametrize("qscale", [8.0, 32.0, 64.0])
def test_scaled_queries(cuda, orc, qscale):
    lens, K, window = [5000, 700, 3000], 2048, 128
    kv, ring, kref, sref, q = _setup(cuda, orc, lens, window, seed=31)
    q = (q * np.float32(qscale)).astype(np.float32)
    idx = _idx(lens, K, 7)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    _check_against_oracle(cuda, orc, kv, ring, kref, sref, seq, q, idx, K, window)


@pytest.mark.parametrize("qscale", [16.0, 64.0])
def test_each_later_tile_holds_a_larger_maximum(cuda, orc, qscale):
    """Row magnitude grows with position and the selection is ascending, so in
    every CTA each later 128-row tile holds a larger logit maximum than the
    earlier ones (8,192 selected rows: several tiles per CTA)."""
    L, K, window = 20000, 8192, 128
    xs = _rows_growing([L], 33, growth=3.0)
    kv, ring, kref, sref, seq = _setup_rows(cuda, orc, xs, window, 34)
    q = (synth.normal_rows(35, "aq", (0,), 0, 16, 512, scale=1 / np.sqrt(512)) * np.float32(qscale))[None]
    idx = np.sort(np.random.default_rng(3).choice(L, K, replace=False)).astype(np.int32)[None]
    _check_against_oracle(cuda, orc, kv, ring, kref, sref, seq, q.astype(np.float32), idx, K, window)


def test_window_holds_the_maximum(cuda, orc):
    """The FP8 window rows are four times larger than the selected rows: the
    maximum of every head lies in the window tile, the selected rows' partials
    are tens of units below it."""
    L, K, window = 6000, 2048, 128
    xs = [synth.normal_rows(36, "ak", (0,), 0, L, 512)]
    kv, ring, kref, sref, seq = _setup_rows(cuda, orc, xs, window, 37, wscale=4.0)
    q = (synth.normal_rows(38, "aq", (0,), 0, 16, 512, scale=1 / np.sqrt(512)) * np.float32(16.0))[None]
    idx = np.sort(np.random.default_rng(4).choice(L - window, K, replace=False)).astype(np.int32)[None]
    _check_against_oracle(cuda, orc, kv, ring, kref, sref, seq, q.astype(np.float32), idx, K, window)


def test_one_selected_row_among_holes(cuda, orc):
    """Every index -1 except one, no window: the output is that row."""
    L, K = 3000, 2048
    xs = [synth.normal_rows(39, "ak", (0,), 0, L, 512)]
    kv, ring, kref, sref, seq = _setup_rows(cuda, orc, xs, 0, 40)
    q = synth.normal_rows(41, "aq", (0,), 0, 16, 512, scale=1 / np.sqrt(512))[None]
    idx = np.full((1, K), -1, np.int32)
    idx[0, 1500] = 1234
    _check_against_oracle(cuda, orc, kv, ring, kref, sref, seq, q, idx, K, 0)
    out, _ = cuda.csa2_sparse_attn(kv, None, torch.from_numpy(q).cuda(), seq, L, torch.from_numpy(idx).cuda(), K, 0)
    row = orc.dequant_fp4(kref[0][0][1234:1235], kref[0][1][1234:1235])[0]
    assert np.array_equal(out[0].cpu().numpy().astype(np.float64), np.broadcast_to(row, (16, 512)))
