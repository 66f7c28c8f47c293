"""Step 1 parity: packed bytes of the CUDA quantiser equal the oracle's, bit for bit."""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth

pytestmark = pytest.mark.gpu


def adversarial_rows(n, C, seed):
    """N(0,1) rows mixed with grid multiples, exact midpoints, zeros, signed
    zeros, tiny (scale underflow), huge (scale saturation) and isolated spikes."""
    rs = np.random.default_rng(seed)
    x = rs.standard_normal((n, C)).astype(np.float32)
    grid = np.array([0, .5, 1, 1.5, 2, 3, 4, 6, .25, .75, 1.25, 1.75, 2.5, 3.5, 5], np.float32)
    for r in range(n):
        kind = r % 9
        if kind == 1:
            s = np.float32(2.0 ** rs.integers(-9, 8))
            x[r] = grid[rs.integers(0, grid.size, C)] * s * np.where(rs.random(C) < .5, -1, 1)
        elif kind == 2:
            x[r] = 0.0
            x[r, rs.integers(0, C, 5)] = -0.0
        elif kind == 3:
            x[r] *= np.float32(1e-30)
        elif kind == 4:
            x[r] *= np.float32(1e30)
        elif kind == 5:
            x[r] = np.float32(1e-3) * x[r]
            x[r, rs.integers(0, C)] = 1e4
        elif kind == 6:
            x[r] = (rs.integers(-(2 ** 20), 2 ** 20, C) * 2.0 ** rs.integers(-40, 20)).astype(np.float32)
        elif kind == 7:
            x[r] = np.float32(6.0) * np.float32(2.0 ** rs.integers(-12, 10))
            x[r, ::3] *= -1
    return x


def random_bit_rows(n, C, seed):
    rs = np.random.default_rng(seed)
    bits = rs.integers(0, 2 ** 32, size=(n, C), dtype=np.uint64).astype(np.uint32)
    x = bits.view(np.float32).copy()
    bad = ~np.isfinite(x)
    x[bad] = 1.0
    return x


@pytest.mark.parametrize("maker", [adversarial_rows, random_bit_rows])
def test_fp4_kv_rows_bit_exact(cuda, orc, maker):
    n = 2048
    x = maker(n, 512, 1)
    cache = cuda.Cache.contiguous(cuda.FMT_FP4_KV, 1, n)
    cuda.csa2_quantize_kv(torch.from_numpy(x)[None].cuda(), cache)
    torch.cuda.synchronize()
    got = cache.data.cpu().numpy().reshape(n, 288)
    qc, qs = orc.quant_fp4(x)
    want = orc.kv_rows(qc, qs)
    assert np.array_equal(got, want), np.argwhere(got != want)[:5]


@pytest.mark.parametrize("maker", [adversarial_rows, random_bit_rows])
def test_fp4_idx_tiles_bit_exact(cuda, orc, maker):
    n = 64 * 70
    x = maker(n, 64, 2)
    cache = cuda.Cache.contiguous(cuda.FMT_FP4_IDX, 1, n)
    cuda.csa2_quantize_kv(torch.from_numpy(x)[None].cuda(), cache)
    torch.cuda.synchronize()
    got = cache.data.cpu().numpy()
    want = np.zeros_like(got)
    qc, qs = orc.quant_fp4(x)
    orc.place_idx(want, np.arange(n), qc, qs)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("maker", [adversarial_rows, random_bit_rows])
def test_fp8_swa_ring_bit_exact(cuda, orc, maker):
    B, W, L = 3, 128, [1000, 77, 128]
    x = maker(B * W, 512, 3).reshape(B, W, 512)
    ring = cuda.Cache.contiguous(cuda.FMT_FP8_SWA, B, W)
    start = torch.tensor([L[b] - min(W, L[b]) for b in range(B)], dtype=torch.int32, device="cuda")
    lens = torch.tensor(L, dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(x).cuda(), ring, start_pos=start, seq_lens=lens)
    torch.cuda.synchronize()
    got = ring.data.cpu().numpy()
    want = np.zeros_like(got)
    for b in range(B):
        n = min(W, L[b])
        pos = np.arange(L[b] - n, L[b])
        c, s = orc.quant_fp8(x[b, :n])
        orc.place_swa(want, B * W, orc.slots_contiguous(b, pos, W, ring=True), c, s)
    assert np.array_equal(got, want)


def test_paged_build_and_append(cuda, orc):
    """Build through a random page table, then append one token per sequence at
    seq_lens-1: the bytes read back through the table equal the oracle's."""
    B, L = 4, [130, 64, 1, 257]
    pages = [(l + 63) // 64 for l in L]
    perm = np.random.default_rng(5).permutation(sum(pages) + 2).astype(np.int32)
    table = np.full((B, max(pages)), -1, np.int32)
    k = 0
    for b in range(B):
        table[b, :pages[b]] = perm[k:k + pages[b]]
        k += pages[b]
    t = torch.from_numpy(table).cuda()
    n_pages = sum(pages) + 2
    kv = cuda.Cache.paged(cuda.FMT_FP4_KV, n_pages, 64, t)
    ik = cuda.Cache.paged(cuda.FMT_FP4_IDX, n_pages, 64, t)
    Lmax = max(L)
    xv = adversarial_rows(B * Lmax, 512, 6).reshape(B, Lmax, 512)
    xk = adversarial_rows(B * Lmax, 64, 7).reshape(B, Lmax, 64)
    lens_m1 = torch.tensor([l - 1 for l in L], dtype=torch.int32, device="cuda")
    lens = torch.tensor(L, dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(xv).cuda(), kv, seq_lens=lens_m1)
    cuda.csa2_quantize_kv(torch.from_numpy(xk).cuda(), ik, seq_lens=lens_m1)
    last_v = torch.from_numpy(np.stack([xv[b, L[b] - 1] for b in range(B)])[:, None]).cuda()
    last_k = torch.from_numpy(np.stack([xk[b, L[b] - 1] for b in range(B)])[:, None]).cuda()
    cuda.csa2_quantize_kv(last_v.contiguous(), kv, start_pos=lens_m1)
    cuda.csa2_quantize_kv(last_k.contiguous(), ik, start_pos=lens_m1)
    st, flags = cuda.csa2_check_device()
    assert st == 0 and flags == 0
    gv = kv.data.cpu().numpy()
    gk = ik.data.cpu().numpy()
    for b in range(B):
        slots = orc.slots_paged(table[b], np.arange(L[b]), 64)
        qc, qs = orc.quant_fp4(xv[b, :L[b]])
        assert np.array_equal(gv.reshape(-1, 288)[slots], orc.kv_rows(qc, qs))
        kc, ks = orc.quant_fp4(xk[b, :L[b]])
        rc, rsc = orc.read_idx(gk, slots)
        assert np.array_equal(rc, kc) and np.array_equal(rsc, ks)


def test_unmapped_page_is_flagged_not_faulted(cuda):
    t = torch.tensor([[0, -1]], dtype=torch.int32, device="cuda")
    kv = cuda.Cache.paged(cuda.FMT_FP4_KV, 2, 64, t)
    x = torch.ones((1, 128, 512), dtype=torch.float32, device="cuda")
    cuda.csa2_quantize_kv(x, kv)
    st, flags = cuda.csa2_check_device()
    assert st == cuda.ERR_INVALID_ARG and (flags & 1)
    # the mapped page was written, the physical page 1 untouched
    d = kv.data.cpu().numpy().reshape(-1, 288)
    assert (d[:64] != 0).any() and (d[64:] == 0).all()
    st, flags = cuda.csa2_check_device()
    assert st == 0 and flags == 0
