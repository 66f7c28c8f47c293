"""Step 2 parity: indexer scores bit-exact and Top-K index sets identical to the
oracle (Full, Reindex over a pool, the Full layer's pool, ties, tiny and
ties that span the select cluster's slices)."""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth

pytestmark = pytest.mark.gpu


def _keys(cuda, orc, xk_list, stride):
    """Build a contiguous FP4 indexer cache for B sequences; return (cache, oracle codes/scales)."""
    B = len(xk_list)
    cache = cuda.Cache.contiguous(cuda.FMT_FP4_IDX, B, stride)
    Lmax = max(x.shape[0] for x in xk_list)
    src = np.zeros((B, max(Lmax, 1), 64), np.float32)
    for b, x in enumerate(xk_list):
        src[b, :x.shape[0]] = x
    lens = torch.tensor([x.shape[0] for x in xk_list], dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(src).cuda(), cache, seq_lens=lens)
    ref = [orc.quant_fp4(x) if x.shape[0] else (np.zeros((0, 32), np.uint8), np.zeros((0, 4), np.uint8))
           for x in xk_list]
    return cache, ref


def _queries(B, seed):
    q = np.stack([synth.normal_rows(seed, "tq", (b,), 0, 4, 64, scale=0.125) for b in range(B)])
    w = np.stack([synth.uniform(seed, "tw", (b,), (4,)) for b in range(B)])
    return q, w


@pytest.mark.parametrize("lens,K", [([1000, 4113], 512), ([37, 1], 64), ([5000, 2500, 64], 1), ([3000], 2048)])
def test_full_scores_and_topk(cuda, orc, lens, K):
    B = len(lens)
    xs = [synth.normal_rows(11, "tk", (b,), 0, L, 64) for b, L in enumerate(lens)]
    Lmax = max(lens)
    cache, ref = _keys(cuda, orc, xs, (Lmax + 63) // 64 * 64)
    q, w = _queries(B, 3)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx, _, sc = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                      seq, Lmax, K, with_scores=True)
    st, flags = cuda.csa2_check_device()
    assert st == 0, flags
    idx = idx.cpu().numpy()
    sc = sc.cpu().numpy()
    for b, L in enumerate(lens):
        want_sc = orc.index_scores(q[b], w[b], ref[b][0], ref[b][1])
        assert np.array_equal(sc[b, :L].view(np.uint32), want_sc.view(np.uint32)), b
        want = orc.topk(want_sc, np.arange(L, dtype=np.int32), K)
        assert np.array_equal(idx[b], want), b


def test_reindex_over_pool_and_full_pool_output(cuda, orc):
    lens = [6000, 3001]
    B, K, P = 2, 256, 1024
    xs = [synth.normal_rows(12, "tk", (b,), 0, L, 64) for b, L in enumerate(lens)]
    cache, ref = _keys(cuda, orc, xs, 6016)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    qf, wf = _queries(B, 4)
    out_pool = torch.empty((B, P), dtype=torch.int32, device="cuda")
    idx_f, pool, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(qf).cuda(),
                                          torch.from_numpy(wf).cuda(), seq, 6000, K, out_pool=out_pool)
    qr, wr = _queries(B, 5)
    idx_r, _, sc = cuda.csa2_index_topk(cuda.MODE_REINDEX, cache, torch.from_numpy(qr).cuda(),
                                        torch.from_numpy(wr).cuda(), seq, 6000, K, pool=pool, with_scores=True)
    st, _ = cuda.csa2_check_device()
    assert st == 0
    pool_h = pool.cpu().numpy()
    for b, L in enumerate(lens):
        s_f = orc.index_scores(qf[b], wf[b], ref[b][0], ref[b][1])
        allpos = np.arange(L, dtype=np.int32)
        assert np.array_equal(idx_f[b].cpu().numpy(), orc.topk(s_f, allpos, K))
        want_pool = orc.topk(s_f, allpos, P)
        assert np.array_equal(pool_h[b], want_pool)
        cand = want_pool[want_pool >= 0]
        s_r = orc.index_scores(qr[b], wr[b], ref[b][0][cand], ref[b][1][cand])
        assert np.array_equal(idx_r[b].cpu().numpy(), orc.topk(s_r, cand, K))
        assert np.array_equal(sc[b, :cand.size].cpu().numpy().view(np.uint32), s_r.view(np.uint32))


def test_ties_take_lower_positions(cuda, orc):
    """Rows repeat in blocks, so equal scores abound; ties go to lower positions."""
    L, K = 4096, 300
    base = synth.normal_rows(13, "tk", (0,), 0, 40, 64)
    x = base[np.random.default_rng(2).integers(0, 40, L)]
    cache, ref = _keys(cuda, orc, [x], L)
    q, w = _queries(1, 6)
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                     seq, L, K)
    s = orc.index_scores(q[0], w[0], ref[0][0], ref[0][1])
    assert np.array_equal(idx[0].cpu().numpy(), orc.topk(s, np.arange(L, dtype=np.int32), K))


def test_all_equal_scores_take_lowest_positions(cuda, orc):
    """20,000 identical keys: every radix digit ties, the tie quota spreads over
    the select cluster's slices, and positions 0..K-1 win."""
    L, K = 20000, 100
    x = np.tile(synth.normal_rows(14, "tk", (0,), 0, 1, 64), (L, 1))
    cache, _ = _keys(cuda, orc, [x], 20032)
    q, w = _queries(1, 7)
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                     seq, L, K)
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)
    assert np.array_equal(idx[0].cpu().numpy(), np.arange(K))
    # a quota that crosses slice boundaries: K larger than one slice (L / 8)
    K2 = 5000
    idx2, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(),
                                      torch.from_numpy(w).cuda(), seq, L, K2)
    assert np.array_equal(idx2[0].cpu().numpy(), np.arange(K2))


@pytest.mark.parametrize("K", [3000, 7777])
def test_few_distinct_scores_over_many_keys(cuda, orc, K):
    """60,000 keys drawn from 40 distinct rows: each score value is shared by
    ~1,500 keys, so the threshold bin overflows the candidate list at every
    digit (coarse, 16-bit, the refining digits) and the ties at the
    threshold are split by position."""
    L = 60000
    rows = synth.normal_rows(15, "tk", (0,), 0, 40, 64)
    pick = np.random.default_rng(15).integers(0, 40, L)
    x = rows[pick]
    cache, ref = _keys(cuda, orc, [x], 60032)
    q, w = _queries(1, 8)
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx, _, sc = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                      seq, L, K, with_scores=True)
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)
    s = orc.index_scores(q[0], w[0], ref[0][0], ref[0][1])
    assert np.array_equal(sc[0].cpu().numpy().view(np.uint32), s.view(np.uint32))
    assert np.array_equal(idx[0].cpu().numpy(), orc.topk(s, np.arange(L, dtype=np.int32), K))


def test_extreme_codes_are_exact(cuda, orc):
    """Keys and queries at the E2M1 extremes (every code +-6, the largest and
    smallest E4M3 scales): the tensor-core block sums stay exact."""
    rs = np.random.default_rng(9)
    L = 2048
    mags = np.array([6.0, -6.0, 0.5, -0.5, 4.0, 3.0], np.float32)
    x = mags[rs.integers(0, mags.size, (L, 64))] * (2.0 ** rs.integers(-9, 7, (L, 1))).astype(np.float32)
    cache, ref = _keys(cuda, orc, [x], L)
    q = (mags[rs.integers(0, mags.size, (1, 4, 64))] * np.float32(2.0 ** 6)).astype(np.float32)
    w = np.ones((1, 4), np.float32)
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx, _, sc = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                      seq, L, 128, with_scores=True)
    s = orc.index_scores(q[0], w[0], ref[0][0], ref[0][1])
    assert np.array_equal(sc[0].cpu().numpy().view(np.uint32), s.view(np.uint32))
    assert np.array_equal(idx[0].cpu().numpy(), orc.topk(s, np.arange(L, dtype=np.int32), 128))


def test_fewer_candidates_than_k_pads(cuda, orc):
    L, K = 10, 64
    x = synth.normal_rows(15, "tk", (0,), 0, L, 64)
    cache, ref = _keys(cuda, orc, [x], 64)
    q, w = _queries(1, 8)
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                     seq, 64, K)
    got = idx[0].cpu().numpy()
    assert np.array_equal(got[:L], np.arange(L)) and (got[L:] == -1).all()


def test_batched_fallback_path(cuda, orc):
    """64 sequences of up to 20,000 keys do not fit one co-resident launch:
    the scan + cluster-select kernels take the call, with the same result."""
    rs = np.random.default_rng(21)
    lens = rs.integers(12000, 20000, 64).tolist()
    xs = [synth.normal_rows(22, "tk", (b,), 0, L, 64) for b, L in enumerate(lens)]
    Lmax = max(lens)
    cache, ref = _keys(cuda, orc, xs, (Lmax + 63) // 64 * 64)
    q, w = _queries(64, 23)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    K = 256
    idx, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                     seq, Lmax, K)
    st, flags = cuda.csa2_check_device()
    assert st == 0, flags
    idx = idx.cpu().numpy()
    for b, L in enumerate(lens):
        s = orc.index_scores(q[b], w[b], ref[b][0], ref[b][1])
        assert np.array_equal(idx[b], orc.topk(s, np.arange(L, dtype=np.int32), K)), b


def test_forced_wait_expiry_reports_timeout(cuda, orc):
    """With the first tile wait limited to zero polls every CTA records a
    timeout, then still waits (normal bound) for its copies: the call reports
    CSA2_ERR_TIMEOUT, its result is still right, and the next call is clean."""
    L, K = 3000, 256
    x = synth.normal_rows(24, "tk", (0,), 0, L, 64)
    cache, ref = _keys(cuda, orc, [x], 3008)
    q, w = _queries(1, 25)
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    want = orc.topk(orc.index_scores(q[0], w[0], ref[0][0], ref[0][1]), np.arange(L, dtype=np.int32), K)
    cuda.csa2_test_set_wait_limit(0)
    try:
        idx, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(),
                                         torch.from_numpy(w).cuda(), seq, L, K)
        st, flags = cuda.csa2_check_device()
    finally:
        cuda.csa2_test_set_wait_limit(-1)
    assert st == cuda.ERR_TIMEOUT and (flags & 2), (st, flags)
    assert np.array_equal(idx[0].cpu().numpy(), want)
    idx, _, _ = cuda.csa2_index_topk(cuda.MODE_FULL, cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(),
                                     seq, L, K)
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)
    assert np.array_equal(idx[0].cpu().numpy(), want)
