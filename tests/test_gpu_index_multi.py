"""Multi-query indexer scoring on the tensor cores (several tokens of one
sequence index at once: Helmcode "DeepSeek V4.1 Flash" explainer, "10 · other
changes": a speculative verification checks several drafted tokens together;
"03 · CSA2": the indexing path in prefill).  Every query row must equal the
oracle's single-query scores bit for bit over its candidates (the causal
prefix, or every position), and its Top-K index set exactly; the rows must
also equal the decode path's single-query call on the same keys."""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth

pytestmark = pytest.mark.gpu


def _keys(cuda, orc, lens, seed, paged=False, const=False):
    B, Lmax = len(lens), max(max(lens), 1)
    xs = [synth.normal_rows(seed, "mk", (b,), 0, L, 64) for b, L in enumerate(lens)]
    if const:  # every key the same: every score ties
        xs = [np.tile(synth.normal_rows(seed, "mk1", (0,), 0, 1, 64), (L, 1)) for L in lens]
    src = np.zeros((B, Lmax, 64), np.float32)
    for b, x in enumerate(xs):
        src[b, :x.shape[0]] = x
    if paged:
        page = 128
        per = (Lmax + page - 1) // page
        perm = np.random.default_rng(seed).permutation(B * per + 3)[:B * per].reshape(B, per)
        cache = cuda.Cache.paged(cuda.FMT_FP4_IDX, B * per + 3, page, torch.from_numpy(perm.astype(np.int32)).cuda())
    else:
        cache = cuda.Cache.contiguous(cuda.FMT_FP4_IDX, B, (Lmax + 63) // 64 * 64)
    lens_t = torch.tensor(lens, dtype=torch.int32, device="cuda")
    cuda.csa2_quantize_kv(torch.from_numpy(src).cuda(), cache, seq_lens=lens_t)
    ref = [orc.quant_fp4(x) if x.shape[0] else (np.zeros((0, 32), np.uint8), np.zeros((0, 4), np.uint8))
           for x in xs]
    return cache, ref


def _queries(B, n_q, seed):
    q = np.stack([synth.normal_rows(seed, "mq", (b,), 0, n_q * 4, 64, scale=0.125).reshape(n_q, 4, 64)
                  for b in range(B)])
    w = np.stack([synth.uniform(seed, "mw", (b,), (n_q, 4)) for b in range(B)]).astype(np.float32)
    return np.ascontiguousarray(q), np.ascontiguousarray(w)


def _check_rows(orc, q, w, ref, lens, K, causal, idx, sc):
    for b, L in enumerate(lens):
        want_sc, want_idx = orc.index_topk_multi(q[b], w[b], ref[b][0], ref[b][1], L, K, causal)
        for i in range(q.shape[1]):
            n = want_sc[i].shape[0]
            if sc is not None:
                assert np.array_equal(sc[b, i, :n].view(np.uint32), want_sc[i].view(np.uint32)), (b, i)
            if idx is not None:
                assert np.array_equal(idx[b, i], want_idx[i]), (b, i)


@pytest.mark.parametrize("lens,n_q,K,causal", [
    ([3000], 8, 256, True),            # a speculative verification of 8 tokens
    ([1000, 4113], 32, 512, True),     # ragged batch, one full query group, ragged last tile
    ([5000], 45, 100, True),           # two query groups, the second partial
    ([700, 300], 5, 2048, False),      # every position, K above the candidates (-1 padding)
    ([10], 16, 4, True),               # more queries than positions: early rows have none
    ([0, 200], 3, 8, True),            # an empty sequence
    ([70000], 32, 2048, True),         # several tiles per CTA
    ([1500, 999], 100, 64, False),     # four query groups per sequence, every position
    ([4097], 33, 4097, True),          # Top-K as large as the context, a one-row second group
])
def test_multi_query_scores_and_topk(cuda, orc, lens, n_q, K, causal):
    B, Lmax = len(lens), max(lens)
    cache, ref = _keys(cuda, orc, lens, 31 + n_q)
    q, w = _queries(B, n_q, 7 + n_q)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx, sc = cuda.csa2_index_topk_multi(cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), seq,
                                         max(Lmax, 1), K, causal=causal, with_scores=True)
    st, flags = cuda.csa2_check_device()
    assert st == 0, (flags, cuda.csa2_last_error())
    _check_rows(orc, q, w, ref, lens, K, causal, idx.cpu().numpy(), sc.cpu().numpy())


def test_paged_keys_and_scores_only(cuda, orc):
    lens = [2500, 1301]
    cache, ref = _keys(cuda, orc, lens, 77, paged=True)
    q, w = _queries(2, 12, 78)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx, sc = cuda.csa2_index_topk_multi(cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), seq,
                                         2560, 64, with_idx=False, with_scores=True)
    assert idx is None
    st, flags = cuda.csa2_check_device()
    assert st == 0, flags
    _check_rows(orc, q, w, ref, lens, 64, True, None, sc.cpu().numpy())
    idx, _ = cuda.csa2_index_topk_multi(cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), seq,
                                        2560, 64)
    _check_rows(orc, q, w, ref, lens, 64, True, idx.cpu().numpy(), None)


def test_all_scores_tied_take_the_lowest_positions(cuda, orc):
    lens = [3333]
    cache, ref = _keys(cuda, orc, lens, 5, const=True)
    q, w = _queries(1, 9, 6)
    seq = torch.tensor(lens, dtype=torch.int32, device="cuda")
    idx, _ = cuda.csa2_index_topk_multi(cache, torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda(), seq,
                                        3333, 1000)
    idx = idx.cpu().numpy()
    _check_rows(orc, q, w, ref, lens, 1000, True, idx, None)
    assert np.array_equal(idx[0, 0], np.arange(1000, dtype=np.int32))


def test_rows_equal_the_single_query_decode_call(cuda, orc):
    """Row i of the multi-query call with causal prefixes = csa2_index_topk
    (Full) for query i with seq_len = its prefix length."""
    L, n_q, K = 4000, 6, 300
    cache, _ = _keys(cuda, orc, [L], 90)
    q, w = _queries(1, n_q, 91)
    qd, wd = torch.from_numpy(q).cuda(), torch.from_numpy(w).cuda()
    seq = torch.tensor([L], dtype=torch.int32, device="cuda")
    idx, sc = cuda.csa2_index_topk_multi(cache, qd, wd, seq, L, K, with_scores=True)
    for i in range(n_q):
        n = L - n_q + i + 1
        one_idx, _, one_sc = cuda.csa2_index_topk(cuda.MODE_FULL, cache, qd[:, i].contiguous(), wd[:, i].contiguous(),
                                                  torch.tensor([n], dtype=torch.int32, device="cuda"), L, K,
                                                  with_scores=True)
        assert torch.equal(idx[0, i], one_idx[0]), i
        assert torch.equal(sc[0, i, :n].view(torch.int32), one_sc[0, :n].view(torch.int32)), i
    st, flags = cuda.csa2_check_device()
    assert st == 0, flags
