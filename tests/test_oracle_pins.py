"""Pins of the CPU oracle to facts outside itself: the format definitions the
pages name (E2M1, E4M3), an independent library codec (torch's float8_e4m3fn),
closed forms, brute force on tiny inputs, and the mode invariants the pages
state (Helmcode explainer "03 · CSA2"; Louis Bouchard's report "Share the
cache and the search work"; 0x0moeen's note on shared indexer keys)."""
import math

import numpy as np
import pytest
import torch

from conftest import read_golden

from csa2_sparse_attention_03_b300 import synth

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _golden_e2m1():
    return {int(c, 16): float(v) for c, v in read_golden("e2m1_codes.txt")}


def _e4m3_lib(codes):
    """Independent E4M3 decode: torch's float8_e4m3fn."""
    t = torch.tensor(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn)
    return t.float().numpy().astype(np.float64)


# ---------------------------------------------------------------- E2M1

def test_e2m1_decode_matches_format_table(orc):
    table = _golden_e2m1()
    for c in range(16):
        v = orc.e2m1_decode(c)
        assert v == table[c] and math.copysign(1, v) == math.copysign(1, table[c]), c


def test_e2m1_roundtrip_all_codes(orc):
    for c in range(16):
        assert orc.e2m1_encode(orc.e2m1_decode(c)) == c


def test_e2m1_rounding_fixture(orc):
    for x, code in read_golden("e2m1_rounding.txt"):
        assert orc.e2m1_encode(float(np.float32(float(x)))) == int(code, 16), x


def test_e2m1_matches_scaled_rint(orc):
    """Independent formulation: on [1, 8) E2M1 is 2-significant-bit rounding,
    i.e. numpy's round-half-even of v * 2^(1-e) at the binade e; below 1 it is
    rint(2v)/2 (subnormal step 0.5)."""
    rs = np.random.default_rng(7)
    xs = np.concatenate([rs.uniform(-7, 7, 20000), rs.uniform(-1, 1, 5000),
                         np.arange(-28, 29) * 0.125, np.arange(-7, 8) * 0.25]).astype(np.float32)
    table = _golden_e2m1()
    for x in xs:
        a = abs(float(x))
        if a < 1.0:
            mag = float(np.rint(2 * a)) / 2
        else:
            e = math.floor(math.log2(a))
            step = 2.0 ** (e - 1)
            mag = float(np.rint(a / step)) * step
        mag = min(mag, 6.0)
        got = table[orc.e2m1_encode(x) & 7]
        assert got == mag, (x, got, mag)
        assert (orc.e2m1_encode(x) >> 3) == int(np.signbit(x))


# ---------------------------------------------------------------- E4M3

def test_e4m3_decode_matches_torch(orc):
    ref = _e4m3_lib(range(256))
    for c in range(256):
        v = orc.e4m3_decode(c)
        if np.isnan(ref[c]):
            assert math.isnan(v), c
        else:
            assert v == ref[c], (c, v, ref[c])
    assert orc.e4m3_decode(0x7E) == 448.0 and orc.e4m3_decode(0x01) == 2.0 ** -9


def test_e4m3_encode_matches_torch_in_range(orc):
    rs = np.random.default_rng(11)
    xs = np.concatenate([
        rs.uniform(-448, 448, 4000), rs.uniform(-1, 1, 4000), rs.uniform(-2 ** -5, 2 ** -5, 4000),
        # every midpoint between neighbouring finite magnitudes (ties)
        (_e4m3_lib(range(0, 126)) + _e4m3_lib(range(1, 127))) / 2,
    ]).astype(np.float32)
    lib = torch.tensor(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, ref in zip(xs, lib):
        assert orc.e4m3_encode(x) == int(ref), (x, orc.e4m3_encode(x), ref)


def test_e4m3_saturates(orc):
    for x in [448.0, 449.0, 463.9, 464.0, 500.0, 1e30, float("inf")]:
        assert orc.e4m3_encode(x) == 0x7E
        assert orc.e4m3_encode(-x) == 0xFE
    assert orc.e4m3_encode(-0.0) == 0x80


def test_e4m3_roundtrip_all_finite(orc):
    for c in range(256):
        if (c & 0x7F) == 0x7F:
            continue
        assert orc.e4m3_encode(orc.e4m3_decode(c)) == c


# ---------------------------------------------------------------- FP4 blocks

def test_fp4_block_exact_when_representable(orc):
    """absmax = 6 s with s an E4M3 value and every entry (E2M1 value) * s:
    the scale comes back as s and every code exactly."""
    table = _golden_e2m1()
    rs = np.random.default_rng(3)
    scodes = [c for c in range(1, 127)]
    for sc in scodes:
        s = float(_e4m3_lib([sc])[0])
        codes = rs.integers(0, 16, size=16)
        codes[rs.integers(0, 16)] = 7 if rs.random() < 0.5 else 15
        x = np.array([table[int(c)] * s for c in codes], np.float32)[None]
        qc, qs = orc.quant_fp4(x)
        assert qs[0, 0] == sc
        got = np.array([(qc[0, i // 2] >> (4 * (i % 2))) & 15 for i in range(16)])
        want = np.where((codes & 7) == 0, codes & 8, codes)  # -0 stays -0
        assert (got == want).all(), (sc, got, want)


def test_fp4_nibble_order_and_row_layout(orc):
    x = np.zeros((1, 512), np.float32)
    x[0, 0] = 6.0   # channel 0 -> low nibble of byte 0
    x[0, 1] = -1.0  # channel 1 -> high nibble of byte 0
    x[0, 17] = 3.0  # block 1, channel 1 -> high nibble of byte 8
    qc, qs = orc.quant_fp4(x)
    assert qc[0, 0] == (0x7 | (0xA << 4))
    assert qs[0, 0] == orc.e4m3_encode(1.0)
    assert qc[0, 8] == 0x70 and qs[0, 1] == orc.e4m3_encode(0.5)
    row = orc.kv_rows(qc, qs)
    assert row.shape == (1, 288) and row[0, 256] == qs[0, 0] and row[0, 0] == qc[0, 0]


def test_fp4_zero_and_underflow_blocks(orc):
    x = np.zeros((3, 16), np.float32)
    x[1, 5] = -0.0
    x[2, :] = 2.0 ** -13  # absmax/6 < 2^-10: scale rounds to 0
    qc, qs = orc.quant_fp4(x)
    assert (qc == 0).all() and (qs == 0).all()


def test_fp4_dequant_error_bound(orc):
    """Each value is within half a grid step of the scaled E2M1 grid, and no
    worse than 6 * scale saturation allows."""
    x = synth.normal_rows(5, "pin", (0,), 0, 256, 512)
    qc, qs = orc.quant_fp4(x)
    deq = orc.dequant_fp4(qc, qs)
    s = np.repeat(_e4m3_lib(qs.reshape(-1)).reshape(qs.shape), 16, axis=1)
    err = np.abs(deq - x)
    # grid gaps are at most 2 * s (between 4 and 6); absmax / s <= 6 * (1 + 2^-4)
    assert (err <= s * 1.0 + 1e-12 + np.abs(x) * 2 ** -3).all()


# ---------------------------------------------------------------- FP8 SWA rows

def test_fp8_rows_roundtrip_and_scale(orc):
    vals = _e4m3_lib(range(0, 127))
    x = np.array([vals * 0.5, -vals * 2.0 ** -3], np.float32)[:, :127]
    x = np.pad(x, ((0, 0), (0, 1)))
    codes, scales = orc.quant_fp8(x)
    assert scales[0] == np.float32(448 * 0.5) / np.float32(448)
    deq = orc.dequant_fp8(codes, scales)
    assert np.array_equal(deq, x.astype(np.float64))


def test_fp8_rows_match_torch(orc):
    x = synth.normal_rows(9, "pin", (1,), 0, 64, 512)
    codes, scales = orc.quant_fp8(x)
    s = (np.abs(x).max(axis=1) / np.float32(448)).astype(np.float32)
    assert np.array_equal(scales, s)
    ref = torch.tensor((x / s[:, None]).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes, ref)


# ---------------------------------------------------------------- footprint

def test_footprint(orc):
    fp = {k: int(v) for k, v in read_golden("footprint.txt")}
    assert fp["kv_row_512ch"] == orc.KV_ROW_BYTES == 256 + 32
    assert fp["idx_row_64ch"] == orc.IDX_ROW_BYTES == 32 + 4
    assert fp["swa_row_512ch"] == orc.SWA_ROW_BYTES == 512 + 4
    assert fp["idx_tile_64tok"] == orc.IDX_TILE_BYTES
    assert fp["kv_page_64tok"] == 64 * orc.KV_ROW_BYTES
    assert fp["idx_page_64tok"] == 64 * orc.IDX_ROW_BYTES
    assert fp["global_bytes_per_token_4_full_layers"] == 4 * (orc.KV_ROW_BYTES + orc.IDX_ROW_BYTES)
    qc, qs = orc.quant_fp4(np.ones((3, 512), np.float32))
    assert orc.kv_rows(qc, qs).nbytes == 3 * 288
    kc, ks = orc.quant_fp4(np.ones((3, 64), np.float32))
    assert kc.nbytes + ks.nbytes == 3 * 36


# ---------------------------------------------------------------- score

def _deq_indep(codes_u8, scales_u8, C):
    table = _golden_e2m1()
    out = np.empty((codes_u8.shape[0], C))
    s = _e4m3_lib(scales_u8.reshape(-1)).reshape(scales_u8.shape)
    for c in range(C):
        nib = (codes_u8[:, c // 2] >> (4 * (c % 2))) & 15
        out[:, c] = np.array([table[int(v)] for v in nib]) * s[:, c // 16]
    return out


def test_score_close_to_fp64_dense(orc):
    """score = sum_h w_h relu(q~_h . k~) within fp32 rounding of its 16 terms,
    with q~, k~ decoded independently (golden E2M1 table, torch E4M3)."""
    x = synth.normal_rows(1, "pin", (2,), 0, 300, 64)
    kc, ks = orc.quant_fp4(x)
    for trial in range(6):
        q = synth.normal_rows(1, "pin", (3, trial), 0, 4, 64, scale=1 / 8)
        w = synth.uniform(1, "pin", (4, trial), (4,))
        got = orc.index_scores(q, w, kc, ks).astype(np.float64)
        qc, qs = orc.quant_fp4(q)
        qd = _deq_indep(qc, qs, 64)
        kd = _deq_indep(kc, ks, 64)
        dots = kd @ qd.T                           # [n, 4]
        ref = (np.maximum(dots, 0) * w.astype(np.float64)).sum(axis=1)
        mag = (np.abs(kd[:, None, :] * qd[None, :, :]).sum(-1) * np.abs(w)).sum(axis=1)
        assert (np.abs(got - ref) <= 6e-7 * mag + 1e-30).all()


def test_score_closed_forms(orc):
    """One nonzero channel per head: score = sum_h w_h relu(q_h k) exactly."""
    q = np.zeros((4, 64), np.float32)
    k = np.zeros((1, 64), np.float32)
    # every block's absmax is 6 x (an E4M3 value), so each value is exact
    q[0, 3], q[1, 20], q[2, 20], q[3, 63] = 3.0, -1.5, 0.375, 6.0
    k[0, 3], k[0, 20], k[0, 63] = 1.5, -3.0, 0.75
    kc, ks = orc.quant_fp4(k)
    w = np.array([0.5, 2.0, 1.0, 0.25], np.float32)
    got = orc.index_scores(q, w, kc, ks)[0]
    assert got == 0.5 * 4.5 + 2.0 * 4.5 + 0.0 + 0.25 * 4.5


def test_score_scaling_and_symmetry(orc):
    x = synth.normal_rows(2, "pin", (5,), 0, 200, 64)
    kc, ks = orc.quant_fp4(x)
    q = synth.normal_rows(2, "pin", (6,), 0, 4, 64, scale=0.125)
    w = np.ones(4, np.float32)
    s1 = orc.index_scores(q, w, kc, ks)
    s2 = orc.index_scores(q * np.float32(4.0), w, kc, ks)
    assert np.array_equal(s2, s1 * np.float32(4.0))           # scales shift exactly
    s3 = orc.index_scores(q, w * np.float32(0.5), kc, ks)
    assert np.array_equal(s3, s1 * np.float32(0.5))
    # one head, weight 1: the score is symmetric in (query, key)
    a = synth.normal_rows(2, "pin", (7,), 0, 2, 64)
    ac, as_ = orc.quant_fp4(a)
    w1 = np.array([1.0], np.float32)
    ab = orc.index_scores(a[:1], w1, ac[1:2], as_[1:2])[0]
    ba = orc.index_scores(a[1:2], w1, ac[0:1], as_[0:1])[0]
    assert ab == ba
    # negating the query swaps which heads survive the relu
    sn = orc.index_scores(-q, w, kc, ks)
    dots = _deq_indep(kc, ks, 64) @ _deq_indep(*orc.quant_fp4(q), 64).T
    both = np.abs(dots).sum(1)
    assert np.allclose(s1.astype(np.float64) + sn, both, rtol=1e-6, atol=1e-30)


def _f32(x):
    """Round an exact rational to the nearest fp32 (ties to even)."""
    return float(np.float32(float(x))) if x == 0 else _round_f32(x)


def _round_f32(x):
    from fractions import Fraction
    x = Fraction(x)
    sign = -1 if x < 0 else 1
    a = abs(x)
    e = math.floor(math.log2(a.numerator) - math.log2(a.denominator))
    # make 2^e <= a < 2^(e+1) exactly
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    q = Fraction(2) ** (e - 23)          # spacing of fp32 values at this binade
    n = a / q
    fl = math.floor(n)
    r = n - fl
    if r > Fraction(1, 2) or (r == Fraction(1, 2) and fl % 2 == 1):
        fl += 1
    return sign * float(fl * q)


def test_score_rounding_points_exact_rational(orc):
    """The score's stated rounding points, evaluated in exact rational
    arithmetic with an fp32 rounding after each step (block sums are exact; the
    head sum rounds after each add; the weighted sum is an fp32 product then
    three fused multiply-adds).  The oracle must agree bit for bit; the
    independent decode uses the golden E2M1 table and torch's E4M3."""
    from fractions import Fraction
    x = synth.normal_rows(5, "pin", (20,), 0, 60, 64)
    kc, ks = orc.quant_fp4(x)
    table = _golden_e2m1()
    for trial in range(4):
        q = synth.normal_rows(5, "pin", (21, trial), 0, 4, 64, scale=1 / 8)
        w = synth.uniform(5, "pin", (22, trial), (4,))
        got = orc.index_scores(q, w, kc, ks)
        qc, qs = orc.quant_fp4(q)
        qsd = _e4m3_lib(qs.reshape(-1)).reshape(qs.shape)
        ksd = _e4m3_lib(ks.reshape(-1)).reshape(ks.shape)
        for p in range(kc.shape[0]):
            r = []
            for h in range(4):
                s = None
                for blk in range(4):
                    P = Fraction(0)
                    for c in range(16 * blk, 16 * blk + 16):
                        qn = (int(qc[h, c // 2]) >> (4 * (c % 2))) & 15
                        kn = (int(kc[p, c // 2]) >> (4 * (c % 2))) & 15
                        P += Fraction(table[qn]) * Fraction(table[kn])
                    t = Fraction(qsd[h, blk]) * Fraction(ksd[p, blk]) * P
                    assert _f32(t) == float(t)              # each block term is exact in fp32
                    s = t if s is None else Fraction(_f32(s + t))
                r.append(max(Fraction(_f32(s)), Fraction(0)))
            acc = Fraction(_f32(Fraction(float(w[0])) * r[0]))
            for h in (1, 2, 3):
                acc = Fraction(_f32(Fraction(float(w[h])) * r[h] + acc))
            assert float(got[p]) == float(acc), (trial, p)


def test_score_zero_is_positive_zero(orc):
    q = -np.ones((4, 64), np.float32)
    kc, ks = orc.quant_fp4(np.ones((1, 64), np.float32))
    s = orc.index_scores(q, np.array([1, -1, 1, 1], np.float32), kc, ks)
    assert s[0] == 0.0 and not np.signbit(s[0])


# ---------------------------------------------------------------- Top-K

def _brute_topk(scores, pos, K):
    """Rank counting: i is selected iff fewer than K candidates beat it."""
    sel = []
    for i in range(len(scores)):
        beat = sum(1 for j in range(len(scores))
                   if scores[j] > scores[i] or (scores[j] == scores[i] and pos[j] < pos[i]))
        if beat < K:
            sel.append(int(pos[i]))
    sel.sort()
    return sel + [-1] * (K - len(sel))


@pytest.mark.parametrize("n,K", [(1, 1), (5, 8), (40, 7), (64, 64), (100, 13), (150, 149)])
def test_topk_brute_force(orc, n, K):
    rs = np.random.default_rng(n * 31 + K)
    for trial in range(4):
        scores = rs.integers(0, 6 if trial % 2 else 1000, size=n).astype(np.float32) * np.float32(0.25)
        pos = rs.permutation(10 * n)[:n].astype(np.int32)
        assert orc.topk(scores, pos, K).tolist() == _brute_topk(scores, pos, K)


def test_topk_ties_take_lower_positions(orc):
    scores = np.array([1, 2, 2, 2, 0, 2], np.float32)
    pos = np.arange(6, dtype=np.int32)
    assert orc.topk(scores, pos, 2).tolist() == [1, 2]
    assert orc.topk(scores, pos, 5).tolist() == [0, 1, 2, 3, 5]


@pytest.mark.parametrize("L,n_q,K,causal", [(40, 6, 5, True), (40, 6, 5, False), (7, 12, 3, True), (1, 1, 2, True)])
def test_multi_query_rows_brute_force(orc, L, n_q, K, causal):
    """Each query row of a multi-query call is an ordinary indexer query over
    its candidates: the causal prefix 0 .. L - n_q + i (rows before position 0
    have none), or all L positions.  Scores per key from the single-query
    function (pinned above); masks and selection by brute force."""
    x = synth.normal_rows(5, "mqk", (L,), 0, L, 64)
    kc, ks = orc.quant_fp4(x)
    q = synth.normal_rows(5, "mqq", (n_q,), 0, n_q * 4, 64, scale=0.125).reshape(n_q, 4, 64)
    w = synth.uniform(5, "mqw", (n_q,), (n_q, 4)).astype(np.float32)
    scores, idx = orc.index_topk_multi(q, w, kc, ks, L, K, causal)
    for i in range(n_q):
        full = orc.index_scores(q[i], w[i], kc, ks)
        last = (L - n_q + i) if causal else (L - 1)
        n = max(0, last + 1)
        assert scores[i].shape == (n,)
        assert np.array_equal(scores[i].view(np.uint32), full[:n].view(np.uint32))
        assert idx[i].tolist() == _brute_topk(full[:n], np.arange(n, dtype=np.int32), K), i
    if causal and n_q <= L:
        # the last row sees every position: the single-query call over all L
        assert idx[-1].tolist() == orc.topk(orc.index_scores(q[-1], w[-1], kc, ks),
                                            np.arange(L, dtype=np.int32), K).tolist()


# ---------------------------------------------------------------- attention

def _dense(q, rows):
    z = q.astype(np.float64) @ rows.T
    m = z.max(axis=1, keepdims=True)
    e = np.exp(z - m)
    return (e @ rows) / e.sum(axis=1, keepdims=True), (m[:, 0] + np.log(e.sum(axis=1)))


def _small_caches(orc, L, seed=1):
    x = synth.normal_rows(seed, "pin", (8,), 0, L, 512)
    kc, ks = orc.quant_fp4(x)
    sw = synth.normal_rows(seed, "pin", (9,), 0, 16, 512)
    wc, wsc = orc.quant_fp8(sw)
    return kc, ks, wc, wsc


def test_attention_dense_when_all_selected(orc):
    """K >= L: the sparse result equals dense softmax attention over every
    dequantised row plus the window rows (an independent numpy softmax)."""
    L = 37
    kc, ks, wc, wsc = _small_caches(orc, L)
    q = synth.normal_rows(1, "pin", (10,), 0, 16, 512, scale=1 / np.sqrt(512))
    idx = np.concatenate([np.arange(L, dtype=np.int32), -np.ones(11, np.int32)])
    out, lse = orc.sparse_attention(q, kc, ks, idx, wc, wsc)
    rows = np.concatenate([_deq_indep(kc, ks, 512), _e4m3_lib(wc.reshape(-1)).reshape(wc.shape) * wsc[:, None]])
    ref, rlse = _dense(q, rows)
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    assert np.allclose(lse, rlse, rtol=1e-12, atol=1e-12)


def test_attention_closed_forms(orc):
    kc, ks, wc, wsc = _small_caches(orc, 9)
    rows = _deq_indep(kc, ks, 512)
    q0 = np.zeros((16, 512), np.float32)
    out, lse = orc.sparse_attention(q0, kc, ks, np.arange(9, dtype=np.int32), wc[:0], wsc[:0])
    assert np.allclose(out, rows.mean(axis=0)[None], atol=1e-12)      # q = 0: plain mean
    assert np.allclose(lse, np.log(9))
    q = synth.normal_rows(1, "pin", (11,), 0, 16, 512, scale=0.05)
    out1, lse1 = orc.sparse_attention(q, kc, ks, np.array([4, -1], np.int32), wc[:0], wsc[:0])
    assert np.allclose(out1, rows[4][None], atol=1e-12)                # one row: that row
    assert np.allclose(lse1, q.astype(np.float64) @ rows[4], atol=1e-12)
    out2, lse2 = orc.sparse_attention(q, kc, ks, np.array([4, 4], np.int32), wc[:0], wsc[:0])
    assert np.allclose(out2, out1, atol=1e-12) and np.allclose(lse2, lse1 + np.log(2))
    # the order of the selected rows does not matter
    a, la = orc.sparse_attention(q, kc, ks, np.array([1, 7, 3], np.int32), wc, wsc)
    b, lb = orc.sparse_attention(q, kc, ks, np.array([7, 3, 1], np.int32), wc, wsc)
    assert np.allclose(a, b, atol=1e-13) and np.allclose(la, lb, atol=1e-13)


# ---------------------------------------------------------------- modes

def _tiny_step(orc, modes, L=300, K=16, P=0, pool=False, same_qidx=False):
    layers = synth.build_layers(modes, pool=pool)
    w = synth.Workload("tiny", 4242, 1, [L], layers, K, pool_len=P)
    caches, per = {}, {}
    for i, ly in enumerate(layers):
        if ly.mode == synth.FULL:
            kc, ks = orc.quant_fp4(synth.kv_values(w, i, 0, 0, L))
            ic, isc = orc.quant_fp4(synth.idx_key_values(w, i, 0, 0, L))
            caches[i] = {0: dict(kv_codes=kc, kv_scales=ks, k_codes=ic, k_scales=isc)}
    for i, ly in enumerate(layers):
        sw = synth.swa_values(w, i, 0)[-min(L, w.window):]
        c, s = orc.quant_fp8(sw)
        qi = synth.index_query(w, 0 if same_qidx else i)
        wt = synth.index_weights(w, 0 if same_qidx else i)
        per[i] = dict(q=synth.query(w, i), q_idx=qi, w=wt, swa_codes=[c], swa_scales=[s])
    return layers, orc.decode_step(layers, [L], K, P, caches, per)


def test_reuse_equals_reindex_with_same_query(orc):
    """Helmcode "03 · CSA2": a Reuse layer reuses the selection; when its
    indexer query equals the Reindex layer's, recomputing gives the same."""
    layers, r = _tiny_step(orc, ["F", "R", "U", "R"], same_qidx=True)
    assert np.array_equal(r[1]["idx"], r[3]["idx"])
    assert np.array_equal(r[2]["idx"], r[1]["idx"])
    # Reindex with the Full layer's own (query, weights) selects what Full selected
    assert np.array_equal(r[0]["idx"], r[1]["idx"])


def test_pool_restricted_equals_unrestricted_when_pool_covers_all(orc):
    """Louis Bouchard, "Share the cache and the search work": later indexing
    layers search the pool; a pool holding every position changes nothing."""
    L = 200
    _, a = _tiny_step(orc, ["F", "R", "R"], L=L, K=24, P=L, pool=True)
    _, b = _tiny_step(orc, ["F", "R", "R"], L=L, K=24, P=0, pool=False)
    for l in (1, 2):
        assert np.array_equal(a[l]["idx"], b[l]["idx"])
        assert np.allclose(a[l]["out"], b[l]["out"], atol=0, rtol=0)
    # a Full layer's Top-K lies inside its own pool
    _, c = _tiny_step(orc, ["F", "R"], L=L, K=24, P=64, pool=True)
    assert set(c[0]["idx"][0].tolist()) <= set(c[0]["pool"][0].tolist())
    assert (np.diff(c[0]["pool"][0]) > 0).all()


def test_swa_only_layer_is_window_attention(orc):
    layers, r = _tiny_step(orc, ["F", "S"], L=50)
    w = synth.Workload("tiny", 4242, 1, [50], layers, 16)
    sw = synth.swa_values(w, 1, 0)[-50:]
    c, s = orc.quant_fp8(sw)
    ref, _ = _dense(synth.query(w, 1)[0], _e4m3_lib(c.reshape(-1)).reshape(c.shape) * s[:, None])
    assert np.allclose(r[1]["out"][0], ref, atol=1e-12)


# ---------------------------------------------------------------- layouts

def test_paged_readback_equals_contiguous(orc):
    """A 64-token paged cache read through its page table holds the same bytes
    as the contiguous encoding."""
    L, page = 300, 64
    x = synth.normal_rows(3, "pin", (12,), 0, L, 64)
    kc, ks = orc.quant_fp4(x)
    n_pages = (L + page - 1) // page
    perm = np.random.default_rng(1).permutation(n_pages + 3)[:n_pages].astype(np.int32)
    cache = np.zeros((n_pages + 3) * page * 36, np.uint8)
    slots = orc.slots_paged(perm, np.arange(L), page)
    orc.place_idx(cache, slots, kc, ks)
    rc, rs_ = orc.read_idx(cache, slots)
    assert np.array_equal(rc, kc) and np.array_equal(rs_, ks)
    contig = np.zeros(n_pages * page * 36, np.uint8)
    orc.place_idx(contig, orc.slots_contiguous(0, np.arange(L), n_pages * page), kc, ks)
    for p in range(n_pages):
        a = contig[p * 2304:(p + 1) * 2304]
        b = cache[perm[p] * 2304:(perm[p] + 1) * 2304]
        assert np.array_equal(a, b)
