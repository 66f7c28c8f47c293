"""CSA2 decode hot path: CPU oracle.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline /
reference legs may import this package.  The product path never does; it
shares no code with the CUDA library (``csa2_oracle.c`` is compiled on its
own with gcc).

Sources are the web pages about DeepSeek V4.1 Flash (see ``csa2_oracle.c``):
[HC] Helmcode explainer ("03 · CSA2", "04 · FP4"), [LB] Louis Bouchard's
KV-cache report ("Share the cache and the search work"), [MO] 0x0moeen's
KV-cache note ("Then every layer stops asking the same question").

Layouts (the pages fix none; stated choices shared with the C interface):
  * main KV row, 512 channels: 256 B of E2M1 codes (channel 2i in the low
    nibble of byte i) then 32 B of E4M3 scales, one per 16 channels: 288 B;
  * indexer keys, 64 channels, stored in tiles of 64 tokens: 64 x 32 B codes
    then 64 x 4 B scales (2,304 B per tile); slot s is row s % 64 of tile s // 64;
  * SWA rows, 512 channels: a plane of 512 B E4M3 codes per slot, then a plane
    of one fp32 scale per slot;
  * slot of (sequence b, position p): contiguous ``b * stride + p`` (SWA ring:
    ``b * stride + p % stride``), or paged ``table[b][p // page] * page + p % page``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "csa2_oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

KV_ROW_BYTES = 288
IDX_ROW_BYTES = 36
IDX_TILE = 64
IDX_TILE_BYTES = IDX_TILE * IDX_ROW_BYTES
SWA_ROW_BYTES = 516


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no FMA contraction, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + ".tmp%d" % os.getpid()
        subprocess.check_call(["gcc", "-std=c11", "-O2", "-ffp-contract=off", "-fno-fast-math", "-fopenmp",
                               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB)
    return _LIB


_lib = None


def lib():
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        P = ctypes.c_void_p
        i32, i64, f32 = ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        L.orc_e2m1_decode.restype = f32
        L.orc_e2m1_decode.argtypes = [ctypes.c_uint32]
        L.orc_e2m1_encode.restype = ctypes.c_uint32
        L.orc_e2m1_encode.argtypes = [f32]
        L.orc_e4m3_decode.restype = f32
        L.orc_e4m3_decode.argtypes = [ctypes.c_uint32]
        L.orc_e4m3_encode.restype = ctypes.c_uint32
        L.orc_e4m3_encode.argtypes = [f32]
        L.orc_quant_fp4_rows.argtypes = [P, i64, i32, P, P]
        L.orc_dequant_fp4_rows.argtypes = [P, P, i64, i32, P]
        L.orc_quant_fp8_rows.argtypes = [P, i64, i32, P, P]
        L.orc_dequant_fp8_rows.argtypes = [P, P, i64, i32, P]
        L.orc_index_scores.argtypes = [P, P, P, i32, i32, P, P, i64, P]
        L.orc_topk.restype = i32
        L.orc_topk.argtypes = [P, P, i64, i32, P]
        L.orc_attend.argtypes = [P, i32, i32, P, i64, P, P]
        L.orc_set_threads.argtypes = [i32]
        L.orc_get_threads.restype = i32
        # single-threaded unless a caller asks for more
        L.orc_set_threads(1)
        _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(ctypes.c_void_p)


def set_threads(n: int) -> None:
    """Threads for the oracle's loops over independent units (results do not
    depend on the count)."""
    lib().orc_set_threads(int(n))


def get_threads() -> int:
    return int(lib().orc_get_threads())


# ---- scalar codecs ----

def e2m1_encode(v: float) -> int:
    return int(lib().orc_e2m1_encode(float(v)))


def e2m1_decode(code: int) -> float:
    return float(lib().orc_e2m1_decode(int(code)))


def e4m3_encode(v: float) -> int:
    return int(lib().orc_e4m3_encode(float(v)))


def e4m3_decode(code: int) -> float:
    return float(lib().orc_e4m3_decode(int(code)))


# ---- row codecs ----

def quant_fp4(x: np.ndarray):
    """[n, C] fp32 -> (codes [n, C/2] u8, scales [n, C/16] u8)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, C = x.shape
    assert C % 16 == 0
    codes = np.empty((n, C // 2), np.uint8)
    scales = np.empty((n, C // 16), np.uint8)
    lib().orc_quant_fp4_rows(_p(x), n, C, _p(codes), _p(scales))
    return codes, scales


def dequant_fp4(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales)
    n, half = codes.shape
    out = np.empty((n, 2 * half), np.float64)
    lib().orc_dequant_fp4_rows(_p(codes), _p(scales), n, 2 * half, _p(out))
    return out


def quant_fp8(x: np.ndarray):
    """[n, C] fp32 -> (codes [n, C] u8, scales [n] fp32)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    n, C = x.shape
    codes = np.empty((n, C), np.uint8)
    scales = np.empty((n,), np.float32)
    lib().orc_quant_fp8_rows(_p(x), n, C, _p(codes), _p(scales))
    return codes, scales


def dequant_fp8(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    codes = np.ascontiguousarray(codes)
    scales = np.ascontiguousarray(scales, dtype=np.float32)
    n, C = codes.shape
    out = np.empty((n, C), np.float64)
    lib().orc_dequant_fp8_rows(_p(codes), _p(scales), n, C, _p(out))
    return out


# ---- layouts ----

def kv_rows(codes: np.ndarray, scales: np.ndarray) -> np.ndarray:
    """[n, 256] codes + [n, 32] scales -> [n, 288] rows."""
    return np.ascontiguousarray(np.concatenate([codes, scales], axis=1))


def kv_rows_split(rows: np.ndarray):
    return rows[:, :256], rows[:, 256:]


def slots_contiguous(b: int, positions: np.ndarray, stride: int, ring: bool = False) -> np.ndarray:
    p = np.asarray(positions, np.int64)
    return b * stride + (p % stride if ring else p)


def slots_paged(table_row: np.ndarray, positions: np.ndarray, page: int) -> np.ndarray:
    p = np.asarray(positions, np.int64)
    return table_row[p // page].astype(np.int64) * page + p % page


def place_kv(cache: np.ndarray, slots: np.ndarray, rows: np.ndarray) -> None:
    """Write [n, 288] rows at the given slots of a flat byte cache."""
    view = cache.reshape(-1, KV_ROW_BYTES)
    view[slots] = rows


def place_idx(cache: np.ndarray, slots: np.ndarray, codes: np.ndarray, scales: np.ndarray) -> None:
    """Write indexer keys ([n, 32] codes, [n, 4] scales) into a tiled cache."""
    tiles = cache.reshape(-1, IDX_TILE_BYTES)
    t = slots // IDX_TILE
    r = slots % IDX_TILE
    for j in range(32):
        tiles[t, r * 32 + j] = codes[:, j]
    for j in range(4):
        tiles[t, IDX_TILE * 32 + r * 4 + j] = scales[:, j]


def read_idx(cache: np.ndarray, slots: np.ndarray):
    tiles = cache.reshape(-1, IDX_TILE_BYTES)
    t = slots // IDX_TILE
    r = slots % IDX_TILE
    codes = np.stack([tiles[t, r * 32 + j] for j in range(32)], axis=1)
    scales = np.stack([tiles[t, IDX_TILE * 32 + r * 4 + j] for j in range(4)], axis=1)
    return codes, scales


def place_swa(cache: np.ndarray, n_slots: int, slots: np.ndarray, codes: np.ndarray,
              scales: np.ndarray) -> None:
    plane = cache[:n_slots * 512].reshape(n_slots, 512)
    plane[slots] = codes
    sc = cache[n_slots * 512:n_slots * 516].view(np.float32)
    sc[slots] = scales


# ---- scoring, selection, attention ----

def index_scores(q_idx: np.ndarray, w: np.ndarray, k_codes: np.ndarray, k_scales: np.ndarray) -> np.ndarray:
    """Scores of n keys for one indexer query q_idx [Hi, Di] (fp32, quantised
    here by the FP4 rule) and head weights w [Hi]."""
    q_idx = np.ascontiguousarray(q_idx, np.float32)
    Hi, Di = q_idx.shape
    qc, qs = quant_fp4(q_idx)
    w = np.ascontiguousarray(w, np.float32)
    k_codes = np.ascontiguousarray(k_codes)
    k_scales = np.ascontiguousarray(k_scales)
    n = k_codes.shape[0]
    out = np.empty((n,), np.float32)
    lib().orc_index_scores(_p(qc), _p(qs), _p(w), Hi, Di, _p(k_codes), _p(k_scales), n, _p(out))
    return out


def topk(scores: np.ndarray, positions: np.ndarray, K: int) -> np.ndarray:
    scores = np.ascontiguousarray(scores, np.float32)
    positions = np.ascontiguousarray(positions, np.int32)
    out = np.empty((K,), np.int32)
    lib().orc_topk(_p(scores), _p(positions), scores.shape[0], K, _p(out))
    return out


def index_topk_multi(q_idx: np.ndarray, w: np.ndarray, k_codes: np.ndarray, k_scales: np.ndarray, L: int,
                     K: int, causal: bool = True):
    """Several indexer queries of one sequence ([HC] "10 · other changes": a
    speculative verification checks several drafted tokens together; [HC]
    "03 · CSA2": the indexing path also runs in prefill): q_idx [n_q, Hi, Di],
    w [n_q, Hi], keys of positions 0..L-1.  Query row i is an ordinary indexer
    query whose candidates are its causal prefix 0 .. L - n_q + i (the queries
    are the sequence's last n_q tokens), or every position < L when not
    causal.  Returns (scores: list of per-row fp32 arrays over the row's
    candidates, idx [n_q, K] ascending positions, -1 padded)."""
    n_q = q_idx.shape[0]
    scores, idx = [], np.full((n_q, K), -1, np.int32)
    for i in range(n_q):
        n = max(0, min(L, L - n_q + i + 1)) if causal else L
        s = index_scores(q_idx[i], w[i], k_codes[:n], k_scales[:n]) if n else np.zeros(0, np.float32)
        scores.append(s)
        idx[i] = topk(s, np.arange(n, dtype=np.int32), K)
    return scores, idx


def attend(q: np.ndarray, rows: np.ndarray):
    """q [H, D] fp32, rows [n, D] fp64 -> (out [H, D] fp64, lse [H] fp64)."""
    q = np.ascontiguousarray(q, np.float32)
    rows = np.ascontiguousarray(rows, np.float64)
    H, D = q.shape
    out = np.empty((H, D), np.float64)
    lse = np.empty((H,), np.float64)
    lib().orc_attend(_p(q), H, D, _p(rows), rows.shape[0], _p(out), _p(lse))
    return out, lse


# ---- one decode step over a static mode schedule ([HC] "03 · CSA2") ----

FULL, REINDEX, REUSE, SWA_ONLY = 0, 1, 2, 3


def window_positions(L: int, window: int) -> np.ndarray:
    return np.arange(max(0, L - window), L, dtype=np.int64)


def sparse_attention(q: np.ndarray, kv_codes: np.ndarray, kv_scales: np.ndarray, idx: np.ndarray,
                     swa_codes: np.ndarray, swa_scales: np.ndarray):
    """One sequence, one layer: softmax over the selected FP4 rows (idx >= 0)
    together with the given FP8 window rows."""
    sel = idx[idx >= 0]
    parts = []
    if sel.size:
        parts.append(dequant_fp4(kv_codes[sel], kv_scales[sel]))
    if swa_codes is not None and swa_codes.shape[0]:
        parts.append(dequant_fp8(swa_codes, swa_scales))
    rows = np.concatenate(parts, axis=0) if parts else np.zeros((0, q.shape[1]))
    return attend(q, rows)


def decode_step(layers, seq_lens, topk_k: int, pool_len: int, caches: dict, per_layer: dict):
    """Run the schedule layer by layer.

    ``layers``: objects with mode, kv_src, idx_src, use_pool (see synth.Layer).
    ``caches[f][b]``: dict(kv_codes [L,256], kv_scales [L,32], k_codes [L,32],
    k_scales [L,4]) in logical position order for FULL layer f.
    ``per_layer[l]``: dict(q [B,16,512], q_idx [B,4,64] or None, w [B,4] or None,
    swa_codes [B] list of [n,512], swa_scales [B] list of [n]).
    Returns per layer: dict(out [B,16,512], lse [B,16], idx [B,K] or None,
    pool [B,P] or None).
    """
    B = len(seq_lens)
    res = {}
    for l, ly in enumerate(layers):
        pl = per_layer[l]
        idx = pool = None
        if ly.mode in (FULL, REINDEX):
            f = ly.kv_src
            idx = np.empty((B, topk_k), np.int32)
            if ly.mode == FULL and pool_len:
                pool = np.empty((B, pool_len), np.int32)
            for b in range(B):
                L = seq_lens[b]
                c = caches[f][b]
                if ly.mode == REINDEX and ly.use_pool:
                    cand = res[f]["pool"][b]
                    cand = cand[cand >= 0]
                else:
                    cand = np.arange(L, dtype=np.int32)
                sc = index_scores(pl["q_idx"][b], pl["w"][b], c["k_codes"][cand], c["k_scales"][cand])
                idx[b] = topk(sc, cand, topk_k)
                if pool is not None:
                    pool[b] = topk(sc, cand, pool_len)
        elif ly.mode == REUSE:
            idx = res[ly.idx_src]["idx"]
        out = np.empty((B,) + pl["q"].shape[1:], np.float64)
        lse = np.empty(pl["q"].shape[:2], np.float64)
        for b in range(B):
            if ly.mode == SWA_ONLY:
                kc = ks = None
                ib = np.zeros((0,), np.int32)
            else:
                c = caches[ly.kv_src][b]
                kc, ks = c["kv_codes"], c["kv_scales"]
                ib = idx[b]
            out[b], lse[b] = sparse_attention(pl["q"][b], kc, ks, ib, pl["swa_codes"][b], pl["swa_scales"][b])
        res[l] = dict(out=out, lse=lse, idx=idx, pool=pool)
    return res
