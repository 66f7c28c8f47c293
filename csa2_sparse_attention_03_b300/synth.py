"""Seeded synthetic inputs for the CSA2 decode hot path.

This module draws random numbers and fixes workload shapes. It holds none of
the method's arithmetic (no quantisation, scoring, selection or attention):
both the CUDA path and the CPU oracle consume exactly what it produces.

Workload recipe (the pages give no data; these are stated synthetic choices):
  * main KV values      N(0, 1) fp32, 512 channels per token
  * indexer keys        N(0, 1) fp32, one 64-channel key per token
  * attention queries   N(0, 1) / sqrt(512) fp32, 16 heads x 512 per layer
  * indexer queries     N(0, 1) / sqrt(64) fp32, 4 heads x 64 per indexing layer
  * indexer head weights U(0, 1) fp32, 4 per indexing layer
  * SWA window values   N(0, 1) fp32, 128 tokens x 512 per layer (each layer has
                        its own local state, DeepSeek V4.1 Flash explainer, "03 CSA2")
  * ragged lengths      integers U[lo, hi] (batch-64 workload)
  * page tables         a seeded random permutation of the physical pages

Every array is drawn from numpy PCG64 streams keyed by (workload seed, stream
name, index tuple), so any slice can be regenerated independently of the rest.
Large arrays are drawn in fixed chunks of ``CHUNK_ROWS`` rows, each chunk from
its own stream, so the values never depend on how a caller batches the work.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import numpy as np

CHUNK_ROWS = 4096  # small enough that a short slice (a window, one row) is cheap to draw

# widths fixed by the workloads
H_Q = 16          # attention heads (MQA over one shared 512-channel row)
D = 512           # main KV / query channels
H_IDX = 4         # indexer heads
D_IDX = 64        # indexer channels
SWA_WINDOW = 128  # local window (tokens)
PAGE = 64         # tokens per page in paged caches

FULL, REINDEX, REUSE, SWA_ONLY = 0, 1, 2, 3
MODE_NAMES = {FULL: "F", REINDEX: "R", REUSE: "U", SWA_ONLY: "S"}


def _stream_key(name: str) -> int:
    return int.from_bytes(hashlib.sha256(name.encode()).digest()[:4], "little")


def rng(seed: int, name: str, *idx: int) -> np.random.Generator:
    """Independent PCG64 stream for (seed, stream name, index tuple)."""
    ss = np.random.SeedSequence([int(seed), _stream_key(name), *[int(i) for i in idx]])
    return np.random.Generator(np.random.PCG64(ss))


def normal_rows(seed: int, name: str, idx: tuple, row0: int, n_rows: int, width: int,
                scale: float = 1.0) -> np.ndarray:
    """Rows [row0, row0+n_rows) of an N(0, scale^2) fp32 matrix of the given width.

    Row r comes from chunk r // CHUNK_ROWS, so any row range is reproducible.
    """
    out = np.empty((n_rows, width), dtype=np.float32)
    r = row0
    end = row0 + n_rows
    while r < end:
        c = r // CHUNK_ROWS
        c0 = c * CHUNK_ROWS
        g = rng(seed, name, *idx, c)
        chunk = g.standard_normal((CHUNK_ROWS, width), dtype=np.float32)
        lo = r - c0
        hi = min(end - c0, CHUNK_ROWS)
        out[r - row0:r - row0 + (hi - lo)] = chunk[lo:hi]
        r = c0 + hi
    if scale != 1.0:
        out *= np.float32(scale)
    return out


def uniform(seed: int, name: str, idx: tuple, shape, lo: float = 0.0, hi: float = 1.0) -> np.ndarray:
    return rng(seed, name, *idx).uniform(lo, hi, size=shape).astype(np.float32)


@dataclass
class Layer:
    mode: int
    kv_src: int = -1     # FULL layer whose caches this layer reads (itself for FULL)
    idx_src: int = -1    # layer whose Top-K this layer reuses (REUSE) / -1
    use_pool: bool = False


@dataclass
class Workload:
    name: str
    seed: int
    batch: int
    seq_lens: list
    layers: list
    topk: int
    pool_len: int = 0          # candidate pool size kept by FULL layers (0 = none)
    paged: bool = False
    append: bool = True        # quantise-and-append one new token per FULL layer per step
    window: int = SWA_WINDOW
    notes: str = ""
    extra: dict = field(default_factory=dict)

    @property
    def max_len(self) -> int:
        return int(max(self.seq_lens))


def schedule_group(n_reuse: int, swa_tail: bool) -> list:
    """[F, R, U x n_reuse, (S)] with sources pointing into the group."""
    return ["F", "R"] + ["U"] * n_reuse + (["S"] if swa_tail else [])


def build_layers(modes: list, pool: bool = False) -> list:
    """Resolve sources for a static mode string: each R/U reads the most recent F's
    caches; each U reuses the most recent indexing layer's Top-K."""
    out = []
    last_full = -1
    last_index = -1
    for i, m in enumerate(modes):
        if m == "F":
            out.append(Layer(FULL, kv_src=i, idx_src=i))
            last_full = i
            last_index = i
        elif m == "R":
            out.append(Layer(REINDEX, kv_src=last_full, idx_src=i, use_pool=pool))
            last_index = i
        elif m == "U":
            out.append(Layer(REUSE, kv_src=last_full, idx_src=last_index))
        elif m == "S":
            out.append(Layer(SWA_ONLY))
        else:
            raise ValueError(m)
    return out


def forty_layer_modes() -> list:
    """4 Full, 4 Reindex, 30 Reuse, 2 SWA-only: Full at 0, 10, 20, 30 each followed
    by one Reindex; SWA-only at 9 and 19 (the group tails)."""
    modes = []
    for g in range(4):
        modes += schedule_group(7 if g < 2 else 8, swa_tail=g < 2)
    assert len(modes) == 40
    return modes


def workload(idx: int, small: bool = False) -> Workload:
    """The five workloads. ``small`` shrinks lengths for quick parity runs while
    keeping every structural feature (schedule, pool, paging, raggedness)."""
    seed = 1000 * idx
    if idx == 0:
        L = 4096 if not small else 1000
        return Workload("B1 L4096 one Full layer K512", seed, 1, [L], build_layers(["F"]), 512)
    if idx == 1:
        L = 32768 if not small else 3000
        modes = schedule_group(7, swa_tail=True)
        return Workload("B8 L32768 [F,R,Ux7,S] K512", seed, 8, [L] * 8, build_layers(modes), 512)
    if idx == 2:
        L = 131072 if not small else 5000
        return Workload("B1 L131072 40-layer 4F/4R/30U/2S K2048", seed, 1, [L],
                        build_layers(forty_layer_modes()), 2048 if not small else 512)
    if idx == 3:
        L = 1048576 if not small else 20000
        P = 16384 if not small else 2048
        K = 2048 if not small else 256
        return Workload("B1 L1048576 hierarchical F(pool16384)+3R K2048", seed, 1, [L],
                        build_layers(["F", "R", "R", "R"], pool=True), K, pool_len=P)
    if idx == 4:
        B = 64 if not small else 4
        lo, hi = (16384, 65536) if not small else (600, 3000)
        lens = rng(seed, "seq_lens").integers(lo, hi + 1, size=B).tolist()
        return Workload("B64 ragged L~U[16384,65536] 40-layer K2048 paged+append", seed, B,
                        [int(x) for x in lens], build_layers(forty_layer_modes()),
                        2048 if not small else 256, paged=True)
    raise ValueError(idx)


# ---- per-tensor draws (names are the stream ids) ----

def kv_values(w: Workload, full_layer: int, b: int, row0: int, n: int) -> np.ndarray:
    return normal_rows(w.seed, "kv", (full_layer, b), row0, n, D)


def idx_key_values(w: Workload, full_layer: int, b: int, row0: int, n: int) -> np.ndarray:
    return normal_rows(w.seed, "idxk", (full_layer, b), row0, n, D_IDX)


def query_scale(w: Workload) -> float:
    """Standard deviation of the attention queries: 1/sqrt(512), times the
    workload's optional ``extra["q_scale"]`` (logits spanning tens of units)."""
    return float(w.extra.get("q_scale", 1.0)) / float(np.sqrt(D))


def query(w: Workload, layer: int) -> np.ndarray:
    """[B, 16, 512] attention query of one layer."""
    return normal_rows(w.seed, "q", (layer,), 0, w.batch * H_Q, D,
                       scale=query_scale(w)).reshape(w.batch, H_Q, D)


def index_query(w: Workload, layer: int) -> np.ndarray:
    """[B, 4, 64] indexer query of one indexing layer."""
    return normal_rows(w.seed, "qidx", (layer,), 0, w.batch * H_IDX, D_IDX,
                       scale=1.0 / np.sqrt(D_IDX)).reshape(w.batch, H_IDX, D_IDX)


def index_weights(w: Workload, layer: int) -> np.ndarray:
    """[B, 4] non-negative indexer head weights."""
    return uniform(w.seed, "widx", (layer,), (w.batch, H_IDX))


def swa_values(w: Workload, layer: int, b: int) -> np.ndarray:
    """[window, 512]: the window rows of one layer/sequence, oldest first."""
    return normal_rows(w.seed, "swa", (layer, b), 0, w.window, D)


def page_permutation(w: Workload, n_pages: int, cache_id: int) -> np.ndarray:
    return rng(w.seed, "pages", cache_id).permutation(n_pages).astype(np.int32)


def device_normal_(t, seed: int, name: str, *idx: int, scale: float = 1.0):
    """Fill a CUDA fp32 tensor in place from a seeded torch generator (bench-size
    inputs where host generation would dominate set-up time)."""
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed((int(seed) * 1_000_003 + _stream_key(name) + sum((i + 1) * 7919 ** (k + 1) for k, i in enumerate(idx))) % (2 ** 63))
    t.normal_(0.0, float(scale), generator=g)
    return t


def device_uniform_(t, seed: int, name: str, *idx: int):
    import torch
    g = torch.Generator(device=t.device)
    g.manual_seed((int(seed) * 1_000_033 + _stream_key(name) + sum((i + 1) * 104729 ** (k + 1) for k, i in enumerate(idx))) % (2 ** 63))
    t.uniform_(0.0, 1.0, generator=g)
    return t
