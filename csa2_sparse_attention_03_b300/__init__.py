"""CSA2 (Compressed Sparse Attention 2) decode hot path on B300.

Thin Python binding of ``libcsa2.so`` (include/csa2.h): argument marshalling
only.  Every step of the path runs in the library's CUDA kernels; PyTorch
supplies device memory and streams.  There is no CPU fallback: without the
compiled library every call raises.
"""
from __future__ import annotations

import ctypes
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libcsa2.so")

# status / modes / formats (include/csa2.h)
OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_WORKSPACE = 0, 1, 2, 3, 4, 5
MODE_FULL, MODE_REINDEX, MODE_REUSE, MODE_SWA_ONLY = 0, 1, 2, 3
FMT_FP4_KV, FMT_FP4_IDX, FMT_FP8_SWA = 0, 1, 2
HEADS, DIM, IDX_HEADS, IDX_DIM = 16, 512, 4, 64


class Csa2Error(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"csa2 status {status}: {message}")
        self.status = status


class csa2_cache(ctypes.Structure):
    _fields_ = [("data", ctypes.c_void_p), ("format", ctypes.c_int32), ("page_size", ctypes.c_int32),
                ("n_slots", ctypes.c_int64), ("seq_stride", ctypes.c_int64),
                ("page_table", ctypes.c_void_p), ("max_pages", ctypes.c_int32),
                ("reserved", ctypes.c_int32)]


class csa2_layer_desc(ctypes.Structure):
    _fields_ = [("mode", ctypes.c_int32), ("kv_src", ctypes.c_int32), ("idx_src", ctypes.c_int32),
                ("use_pool", ctypes.c_int32),
                ("kv", ctypes.POINTER(csa2_cache)), ("idx_keys", ctypes.POINTER(csa2_cache)),
                ("swa", ctypes.POINTER(csa2_cache)),
                ("q", ctypes.c_void_p), ("q_idx", ctypes.c_void_p), ("w", ctypes.c_void_p),
                ("new_kv", ctypes.c_void_p), ("new_idx_key", ctypes.c_void_p), ("new_swa", ctypes.c_void_p),
                ("out", ctypes.c_void_p), ("lse", ctypes.c_void_p), ("idx_out", ctypes.c_void_p),
                ("pool_out", ctypes.c_void_p)]


class csa2_footprint(ctypes.Structure):
    _fields_ = [("global_bytes_per_token", ctypes.c_int64), ("cache_bytes", ctypes.c_int64),
                ("step_bytes", ctypes.c_int64), ("sessions", ctypes.c_int64)]


class csa2_cost(ctypes.Structure):
    _fields_ = [("index_flops", ctypes.c_double), ("attn_flops", ctypes.c_double),
                ("weighted_flops", ctypes.c_double), ("bytes_sequential", ctypes.c_double)]


_lib = None


def load():
    """Load libcsa2.so; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"{LIB_PATH} is missing: build it with __graft_entry__.build() "
                          "(csa2_sparse_attention_03_b300/build.py)")
    L = ctypes.CDLL(LIB_PATH)
    P, i32, i64, sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_size_t
    C = ctypes.POINTER(csa2_cache)
    L.csa2_cache_bytes.restype = sz
    L.csa2_cache_bytes.argtypes = [i32, i64]
    L.csa2_quantize_kv.restype = i32
    L.csa2_quantize_kv.argtypes = [P, i32, i64, P, P, C, P]
    L.csa2_index_topk_workspace.restype = sz
    L.csa2_index_topk_workspace.argtypes = [i32, i32, i32, i32, i32]
    L.csa2_index_topk.restype = i32
    L.csa2_index_topk.argtypes = [i32, C, P, P, i32, i32, i32, P, i32, P, i32, i32, P, P, i32, P, P, sz, P]
    L.csa2_index_topk_multi_workspace.restype = sz
    L.csa2_index_topk_multi_workspace.argtypes = [i32, i32, i32]
    L.csa2_index_topk_multi.restype = i32
    L.csa2_index_topk_multi.argtypes = [C, P, P, i32, i32, i32, i32, P, i32, i32, i32, P, P, P, sz, P]
    L.csa2_sparse_attn_workspace.restype = sz
    L.csa2_sparse_attn_workspace.argtypes = [i32, i32, i32]
    L.csa2_sparse_attn.restype = i32
    L.csa2_sparse_attn.argtypes = [C, C, P, i32, i32, i32, P, i32, P, i32, i32, P, P, P, sz, P]
    L.csa2_sparse_attn_noalloc.restype = i32
    L.csa2_sparse_attn_noalloc.argtypes = [C, C, P, i32, i32, i32, P, i32, P, i32, i32, P, P, P]
    L.csa2_decode_layers_workspace.restype = sz
    L.csa2_decode_layers_workspace.argtypes = [ctypes.POINTER(csa2_layer_desc), i32, i32, i32, i32, i32, i32]
    L.csa2_decode_layers.restype = i32
    L.csa2_decode_layers.argtypes = [ctypes.POINTER(csa2_layer_desc), i32, i32, P, i32, i32, i32, i32, P, sz, P]
    L.csa2_decode_layer_workspace.restype = sz
    L.csa2_decode_layer_workspace.argtypes = [ctypes.POINTER(csa2_layer_desc), i32, i32, i32, i32, i32, i32]
    L.csa2_decode_layer.restype = i32
    L.csa2_decode_layer.argtypes = [ctypes.POINTER(csa2_layer_desc), i32, i32, i32, P, i32, i32, i32, i32, P, sz,
                                    P]
    L.csa2_plan_footprint.restype = i32
    L.csa2_plan_footprint.argtypes = [P, i32, i64, i32, i32, i32, i64, ctypes.POINTER(csa2_footprint)]
    L.csa2_plan_cost.restype = i32
    L.csa2_plan_cost.argtypes = [P, i32, i64, i32, i32, i32, ctypes.POINTER(csa2_cost)]
    L.csa2_test_set_wait_limit.restype = i32
    L.csa2_test_set_wait_limit.argtypes = [i32]
    L.csa2_last_error.restype = ctypes.c_char_p
    L.csa2_last_error.argtypes = []
    L.csa2_check_device.restype = i32
    L.csa2_check_device.argtypes = [P]
    L.csa2_last_device_flags.restype = i32
    L.csa2_last_device_flags.argtypes = []
    L.csa2_set_phase_events.restype = i32
    L.csa2_set_phase_events.argtypes = [ctypes.POINTER(ctypes.c_void_p), i32]
    L.csa2_launch_count.restype = i64
    L.csa2_launch_count.argtypes = []
    L.csa2_version.restype = i32
    L.csa2_version.argtypes = []
    _lib = L
    return L


def _check(status):
    if status != OK:
        raise Csa2Error(status, load().csa2_last_error().decode())


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def cache_bytes(fmt: int, n_slots: int) -> int:
    return int(load().csa2_cache_bytes(fmt, n_slots))


class Cache:
    """A packed cache in device memory plus its csa2_cache descriptor."""

    def __init__(self, fmt, n_slots, device="cuda", seq_stride=0, page_size=0, page_table=None):
        import torch
        nbytes = cache_bytes(fmt, n_slots)
        if nbytes == 0:
            raise ValueError(f"invalid cache: format {fmt}, {n_slots} slots")
        self.data = torch.zeros(nbytes, dtype=torch.uint8, device=device)
        self.page_table = page_table
        self.desc = csa2_cache(self.data.data_ptr(), fmt, page_size, n_slots, seq_stride,
                               page_table.data_ptr() if page_table is not None else None,
                               page_table.shape[1] if page_table is not None else 0, 0)

    @classmethod
    def contiguous(cls, fmt, batch, seq_stride, device="cuda"):
        return cls(fmt, batch * seq_stride, device, seq_stride=seq_stride)

    @classmethod
    def paged(cls, fmt, n_pages, page_size, page_table, device="cuda"):
        return cls(fmt, n_pages * page_size, device, page_size=page_size, page_table=page_table)

    @property
    def ref(self):
        return ctypes.byref(self.desc)

    def seq_view(self, b: int) -> "csa2_cache":
        """Descriptor addressing only sequence b as sequence 0 (FP4 formats)."""
        d = self.desc
        if d.format == FMT_FP8_SWA:
            raise ValueError("SWA rings have shared planes; address them with the full descriptor")
        if d.page_size:
            return csa2_cache(d.data, d.format, d.page_size, d.n_slots, 0,
                              d.page_table + 4 * b * d.max_pages, d.max_pages, 0)
        row = 288 if d.format == FMT_FP4_KV else 36
        return csa2_cache(d.data + b * d.seq_stride * row, d.format, 0, d.seq_stride, d.seq_stride,
                          None, 0, 0)


def csa2_quantize_kv(src, cache, start_pos=None, seq_lens=None, stream=None):
    """src: CUDA fp32 [n_seqs, rows_per_seq, C] -> packed rows in ``cache``
    (a Cache, or a csa2_cache descriptor such as Cache.seq_view(b))."""
    ref = cache.ref if isinstance(cache, Cache) else ctypes.byref(cache)
    _check(load().csa2_quantize_kv(_ptr(src), src.shape[0], src.shape[1], _ptr(start_pos), _ptr(seq_lens),
                                   ref, _stream(stream)))


def csa2_index_topk(mode, keys: Cache, q_idx, w, seq_lens, max_seq_len, topk, pool=None, out_idx=None,
                    out_pool=None, with_scores=False, workspace=None, stream=None):
    """Returns (idx [B, topk], pool [B, P] or None, scores or None)."""
    import torch
    L = load()
    B = q_idx.shape[0]
    dev = q_idx.device
    pool_len = pool.shape[1] if pool is not None else 0
    if out_idx is None:
        out_idx = torch.empty((B, topk), dtype=torch.int32, device=dev)
    P = out_pool.shape[1] if out_pool is not None else 0
    scores = None
    if with_scores:
        scores = torch.full((B, pool_len if pool is not None else max_seq_len), float("nan"),
                            dtype=torch.float32, device=dev)
    need = L.csa2_index_topk_workspace(B, max_seq_len, pool_len, topk, P)
    if workspace is None:
        workspace = new_workspace(need, dev)
    _check(L.csa2_index_topk(mode, keys.ref, _ptr(q_idx), _ptr(w), B, q_idx.shape[1], q_idx.shape[2],
                             _ptr(seq_lens), max_seq_len, _ptr(pool), pool_len, topk, _ptr(out_idx),
                             _ptr(out_pool), P, _ptr(scores), _ptr(workspace), workspace.numel(),
                             _stream(stream)))
    return out_idx, out_pool, scores


def csa2_index_topk_multi_workspace(batch, n_q, max_seq_len) -> int:
    return int(load().csa2_index_topk_multi_workspace(batch, n_q, max_seq_len))


def csa2_index_topk_multi(keys: Cache, q_idx, w, seq_lens, max_seq_len, topk, causal=True, out_idx=None,
                          with_idx=True, with_scores=False, workspace=None, stream=None):
    """Many queries per sequence: q_idx [B, n_q, 4, 64], w [B, n_q, 4].
    Returns (idx [B, n_q, topk] or None, scores [B, n_q, max_seq_len] or None)."""
    import torch
    L = load()
    B, nq = q_idx.shape[0], q_idx.shape[1]
    dev = q_idx.device
    if with_idx and out_idx is None:
        out_idx = torch.empty((B, nq, topk), dtype=torch.int32, device=dev)
    if not with_idx:
        out_idx = None
    scores = None
    if with_scores:
        scores = torch.full((B, nq, max_seq_len), float("nan"), dtype=torch.float32, device=dev)
    need = L.csa2_index_topk_multi_workspace(B, nq, max_seq_len)
    if workspace is None:
        workspace = new_workspace(need, dev)
    _check(L.csa2_index_topk_multi(keys.ref, _ptr(q_idx), _ptr(w), B, nq, q_idx.shape[2], q_idx.shape[3],
                                   _ptr(seq_lens), max_seq_len, 1 if causal else 0, topk, _ptr(out_idx),
                                   _ptr(scores), _ptr(workspace), workspace.numel(), _stream(stream)))
    return out_idx, scores


def csa2_sparse_attn(kv, swa, q, seq_lens, max_seq_len, idx, topk, swa_window, out=None, lse=None,
                     workspace=None, stream=None):
    """Returns (out [B, 16, 512], lse [B, 16])."""
    import torch
    L = load()
    B = q.shape[0]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, q.shape[1]), dtype=torch.float32, device=q.device)
    need = int(L.csa2_sparse_attn_workspace(B, topk if idx is not None else 0, swa_window))
    if workspace is None and need > 0:
        workspace = new_workspace(need, q.device)
    _check(L.csa2_sparse_attn(kv.ref if kv is not None else None, swa.ref if swa is not None else None,
                              _ptr(q), B, q.shape[1], q.shape[2], _ptr(seq_lens), max_seq_len, _ptr(idx),
                              topk, swa_window, _ptr(out), _ptr(lse), _ptr(workspace),
                              workspace.numel() if workspace is not None else 0, _stream(stream)))
    return out, lse


def csa2_sparse_attn_noalloc(kv, swa, q, seq_lens, max_seq_len, idx, topk, swa_window, out=None, lse=None,
                             stream=None):
    """csa2_sparse_attn without a workspace (the library's fixed scratch
    array stands in for it).  Returns (out [B, 16, 512], lse [B, 16])."""
    import torch
    L = load()
    B = q.shape[0]
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((B, q.shape[1]), dtype=torch.float32, device=q.device)
    _check(L.csa2_sparse_attn_noalloc(kv.ref if kv is not None else None, swa.ref if swa is not None else None,
                                      _ptr(q), B, q.shape[1], q.shape[2], _ptr(seq_lens), max_seq_len, _ptr(idx),
                                      topk, swa_window, _ptr(out), _ptr(lse), _stream(stream)))
    return out, lse


def layer_array(descs):
    arr = (csa2_layer_desc * len(descs))()
    for i, d in enumerate(descs):
        arr[i] = d
    return arr


def csa2_decode_layers_workspace(descs, batch, max_seq_len, topk, pool_len, swa_window) -> int:
    arr = layer_array(descs)
    return int(load().csa2_decode_layers_workspace(arr, len(descs), batch, max_seq_len, topk, pool_len,
                                                   swa_window))


def csa2_decode_layers(descs, batch, seq_lens, max_seq_len, topk, pool_len, swa_window, workspace,
                       stream=None, arr=None):
    """One decode step over the schedule described by ``descs`` (csa2_layer_desc)."""
    if arr is None:
        arr = layer_array(descs)
    _check(load().csa2_decode_layers(arr, len(descs), batch, _ptr(seq_lens), max_seq_len, topk, pool_len,
                                     swa_window, _ptr(workspace), workspace.numel(), _stream(stream)))


def csa2_decode_layer_workspace(descs, batch, max_seq_len, topk, pool_len, swa_window) -> int:
    arr = layer_array(descs)
    return int(load().csa2_decode_layer_workspace(arr, len(descs), batch, max_seq_len, topk, pool_len,
                                                  swa_window))


def csa2_decode_layer(descs, layer, batch, seq_lens, max_seq_len, topk, pool_len, swa_window, workspace,
                      stream=None, arr=None):
    """Layer ``layer`` of the schedule ``descs`` alone (appends, indexing, attention)."""
    if arr is None:
        arr = layer_array(descs)
    _check(load().csa2_decode_layer(arr, len(descs), layer, batch, _ptr(seq_lens), max_seq_len, topk, pool_len,
                                    swa_window, _ptr(workspace), workspace.numel(), _stream(stream)))


def csa2_test_set_wait_limit(polls: int):
    """Test hook: polls of each fused indexing CTA's first tile wait (< 0: normal)."""
    _check(load().csa2_test_set_wait_limit(int(polls)))


def new_workspace(nbytes, device):
    """A workspace as the C interface wants it: zero-filled before first use."""
    import torch
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)


def _modes_arr(modes):
    arr = (ctypes.c_int32 * len(modes))(*[int(m) for m in modes])
    return arr


def csa2_plan_footprint(modes, context, topk, pool_len, window, hbm_bytes) -> dict:
    """Footprint of one session (see include/csa2.h); modes: CSA2_MODE_* per layer."""
    out = csa2_footprint()
    _check(load().csa2_plan_footprint(_modes_arr(modes), len(modes), int(context), int(topk), int(pool_len),
                                      int(window), int(hbm_bytes), ctypes.byref(out)))
    return {k: int(getattr(out, k)) for k, _ in csa2_footprint._fields_}


def csa2_plan_cost(modes, context, topk, pool_len, window) -> dict:
    """Compute and traffic of one decode token (see include/csa2.h)."""
    out = csa2_cost()
    _check(load().csa2_plan_cost(_modes_arr(modes), len(modes), int(context), int(topk), int(pool_len),
                                 int(window), ctypes.byref(out)))
    return {k: float(getattr(out, k)) for k, _ in csa2_cost._fields_}


def csa2_check_device(stream=None):
    """Synchronise and return (status, raw flag bits) of the device flag word."""
    L = load()
    st = L.csa2_check_device(_stream(stream))
    return st, int(L.csa2_last_device_flags())


def csa2_set_phase_events(events):
    L = load()
    n = len(events)
    arr = (ctypes.c_void_p * max(n, 1))(*[ctypes.c_void_p(e.cuda_event) for e in events])
    _check(L.csa2_set_phase_events(arr, n))


def csa2_launch_count() -> int:
    return int(load().csa2_launch_count())


def csa2_last_error() -> str:
    return load().csa2_last_error().decode()
