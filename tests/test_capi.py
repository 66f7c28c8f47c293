"""C interface checks that need no GPU: the library loads, exports every
function include/csa2.h declares, and rejects bad arguments on the host
before touching the device."""
import ctypes
import os
import re

import pytest

from conftest import ROOT

import csa2_sparse_attention_03_b300 as csa2


def _declared():
    text = open(os.path.join(ROOT, "include", "csa2.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(csa2_[a-z0-9_]+)\s*\(", text)))


@pytest.fixture(scope="module")
def lib():
    from csa2_sparse_attention_03_b300 import build
    build.build()
    return csa2.load()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert len(names) >= 12
    for n in names:
        assert hasattr(lib, n), n


def test_version_and_sizes(lib):
    assert lib.csa2_version() >= 100
    assert lib.csa2_cache_bytes(csa2.FMT_FP4_KV, 10) == 2880
    assert lib.csa2_cache_bytes(csa2.FMT_FP4_IDX, 128) == 2 * 2304
    assert lib.csa2_cache_bytes(csa2.FMT_FP4_IDX, 100) == 0
    assert lib.csa2_cache_bytes(csa2.FMT_FP8_SWA, 128) == 128 * 516
    assert lib.csa2_cache_bytes(7, 128) == 0


def _fake_cache(fmt, n_slots, stride, data=0x10000):
    return csa2.csa2_cache(data, fmt, 0, n_slots, stride, None, 0, 0)


def test_index_topk_rejects_bad_arguments(lib):
    P = ctypes.c_void_p
    keys = _fake_cache(csa2.FMT_FP4_IDX, 1024, 1024)
    buf = P(0x20000)

    def call(mode=csa2.MODE_FULL, k=keys, heads=4, dim=64, B=1, L=1000, topk=64, ws=P(0x40000), wsb=1 << 30):
        return lib.csa2_index_topk(mode, ctypes.byref(k), buf, buf, B, heads, dim, buf, L, None, 0, topk, buf,
                                   None, 0, None, ws, wsb, None)

    assert call(mode=csa2.MODE_REUSE) == csa2.ERR_INVALID_ARG
    assert call(heads=8) == csa2.ERR_UNSUPPORTED
    assert call(topk=0) == csa2.ERR_INVALID_ARG
    assert call(topk=70000) == csa2.ERR_INVALID_ARG
    assert call(B=0) == csa2.ERR_INVALID_ARG
    assert call(L=2000) == csa2.ERR_INVALID_ARG           # seq_stride 1024 < max_seq_len
    assert call(k=_fake_cache(csa2.FMT_FP4_KV, 1024, 1024)) == csa2.ERR_INVALID_ARG
    assert call(k=_fake_cache(csa2.FMT_FP4_IDX, 1000, 1000)) == csa2.ERR_INVALID_ARG
    assert call(k=_fake_cache(csa2.FMT_FP4_IDX, 1024, 1024, data=0x10001)) == csa2.ERR_INVALID_ARG
    assert call(ws=None) == csa2.ERR_WORKSPACE
    assert call(ws=P(0x40010)) == csa2.ERR_WORKSPACE
    assert call(wsb=16) == csa2.ERR_WORKSPACE
    assert "workspace" in lib.csa2_last_error().decode()


def test_sparse_attn_and_quantize_reject_bad_arguments(lib):
    P = ctypes.c_void_p
    kv = _fake_cache(csa2.FMT_FP4_KV, 4096, 4096)
    swa = _fake_cache(csa2.FMT_FP8_SWA, 128, 128)
    buf = P(0x20000)
    ws = P(0x40000)
    assert lib.csa2_sparse_attn(ctypes.byref(kv), ctypes.byref(swa), buf, 1, 8, 512, buf, 4096, buf, 64, 128,
                                buf, None, ws, 1 << 30, None) == csa2.ERR_UNSUPPORTED
    assert lib.csa2_sparse_attn(ctypes.byref(kv), ctypes.byref(swa), P(0x20004), 1, 16, 512, buf, 4096, buf, 64,
                                128, buf, None, ws, 1 << 30, None) == csa2.ERR_INVALID_ARG
    small = _fake_cache(csa2.FMT_FP8_SWA, 64, 64)
    assert lib.csa2_sparse_attn(ctypes.byref(kv), ctypes.byref(small), buf, 1, 16, 512, buf, 4096, buf, 64, 128,
                                buf, None, ws, 1 << 30, None) == csa2.ERR_INVALID_ARG  # ring < window
    assert lib.csa2_quantize_kv(buf, 1, 10, None, None, None, None) == csa2.ERR_INVALID_ARG
    assert lib.csa2_quantize_kv(P(0x20008), 1, 10, None, None, ctypes.byref(kv), None) == csa2.ERR_INVALID_ARG
    bad = _fake_cache(9, 4096, 4096)
    assert lib.csa2_quantize_kv(buf, 1, 10, None, None, ctypes.byref(bad), None) == csa2.ERR_INVALID_ARG
    assert lib.csa2_quantize_kv(buf, 0, 10, None, None, ctypes.byref(kv), None) == csa2.OK  # nothing to do


def test_decode_layers_rejects_bad_schedules(lib):
    P = ctypes.c_void_p
    kv = _fake_cache(csa2.FMT_FP4_KV, 4096, 4096)
    ik = _fake_cache(csa2.FMT_FP4_IDX, 4096, 4096)
    swa = _fake_cache(csa2.FMT_FP8_SWA, 128, 128)
    buf = 0x20000

    def desc(mode, kv_src=-1, idx_src=-1, use_pool=0):
        d = csa2.csa2_layer_desc()
        d.mode, d.kv_src, d.idx_src, d.use_pool = mode, kv_src, idx_src, use_pool
        d.kv, d.idx_keys, d.swa = ctypes.pointer(kv), ctypes.pointer(ik), ctypes.pointer(swa)
        d.q = d.q_idx = d.w = d.out = d.idx_out = d.pool_out = buf
        return d

    ok = [desc(csa2.MODE_FULL, 0, 0), desc(csa2.MODE_REINDEX, 0), desc(csa2.MODE_REUSE, 0, 1),
          desc(csa2.MODE_SWA_ONLY)]
    arr = csa2.layer_array(ok)
    assert lib.csa2_decode_layers_workspace(arr, 4, 1, 4096, 512, 0, 128) > 0
    cases = [
        [desc(csa2.MODE_REUSE, 0, 0)],                                    # no earlier FULL
        [desc(csa2.MODE_FULL, 1, 0)],                                     # FULL must name itself
        [desc(csa2.MODE_FULL, 0, 0), desc(csa2.MODE_REUSE, 0, 3)],        # forward source
        [desc(csa2.MODE_FULL, 0, 0), desc(csa2.MODE_REINDEX, 0, use_pool=1)],  # pool without pool_len
        [desc(7)],
    ]
    for c in cases:
        a = csa2.layer_array(c)
        assert lib.csa2_decode_layers(a, len(c), 1, P(buf), 4096, 512, 0, 128, P(0x40000), 1 << 30, None) \
            == csa2.ERR_INVALID_ARG, lib.csa2_last_error()
    assert lib.csa2_decode_layers(arr, 4, 1, P(buf), 4096, 512, 0, 128, P(0x40000), 16, None) == csa2.ERR_WORKSPACE


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(csa2, "_lib", None)
    monkeypatch.setattr(csa2, "LIB_PATH", "/nonexistent/libcsa2.so")
    with pytest.raises(ImportError):
        csa2.load()
