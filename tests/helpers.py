"""Test helpers: oracle-side inputs of a workload from the same seeded streams
the GPU path consumes, and the attention tolerance."""
import numpy as np

from csa2_sparse_attention_03_b300 import synth

# Attention outputs: |gpu - ref| <= ATOL + RTOL * |ref| elementwise (fp32
# accumulation of fp16 operands against the fp64 oracle).
ATOL, RTOL = 2e-3, 1e-2


def within_tol(got, ref, atol=ATOL, rtol=RTOL):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    excess = np.abs(got - ref) - (atol + rtol * np.abs(ref))
    return bool((excess <= 0).all()), float(excess.max()) if excess.size else 0.0


def oracle_inputs(orc, w: synth.Workload, layers_needed=None):
    """caches[f][b] and per_layer[l] for oracle.decode_step, in logical order."""
    caches, per = {}, {}
    for f, ly in enumerate(w.layers):
        if ly.mode != synth.FULL:
            continue
        caches[f] = {}
        for b, L in enumerate(w.seq_lens):
            kc, ks = orc.quant_fp4(synth.kv_values(w, f, b, 0, L))
            ic, isc = orc.quant_fp4(synth.idx_key_values(w, f, b, 0, L))
            caches[f][b] = dict(kv_codes=kc, kv_scales=ks, k_codes=ic, k_scales=isc)
    for l, ly in enumerate(w.layers):
        codes, scales = [], []
        for b, L in enumerate(w.seq_lens):
            n = min(w.window, L)
            c, s = orc.quant_fp8(synth.swa_values(w, l, b)[w.window - n:])
            codes.append(c)
            scales.append(s)
        pl = dict(q=synth.query(w, l), swa_codes=codes, swa_scales=scales, q_idx=None, w=None)
        if ly.mode in (synth.FULL, synth.REINDEX):
            pl["q_idx"] = synth.index_query(w, l)
            pl["w"] = synth.index_weights(w, l)
        per[l] = pl
    return caches, per


def oracle_step(orc, w: synth.Workload):
    caches, per = oracle_inputs(orc, w)
    return orc.decode_step(w.layers, list(w.seq_lens), w.topk, w.pool_len, caches, per), caches, per


def oracle_inputs_seq(orc, w: synth.Workload, b: int, chunk=synth.CHUNK_ROWS):
    """caches[f][0] and per_layer[l] of sequence b alone (a batch of one), from
    the same streams the GPU path draws sequence b from; the main KV is
    quantised chunk by chunk so long contexts stay within memory."""
    L = int(w.seq_lens[b])
    caches, per = {}, {}
    for f, ly in enumerate(w.layers):
        if ly.mode != synth.FULL:
            continue
        kc = np.empty((L, 256), np.uint8)
        ks = np.empty((L, 32), np.uint8)
        for r0 in range(0, L, chunk):
            n = min(chunk, L - r0)
            kc[r0:r0 + n], ks[r0:r0 + n] = orc.quant_fp4(synth.kv_values(w, f, b, r0, n))
        ic = np.empty((L, 32), np.uint8)
        isc = np.empty((L, 4), np.uint8)
        for r0 in range(0, L, chunk):
            n = min(chunk, L - r0)
            ic[r0:r0 + n], isc[r0:r0 + n] = orc.quant_fp4(synth.idx_key_values(w, f, b, r0, n))
        caches[f] = {0: dict(kv_codes=kc, kv_scales=ks, k_codes=ic, k_scales=isc)}
    for l, ly in enumerate(w.layers):
        n = min(w.window, L)
        c, s = orc.quant_fp8(synth.swa_values(w, l, b)[w.window - n:])
        pl = dict(q=synth.query(w, l)[b:b + 1], swa_codes=[c], swa_scales=[s], q_idx=None, w=None)
        if ly.mode in (synth.FULL, synth.REINDEX):
            pl["q_idx"] = synth.index_query(w, l)[b:b + 1]
            pl["w"] = synth.index_weights(w, l)[b:b + 1]
        per[l] = pl
    return caches, per


def oracle_step_seq(orc, w: synth.Workload, b: int):
    caches, per = oracle_inputs_seq(orc, w, b)
    return orc.decode_step(w.layers, [int(w.seq_lens[b])], w.topk, w.pool_len, caches, per)
