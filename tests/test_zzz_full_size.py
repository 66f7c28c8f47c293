"""Parity at the workloads' full sizes.

* The L = 131,072, 40-layer schedule (4 Full / 4 Reindex / 30 Reuse / 2
  SWA-only) at Top-K 2,048 -- the benchmark's workload -- through both launch
  sequences the bench times: the layer-sequential one (csa2_decode_layer per
  layer) and the phased one (csa2_decode_layers).  Every index set bit for bit,
  every layer's output and LSE within the attention tolerance, the appended
  token's packed bytes.  A second step with the queries scaled by 16 (logits
  spanning tens of units) checks the softmax rescale path at full size.
* The hierarchical workload: L = 1,048,576, the Full layer's 16,384-entry pool,
  three Reindex layers inside it, Top-K 2,048.
* The batch-64 ragged, paged workload (contexts 16K..64K, 40 layers, append):
  all 64 sequences run on the GPU; three of them are built from the host
  streams and followed by the oracle one by one (every index set and every
  layer's output of those sequences).
The inputs come from the same seeded host streams on both sides.  Slow, so the
file is named to run last.
"""
import os

import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth
from csa2_sparse_attention_03_b300.schedule import DecodeStep
from helpers import oracle_step_seq, within_tol

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


@pytest.fixture(autouse=True)
def _oracle_threads(orc):
    orc.set_threads(os.cpu_count() or 1)
    yield
    orc.set_threads(1)


def _compare_seq(step, ref, w, b, what):
    for l, ly in enumerate(w.layers):
        if ly.mode in (synth.FULL, synth.REINDEX):
            assert np.array_equal(step.idx[l][b].cpu().numpy(), ref[l]["idx"][0]), f"{what}: layer {l} indices"
        if ref[l]["pool"] is not None:
            assert np.array_equal(step.pool[l][b].cpu().numpy(), ref[l]["pool"][0]), f"{what}: layer {l} pool"
        ok, ex = within_tol(step.out[l][b].cpu().numpy(), ref[l]["out"][0])
        assert ok, f"{what}: layer {l} output excess {ex:.3e}"
        assert np.allclose(step.lse[l][b].cpu().numpy(), ref[l]["lse"][0], atol=2e-3, rtol=1e-5), \
            f"{what}: layer {l} lse"


def _clear(step):
    for t in step.step_outputs():
        t.fill_(0)


def test_full_size_decode_step(cuda, orc):
    w = synth.workload(2)
    assert (w.batch, w.max_len, len(w.layers), w.topk) == (1, 131072, 40, 2048)
    step = DecodeStep(w, fill="host")
    ref = oracle_step_seq(orc, w, 0)
    for order in ("layer-sequential", "phased"):
        _clear(step)
        step.run_sequential() if order == "layer-sequential" else step.run()
        st, flags = cuda.csa2_check_device()
        assert st == 0, (order, st, flags, cuda.csa2_last_error())
        _compare_seq(step, ref, w, 0, order)
    # the step appended position L-1 of every Full layer: its packed bytes match the oracle's
    L = int(w.seq_lens[0])
    for f, (kv, ik) in step.caches.items():
        slot = orc.slots_contiguous(0, np.array([L - 1]), kv.desc.seq_stride)
        got_kv = kv.data.cpu().numpy().reshape(-1, 288)[slot]
        kc, ks = orc.quant_fp4(synth.kv_values(w, f, 0, L - 1, 1))
        assert np.array_equal(got_kv, orc.kv_rows(kc, ks))
        rc, rs = orc.read_idx(ik.data.cpu().numpy(), slot)
        ic, isc = orc.quant_fp4(synth.idx_key_values(w, f, 0, L - 1, 1))
        assert np.array_equal(rc, ic) and np.array_equal(rs, isc)


def test_full_size_decode_step_scaled_queries(cuda, orc):
    """The same workload with every attention query scaled by 16 (another
    seed): logits span tens of units, so maxima move between tiles and the
    cluster's partials sit far apart."""
    w = synth.workload(2)
    w.seed += 7
    w.extra["q_scale"] = 16.0
    step = DecodeStep(w, fill="host")
    ref = oracle_step_seq(orc, w, 0)
    step.run_sequential()
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)
    _compare_seq(step, ref, w, 0, "scaled queries")


def test_full_size_hierarchical_pool(cuda, orc):
    w = synth.workload(3)
    assert (w.max_len, w.pool_len, w.topk, len(w.layers)) == (1 << 20, 16384, 2048, 4)
    step = DecodeStep(w, fill="host")
    ref = oracle_step_seq(orc, w, 0)
    for order in ("layer-sequential", "phased"):
        _clear(step)
        step.run_sequential() if order == "layer-sequential" else step.run()
        st, flags = cuda.csa2_check_device()
        assert st == 0, (order, st, flags, cuda.csa2_last_error())
        _compare_seq(step, ref, w, 0, order)


def test_full_size_batch64_ragged_paged(cuda, orc):
    w = synth.workload(4)
    assert w.batch == 64 and w.paged and len(w.layers) == 40
    sampled = [0, 31, 63]
    step = DecodeStep(w, fill="sampled", host_seqs=sampled)
    refs = {b: oracle_step_seq(orc, w, b) for b in sampled}
    for order in ("layer-sequential", "phased"):
        _clear(step)
        step.run_sequential() if order == "layer-sequential" else step.run()
        st, flags = cuda.csa2_check_device()
        assert st == 0, (order, st, flags, cuda.csa2_last_error())
        for b in sampled:
            _compare_seq(step, refs[b], w, b, f"{order}, sequence {b} (L={w.seq_lens[b]})")
