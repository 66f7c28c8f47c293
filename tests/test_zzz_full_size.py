"""Parity at the benchmark's full size.

One decode step of the L = 131,072, 40-layer schedule (4 Full / 4 Reindex /
30 Reuse / 2 SWA-only) at Top-K 2,048 -- the workload and the single
csa2_decode_layers launch sequence that bench.py times -- against the oracle
layer by layer: every Full and Reindex index set bit for bit, every layer's
output and LSE within the attention tolerance, and the appended token's packed
bytes in every Full layer's caches.  The inputs come from the same seeded host
streams on both sides (the bench fills its caches on the device only to save
set-up time).  Slow (about two minutes, most of it the oracle), so it is
named to run last.
"""
import numpy as np
import pytest

from csa2_sparse_attention_03_b300 import synth
from csa2_sparse_attention_03_b300.schedule import DecodeStep
from helpers import oracle_step, within_tol

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def test_full_size_decode_step(cuda, orc):
    w = synth.workload(2)
    assert (w.batch, w.max_len, len(w.layers), w.topk) == (1, 131072, 40, 2048)
    step = DecodeStep(w, fill="host")
    step.run()
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags, cuda.csa2_last_error())
    ref, caches, _ = oracle_step(orc, w)
    for l, ly in enumerate(w.layers):
        if ly.mode in (synth.FULL, synth.REINDEX):
            assert np.array_equal(step.idx[l].cpu().numpy(), ref[l]["idx"]), f"layer {l}: indices differ"
        ok, ex = within_tol(step.out[l].cpu().numpy(), ref[l]["out"])
        assert ok, f"layer {l}: output excess {ex:.3e}"
        assert np.allclose(step.lse[l].cpu().numpy(), ref[l]["lse"], atol=2e-3, rtol=1e-3), f"layer {l}: lse"
    # the step appended position L-1 of every Full layer: its packed bytes match the oracle's
    L = int(w.seq_lens[0])
    for f, (kv, ik) in step.caches.items():
        slot = orc.slots_contiguous(0, np.array([L - 1]), kv.desc.seq_stride)
        c = caches[f][0]
        got_kv = kv.data.cpu().numpy().reshape(-1, 288)[slot]
        assert np.array_equal(got_kv, orc.kv_rows(c["kv_codes"][L - 1:L], c["kv_scales"][L - 1:L]))
        rc, rs = orc.read_idx(ik.data.cpu().numpy(), slot)
        assert np.array_equal(rc, c["k_codes"][L - 1:L]) and np.array_equal(rs, c["k_scales"][L - 1:L])
