"""bench.py's algorithmic byte counts, recomputed by hand for the L = 131,072,
40-layer workload (B 1, Top-K 2,048, window 128; 4 Full, 4 Reindex, 30 Reuse,
2 SWA-only layers).  These totals are the numerators of every GB/s and roofline
fraction the bench reports."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from csa2_sparse_attention_03_b300 import synth  # noqa: E402

L, K, W = 131072, 2048, 128
KV, IDX, SWA = 288, 36, 516            # packed row bytes: FP4 main, FP4 indexer key, FP8 window
Q = OUT = 16 * 512 * 4                 # per layer and sequence, fp32
LSE = 16 * 4
IDXQ = 4 * 64 * 4 + 4 * 4              # indexer query and head weights


def test_step_bytes_l131072():
    import bench

    w = synth.workload(2)
    p = bench.step_bytes(w)
    n_full, n_reindex, n_swa_only = 4, 4, 2
    n_layers = 40
    # one key pass per Full layer: its pool-free Reindex partner scores in the same pass
    assert p["scan"] == n_full * L * IDX
    assert p["gather"] == (n_layers - n_swa_only) * K * KV
    assert p["swa"] == n_layers * W * SWA
    io = (n_layers * (Q + OUT + LSE)
          + (n_full + n_reindex) * (IDXQ + K * 4)          # indexer inputs, indices written
          + (n_layers - n_swa_only) * K * 4                # indices read by attention
          + n_full * (512 * 4 + KV + 64 * 4 + IDX)         # the appended token: fp32 in, packed out
          + n_layers * (512 * 4 + SWA))                    # each layer's window append
    assert p["io"] == io
    assert p["total"] == p["scan"] + p["gather"] + p["swa"] + p["io"] == 47_051_824


def test_attention_bytes_l131072():
    import bench

    w = synth.workload(2)
    assert bench.attention_bytes(w) == (38 * (K * KV + K * 4) + 40 * W * SWA + 40 * (Q + OUT + LSE))
