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
N_FULL, N_REINDEX, N_SWA_ONLY, N_LAYERS = 4, 4, 2, 40


def test_layer_sequential_step_bytes_l131072():
    """Every Full and every Reindex layer reads all 131,072 keys (each key pass
    counted), every layer but the SWA-only ones gathers its 2,048 rows."""
    import bench

    w = synth.workload(2)
    p = bench.step_bytes(w)
    assert p["scan"] == (N_FULL + N_REINDEX) * L * IDX == 37_748_736
    assert p["gather"] == (N_LAYERS - N_SWA_ONLY) * K * KV == 22_413_312
    assert p["swa"] == N_LAYERS * W * SWA
    io = (N_LAYERS * (Q + OUT + LSE)
          + (N_FULL + N_REINDEX) * (IDXQ + K * 4)          # indexer inputs, indices written
          + (N_LAYERS - N_SWA_ONLY) * K * 4                # indices read by attention
          + N_FULL * (512 * 4 + KV + 64 * 4 + IDX)         # the appended token: fp32 in, packed out
          + N_LAYERS * (512 * 4 + SWA))                    # each layer's window append
    assert p["io"] == io
    assert p["total"] == p["scan"] + p["gather"] + p["swa"] + p["io"] == 65_926_192


def test_fused_step_bytes_l131072():
    """The phased launch sequence: one key pass per Full/Reindex pair, and the
    rows of a selection gathered once per unit of two layers (a Full layer
    alone: 1 unit; Reindex + its Reuse layers, 8 or 9 layers: 4 or 5 units)."""
    import bench

    w = synth.workload(2)
    p = bench.fused_step_bytes(w)
    assert p["scan"] == N_FULL * L * IDX
    # groups: F alone x4 (1 unit each); R + 7 U (8 layers, 4 units) x2; R + 8 U (9 layers, 5 units) x2
    units = 4 * 1 + 2 * 4 + 2 * 5
    assert p["gather"] == units * K * KV
    assert p["total"] == p["scan"] + p["gather"] + p["swa"] + p["io"]


def test_launch_bytes_l131072():
    import bench

    w = synth.workload(2)
    reuse = w.layers[2]
    assert reuse.mode == synth.REUSE
    assert bench.attention_launch_bytes(w, reuse) == K * KV + W * SWA + Q + OUT + LSE + K * 4
    full = w.layers[0]
    assert bench.index_launch_bytes(w, full) == L * IDX + IDXQ + K * 4 + 512 * 4 + KV + 64 * 4 + IDX
