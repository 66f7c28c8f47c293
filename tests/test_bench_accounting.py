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


def test_traffic_record_is_read_only_for_unchanged_kernel_sources(tmp_path):
    """roofline.traffic comes from a committed ncu summary line, and is null
    once the kernel's sources differ from those the counters were taken on."""
    import bench

    sha = bench.kernel_source_sha16("attn_kernel")
    wl = "B1 L131072 40-layer 4F/4R/30U/2S K2048"
    (tmp_path / "a.md").write_text(
        "some text\n"
        f"traffic-record: kernel=attn_kernel workload={wl.replace(' ', '_')} launches=40 "
        f"dram_bytes_per_launch=123456.5 source_sha16={sha}\n")
    v, src = bench.recorded_traffic("attn_kernel", wl, str(tmp_path))
    assert v == 123456.5 and src.endswith("a.md")
    assert bench.recorded_traffic("attn_kernel", "another workload", str(tmp_path)) == (None, None)
    (tmp_path / "a.md").write_text(
        f"traffic-record: kernel=attn_kernel workload={wl.replace(' ', '_')} launches=40 "
        "dram_bytes_per_launch=1 source_sha16=0000000000000000\n")
    v, src = bench.recorded_traffic("attn_kernel", wl, str(tmp_path))
    assert v is None and "changed" in src
