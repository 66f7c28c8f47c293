"""The static layer schedules, pinned independently of the code that builds
them: the 40-layer schedule against a hand-written table (tests/golden/
schedule_40.txt, from the Helmcode explainer's "03 · CSA2" counts and the
stated placement reading), and the 10-layer and hierarchical schedules of the
other workloads against their stated shapes.  Both the oracle's decode step
and the GPU descriptors consume these sources, so a wrong source rule would
otherwise pass parity on both sides."""
from collections import Counter

from conftest import read_golden

from csa2_sparse_attention_03_b300 import synth

NAMES = {"F": synth.FULL, "R": synth.REINDEX, "U": synth.REUSE, "S": synth.SWA_ONLY}


def test_forty_layer_schedule_matches_the_golden_table():
    rows = read_golden("schedule_40.txt")
    assert len(rows) == 40
    modes = synth.forty_layer_modes()
    layers = synth.build_layers(modes)
    for (i, m, kv, ix), ly, mode_str in zip(rows, layers, modes):
        assert mode_str == m, i
        assert ly.mode == NAMES[m], i
        if m != "S":
            assert (ly.kv_src, ly.idx_src) == (int(kv), int(ix)), i
        assert not ly.use_pool
    # the counts the explainer gives
    assert Counter(modes) == Counter({"U": 30, "F": 4, "R": 4, "S": 2})


def test_every_workload_schedule_is_the_stated_one():
    w0 = synth.workload(0)
    assert [(ly.mode, ly.kv_src, ly.idx_src) for ly in w0.layers] == [(synth.FULL, 0, 0)]
    w1 = synth.workload(1)
    want1 = [(synth.FULL, 0, 0), (synth.REINDEX, 0, 1)] + [(synth.REUSE, 0, 1)] * 7
    assert [(ly.mode, ly.kv_src, ly.idx_src) for ly in w1.layers[:9]] == want1
    assert w1.layers[9].mode == synth.SWA_ONLY and len(w1.layers) == 10
    w3 = synth.workload(3)
    assert [(ly.mode, ly.kv_src, ly.use_pool) for ly in w3.layers] == \
        [(synth.FULL, 0, False)] + [(synth.REINDEX, 0, True)] * 3
    assert w3.pool_len == 16384 and w3.topk == 2048 and w3.max_len == 1 << 20
    for cfg in (2, 4):
        w = synth.workload(cfg)
        assert "".join(synth.MODE_NAMES[ly.mode] for ly in w.layers) == \
            "".join(r[1] for r in read_golden("schedule_40.txt"))
