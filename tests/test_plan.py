"""The planning calculators (csa2_plan_footprint, csa2_plan_cost) against the
oracle's independent restatement (oracle/plan.py) and against closed forms:
the packed-layout fixture, the benchmark's byte count, and hand sums."""
import numpy as np
import pytest

from conftest import read_golden

import csa2_sparse_attention_03_b300 as csa2
from csa2_sparse_attention_03_b300 import synth
from oracle import plan as oplan

F, R, U, S = 0, 1, 2, 3


@pytest.fixture(scope="module")
def lib():
    from csa2_sparse_attention_03_b300 import build
    build.build()
    return csa2.load()


def _forty():
    return [{"F": F, "R": R, "U": U, "S": S}[m] for m in synth.forty_layer_modes()]


def test_matches_the_oracle_on_random_schedules(lib):
    rs = np.random.default_rng(5)
    for _ in range(300):
        n = int(rs.integers(1, 48))
        modes = [F] + rs.integers(0, 4, n - 1).tolist()
        ctx = int(rs.integers(0, 1 << 21))
        topk = int(rs.integers(0, 65537))
        pool = int(rs.choice([0, int(rs.integers(1, 65537))]))
        win = int(rs.integers(0, 1000))
        hbm = int(rs.integers(0, 300 << 30))
        assert csa2.csa2_plan_footprint(modes, ctx, topk, pool, win, hbm) == \
            oplan.footprint(modes, ctx, topk, pool, win, hbm)
        got = csa2.csa2_plan_cost(modes, ctx, topk, pool, win)
        want = oplan.cost(modes, ctx, topk, pool, win)
        for k in want:
            assert got[k] == pytest.approx(want[k], rel=1e-12, abs=0.0), k


def test_footprint_closed_forms(lib):
    fx = {k: int(v) for k, v in read_golden("footprint.txt")}
    modes = _forty()
    f = csa2.csa2_plan_footprint(modes, 131072, 2048, 0, 128, 275_040 << 20)
    assert f["global_bytes_per_token"] == fx["global_bytes_per_token_4_full_layers"] == 4 * (288 + 36)
    assert f["cache_bytes"] == 131072 * 1296 + 40 * 128 * 516
    assert f["step_bytes"] == 40 * (2 * 16 * 512 * 4 + 64) + 8 * 2048 * 4
    assert f["sessions"] == (275_040 << 20) // (f["cache_bytes"] + f["step_bytes"])
    # a million tokens of global KV in this layout: 1.36 GB (the pages quote 0.89 GB for their 890 B/token)
    one_m = csa2.csa2_plan_footprint(modes, 1_000_000, 2048, 0, 0, 0)
    assert one_m["cache_bytes"] == (1_000_000 + 64 - 1) // 64 * 64 * 1296


def test_cost_closed_forms(lib):
    import bench

    modes = _forty()
    c = csa2.csa2_plan_cost(modes, 131072, 2048, 0, 128)
    # the benchmark's own count of the same step
    assert c["bytes_sequential"] == bench.step_bytes(synth.workload(2))["total"] == 65_926_192
    assert c["index_flops"] == 8 * 131072 * 2 * 4 * 64
    assert c["attn_flops"] == (38 * 2048 + 40 * 128) * 4 * 16 * 512
    assert c["weighted_flops"] == 0.25 * c["index_flops"] + 0.25 * 38 * 2048 * 4 * 16 * 512 + \
        0.5 * 40 * 128 * 4 * 16 * 512
    # hierarchical: Reindex layers score the 16,384-entry pool, not the context
    h = csa2.csa2_plan_cost([F, R, R, R], 1 << 20, 2048, 16384, 128)
    assert h["index_flops"] == ((1 << 20) + 3 * 16384) * 2 * 4 * 64
    assert h["bytes_sequential"] == bench.step_bytes(synth.workload(3))["total"]


def test_cost_grows_with_context_only_through_the_scan(lib):
    modes = _forty()
    a = csa2.csa2_plan_cost(modes, 4096, 2048, 0, 128)
    b = csa2.csa2_plan_cost(modes, 1 << 20, 2048, 0, 128)
    assert b["attn_flops"] == a["attn_flops"]
    assert b["index_flops"] == a["index_flops"] * 256


def test_rejects_bad_arguments(lib):
    import ctypes
    out = csa2.csa2_footprint()
    assert lib.csa2_plan_footprint(None, 1, 10, 1, 0, 0, 0, ctypes.byref(out)) == csa2.ERR_INVALID_ARG
    bad = (ctypes.c_int32 * 1)(9)
    assert lib.csa2_plan_footprint(bad, 1, 10, 1, 0, 0, 0, ctypes.byref(out)) == csa2.ERR_INVALID_ARG
    c = csa2.csa2_cost()
    assert lib.csa2_plan_cost(bad, 1, 10, 1, 0, 0, ctypes.byref(c)) == csa2.ERR_INVALID_ARG
