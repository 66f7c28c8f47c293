"""Step 4 parity: one decode step over each workload's schedule (shrunk
lengths), against the oracle layer by layer; graph capture and determinism."""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import synth
from csa2_sparse_attention_03_b300.schedule import DecodeStep
from helpers import oracle_step, within_tol

pytestmark = pytest.mark.gpu


def _compare(step, ref, w):
    for l, ly in enumerate(w.layers):
        if ly.mode in (synth.FULL, synth.REINDEX):
            got = step.idx[l].cpu().numpy()
            assert np.array_equal(got, ref[l]["idx"]), f"layer {l}: indices differ"
        if ref[l]["pool"] is not None:
            assert np.array_equal(step.pool[l].cpu().numpy(), ref[l]["pool"]), f"layer {l}: pool differs"
        ok, ex = within_tol(step.out[l].cpu().numpy(), ref[l]["out"])
        assert ok, f"layer {l}: output excess {ex:.3e}"
        lse = step.lse[l].cpu().numpy()
        assert np.allclose(lse, ref[l]["lse"], atol=2e-3, rtol=1e-3), f"layer {l}: lse"


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_decode_step_small(cuda, orc, cfg):
    w = synth.workload(cfg, small=True)
    step = DecodeStep(w, fill="host")
    step.run()
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags, cuda.csa2_last_error())
    ref, caches, _ = oracle_step(orc, w)
    _compare(step, ref, w)
    # after the step the caches hold every token, appended one included
    for f, (kv, ik) in step.caches.items():
        gv = kv.data.cpu().numpy().reshape(-1, 288)
        gk = ik.data.cpu().numpy()
        for b, L in enumerate(w.seq_lens):
            if w.paged:
                slots = orc.slots_paged(step.page_tables[f][b].cpu().numpy(), np.arange(L), 64)
            else:
                slots = orc.slots_contiguous(b, np.arange(L), kv.desc.seq_stride)
            c = caches[f][b]
            assert np.array_equal(gv[slots], orc.kv_rows(c["kv_codes"], c["kv_scales"]))
            rc, rs = orc.read_idx(gk, slots)
            assert np.array_equal(rc, c["k_codes"]) and np.array_equal(rs, c["k_scales"])


def test_graph_replay_and_determinism(cuda, orc):
    w = synth.workload(1, small=True)
    step = DecodeStep(w, fill="host")
    step.run()
    torch.cuda.synchronize()
    first = [t.clone() for t in step.step_outputs()]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step.run(stream=s)  # warm-up on the capture stream
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step.run(stream=s)
    for _ in range(3):
        for t in step.step_outputs():
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(first, step.step_outputs()):
            assert torch.equal(a, b)
    st, flags = cuda.csa2_check_device()
    assert st == 0


@pytest.mark.parametrize("cfg", [0, 1, 2, 3, 4])
def test_decode_step_layer_sequential_small(cuda, orc, cfg):
    """The same step through csa2_decode_layer, one call per layer in schedule
    order (the order a model runs it in), against the oracle layer by layer."""
    w = synth.workload(cfg, small=True)
    step = DecodeStep(w, fill="host")
    step.run_sequential()
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags, cuda.csa2_last_error())
    ref, _, _ = oracle_step(orc, w)
    _compare(step, ref, w)


def test_layer_sequential_graph_replays_identically(cuda, orc):
    w = synth.workload(2, small=True)
    step = DecodeStep(w, fill="host")
    step.run_sequential()
    torch.cuda.synchronize()
    first = [t.clone() for t in step.step_outputs()]
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        step.run_sequential(stream=s)
        torch.cuda.synchronize()
        with torch.cuda.graph(g, stream=s):
            step.run_sequential(stream=s)
    for _ in range(3):
        for t in step.step_outputs():
            t.zero_()
        g.replay()
        torch.cuda.synchronize()
        for a, b in zip(first, step.step_outputs()):
            assert torch.equal(a, b)
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags)


def test_pipelined_serving_step_copies_every_output(cuda, orc):
    """DecodeStep.capture_sequential: the inputs come in from pinned host memory
    by groups of layers and the outputs go back by groups, overlapping the
    kernels.  The host copy of the outputs equals what the plain layer-
    sequential step writes on the device, bit for bit, and matches the oracle;
    the device inputs equal the host inputs."""
    w = synth.workload(2, small=True)
    step = DecodeStep(w, fill="host")
    ref, _, _ = oracle_step(orc, w)
    h_in = step.arena_in.detach().cpu().pin_memory()
    step.run_sequential()
    torch.cuda.synchronize()
    want = step.arena_out.detach().cpu().clone()
    h_out = torch.zeros(step.arena_out.shape, dtype=step.arena_out.dtype, pin_memory=True)
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        g = step.capture_sequential(s, h_in, h_out)
    for _ in range(2):
        step.arena_in.zero_()
        step.arena_out.zero_()
        h_out.zero_()
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(step.arena_in.cpu(), h_in)
        assert torch.equal(h_out, want)
    _compare(step, ref, w)
    st, flags = cuda.csa2_check_device()
    assert st == 0, (st, flags, cuda.csa2_last_error())
