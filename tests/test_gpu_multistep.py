"""Several decode steps in a row over the same caches: the appended main-KV
row, indexer key and window row of each step are where the next step finds
them, and the FP8 window ring (128 slots, position p in slot p mod 128) wraps
correctly.  Each step is checked against the oracle run on the whole logical
history up to that step (Helmcode "DeepSeek V4.1 Flash" explainer, "03 ·
CSA2": each layer keeps its own window state; Louis Bouchard's KV-cache
report, "Share the cache and the search work": the 128-token local window).
Steps alternate between the layer-sequential and the phased entry points."""
import numpy as np
import pytest
import torch

from csa2_sparse_attention_03_b300 import csa2_decode_layers_workspace, new_workspace, synth
from csa2_sparse_attention_03_b300.schedule import DecodeStep
from helpers import within_tol

pytestmark = pytest.mark.gpu

N_STEPS = 4


def _workload(paged):
    # lengths chosen so that N_STEPS - 1 more tokens stay inside each
    # sequence's last 64-token page (paged) and inside the contiguous stride
    lens = [300, 251]
    return synth.Workload("multistep", 4242 + int(paged), 2, lens,
                          synth.build_layers(["F", "R", "U", "U", "S"]), 64, paged=paged)


def _step_draws(w, s):
    """Per-step inputs of step s >= 1 (step 0 uses the workload's own draws)."""
    B = w.batch
    q = {l: synth.normal_rows(w.seed, "ms_q", (l, s), 0, B * 16, 512, scale=1 / np.sqrt(512)).reshape(B, 16, 512)
         for l in range(len(w.layers))}
    qi = {l: synth.normal_rows(w.seed, "ms_qi", (l, s), 0, B * 4, 64, scale=1 / 8).reshape(B, 4, 64)
          for l, ly in enumerate(w.layers) if ly.mode in (synth.FULL, synth.REINDEX)}
    wt = {l: synth.uniform(w.seed, "ms_w", (l, s), (B, 4)).astype(np.float32) for l in qi}
    swa_new = {l: synth.normal_rows(w.seed, "ms_swa", (l, s), 0, B, 512) for l in range(len(w.layers))}
    return q, qi, wt, swa_new


def _oracle(orc, w, lens, q, qi, wt, windows):
    caches, per = {}, {}
    for f, ly in enumerate(w.layers):
        if ly.mode != synth.FULL:
            continue
        caches[f] = {}
        for b, L in enumerate(lens):
            kc, ks = orc.quant_fp4(synth.kv_values(w, f, b, 0, L))
            ic, isc = orc.quant_fp4(synth.idx_key_values(w, f, b, 0, L))
            caches[f][b] = dict(kv_codes=kc, kv_scales=ks, k_codes=ic, k_scales=isc)
    for l, ly in enumerate(w.layers):
        codes, scales = [], []
        for b in range(w.batch):
            c, s_ = orc.quant_fp8(windows[l][b][-w.window:])
            codes.append(c)
            scales.append(s_)
        per[l] = dict(q=q[l], swa_codes=codes, swa_scales=scales, q_idx=qi.get(l), w=wt.get(l))
    return orc.decode_step(w.layers, list(lens), w.topk, w.pool_len, caches, per)


@pytest.mark.parametrize("paged", [False, True])
def test_consecutive_steps_append_and_wrap_the_window(cuda, orc, paged):
    w = _workload(paged)
    B = w.batch
    step = DecodeStep(w, fill="host")
    # room for the later steps: the caches hold them already (stride / pages)
    step.Lmax = max(w.seq_lens) + N_STEPS - 1
    step.ws_bytes = csa2_decode_layers_workspace(step.descs, B, step.Lmax, step.topk, step.pool_len, step.window)
    step.workspace = new_workspace(step.ws_bytes, step.device)
    lens = list(w.seq_lens)
    # logical window history per layer and sequence, oldest first
    windows = {l: [synth.swa_values(w, l, b).astype(np.float32) for b in range(B)] for l in range(len(w.layers))}
    q = {l: synth.query(w, l) for l in range(len(w.layers))}
    qi = {l: synth.index_query(w, l) for l, ly in enumerate(w.layers) if ly.mode in (synth.FULL, synth.REINDEX)}
    wt = {l: synth.index_weights(w, l) for l in qi}
    for s in range(N_STEPS):
        if s > 0:
            lens = [L + 1 for L in lens]
            q, qi, wt, swa_new = _step_draws(w, s)
            for l in range(len(w.layers)):
                step.q[l].copy_(torch.from_numpy(q[l]))
                step.new_rows[("swa", l)].copy_(torch.from_numpy(swa_new[l]))
                for b in range(B):
                    windows[l][b] = np.concatenate([windows[l][b], swa_new[l][b:b + 1]])
            for l in qi:
                step.q_idx[l].copy_(torch.from_numpy(qi[l]))
                step.wts[l].copy_(torch.from_numpy(wt[l]))
            for f in step.caches:
                for b, L in enumerate(lens):
                    step.new_rows[("kv", f)][b].copy_(torch.from_numpy(synth.kv_values(w, f, b, L - 1, 1)[0]))
                    step.new_rows[("idxk", f)][b].copy_(torch.from_numpy(synth.idx_key_values(w, f, b, L - 1, 1)[0]))
            step.seq_lens.copy_(torch.tensor(lens, dtype=torch.int32))
        if s % 2 == 0:
            step.run_sequential()
        else:
            step.run()
        st, flags = cuda.csa2_check_device()
        assert st == 0, (s, st, flags, cuda.csa2_last_error())
        ref = _oracle(orc, w, lens, q, qi, wt, windows)
        for l, ly in enumerate(w.layers):
            if ly.mode in (synth.FULL, synth.REINDEX):
                assert np.array_equal(step.idx[l].cpu().numpy(), ref[l]["idx"]), f"step {s}, layer {l}: indices"
            ok, ex = within_tol(step.out[l].cpu().numpy(), ref[l]["out"])
            assert ok, f"step {s}, layer {l}: output excess {ex:.3e}"
            assert np.allclose(step.lse[l].cpu().numpy(), ref[l]["lse"], atol=2e-3, rtol=1e-3), f"step {s}, layer {l}"
