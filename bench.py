#!/usr/bin/env python3
"""Benchmark of one CSA2 decode step on B300.

A step is one pass of the whole decode path over one batch: the quantise-and-
append of the new token into every Full layer's FP4 caches and every layer's
FP8 window ring, indexer scoring and Top-K of the Full and Reindex layers,
and the gather-attention (FP4 selected rows + FP8 window) of every layer,
over the static 40-layer schedule (4 Full, 4 Reindex, 30 Reuse, 2 SWA-only)
at batch 1, context 131,072 and Top-K 2,048 (the workload the headline
metric is quoted on).  The step runs through ``csa2_decode_layers``, captured
once in a CUDA graph and replayed.

Timing: W untimed warm-up steps, then K timed steps.  Before every step a
256 MB buffer is written to flush L2 (outside the timed events); each step is
bracketed by CUDA events on the stream it runs on.  Phase events recorded by
the library inside the graph give each kernel's duration.

Output: one JSON line (rank 0).  ``value`` = query-tokens/s (batch / step
time); ``hbm`` gives the algorithmic bytes per step and the achieved GB/s
against the measured copy bandwidth; ``roofline`` covers the dominant kernel;
``e2e`` repeats the metric through the Python binding of the C interface with
host buffers, copying the step's inputs in and outputs out every step;
``cpu_baseline`` times the CPU oracle on a bounded sample of the workload.

``--impl reference`` times the CPU oracle instead (there is no runnable
reference implementation of this method): each step is one layer of each mode
at the full context, composed into the 40-layer schedule.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "CSA2 decode query-tokens/s and achieved HBM GB/s (% of peak) at L=128K, FP4 KV"
UNIT = "query-tokens/s"
FALLBACK_HBM_GBS = 6400.0

# bytes per unit (layouts of include/csa2.h)
KV_ROW = 288        # FP4 main-KV row: 256 B codes + 32 B E4M3 scales
IDX_ROW = 36        # FP4 indexer key: 32 B codes + 4 B scales
SWA_ROW = 516       # FP8 window row: 512 B codes + 4 B fp32 scale
Q_BYTES = 16 * 512 * 4
OUT_BYTES = 16 * 512 * 4
LSE_BYTES = 16 * 4


def parse():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="csa2", choices=["csa2", "reference"])
    ap.add_argument("--config", type=int, default=2, help="workload index (default: the L=131072 40-layer step)")
    ap.add_argument("--e2e-steps", type=int, default=50)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0, help="CPU work budget of the oracle baseline")
    return ap.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# ---------------------------------------------------------------------------
# algorithmic bytes
# ---------------------------------------------------------------------------

def step_bytes(w):
    """Algorithmic bytes of one decode step, by part.

    scan:   36 B per (position, key pass).  A Full layer and the pool-free
            Reindex layer over the same keys share one pass in this step
            (their queries are both known when the step starts), so a
            position of such a pair is counted once; pool-restricted
            Reindex layers read 36 B (+4 B pool entry) per pool position.
    gather: 288 B per selected row per non-SWA-only layer.
    swa:    516 B per window row per layer.
    io:     q and out (32 KiB each), lse, indexer q and weights, indices
            written (4 B per Top-K / pool entry) and read by attention, and
            the appended rows (fp32 read, packed write).
    """
    from csa2_sparse_attention_03_b300 import synth
    B = w.batch
    Ls = [int(x) for x in w.seq_lens]
    parts = dict(scan=0, gather=0, swa=0, io=0)
    layers = w.layers
    paired = set()
    for l, ly in enumerate(layers):
        if ly.mode == synth.FULL:
            partner = [r for r in range(len(layers)) if layers[r].mode == synth.REINDEX
                       and layers[r].kv_src == l and not layers[r].use_pool]
            n_pass = 1 + max(0, len(partner) - 1)
            paired.update(partner[:1])
            parts["scan"] += n_pass * IDX_ROW * sum(Ls)
            parts["io"] += B * (4 * 64 * 4 + 16)       # q_idx + w
            parts["io"] += B * w.topk * 4               # indices written
            if w.pool_len:
                parts["io"] += B * w.pool_len * 4
        elif ly.mode == synth.REINDEX:
            if ly.use_pool:
                parts["scan"] += B * w.pool_len * (IDX_ROW + 4)
            parts["io"] += B * (4 * 64 * 4 + 16) + B * w.topk * 4
        if ly.mode != synth.SWA_ONLY:
            sel = sum(min(w.topk, L) for L in Ls)
            parts["gather"] += sel * KV_ROW
            parts["io"] += B * w.topk * 4               # indices read
        parts["swa"] += sum(min(w.window, L) for L in Ls) * SWA_ROW
        parts["io"] += B * (Q_BYTES + OUT_BYTES + LSE_BYTES)
        # appends: the new token's fp32 rows in, packed rows out
        if ly.mode == synth.FULL and w.append:
            parts["io"] += B * (512 * 4 + KV_ROW + 64 * 4 + IDX_ROW)
        if w.append:
            parts["io"] += B * (512 * 4 + SWA_ROW)
    parts["total"] = sum(parts.values())
    return parts


def attention_bytes(w):
    """Algorithmic bytes of the attention kernel (one launch covers every layer)."""
    from csa2_sparse_attention_03_b300 import synth
    Ls = [int(x) for x in w.seq_lens]
    B = w.batch
    tot = 0
    for ly in w.layers:
        if ly.mode != synth.SWA_ONLY:
            tot += sum(min(w.topk, L) for L in Ls) * KV_ROW + B * w.topk * 4
        tot += sum(min(w.window, L) for L in Ls) * SWA_ROW
        tot += B * (Q_BYTES + OUT_BYTES + LSE_BYTES)
    return tot


def scan_bytes(w):
    p = step_bytes(w)
    from csa2_sparse_attention_03_b300 import synth
    n_idx = sum(1 for ly in w.layers if ly.mode in (synth.FULL, synth.REINDEX))
    return p["scan"] + n_idx * w.batch * (4 * 64 * 4 + 16)


# ---------------------------------------------------------------------------
# clocks
# ---------------------------------------------------------------------------

class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu = gpu_id
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.Q,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (self.out or "").splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), max=float(f[2]), power=float(f[3]),
                                 hw=f[5], hwt=f[6], swt=f[7], pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        loaded = [r["sm"] for r in rows if r["power"] > 200.0] or [r["sm"] for r in rows]
        return {"sm_mhz": statistics.median(loaded), "sm_max_mhz": max(r["max"] for r in rows),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(r["power"] for r in rows)}


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and --impl reference)
# ---------------------------------------------------------------------------

class OracleSample:
    """One layer of each mode at the workload's full context, on the CPU oracle.

    Set-up (not timed) draws the inputs from the seeded streams and quantises
    them with the oracle; only what the sampled layers read is quantised (the
    indexer keys of the whole context, the main-KV rows the selections and
    windows touch).  ``run()`` times the oracle's per-layer decode work:
    scoring + Top-K (Full, Reindex), gather-dequantise-attend (every mode).
    """

    def __init__(self, w):
        import numpy as np
        import oracle
        from csa2_sparse_attention_03_b300 import synth
        self.np, self.orc, self.synth, self.w = np, oracle, synth, w
        oracle.build()
        b = 0
        L = int(w.seq_lens[b])
        self.L = L
        f = next(i for i, ly in enumerate(w.layers) if ly.mode == synth.FULL)
        r = next((i for i, ly in enumerate(w.layers) if ly.mode == synth.REINDEX), None)
        u = next((i for i, ly in enumerate(w.layers) if ly.mode == synth.REUSE), None)
        s = next((i for i, ly in enumerate(w.layers) if ly.mode == synth.SWA_ONLY), None)
        self.sample_layers = {"F": f, "R": r, "U": u, "S": s}
        self.counts = {"F": 0, "R": 0, "U": 0, "S": 0}
        for ly in w.layers:
            self.counts[synth.MODE_NAMES[ly.mode]] += 1
        self.k_codes, self.k_scales = oracle.quant_fp4(synth.idx_key_values(w, f, b, 0, L))
        self.q_idx = {m: synth.index_query(w, l)[b] for m, l in self.sample_layers.items()
                      if l is not None and m in "FR"}
        self.wts = {m: synth.index_weights(w, l)[b] for m, l in self.sample_layers.items()
                    if l is not None and m in "FR"}
        self.q = {m: synth.query(w, l)[b] for m, l in self.sample_layers.items() if l is not None}
        self.swa = {}
        for m, l in self.sample_layers.items():
            if l is None:
                continue
            n = min(w.window, L)
            self.swa[m] = oracle.quant_fp8(synth.swa_values(w, l, b)[w.window - n:])
        # main-KV rows every sampled layer may touch: run the selections once untimed
        self.cand = np.arange(L, dtype=np.int32)
        sel = set()
        for m in "FR":
            if m in self.q_idx:
                sc = oracle.index_scores(self.q_idx[m], self.wts[m], self.k_codes, self.k_scales)
                sel.update(int(x) for x in oracle.topk(sc, self.cand, w.topk) if x >= 0)
        rows = np.array(sorted(sel), dtype=np.int64)
        self.kv_codes = np.zeros((L, 256), np.uint8)
        self.kv_scales = np.zeros((L, 32), np.uint8)
        lo = 0
        while lo < rows.size:  # quantise the touched rows chunk by chunk of the value stream
            c0 = int(rows[lo]) // synth.CHUNK_ROWS * synth.CHUNK_ROWS
            hi = int(np.searchsorted(rows, c0 + synth.CHUNK_ROWS))
            vals = synth.kv_values(w, f, b, c0, min(synth.CHUNK_ROWS, L - c0))
            kc, ks = oracle.quant_fp4(vals[rows[lo:hi] - c0])
            self.kv_codes[rows[lo:hi]] = kc
            self.kv_scales[rows[lo:hi]] = ks
            lo = hi

    def layer(self, m, idx_in=None):
        orc, w = self.orc, self.w
        idx = idx_in
        if m in "FR":
            sc = orc.index_scores(self.q_idx[m], self.wts[m], self.k_codes, self.k_scales)
            idx = orc.topk(sc, self.cand, w.topk)
        if m == "S":
            orc.sparse_attention(self.q[m], None, None, self.np.zeros((0,), self.np.int32), *self.swa[m])
        else:
            orc.sparse_attention(self.q[m], self.kv_codes, self.kv_scales, idx, *self.swa[m])
        return idx

    def run(self):
        """Times one layer per mode; returns (seconds of a composed 40-layer step, per-mode seconds)."""
        t = {}
        idx = None
        for m in "FRUS":
            if self.sample_layers[m] is None:
                continue
            t0 = time.perf_counter()
            out = self.layer(m, idx)
            t[m] = time.perf_counter() - t0
            if m in "FR":
                idx = out
        step = sum(self.counts[m] * t.get(m, 0.0) for m in "FRUS")
        return step, t, sum(t.values())


def cpu_baseline(w, budget_s):
    samp = OracleSample(w)
    steps, work = [], 0.0
    while work < budget_s or not steps:
        s, _, spent = samp.run()
        steps.append(s)
        work += spent
    step_s = statistics.median(steps)
    return {"value": w.batch / step_s, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"one layer of each mode (F, R, U, S) at B={w.batch}, L={samp.L}, K={w.topk}, "
                       f"single-threaded C oracle, repeated {len(steps)}x ({work:.1f} s of CPU work); "
                       f"step time composed as {samp.counts['F']}F+{samp.counts['R']}R+"
                       f"{samp.counts['U']}U+{samp.counts['S']}S layer times (median)"),
            "seconds_per_step": step_s}


# ---------------------------------------------------------------------------
# ranks: one replica of the workload per GPU
# ---------------------------------------------------------------------------

def replica_seed(seed, rank):
    """Workload seed of a rank's replica (independent draws per rank)."""
    return seed + 100000 * rank


def max_over_ranks(pg, values, device="cpu"):
    """Element-wise max of this rank's floats over the process group (the
    slowest rank's times); the values themselves without a group."""
    if pg is None:
        return [float(v) for v in values]
    import torch
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(v) for v in t.tolist()]


def whole_job_value(world, batch, ms_per_step):
    """Query tokens per second of all ranks together: every rank decodes
    `batch` sequences per step, a step lasting the slowest rank's time."""
    return world * batch / (ms_per_step * 1e-3)


# ---------------------------------------------------------------------------
# reference arm: the CPU oracle, timed
# ---------------------------------------------------------------------------

def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from csa2_sparse_attention_03_b300 import synth
    w = synth.workload(args.config)
    samp = OracleSample(w)
    # warm-up (at most 2 samples, untimed) also estimates one sample's cost; the
    # timed steps are capped at about 90 s of oracle work so the arm ends in minutes
    est = None
    for _ in range(max(1, min(args.warmup, 2))):
        t = time.perf_counter()
        samp.run()
        est = time.perf_counter() - t
    n_timed = args.steps if args.steps * est <= 90.0 else max(3, int(90.0 / est))
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(n_timed):
        s, _, _ = samp.run()
        total += s
    wall = time.perf_counter() - t0
    ms = 1e3 * total / n_timed
    value = w.batch / (total / n_timed)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "timed_steps": n_timed, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.max_len, "layers": len(w.layers),
                   "topk": w.topk, "window": w.window},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": (f"each step: one layer of each mode (F, R, U, S) at the full context on the "
                                    f"single-threaded C oracle, composed as {samp.counts['F']}F+"
                                    f"{samp.counts['R']}R+{samp.counts['U']}U+{samp.counts['S']}S; "
                                    f"{n_timed} of the {args.steps} requested steps timed "
                                    f"(capped near 90 s of oracle work), {wall:.1f} s wall")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def run_csa2(args):
    import numpy as np
    import torch

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1

    # the CPU oracle leg runs before any GPU work (rank 0, one GPU only)
    from csa2_sparse_attention_03_b300 import synth
    w = synth.workload(args.config)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w, args.cpu_seconds)

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
        pg = dist

    import csa2_sparse_attention_03_b300 as csa2
    from csa2_sparse_attention_03_b300.schedule import DecodeStep
    csa2.load()

    # each rank runs an independent replica of the workload (sequences are
    # independent units; nothing is exchanged on the data path)
    w.seed = replica_seed(w.seed, rank)
    step = DecodeStep(w, device=dev, fill="device")
    stream = torch.cuda.Stream(device=dev)
    props = torch.cuda.get_device_properties(dev)
    # L2 flush: write one buffer of twice the L2 size, then read another, so
    # the step starts with L2 holding clean lines of neither its inputs nor
    # the flush's own dirty data
    flush = torch.empty(2 * max(props.L2_cache_size, 64 << 20), dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(flush.numel() // 8, dtype=torch.int64, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)

    # phase events inside the graph (recorded as external event nodes)
    n_ph = 6
    ph = [torch.cuda.Event(enable_timing=True) for _ in range(n_ph)]
    t_start = torch.cuda.Event(enable_timing=True)
    t_end = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        for e in ph:  # torch only times events it has seen recorded once
            e.record(stream)
    csa2.csa2_set_phase_events(ph)
    with torch.cuda.stream(stream):
        step.run(stream=stream)
        stream.synchronize()
        st, flags = csa2.csa2_check_device(stream)
        if st != 0:
            raise RuntimeError(f"device flags after the first step: status {st}, bits {flags}")
        # the phase breakdown comes from a graph with event nodes between the
        # kernels; the timed value from a second graph without them
        g_phases = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g_phases, stream=stream):
            step.run(stream=stream)
        csa2.csa2_set_phase_events([])
        n0 = csa2.csa2_launch_count()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            step.run(stream=stream)
        launches_per_step = csa2.csa2_launch_count() - n0
    torch.cuda.synchronize()

    def one_step(timed, phased=False):
        with torch.cuda.stream(stream):
            flush.fill_(1)
            torch.sum(flush_rd, dim=0, out=flush_sink)
            t_start.record(stream)
            (g_phases if phased else graph).replay()
            t_end.record(stream)
        t_end.synchronize()
        if not timed:
            return None
        tot = t_start.elapsed_time(t_end)
        if not phased:
            return tot, None
        marks = [t_start] + ph
        phases = [marks[i].elapsed_time(marks[i + 1]) for i in range(n_ph)]
        return tot, phases

    for _ in range(max(args.warmup, 3)):
        one_step(False)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    times, phase_sum = [], [0.0] * n_ph
    uuid = str(getattr(props, "uuid", "") or "")
    gpu_id = ("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(local))
    with ClockSampler(gpu_id) as clk:
        for _ in range(args.steps):
            tot, _ = one_step(True)
            times.append(tot)
    torch.cuda.synchronize()
    # phase breakdown (separate replays of the graph with event nodes)
    n_phased = max(1, min(args.steps, 100))
    for _ in range(3):
        one_step(False, phased=True)
    phased_tot = 0.0
    for _ in range(n_phased):
        tot, phases = one_step(True, phased=True)
        phased_tot += tot
        for i in range(n_ph):
            phase_sum[i] += phases[i]

    # the layer-sequential order (per-layer entry points, as a model calls them),
    # timed the same way from its own graph; one GPU only (a rank failing here
    # must not leave the others in a collective)
    st0, fl0 = csa2.csa2_check_device(stream)
    if st0 != 0:
        raise RuntimeError(f"device flags after the timed steps: status {st0}, bits {fl0}")

    # the quantise step's cache build: one Full layer's main KV and indexer keys
    # over the whole context (fp32 rows in, packed rows out), L2 flushed first
    build = None
    if pg is None:
        try:
            Lb = int(w.max_len)
            build = {}
            for kind, fmt, ch, row in (("main_kv", csa2.FMT_FP4_KV, 512, KV_ROW), ("indexer_keys", csa2.FMT_FP4_IDX, 64,
                                                                                   IDX_ROW)):
                src = torch.empty((1, Lb, ch), dtype=torch.float32, device=dev).normal_()
                cache = csa2.Cache.contiguous(fmt, 1, (Lb + 63) // 64 * 64, dev)
                b_ms = []
                for it in range(6):
                    with torch.cuda.stream(stream):
                        flush.fill_(1)
                        torch.sum(flush_rd, dim=0, out=flush_sink)
                        t_start.record(stream)
                        csa2.csa2_quantize_kv(src, cache, stream=stream)
                        t_end.record(stream)
                    t_end.synchronize()
                    if it >= 3:
                        b_ms.append(t_start.elapsed_time(t_end))
                ms_b = sum(b_ms) / len(b_ms)
                nbytes = Lb * (ch * 4 + row)
                build[kind] = {"rows": Lb, "ms": ms_b, "algorithmic_bytes": nbytes,
                               "achieved_gbs": nbytes / (ms_b * 1e-3) / 1e9,
                               "frac": nbytes / (ms_b * 1e-3) / 1e9 / peaks()[0]}
                del src, cache
            bst, bfl = csa2.csa2_check_device(stream)
            if bst != 0:
                build = {"error": f"device flags after the cache builds: status {bst}, bits {bfl}"}
        except Exception as exc:  # reported, never fatal to the main measurement
            build = {"error": repr(exc)[:300]}
    seq = None
    if pg is None:
        try:
            with torch.cuda.stream(stream):
                step.run_sequential(stream=stream)
                stream.synchronize()
                n0s = csa2.csa2_launch_count()
                g_seq = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g_seq, stream=stream):
                    step.run_sequential(stream=stream)
                seq_launches = csa2.csa2_launch_count() - n0s
            torch.cuda.synchronize()

            def seq_step():
                with torch.cuda.stream(stream):
                    flush.fill_(1)
                    torch.sum(flush_rd, dim=0, out=flush_sink)
                    t_start.record(stream)
                    g_seq.replay()
                    t_end.record(stream)
                t_end.synchronize()
                return t_start.elapsed_time(t_end)

            for _ in range(3):
                seq_step()
            st_ms = [seq_step() for _ in range(max(1, min(args.steps, 100)))]
            s_ms = sum(st_ms) / len(st_ms)
            seq = {"ms_per_step": s_ms, "value": whole_job_value(world, w.batch, s_ms), "unit": UNIT,
                   "launches_per_step": int(seq_launches),
                   "how": "each layer in schedule order: its appends, its indexing, its attention, through "
                          "csa2_quantize_kv / csa2_index_topk / csa2_sparse_attn, one CUDA graph per step"}
            sst, sfl = csa2.csa2_check_device(stream)
            if sst != 0:
                seq = {"error": f"device flags after the layer-sequential steps: status {sst}, bits {sfl}"}
        except Exception as exc:  # reported, never fatal to the main measurement
            seq = {"error": repr(exc)[:300]}
    if pg:
        pg.barrier()
    ms_total = max_over_ranks(pg, [sum(times)], dev)[0]
    ms = ms_total / args.steps
    value = whole_job_value(world, w.batch, ms)

    # dominant kernel: the phase with the largest share
    names = ["append (quantize)", "scan", "select", "level-1 scan+select", "attention", "merge"]
    kern = ["quantize_kernel", "scan_kernel", "select_kernel", "scan_kernel+select_kernel (pool)",
            "attn_tc_kernel + attn_merge_kernel", "attn_tc_kernel + attn_merge_kernel"]
    ph_ms = [p / n_phased for p in phase_sum]
    # attention is one unit: the gather/softmax kernel and the merge that writes the outputs
    unit_ms = ph_ms[:4] + [ph_ms[4] + ph_ms[5]]
    top = int(np.argmax(unit_ms))
    peak, peak_kind = peaks()
    sb = step_bytes(w)
    if top == 4:
        kbytes = attention_bytes(w)
    elif top == 1:
        kbytes = scan_bytes(w)
    else:
        kbytes = None
    roof = {"kernel": kern[top], "bound": "hbm", "unit": "GB/s", "peak": peak,
            "peak_source": f"{peak_kind} copy bandwidth", "traffic": None,
            "ms_per_launch": unit_ms[top],
            "timing": "phase events inside a separate graph replay of the same step"}
    if kbytes is not None:
        ach = kbytes / (unit_ms[top] * 1e-3) / 1e9
        roof.update(achieved=ach, frac=ach / peak, algorithmic_bytes=kbytes)
    else:
        roof.update(achieved=None, frac=None, algorithmic_bytes=None)

    # end to end: host inputs -> device -> step -> host outputs, as one graph replay
    e2e = None
    if args.e2e_steps > 0:
        ins = step.step_inputs()
        outs = step.step_outputs()
        h_in = [t.detach().cpu().pin_memory() for t in ins]
        h_out = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
        bi = sum(t.numel() * t.element_size() for t in h_in)
        bo = sum(t.numel() * t.element_size() for t in h_out)
        csa2.csa2_set_phase_events([])
        e_s = torch.cuda.Event(enable_timing=True)
        e_e = torch.cuda.Event(enable_timing=True)

        # the serving step as one replay: host inputs in, the step, host outputs out
        g_e2e = step.capture(stream, h_in[0], h_out[0])

        def e2e_step(timed, direct=False):
            with torch.cuda.stream(stream):
                flush.fill_(1)
                torch.sum(flush_rd, dim=0, out=flush_sink)
                e_s.record(stream)
                if direct:
                    for d, h in zip(ins, h_in):
                        d.copy_(h, non_blocking=True)
                    step.run(stream=stream)
                    for h, d in zip(h_out, outs):
                        h.copy_(d, non_blocking=True)
                else:
                    g_e2e.replay()
                e_e.record(stream)
            e_e.synchronize()
            return e_s.elapsed_time(e_e) if timed else None

        for _ in range(3):
            e2e_step(False)
            e2e_step(False, direct=True)
        et = [e2e_step(True) for _ in range(args.e2e_steps)]
        dt = [e2e_step(True, direct=True) for _ in range(args.e2e_steps)]
        e_ms, d_ms = max_over_ranks(pg, [sum(et) / len(et), sum(dt) / len(dt)], dev)
        e2e = {"value": whole_job_value(world, w.batch, e_ms), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": e_ms,
               "how": "DecodeStep.capture: one CUDA graph per step that copies the pinned host input arena "
                      "in, runs csa2_decode_layers and copies the output arena (out, lse, indices) back; "
                      "all inside the CUDA-event region",
               "direct_call_ms_per_step": d_ms}

    st, flags = csa2.csa2_check_device(stream)
    if st != 0:
        raise RuntimeError(f"device flags after the timed steps: status {st}, bits {flags}")

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (FP4/FP8 storage, fp16 MMA operands)", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "seq_len": w.max_len, "layers": len(w.layers),
                       "schedule": "".join(synth.MODE_NAMES[ly.mode] for ly in w.layers), "topk": w.topk,
                       "window": w.window, "pool": w.pool_len,
                       "execution": "csa2_decode_layers captured in one CUDA graph, replayed",
                       "l2": f"flushed before every timed step ({flush.numel() >> 20} MB write, then a {flush.numel() >> 20} MB read of another buffer)",
                       "parallelism": f"replicas x{world}"},
            "hbm": {"algorithmic_bytes_per_step": sb["total"], "parts": {k: v for k, v in sb.items() if k != "total"},
                    "achieved_gbs": sb["total"] / (ms * 1e-3) / 1e9,
                    "frac": sb["total"] / (ms * 1e-3) / 1e9 / peak, "peak_gbs": peak,
                    "peak_source": f"{peak_kind} copy bandwidth"},
            "phases_ms": {names[i]: ph_ms[i] for i in range(n_ph)},
            "phased_ms_per_step": phased_tot / n_phased,
            "layer_sequential": seq,
            "cache_build": build,
            "roofline": roof,
            "gpu_launches": int(launches_per_step) * args.steps,
            "launches_per_step": int(launches_per_step),
            "clocks": clk.summary(),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.impl == "reference":
        return run_reference(args)
    return run_csa2(args)


if __name__ == "__main__":
    sys.exit(main())
