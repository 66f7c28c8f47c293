#!/usr/bin/env python3
"""Benchmark of one CSA2 decode step on B300.

A step is one pass of the whole decode path over one batch: the quantise-and-
append of the new token into every Full layer's FP4 caches and every layer's
FP8 window ring, indexer scoring and Top-K of the Full and Reindex layers,
and the gather-attention (FP4 selected rows + FP8 window) of every layer,
over the static 40-layer schedule (4 Full, 4 Reindex, 30 Reuse, 2 SWA-only)
at batch 1, context 131,072 and Top-K 2,048 (the workload the headline
metric is quoted on; ``--config`` picks another).

Headline: the *layer-sequential* step -- one ``csa2_decode_layer`` call per
layer in schedule order, the order a model runs it in (layer l+1's queries
do not exist before layer l is done) -- captured once in a CUDA graph and
replayed.  The *phased* step (``csa2_decode_layers``: every layer's indexing,
then every attention, valid only when all queries are known up front) is
reported beside it under ``phased``.

Timing: W untimed warm-up steps, then K timed steps.  Before every step a
buffer of twice the L2 size is written and another read (outside the timed
events); each step is bracketed by CUDA events on the stream it runs on.
The attention and indexing kernels are also timed alone (every layer's
attention, or every indexing layer, in one graph) for the roofline.

Output: one JSON line (rank 0).  ``value`` = query-tokens/s (batch / step
time); ``hbm`` gives the algorithmic bytes per step and the achieved GB/s
against the measured copy bandwidth; ``roofline`` covers the dominant
kernel; ``e2e`` repeats the metric through the Python binding of the C
interface with host buffers, copying the step's inputs in and outputs out
every step; ``cpu_baseline`` times the CPU oracle on one whole decode step of
the same workload (one thread and all host cores).

``--impl reference`` times the CPU oracle instead (there is no runnable
reference implementation of this method): each step is one whole decode step
of the workload on the host cores.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

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
    ap.add_argument("--only-sequential", action="store_true",
                    help="time the layer-sequential step alone and print its time (no other measurements; "
                         "the command the committed launch-list and kernel profiles were taken with)")
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

KERNEL_SOURCES = {  # the device code a kernel is compiled from (a change voids its ncu counters)
    "attn_kernel": ("attention.cu", "tc.cuh", "common.cuh"),
    "index_fused_kernel": ("index_fused.cu", "scan.cuh", "tc.cuh", "common.cuh"),
}


def kernel_source_sha16(kernel):
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "csa2_sparse_attention_03_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(kernel, workload, pdir=None):
    """DRAM bytes (read + write) per launch of ``kernel`` from the committed ncu
    summaries: a line ``traffic-record: kernel=K workload=W launches=N
    dram_bytes_per_launch=B source_sha16=S`` (W with '_' for ' ').  None when
    no record matches the workload or the kernel's sources changed since."""
    pdir = pdir or os.path.join(ROOT, "profiles")
    if not os.path.isdir(pdir):
        return None, None
    want = kernel_source_sha16(kernel)
    for fn in sorted(os.listdir(pdir)):
        if not fn.endswith((".md", ".txt")):
            continue
        with open(os.path.join(pdir, fn)) as f:
            for line in f:
                if not line.strip().startswith("traffic-record:"):
                    continue
                kv = dict(t.split("=", 1) for t in line.split(":", 1)[1].split() if "=" in t)
                if kv.get("kernel") == kernel and kv.get("workload", "").replace("_", " ") == workload:
                    if kv.get("source_sha16") != want:
                        return None, f"profiles/{fn}: kernel sources changed since the capture"
                    return float(kv["dram_bytes_per_launch"]), f"profiles/{fn}"
    return None, None


def _layer_parts(w, ly):
    """Bytes one layer moves in the layer-sequential order, by part: its key
    pass (36 B per position scored, or 36 B + 4 B per pool entry), its
    gathered rows (288 B per selected row), its window rows (516 B), and io
    (q, out, lse, the indexer query and weights, indices written and read,
    the appended rows: fp32 in, packed out)."""
    from csa2_sparse_attention_03_b300 import synth
    B = w.batch
    Ls = [int(x) for x in w.seq_lens]
    p = dict(scan=0, gather=0, swa=0, io=0)
    if ly.mode in (synth.FULL, synth.REINDEX):
        if ly.mode == synth.REINDEX and ly.use_pool:
            p["scan"] += B * w.pool_len * (IDX_ROW + 4)
        else:
            p["scan"] += IDX_ROW * sum(Ls)
        p["io"] += B * (4 * 64 * 4 + 16) + B * w.topk * 4
        if ly.mode == synth.FULL and w.pool_len:
            p["io"] += B * w.pool_len * 4
    if ly.mode != synth.SWA_ONLY:
        p["gather"] += sum(min(w.topk, L) for L in Ls) * KV_ROW
        p["io"] += B * w.topk * 4
    p["swa"] += sum(min(w.window, L) for L in Ls) * SWA_ROW
    p["io"] += B * (Q_BYTES + OUT_BYTES + LSE_BYTES)
    if ly.mode == synth.FULL and w.append:
        p["io"] += B * (512 * 4 + KV_ROW + 64 * 4 + IDX_ROW)
    if w.append:
        p["io"] += B * (512 * 4 + SWA_ROW)
    return p


def step_bytes(w):
    """Algorithmic bytes of one decode step in the layer-sequential order, by
    part: every Full and every Reindex layer reads its keys (each key pass is
    counted), every non-SWA-only layer gathers its selected rows, every layer
    reads its window, q, out, indices and appended rows."""
    parts = dict(scan=0, gather=0, swa=0, io=0)
    for ly in w.layers:
        for k, v in _layer_parts(w, ly).items():
            parts[k] += v
    parts["total"] = sum(parts.values())
    return parts


def fused_step_bytes(w):
    """The same step as the phased launch sequence reads it: a Full layer and
    its pool-free Reindex partner score in one key pass, and two layers that
    share a selection (the attention's unit) gather its rows once."""
    from csa2_sparse_attention_03_b300 import synth
    parts = step_bytes(w)
    layers = w.layers
    B = w.batch
    Ls = [int(x) for x in w.seq_lens]
    for l, ly in enumerate(layers):
        if ly.mode == synth.REINDEX and not ly.use_pool:
            parts["scan"] -= IDX_ROW * sum(Ls)  # shares its Full layer's pass
    groups = {}
    for l, ly in enumerate(layers):
        if ly.mode == synth.SWA_ONLY:
            continue
        src = l if ly.mode in (synth.FULL, synth.REINDEX) else ly.idx_src
        groups[src] = groups.get(src, 0) + 1
    sel = sum(min(w.topk, L) for L in Ls) * KV_ROW
    for n in groups.values():
        parts["gather"] -= (n - (n + 1) // 2) * sel  # units of two layers
    parts["total"] = parts["scan"] + parts["gather"] + parts["swa"] + parts["io"]
    return parts


def attention_launch_bytes(w, ly):
    """One layer's attention launch: selected rows, window rows, q/out/lse,
    indices read, the appended window row."""
    p = _layer_parts(w, ly)
    from csa2_sparse_attention_03_b300 import synth
    B = w.batch
    io = B * (Q_BYTES + OUT_BYTES + LSE_BYTES) + (B * w.topk * 4 if ly.mode != synth.SWA_ONLY else 0)
    return p["gather"] + p["swa"] + io


def index_launch_bytes(w, ly):
    """One indexing layer's launch: its key pass, indexer q and weights,
    indices (and pool) written, a Full layer's appended row and key."""
    from csa2_sparse_attention_03_b300 import synth
    p = _layer_parts(w, ly)
    B = w.batch
    io = B * (4 * 64 * 4 + 16) + B * w.topk * 4
    if ly.mode == synth.FULL:
        io += (B * w.pool_len * 4 if w.pool_len else 0) + (B * (512 * 4 + KV_ROW + 64 * 4 + IDX_ROW) if w.append else 0)
    return p["scan"] + io


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

class OracleStep:
    """One whole decode step of a workload on the CPU oracle.

    Set-up (not timed) draws the inputs from the seeded host streams and
    quantises the caches with the oracle, using every host core (the result
    does not depend on the thread count).  ``run(threads)`` times the oracle's
    decode step -- every layer's scoring, Top-K and gather-attention -- with
    the given number of threads and returns (seconds, outputs).  Sequences
    beyond ``max_seqs`` are left out (a bounded sample of the batch)."""

    def __init__(self, w, max_seqs=None):
        import copy

        import oracle
        from csa2_sparse_attention_03_b300 import synth
        self.orc, self.synth = oracle, synth
        oracle.build()
        w = copy.copy(w)
        if max_seqs is not None and w.batch > max_seqs:
            w.seq_lens = list(w.seq_lens)[:max_seqs]
            w.batch = max_seqs
        self.w = w
        self.cores = os.cpu_count() or 1
        oracle.set_threads(self.cores)
        caches, per = {}, {}
        for f, ly in enumerate(w.layers):
            if ly.mode != synth.FULL:
                continue
            caches[f] = {}
            for b, L in enumerate(w.seq_lens):
                kc = np.empty((L, 256), np.uint8)
                ks = np.empty((L, 32), np.uint8)
                for r0 in range(0, L, synth.CHUNK_ROWS):
                    n = min(synth.CHUNK_ROWS, L - r0)
                    kc[r0:r0 + n], ks[r0:r0 + n] = oracle.quant_fp4(synth.kv_values(w, f, b, r0, n))
                ic, isc = oracle.quant_fp4(synth.idx_key_values(w, f, b, 0, L))
                caches[f][b] = dict(kv_codes=kc, kv_scales=ks, k_codes=ic, k_scales=isc)
        for l, ly in enumerate(w.layers):
            codes, scales = [], []
            for b, L in enumerate(w.seq_lens):
                n = min(w.window, L)
                c, sc = oracle.quant_fp8(synth.swa_values(w, l, b)[w.window - n:])
                codes.append(c)
                scales.append(sc)
            pl = dict(q=synth.query(w, l), swa_codes=codes, swa_scales=scales, q_idx=None, w=None)
            if ly.mode in (synth.FULL, synth.REINDEX):
                pl["q_idx"] = synth.index_query(w, l)
                pl["w"] = synth.index_weights(w, l)
            per[l] = pl
        self.caches, self.per = caches, per

    def run(self, threads):
        self.orc.set_threads(threads)
        t0 = time.perf_counter()
        res = self.orc.decode_step(self.w.layers, list(self.w.seq_lens), self.w.topk, self.w.pool_len,
                                   self.caches, self.per)
        return time.perf_counter() - t0, res

    @staticmethod
    def same(a, b):
        """Byte-identical outputs of two runs (indices, outputs, lse)."""
        for l in a:
            for k in ("idx", "pool", "out", "lse"):
                x, y = a[l][k], b[l][k]
                if (x is None) != (y is None) or (x is not None and not np.array_equal(x, y)):
                    return False
        return True


def cpu_baseline(w, budget_s):
    """The oracle's whole decode step, single-threaded and on every host core
    (checked byte-identical), on a bounded sample of the batch."""
    max_seqs = 1 if w.batch > 1 else None
    t0 = time.perf_counter()
    st = OracleStep(w, max_seqs=max_seqs)
    setup_s = time.perf_counter() - t0
    t1, r1 = st.run(1)
    tn, rn = st.run(st.cores)
    ident = OracleStep.same(r1, rn)
    runs = [tn]
    while sum(runs) + t1 < budget_s and len(runs) < 5:
        runs.append(st.run(st.cores)[0])
    step_s = statistics.median(runs)
    b = st.w.batch
    return {"value": b / step_s, "unit": UNIT, "cores": st.cores, "kind": "oracle",
            "sample": (f"whole decode step of the workload ({len(st.w.layers)} layers, K={st.w.topk}) on "
                       f"{b} of its {w.batch} sequence(s), L={max(st.w.seq_lens)}: the C oracle on {st.cores} host "
                       f"threads, median of {len(runs)} steps; set-up (input draws, cache quantisation) "
                       f"{setup_s:.1f} s untimed"),
            "seconds_per_step": step_s,
            "single_thread": {"value": b / t1, "seconds_per_step": t1, "cores": 1},
            "threads_identical": ident}


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
    st = OracleStep(w, max_seqs=1 if w.batch > 1 else None)
    cores = st.cores
    est = None
    for _ in range(max(1, min(args.warmup, 2))):
        est = st.run(cores)[0]
    # timed steps capped at about 90 s of oracle work so the arm ends in minutes
    n_timed = args.steps if args.steps * est <= 90.0 else max(3, int(90.0 / est))
    t0 = time.perf_counter()
    total = 0.0
    for _ in range(n_timed):
        total += st.run(cores)[0]
    wall = time.perf_counter() - t0
    ms = 1e3 * total / n_timed
    b = st.w.batch
    value = b / (total / n_timed)
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "timed_steps": n_timed, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "seq_len": w.max_len, "layers": len(w.layers),
                   "topk": w.topk, "window": w.window},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": (f"each step: the whole decode step of the workload on {b} of its {w.batch} "
                                    f"sequence(s) by the C oracle on {cores} host threads; {n_timed} of the "
                                    f"{args.steps} requested steps timed (capped near 90 s of oracle work), "
                                    f"{wall:.1f} s wall")},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# the CUDA path
# ---------------------------------------------------------------------------

def _flush_buffers(torch, dev):
    props = torch.cuda.get_device_properties(dev)
    flush = torch.empty(2 * max(props.L2_cache_size, 64 << 20), dtype=torch.uint8, device=dev)
    flush_rd = torch.ones(flush.numel() // 8, dtype=torch.int64, device=dev)
    flush_sink = torch.empty((), dtype=torch.int64, device=dev)
    return flush, flush_rd, flush_sink


class GraphTimer:
    """Replays a CUDA graph after an L2 flush (a write of twice the L2 size,
    then a read of another buffer), CUDA events around the replay only."""

    def __init__(self, torch, dev, stream):
        self.torch, self.stream = torch, stream
        self.flush, self.flush_rd, self.sink = _flush_buffers(torch, dev)
        self.t0 = torch.cuda.Event(enable_timing=True)
        self.t1 = torch.cuda.Event(enable_timing=True)

    def capture(self, fn):
        torch = self.torch
        with torch.cuda.stream(self.stream):
            fn()  # once outside the capture (planning, attribute set-up)
            self.stream.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=self.stream):
                fn()
        torch.cuda.synchronize()
        return g

    def time(self, g, n, warm=3):
        torch = self.torch
        out = []
        for i in range(warm + n):
            with torch.cuda.stream(self.stream):
                self.flush.fill_(1)
                torch.sum(self.flush_rd, dim=0, out=self.sink)
                self.t0.record(self.stream)
                g.replay()
                self.t1.record(self.stream)
            self.t1.synchronize()
            if i >= warm:
                out.append(self.t0.elapsed_time(self.t1))
        return out


def multi_query_timing(csa2, torch, step, w, timer, stream, dev, n_small):
    """csa2_index_topk_multi at n_q = 8 and 32 causal query rows per sequence
    over the first Full layer's indexer keys (Top-K = the workload's).
    Useful tensor work: 2 x 4 heads x 64 channels per (row, candidate)."""
    if not step.caches:
        return None
    ik = step.caches[min(step.caches)][1]
    B, L, K = w.batch, int(w.max_len), int(w.topk)
    lens = [int(x) for x in w.seq_lens]
    gen = torch.Generator(device=dev)
    gen.manual_seed(w.seed + 7)
    res = {}
    for nq in (8, 32):
        q = torch.randn((B, nq, 4, 64), generator=gen, device=dev) * 0.125
        wt = torch.rand((B, nq, 4), generator=gen, device=dev)
        idx = torch.empty((B, nq, K), dtype=torch.int32, device=dev)
        ws = csa2.new_workspace(csa2.csa2_index_topk_multi_workspace(B, nq, L), dev)
        n0 = csa2.csa2_launch_count()
        g = timer.capture(lambda: csa2.csa2_index_topk_multi(ik, q, wt, step.seq_lens, L, K, out_idx=idx,
                                                             workspace=ws, stream=stream))
        launches = (csa2.csa2_launch_count() - n0) // 2
        t = statistics.mean(timer.time(g, n_small))
        cand = sum(max(0, min(Lb, Lb - nq + i + 1)) for Lb in lens for i in range(nq))
        flops = 2 * 4 * 64 * cand
        nbytes = sum(lens) * IDX_ROW + B * nq * (4 * 64 * 4 + 16 + K * 4)
        res[f"n_q={nq}"] = {"ms": t, "query_tokens_per_s": B * nq / (t * 1e-3), "launches": int(launches),
                            "useful_tflops": flops / (t * 1e-3) / 1e12, "keys_gbs": nbytes / (t * 1e-3) / 1e9}
        del g
    res["how"] = ("csa2_index_topk_multi (tcgen05 kind::f16 scoring, one MMA per 16-channel block, then the "
                  "cluster select), causal rows, CUDA events around a graph of the call, L2 flushed before each")
    return res


def run_csa2(args):
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
    if rank == 0 and world == 1 and not args.no_cpu_baseline and not args.only_sequential:
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
    timer = GraphTimer(torch, dev, stream)

    def check(what):
        st, flags = csa2.csa2_check_device(stream)
        if st != 0:
            raise RuntimeError(f"device flags after {what}: status {st}, bits {flags}")

    # the headline: the layer-sequential step, one graph
    n0 = csa2.csa2_launch_count()
    g_seq = timer.capture(lambda: step.run_sequential(stream=stream))
    seq_launches = (csa2.csa2_launch_count() - n0) // 2  # once eagerly, once captured
    check("the layer-sequential step")
    for _ in range(max(args.warmup, 3)):
        timer.time(g_seq, 0, warm=1)
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    uuid = str(getattr(torch.cuda.get_device_properties(dev), "uuid", "") or "")
    gpu_id = ("GPU-" + uuid) if uuid and not uuid.startswith("GPU-") else (uuid or str(local))
    with ClockSampler(gpu_id) as clk:
        times = timer.time(g_seq, args.steps, warm=0)
    torch.cuda.synchronize()
    check("the timed steps")
    if pg:
        pg.barrier()
    ms_total = max_over_ranks(pg, [sum(times)], dev)[0]
    ms = ms_total / args.steps
    value = whole_job_value(world, w.batch, ms)
    n_small = max(1, min(args.steps, 100))
    if args.only_sequential:
        if rank == 0:
            print(json.dumps({"metric": METRIC, "value": value, "unit": UNIT, "ms_per_step": ms, "steps": args.steps,
                              "warmup": args.warmup, "launches_per_step": int(seq_launches),
                              "note": "layer-sequential step only (profiling run)"}))
        return 0

    # the phased step (csa2_decode_layers), same timing
    n0 = csa2.csa2_launch_count()
    g_ph = timer.capture(lambda: step.run(stream=stream))
    ph_launches = (csa2.csa2_launch_count() - n0) // 2
    ph_ms = statistics.mean(timer.time(g_ph, n_small))
    check("the phased step")
    fsb = fused_step_bytes(w)
    phased = {"ms_per_step": ph_ms, "value": whole_job_value(world, w.batch, ph_ms), "unit": UNIT,
              "launches_per_step": int(ph_launches),
              "hbm": {"algorithmic_bytes_per_step": fsb["total"],
                      "parts": {k: v for k, v in fsb.items() if k != "total"},
                      "achieved_gbs": fsb["total"] / (ph_ms * 1e-3) / 1e9},
              "how": "csa2_decode_layers: every layer's indexing, then every layer's attention (valid only "
                     "when every query is an input of the step); bytes counted as that launch sequence reads "
                     "them (a Full layer and its Reindex partner in one key pass, two layers per gather)"}

    # the dominant kernels alone: every layer's attention; every indexing layer
    peak, peak_kind = peaks()
    attn_layers = list(range(len(w.layers)))
    idx_layers = [l for l, ly in enumerate(w.layers) if ly.mode in (synth.FULL, synth.REINDEX)]

    def attn_only():
        for l in attn_layers:
            step.attention_only(l, stream=stream)

    def index_only():
        for l in idx_layers:
            step.index_only(l, stream=stream)

    kernels = {}
    for name, fn, layers_, bytes_fn in (("attention (attn_kernel)", attn_only, attn_layers, attention_launch_bytes),
                                        ("indexing (index_fused_kernel)", index_only, idx_layers, index_launch_bytes)):
        if not layers_:
            continue
        n0 = csa2.csa2_launch_count()
        g = timer.capture(fn)
        nl = (csa2.csa2_launch_count() - n0) // 2
        t = statistics.mean(timer.time(g, n_small))
        by = sum(bytes_fn(w, w.layers[l]) for l in layers_)
        kernels[name] = {"launches": int(nl), "ms_all_launches": t, "ms_per_launch": t / max(1, nl),
                         "algorithmic_bytes_per_launch": by / max(1, nl),
                         "achieved_gbs": by / (t * 1e-3) / 1e9, "frac": by / (t * 1e-3) / 1e9 / peak}
        del g
    check("the kernel timings")

    # many queries per sequence (a speculative verification, a prefill chunk):
    # the tensor-core multi-query scoring and its Top-K over the first Full
    # layer's indexer keys, causal rows
    multi = multi_query_timing(csa2, torch, step, w, timer, stream, dev, n_small)
    check("the multi-query indexing")
    # dominant kernel: the larger share of the step (its launches x their time)
    top = max(kernels, key=lambda k: kernels[k]["ms_all_launches"]) if kernels else None
    roof = None
    if top:
        kd = kernels[top]
        kname = top.split("(")[-1].rstrip(")")
        traffic, traffic_src = recorded_traffic(kname, w.name)
        roof = {"kernel": top, "bound": "hbm", "unit": "GB/s", "peak": peak,
                "peak_source": f"{peak_kind} copy bandwidth", "achieved": kd["achieved_gbs"], "frac": kd["frac"],
                "traffic": traffic, "traffic_source": traffic_src,
                "algorithmic_bytes_per_launch": kd["algorithmic_bytes_per_launch"],
                "ms_per_launch": kd["ms_per_launch"],
                "timing": "CUDA events around a graph of this kernel's launches for every layer of the step, "
                          "L2 flushed before each replay"}

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
                g = timer.capture(lambda: csa2.csa2_quantize_kv(src, cache, stream=stream))
                ms_b = statistics.mean(timer.time(g, 5))
                nbytes = Lb * (ch * 4 + row)
                build[kind] = {"rows": Lb, "ms": ms_b, "algorithmic_bytes": nbytes,
                               "achieved_gbs": nbytes / (ms_b * 1e-3) / 1e9,
                               "frac": nbytes / (ms_b * 1e-3) / 1e9 / peak}
                del src, cache, g
            check("the cache builds")
        except Exception as exc:  # reported, never fatal to the main measurement
            build = {"error": repr(exc)[:300]}

    # end to end: host inputs -> device -> the layer-sequential step -> host outputs
    e2e = None
    if args.e2e_steps > 0:
        h_in = step.arena_in.detach().cpu().pin_memory()
        h_out = torch.empty(step.arena_out.shape, dtype=step.arena_out.dtype, pin_memory=True)
        bi = h_in.numel() * h_in.element_size()
        bo = h_out.numel() * h_out.element_size()

        def serve():
            step.arena_in.copy_(h_in, non_blocking=True)
            step.run_sequential(stream=stream)
            h_out.copy_(step.arena_out, non_blocking=True)

        # the serving step as DecodeStep.capture_sequential builds it: groups of
        # layers' inputs copied in on a side stream ahead of the layers that
        # need them, groups of outputs copied back as soon as they are done
        with torch.cuda.stream(stream):
            g_e2e = step.capture_sequential(stream, h_in, h_out)
        torch.cuda.synchronize()
        et = timer.time(g_e2e, args.e2e_steps)

        dt = []
        for i in range(3 + args.e2e_steps):
            with torch.cuda.stream(stream):
                timer.flush.fill_(1)
                torch.sum(timer.flush_rd, dim=0, out=timer.sink)
                timer.t0.record(stream)
                serve()
                timer.t1.record(stream)
            timer.t1.synchronize()
            if i >= 3:
                dt.append(timer.t0.elapsed_time(timer.t1))
        e_ms, d_ms = max_over_ranks(pg, [statistics.mean(et), statistics.mean(dt)], dev)
        e2e = {"value": whole_job_value(world, w.batch, e_ms), "unit": UNIT, "h2d_bytes_per_step": bi,
               "d2h_bytes_per_step": bo, "ms_per_step": e_ms,
               "how": "one CUDA graph per step (DecodeStep.capture_sequential): the pinned host input arena "
                      "(queries, indexer queries, weights, appended rows) copied in by groups of layers on a "
                      "second stream, each layer waiting only for its group; the layer-sequential step "
                      "(csa2_decode_layer per layer); the output arena (out, lse, indices) copied back by "
                      "groups of layers on a third stream as they finish; all inside the CUDA events",
               "direct_call_ms_per_step": d_ms,
               "direct_call_how": "the same step as direct calls, one whole-arena copy in, then every layer, "
                                  "then one whole-arena copy out, no graph"}
        check("the end-to-end steps")

    if rank == 0:
        sb = step_bytes(w)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f32 (FP4/FP8 storage, fp16 MMA operands)", "data": "synthetic",
            "config": {"workload": w.name, "batch": w.batch, "seq_len": w.max_len, "layers": len(w.layers),
                       "schedule": "".join(synth.MODE_NAMES[ly.mode] for ly in w.layers), "topk": w.topk,
                       "window": w.window, "pool": w.pool_len,
                       "execution": "layer-sequential: csa2_decode_layer for each layer in schedule order, "
                                    "captured in one CUDA graph, replayed",
                       "l2": f"flushed before every timed step ({timer.flush.numel() >> 20} MB write, then a "
                             f"{timer.flush.numel() >> 20} MB read of another buffer)",
                       "parallelism": f"replicas x{world}"},
            "hbm": {"algorithmic_bytes_per_step": sb["total"], "parts": {k: v for k, v in sb.items() if k != "total"},
                    "achieved_gbs": sb["total"] / (ms * 1e-3) / 1e9,
                    "frac": sb["total"] / (ms * 1e-3) / 1e9 / peak, "peak_gbs": peak,
                    "peak_source": f"{peak_kind} copy bandwidth"},
            "phased": phased,
            "kernels": kernels,
            "multi_query_index": multi,
            "cache_build": build,
            "roofline": roof,
            "gpu_launches": int(seq_launches) * args.steps,
            "launches_per_step": int(seq_launches),
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
