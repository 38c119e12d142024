#!/usr/bin/env python3
"""Benchmark of the QSA hot path on GB300; prints ONE JSON line.

Headline: prefill tokens/s on the ragged batch (B=4, padded S=16384, live
lengths ~ U[4096, 16384] drawn with seed 1003, Hq=32, Hkv=4, D=128, indexer
8 x 128, rot 64, ratio 4, budget 512, topK 2051): one step is
qsa_indexer_prefill + qsa_sparse_prefill over one batch already resident in
HBM, timed with CUDA events per step on the launching stream, L2 flushed
between steps outside the timed events (a 512 MB write, then a 256 MB read
of another buffer, so that L2 holds neither the step's data nor dirty lines
whose write-back the step would pay); value = sum of live lengths / time.
The same line carries the 8K and 28K prefill workloads as side lines, the
decode us/step of the two decode workloads (one CUDA-graph replay of
qsa_indexer_decode + qsa_sparse_decode), the roofline of the dominant kernel
against an L2 read bandwidth measured in the same run (libqsa_peaks.so), an
end-to-end figure through the C ABI with host buffers, the CPU oracle
baseline and the SM clocks sampled during the timed regions.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

With N > 1 (launched by torch.distributed.run) every rank runs the same
workload on its own GPU (replicas: the path shards by sequence with no
exchange); value is the sum over ranks, time the max over ranks.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

from block_sparse_gqa_qsa_gb300 import synthetic as syn  # noqa: E402

METRIC = "QSA prefill tokens/s & decode us/step; % of HBM/tensor roofline on 1 GB300"
UNIT = "tokens/s"
HEADLINE = syn.PREFILL_RAGGED
SIDE_PREFILLS = (syn.PREFILL_8K, syn.PREFILL_28K)
DECODES = (syn.DECODE_32, syn.DECODE_LONG)
FLUSH_BYTES = 512 << 20  # > 129 MB L2
L2_PROBE_BYTES = 32 << 20  # stays resident in the 129 MB L2


def f32(x):
    return float(np.float32(x))


# DRAM read+write bytes of one sparse_prefill_kernel launch on the headline workload, from the ncu
# capture summarised under profiles/.  Reported only while the kernel's sources hash to the value
# they had when the counters were taken (None: no capture of the current sources yet).
PROFILED_TRAFFIC = {"bytes": 823_708_160 + 514_016_000, "sources": ("qsa_attention.cu", "qsa_device.cuh"),
                    "sha256": "3ce07eda46bb9934e1a396ba9a9eb5df759ba968a49b4f70b5cbe3374d543f5e"}


def profiled_traffic():
    import hashlib
    h = hashlib.sha256()
    try:
        for name in PROFILED_TRAFFIC["sources"]:
            with open(os.path.join(ROOT, "block_sparse_gqa_qsa_gb300", "csrc", name), "rb") as f:
                h.update(f.read())
    except OSError:
        return None
    return PROFILED_TRAFFIC["bytes"] if h.hexdigest() == PROFILED_TRAFFIC["sha256"] else None


class Probes:
    """Roofline denominators measured live on this GPU (libqsa_peaks.so): L2 -> SM read bandwidth and
    the CUDA-core fp32 FMA rate, each the best of several CUDA-event-timed launches."""

    def __init__(self, dev):
        import ctypes
        from block_sparse_gqa_qsa_gb300 import build
        self.lib = ctypes.CDLL(build.PEAKS_LIB)
        self.lib.qsa_peaks_l2_read.argtypes = [ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int, ctypes.c_void_p,
                                               ctypes.c_int, ctypes.c_void_p]
        self.lib.qsa_peaks_l2_cpasync.argtypes = self.lib.qsa_peaks_l2_read.argtypes
        self.lib.qsa_peaks_ffma.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int, ctypes.c_void_p]
        self.dev = dev
        self.sms = torch.cuda.get_device_properties(dev).multi_processor_count

    def _time(self, launch, reps=10):
        st = torch.cuda.current_stream()
        for _ in range(3):
            launch(st.cuda_stream)
        torch.cuda.synchronize()
        ts = []
        for _ in range(reps):
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            launch(st.cuda_stream)
            e1.record()
            e1.synchronize()
            ts.append(e0.elapsed_time(e1) / 1000.0)
        return min(ts), statistics.median(ts)

    def l2_read(self):
        """The larger of two L2 -> SM read probes (register loads, cp.async into shared memory)."""
        buf = torch.randint(0, 1 << 30, (L2_PROBE_BYTES // 4,), dtype=torch.int32, device=self.dev)
        sink = torch.zeros(4, dtype=torch.int32, device=self.dev)
        passes = 32
        nbytes = passes * L2_PROBE_BYTES
        out = {}
        for name, fn, grid in (("ld_global_cg", self.lib.qsa_peaks_l2_read, 4 * self.sms),
                               ("cp_async_cg", self.lib.qsa_peaks_l2_cpasync, 3 * self.sms)):
            def launch(stream, fn=fn, grid=grid):
                rc = fn(buf.data_ptr(), L2_PROBE_BYTES, passes, sink.data_ptr(), grid, stream)
                if rc:
                    raise RuntimeError(f"L2 probe {name}: CUDA error {rc}")

            best, med = self._time(launch)
            out[name] = {"gbs": round(nbytes / best / 1e9, 1), "median_gbs": round(nbytes / med / 1e9, 1)}
        peak = max(v["gbs"] for v in out.values())
        return {"gbs": peak, "probes": out,
                "how": f"a {L2_PROBE_BYTES >> 20} MB buffer (L2-resident) re-read {passes} times per launch with "
                       f"16-byte accesses, 8 in flight per thread: ld.global.cg by {4 * self.sms} CTAs x 512 "
                       f"threads, and cp.async.cg into a 64 KB shared ring by {3 * self.sms} CTAs x 512; best of 10 "
                       f"launches each (CUDA events); the peak is the larger"}

    def ffma(self):
        out = torch.zeros(4, dtype=torch.float32, device=self.dev)
        iters, grid = 4096, 8 * self.sms

        def launch(stream):
            rc = self.lib.qsa_peaks_ffma(out.data_ptr(), iters, grid, stream)
            if rc:
                raise RuntimeError(f"qsa_peaks_ffma: CUDA error {rc}")

        best, med = self._time(launch)
        fma = grid * 256 * 16 * iters
        return {"tfma_s": round(fma / best / 1e12, 2), "median_tfma_s": round(fma / med / 1e12, 2),
                "how": f"16 independent fmaf chains x {iters} steps per thread, {grid} CTAs x 256 threads; best of 10"}


def max_over_ranks(x, world, device):
    """The largest of each rank's x (the slowest replica's time); x itself on one rank."""
    if world <= 1:
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank, world, ms):
    """Units per second of the whole job: every rank's units over the slowest rank's time."""
    return world * units_per_rank / (ms / 1000.0)


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p.get("bf16_tflops"), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


# ------------------------------------------------------------ algorithmic work
def prefill_work(cfg, ctx):
    """Sum of live tokens, sum of list lengths cnt(t), gathered bytes and MMA flops of the attention."""
    r, beta = cfg.ratio, cfg.budget
    tok = 0
    cnt = 0
    for L in ctx:
        L = int(L)
        t = np.arange(L, dtype=np.int64)
        n_c = (t + 1) // r
        cnt += int(np.sum(np.minimum(n_c, beta) * r + (t + 1 - n_c * r)))
        tok += L
    kv = cfg.Hkv * cnt * 2 * cfg.D * 2
    qo = 2 * tok * cfg.Hq * cfg.D * 2
    lists = cfg.B * cfg.S * cfg.topK * 4
    flops = 4 * cnt * cfg.Hq * cfg.D
    return tok, cnt, kv + qo + lists, flops


def indexer_fma(cfg, ctx):
    """FMAs of the prefill block scores: every row that selects (n_c > budget) scores its n_c blocks
    against Hi query heads of di dims."""
    r, beta = cfg.ratio, cfg.budget
    tot = 0
    for L in ctx:
        n_c = (np.arange(int(L), dtype=np.int64) + 1) // r
        tot += int(np.sum(n_c[n_c > beta]))
    return tot * cfg.Hi * cfg.di


def decode_work(cfg, ctx):
    """Bytes one decode step must move: block keys, gathered K/V rows, q/o/lists."""
    r, beta = cfg.ratio, cfg.budget
    kbar = sum((int(L) // r) * cfg.di * 2 for L in ctx)
    cnt = sum(min(int(L) // r, beta) * r + (int(L) - (int(L) // r) * r) for L in ctx)
    kv = cfg.Hkv * cnt * 2 * cfg.D * 2
    small = cfg.B * (2 * cfg.Hq * cfg.D * 2 + cfg.Hi * cfg.di * 2 + cfg.topK * 4 * 2)
    return kbar, kv, kbar + kv + small


# ------------------------------------------------------------------- clocks
class ClockSampler:
    """nvidia-smi sampling (read-only queries) around the timed regions.

    The sampler runs from before the warm-up to after the last timed region;
    `window()` brackets each timed region with host timestamps, and the summary
    keeps the samples that fall inside a window (all samples if the windows are
    too short to contain one, which the summary then says)."""
    FIELDS = "timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active"

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.windows = []
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.5)  # let the first samples arrive before anything is timed
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except Exception:
                self.proc.kill()
                out = ""
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    class _Window:
        def __init__(self, owner):
            self.owner = owner

        def __enter__(self):
            self.t0 = time.time()

        def __exit__(self, *a):
            self.owner.windows.append((self.t0, time.time()))

    def window(self):
        return ClockSampler._Window(self)

    def summary(self):
        import datetime
        rows = []
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                r = int(parts[4], 16) if parts[4].startswith("0x") else int(parts[4])
                rows.append((ts, float(parts[1]), float(parts[2]), r))
            except (ValueError, IndexError):
                pass
        inside = [r for r in rows if any(t0 - 0.05 <= r[0] <= t1 + 0.05 for t0, t1 in self.windows)]
        use = inside or rows
        names = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap", 0x8: "hw_slowdown",
                 0x20: "sw_thermal_slowdown", 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
                 0x100: "display_clock_setting"}
        reasons = 0
        for r in use:
            reasons |= r[3]
        return {"sm_mhz": statistics.median(r[1] for r in use) if use else None,
                "sm_max_mhz": max(r[2] for r in use) if use else None,
                "reasons": [n for bit, n in names.items() if reasons & bit], "samples": len(use),
                "samples_in_timed_windows": len(inside)}


# ------------------------------------------------------------------ our arm
class Prefill:
    def __init__(self, cfg, dev):
        from block_sparse_gqa_qsa_gb300 import _binding as qb
        self.qb, self.cfg, self.dev = qb, cfg, dev
        self.host = syn.make_prefill(cfg)
        self.t = {k: v.to(dev) for k, v in self.host.items()}
        self.ws = qb.alloc_workspace(qb.indexer_prefill_workspace_size(cfg.B, cfg.S, cfg.di, cfg.ratio), dev)
        self.ind = torch.empty((cfg.B, cfg.S, cfg.topK), dtype=torch.int32, device=dev)
        self.out = torch.empty((cfg.B, cfg.S, cfg.Hq, cfg.D), dtype=torch.float16, device=dev)

    def indexer(self, t=None):
        c, t = self.cfg, t or self.t
        self.qb.indexer_prefill(t["idxQ"], t["idxK"], t["wq"], t["wk"], t["ctx"], self.ind, self.ws, rot=c.rot,
                                ratio=c.ratio, budget=c.budget, topK=c.topK, theta=c.theta, eps=c.eps)

    def attention(self, t=None, out=None):
        c, t = self.cfg, t or self.t
        self.qb.sparse_prefill(t["q"], t["k"], t["v"], self.ind, t["ctx"], self.out if out is None else out,
                               f32(c.scale))


class Decode:
    def __init__(self, cfg, dev):
        from block_sparse_gqa_qsa_gb300 import _binding as qb
        self.qb, self.cfg, self.dev = qb, cfg, dev
        d = syn.make_decode(cfg, device=dev)
        self.ctx_host = d["ctx"].clone()
        self.d = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        self.ws = qb.alloc_workspace(qb.indexer_decode_workspace_size(cfg.B, cfg.maxPagesPerSeq, cfg.ratio,
                                                                      cfg.budget), dev)
        po, ps, pc = qb.sparse_decode_workspace_elems(cfg.B, cfg.Hkv, cfg.D)
        self.parts = (torch.zeros(po, device=dev), torch.zeros(ps, device=dev),
                      torch.zeros(pc, dtype=torch.int32, device=dev))
        self.ind = torch.empty((cfg.B, 1, cfg.topK), dtype=torch.int32, device=dev)
        self.out = torch.empty((cfg.B, 1, cfg.Hq, cfg.D), dtype=torch.float16, device=dev)

    def step(self):
        c, d = self.cfg, self.d
        self.qb.indexer_decode(d["idxQ"], d["idxK"], d["wq"], d["wk"], d["pool"], d["page_table"], d["ctx"],
                               self.ind, self.ws, D=c.D, rot=c.rot, ratio=c.ratio, budget=c.budget, topK=c.topK,
                               theta=c.theta, eps=c.eps)
        self.qb.sparse_decode(d["q"], d["pool"], d["page_table"], self.ind, d["ctx"], self.out, *self.parts, D=c.D,
                              scale=f32(c.scale))


class L2Flush:
    """Evicts everything from L2 between timed steps: a write of FLUSH_BYTES (> L2), then a read of
    half as much from a second buffer, which turns the written buffer's dirty lines into clean,
    unrelated ones."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.r = torch.zeros(FLUSH_BYTES // 8, dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.add_(1)
        self.r.sum()


def time_graph(fn, flush, clk, reps=50, warm=10):
    """Median us of one CUDA-graph replay of fn(), L2 flushed before each replay (outside the events)."""
    for _ in range(3):
        fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    for _ in range(warm):
        g.replay()
    torch.cuda.synchronize()
    times = []
    with clk.window():
        for _ in range(reps):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            g.replay()
            e1.record()
            e1.synchronize()
            times.append(e0.elapsed_time(e1) * 1000.0)
    return statistics.median(times), times


def time_decode(dec, flush, clk, reps=50, warm=10):
    return time_graph(dec.step, flush, clk, reps, warm)


def decode_gather_ab(dec, flush, clk):
    """The attention half of a decode step two ways on the list the step just produced: the split-K decode
    gathering through the page table (A), and qsa_gather_selected into contiguous scratch followed by the
    same decode on the scratch (B)."""
    qb, c, d = dec.qb, dec.cfg, dec.d
    out_b = torch.empty_like(dec.out)
    parts_b = tuple(torch.zeros_like(t) for t in dec.parts)
    sc = qb.gather_scratch(c.B, c.Hkv, c.D, c.topK, device=dec.dev)

    def a():
        qb.sparse_decode(d["q"], d["pool"], d["page_table"], dec.ind, d["ctx"], dec.out, *dec.parts, D=c.D,
                         scale=f32(c.scale))

    def gather():
        qb.gather_selected(d["pool"], d["page_table"], dec.ind, d["ctx"], *sc, D=c.D)

    def b():
        gather()
        qb.sparse_decode(d["q"], sc[0], sc[1], sc[2], sc[3], out_b, *parts_b, D=c.D, scale=f32(c.scale))

    ta, _ = time_graph(a, flush, clk)
    tg, _ = time_graph(gather, flush, clk)
    tb, _ = time_graph(b, flush, clk)
    torch.cuda.synchronize()
    same = bool(torch.equal(out_b.view(torch.int16), dec.out.view(torch.int16)))
    valid = int((dec.ind >= 0).sum())
    row = c.Hkv * c.D * 2
    return {"in_kernel_gather_us": round(ta, 2), "gather_us": round(tg, 2), "gather_then_decode_us": round(tb, 2),
            "gather_bytes": 4 * valid * row, "outputs_bit_identical": same}


def time_prefill(pf, flush, clk, steps):
    """Per-step CUDA-event times (ms) of the indexer, the attention and the whole step, L2 flushed
    before each step outside the events."""
    t_idx, t_att, t_step = [], [], []
    with clk.window():
        for _ in range(steps):
            flush()
            e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
            e[0].record()
            pf.indexer()
            e[1].record()
            pf.attention()
            e[2].record()
            e[2].synchronize()
            t_idx.append(e[0].elapsed_time(e[1]))
            t_att.append(e[1].elapsed_time(e[2]))
            t_step.append(e[0].elapsed_time(e[2]))
    return t_idx, t_att, t_step


def live_copies(cfg, ctx, dst, src):
    """(destination, source) views of one tensor's copy in an end-to-end step: the live rows
    [0, L) of each sequence for the [B, S, ...] tensors (rows at or past L are padding that no
    kernel reads), the whole tensor otherwise."""
    if src.dim() >= 2 and tuple(src.shape[:2]) == (cfg.B, cfg.S):
        return [(dst[b, :L], src[b, :L]) for b, L in enumerate(ctx) if L > 0]
    return [(dst, src)]


def attention_roofline(gbytes, flops, att_ms, l2_gbs, hbm_peak, mma_peak, traffic):
    """The attention kernel against the resource that binds it: its gathered K/V rows come from L2
    (one sequence's K/V is at most 16.8 MB here), so achieved = algorithmic bytes / kernel time is set
    against the measured L2 read bandwidth; DRAM bytes and MMA rate are reported beside it."""
    achieved = gbytes / (att_ms / 1000.0) / 1e9
    out = {"kernel": "sparse_prefill_kernel", "bound": "l2", "achieved": round(achieved, 1), "peak": l2_gbs,
           "unit": "GB/s", "frac": round(achieved / l2_gbs, 4), "traffic": traffic, "algorithmic_bytes": gbytes,
           "peak_source": "measured in this run: L2 read probe (libqsa_peaks.so)",
           "hbm": {"algorithmic_frac": round(achieved / hbm_peak, 4),
                   "dram_gbs": None if traffic is None else round(traffic / (att_ms / 1000.0) / 1e9, 1),
                   "dram_frac": None if traffic is None else round(traffic / (att_ms / 1000.0) / 1e9 / hbm_peak, 4),
                   "peak_gbs": hbm_peak},
           "tensor": {"flops": flops, "achieved_tflops": round(flops / (att_ms / 1000.0) / 1e12, 1),
                      "peak_tflops": mma_peak, "frac": round(flops / (att_ms / 1000.0) / 1e12 / mma_peak, 4),
                      "note": "fp16 MMA at the measured bf16 burst rate (same nominal rate)"}}
    return out


def run_ours(args, rank, world, dev):
    from block_sparse_gqa_qsa_gb300 import _binding as qb
    qb.lib()
    hbm_peak, mma_peak, peak_kind = peaks()
    probes = Probes(dev)
    l2 = probes.l2_read()
    fma = probes.ffma()
    cfg = HEADLINE
    pf = Prefill(cfg, dev)
    flush = L2Flush(dev)
    clk = ClockSampler(torch.cuda.current_device())
    clk.__enter__()
    for _ in range(max(args.warmup, 3)):
        pf.indexer()
        pf.attention()
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t_idx, t_att, t_step = time_prefill(pf, flush, clk, args.steps)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    ms = max_over_ranks(statistics.mean(t_step), world, dev)
    ctx = pf.host["ctx"].tolist()
    tok, cnt, gbytes, flops = prefill_work(cfg, ctx)
    value = whole_job_rate(tok, world, ms)
    att_ms = statistics.mean(t_att)
    idx_ms = statistics.mean(t_idx)
    roof = attention_roofline(gbytes, flops, att_ms, l2["gbs"], hbm_peak, mma_peak, profiled_traffic())
    ifma = indexer_fma(cfg, ctx)

    # End to end through the C ABI: every step copies its inputs from pinned host memory and its output back.
    # The inputs are the live rows of the [B, S, ...] tensors (rows t >= L are padding that no kernel reads),
    # the norm weights and the lengths; the output is the live rows of O.  Two device buffer sets; one copy
    # stream moves step i+1's inputs and another step i's output while step i computes on the compute stream,
    # so the two directions use separate copy engines (events order the reuse of each set).
    pinned = {k: v.pin_memory() for k, v in pf.host.items()}
    out_host = [torch.empty(pf.out.shape, dtype=pf.out.dtype).pin_memory() for _ in range(2)]
    dev_in = [{k: torch.empty_like(v, device=dev) for k, v in pf.host.items()} for _ in range(2)]
    dev_out = [torch.empty_like(pf.out) for _ in range(2)]

    in_pairs = [[p for k in pinned for p in live_copies(cfg, ctx, dev_in[j][k], pinned[k])] for j in range(2)]
    out_pairs = [live_copies(cfg, ctx, out_host[j], dev_out[j]) for j in range(2)]
    h2d = sum(s_.numel() * s_.element_size() for _, s_ in in_pairs[0])
    d2h = sum(s_.numel() * s_.element_size() for _, s_ in out_pairs[0])
    comp, copy_in, copy_out = torch.cuda.current_stream(), torch.cuda.Stream(), torch.cuda.Stream()
    n_e2e = max(args.steps, 4)

    def e2e_run(n):
        in_ready = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]
        out_done = [torch.cuda.Event() for _ in range(2)]
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        copy_in.wait_stream(comp)
        copy_out.wait_stream(comp)
        e0.record(copy_in)

        def h2d_step(i):
            with torch.cuda.stream(copy_in):
                if i >= 2:
                    copy_in.wait_event(done[i % 2])  # set i % 2 was read by step i - 2
                for d_, s_ in in_pairs[i % 2]:
                    d_.copy_(s_, non_blocking=True)
                in_ready[i % 2].record(copy_in)

        h2d_step(0)
        for i in range(n):
            if i + 1 < n:
                h2d_step(i + 1)
            comp.wait_event(in_ready[i % 2])
            if i >= 2:
                comp.wait_event(out_done[i % 2])  # step i - 2's output has left dev_out[i % 2]
            pf.indexer(dev_in[i % 2])
            pf.attention(dev_in[i % 2], dev_out[i % 2])
            done[i % 2].record(comp)
            with torch.cuda.stream(copy_out):
                copy_out.wait_event(done[i % 2])
                for d_, s_ in out_pairs[i % 2]:
                    d_.copy_(s_, non_blocking=True)
                out_done[i % 2].record(copy_out)
        copy_out.wait_stream(copy_in)
        e1.record(copy_out)
        e1.synchronize()
        comp.wait_stream(copy_out)
        return e0.elapsed_time(e1) / n

    e2e_run(3)  # warm-up
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    with clk.window():
        e2e_ms = e2e_run(n_e2e)
    torch.cuda.synchronize()
    e2e_value = whole_job_rate(tok, world, max_over_ranks(e2e_ms, world, dev))
    del pinned, out_host, dev_in, dev_out, in_pairs, out_pairs

    # bf16 surface of the prefill attention: the same workload and lists with bfloat16 Q/K/V/O
    t16 = {n: pf.t[n].to(torch.bfloat16) for n in ("q", "k", "v")}
    out16 = torch.empty(pf.out.shape, dtype=torch.bfloat16, device=dev)
    pf.indexer()
    ts = []
    with clk.window():
        for i in range(args.steps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pf.qb.sparse_prefill(t16["q"], t16["k"], t16["v"], pf.ind, pf.t["ctx"], out16, f32(cfg.scale))
            e1.record()
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1))
    bf16_ms = statistics.mean(ts)

    # the attention on the tcgen05 tensor cores (qsa_sparse_prefill_tcgen05) on the same lists: an A/B
    out_tc = torch.empty_like(pf.out)
    ts = []
    with clk.window():
        for i in range(args.steps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pf.qb.sparse_prefill(pf.t["q"], pf.t["k"], pf.t["v"], pf.ind, pf.t["ctx"], out_tc, f32(cfg.scale),
                                 impl="tcgen05")
            e1.record()
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1))
    pf.attention()
    torch.cuda.synchronize()
    tc_ms = statistics.mean(ts)
    impl_ab = {"workload": cfg.name, "mma_sync_ms": round(att_ms, 4), "tcgen05_ms": round(tc_ms, 4),
               "tcgen05_l2_frac": round(gbytes / (tc_ms / 1000.0) / 1e9 / l2["gbs"], 4),
               "max_abs_diff": float((out_tc.float() - pf.out.float()).abs().max()),
               "note": "the same lists through qsa_sparse_prefill (mma.sync tiles) and qsa_sparse_prefill_tcgen05 "
                       "(tcgen05.mma, TMEM accumulators); the headline uses the faster"}
    del out_tc
    bf16 = {"workload": cfg.name, "kernel": "sparse_prefill_kernel (bf16)", "ms": round(bf16_ms, 4),
            "achieved_gbs": round(gbytes / (bf16_ms / 1000.0) / 1e9, 1),
            "l2_frac": round(gbytes / (bf16_ms / 1000.0) / 1e9 / l2["gbs"], 4)}
    del t16, out16, pf
    torch.cuda.empty_cache()

    # side prefill workloads: the 8K sequence and the 28K sequence the qsa.rs page times its scorer on
    side = []
    pf8 = None
    for sc in SIDE_PREFILLS:
        spf = Prefill(sc, dev)
        for _ in range(3):
            spf.indexer()
            spf.attention()
        torch.cuda.synchronize()
        si, sa, st = time_prefill(spf, flush, clk, max(3, args.steps // 2))
        stok, scnt, sbytes, sflops = prefill_work(sc, spf.host["ctx"].tolist())
        sfma = indexer_fma(sc, spf.host["ctx"].tolist())
        sa_ms, si_ms = statistics.mean(sa), statistics.mean(si)
        side.append({"workload": sc.name, "tokens_per_s": round(stok / (statistics.mean(st) / 1000.0), 1),
                     "ms_per_step": round(statistics.mean(st), 4), "indexer_ms": round(si_ms, 4),
                     "attention_ms": round(sa_ms, 4),
                     "attention_l2_frac": round(sbytes / (sa_ms / 1000.0) / 1e9 / l2["gbs"], 4),
                     "indexer_score_tfma_s": round(sfma / (si_ms / 1000.0) / 1e12, 2),
                     "indexer_fma_frac": round(sfma / (si_ms / 1000.0) / 1e12 / fma["tfma_s"], 4)})
        if sc is syn.PREFILL_8K:
            pf8 = spf
        else:
            del spf
        torch.cuda.empty_cache()

    # prefill -> decode hand-off of the indexer state (the 8K sequence into a pool of Hkv 4, D 128)
    handoff = None
    c8 = syn.PREFILL_8K
    L = int(pf8.host["ctx"][0])
    npg = -(-(L + 1) // syn.TOKENS_PER_PAGE)
    pool = torch.zeros((2 * npg, syn.TOKENS_PER_PAGE, c8.Hkv, c8.D + c8.di), dtype=torch.float16, device=dev)
    ids = torch.arange(npg, dtype=torch.int32, device=dev)
    pt = torch.stack([ids, ids + npg])[None].contiguous()
    pf8.indexer()
    ts = []
    with clk.window():
        for i in range(args.steps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pf8.qb.indexer_prefill_handoff(pf8.t["idxK"], pf8.t["ctx"], pf8.ws, pool, pt, D=c8.D, ratio=c8.ratio)
            e1.record()
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) * 1000.0)
    nb = L // c8.ratio
    moved = 2 * nb * c8.di * 2 + 2 * (L - nb * c8.ratio) * c8.di * 2  # block keys and tail keys, read + write
    handoff = {"workload": f"{c8.name} -> paged pool", "us": round(statistics.median(ts), 2), "bytes": moved,
               "blocks": nb}
    del pool

    # upstream q/k norm + partial RoPE of the 8K workload's packed QKV (dense q/k/v outputs)
    qkv = torch.cat([pf8.t["q"], pf8.t["k"], pf8.t["v"]], dim=2).contiguous()
    qo = torch.empty_like(pf8.t["q"])
    ko, vo = torch.empty_like(pf8.t["k"]), torch.empty_like(pf8.t["v"])
    ts = []
    with clk.window():
        for i in range(args.steps + 3):
            flush()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            pf8.qb.rope_qkv(qkv, pf8.t["wq"], pf8.t["wk"], pf8.t["ctx"], qo, Hq=c8.Hq, Hkv=c8.Hkv, rot=c8.rot,
                            theta=c8.theta, eps=c8.eps, k_out=ko, v_out=vo)
            e1.record()
            e1.synchronize()
            if i >= 3:
                ts.append(e0.elapsed_time(e1) * 1000.0)
    rope_bytes = 2 * qkv.numel() * qkv.element_size()  # read once, written once (q, k, v)
    rope_us = statistics.median(ts)
    rope = {"workload": f"{c8.name} packed QKV", "us": round(rope_us, 2), "bytes": rope_bytes,
            "achieved_gbs": round(rope_bytes / (rope_us * 1e-6) / 1e9, 1),
            "frac": round(rope_bytes / (rope_us * 1e-6) / 1e9 / hbm_peak, 4)}
    del qkv, qo, ko, vo, pf8
    torch.cuda.empty_cache()

    # decode workloads: one graph replay per step
    decode = []
    for dc in DECODES:
        dec = Decode(dc, dev)
        us, _ = time_decode(dec, flush, clk)
        kbar, kv, total = decode_work(dc, dec.ctx_host.tolist())
        ab = decode_gather_ab(dec, flush, clk)
        decode.append({"workload": dc.name, "us_per_step": round(us, 2), "bytes_per_step": total,
                       "roofline_us": round(total / (hbm_peak * 1e9) * 1e6, 2),
                       "frac": round(total / (hbm_peak * 1e9) * 1e6 / us, 4), "kernels_per_step": 4,
                       "attention_gather_ab": ab})
        del dec
        torch.cuda.empty_cache()
    clk.__exit__(None, None, None)
    return {
        "value": value, "ms": ms, "tok": tok, "t_idx": idx_ms, "t_att": att_ms, "roofline": roof,
        "indexer": {"score_fma": ifma, "tfma_s": round(ifma / (idx_ms / 1000.0) / 1e12, 2),
                    "fma_frac": round(ifma / (idx_ms / 1000.0) / 1e12 / fma["tfma_s"], 4),
                    "note": "indexer call time (pool + select kernels) against the probe's fp32 FMA rate"},
        "peaks": {"l2_read": l2, "ffma": fma, "hbm_gbs": hbm_peak, "bf16_tflops": mma_peak, "hbm_source": peak_kind},
        "e2e": e2e_value, "h2d": h2d, "d2h": d2h, "clocks": clk.summary(), "side_prefill": side,
        "decode": decode, "handoff": handoff, "bf16_prefill_attention": bf16, "rope_qkv": rope,
        "attention_impl_ab": impl_ab,
        # per timed prefill step: block_pool, prefill_select, sparse_prefill
        "launches": 3 * args.steps,
    }


# --------------------------------------------------------- the CPU oracle
def headline_config(cfg, ctx):
    """The workload description both arms print (identical keys and values)."""
    return {"workload": cfg.name, "B": cfg.B, "S": cfg.S, "Hq": cfg.Hq, "Hkv": cfg.Hkv, "D": cfg.D,
            "indexer": f"{cfg.Hi}x{cfg.di} rot {cfg.rot}", "ratio": cfg.ratio, "budget": cfg.budget,
            "topK": cfg.topK, "context_lengths": [int(x) for x in ctx],
            "context_lengths_drawn": f"U[{cfg.ctx_lo}, {cfg.ctx_hi}], seed {cfg.seed + 1}" if cfg.ctx_lo else "full",
            "l2": "GPU steps: flushed between steps (512 MB write, then 256 MB read)", "parallelism": "replicas"}


def live_rows(cfg, ctx, nrows):
    """`nrows` flat rows b*S + t spread evenly over the live rows t < L_b of every sequence."""
    flat = np.concatenate([b * cfg.S + np.arange(int(L), dtype=np.int64) for b, L in enumerate(ctx)])
    pick = np.linspace(0, len(flat) - 1, min(nrows, len(flat))).astype(np.int64)
    return flat[pick]


def oracle_sample(cfg, t_np, nrows, nthreads=0):
    """Oracle prefill (indexer + attention) on `nrows` live rows spread over the batch; returns (rows, seconds)."""
    import oracle
    rows = live_rows(cfg, t_np["ctx"], nrows)
    t0 = time.perf_counter()
    ind = oracle.indexer_prefill(t_np["idxQ"], t_np["idxK"], t_np["wq"], t_np["wk"], t_np["ctx"], rot=cfg.rot,
                                 ratio=cfg.ratio, budget=cfg.budget, topK=cfg.topK, theta=cfg.theta,
                                 eps=f32(cfg.eps), rows=rows, nthreads=nthreads)
    oracle.sparse_prefill(t_np["q"], t_np["k"], t_np["v"], ind, t_np["ctx"], f32(cfg.scale), rows=rows,
                          nthreads=nthreads)
    return len(rows), time.perf_counter() - t0


def cpu_baseline(cfg, t_np, target_s=12.0):
    cores = os.cpu_count() or 1
    n, s = oracle_sample(cfg, t_np, 64)
    total = int(np.sum(t_np["ctx"]))
    nrows = int(min(total, max(64, 64 * target_s / max(s, 1e-3))))
    n, s = oracle_sample(cfg, t_np, nrows)
    return {"value": n / s, "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of the {total} live rows of {cfg.name}, spread over its {cfg.B} sequences (indexer + "
                      f"attention for those rows, f64, {cores} threads), {s:.1f} s"}


def run_reference(args, rank, world):
    """Reference arm: the fp64 CPU oracle on the host cores, same metric and workload."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    cfg = HEADLINE
    t = syn.make_prefill(cfg)
    t_np = {k: v.numpy() for k, v in t.items()}
    cores = os.cpu_count() or 1
    # each step: a bounded sample of the workload's live rows
    nrows = 192
    for _ in range(args.warmup):
        oracle_sample(cfg, t_np, 32)
    times = []
    for _ in range(args.steps):
        n, s = oracle_sample(cfg, t_np, nrows)
        times.append(s)
    per = statistics.mean(times)
    value = nrows / per
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": per * 1000.0, "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic", "impl": "reference",
            "config": headline_config(cfg, t["ctx"].tolist()),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": f"{nrows} live rows per step, spread over the {cfg.B} sequences"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if args.impl == "reference":
        run_reference(args, rank, world)
        return
    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(dev))
    r = run_ours(args, rank, world, dev)
    if rank == 0:
        cfg = HEADLINE
        cpu = None
        host = syn.make_prefill(cfg)
        if not args.no_cpu_baseline and world == 1:
            t_np = {k: v.numpy() for k, v in host.items()}
            cpu = cpu_baseline(cfg, t_np)
        line = {
            "metric": METRIC, "value": r["value"], "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": max(args.warmup, 3), "ms_per_step": r["ms"], "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "fp16", "data": "synthetic",
            "config": headline_config(cfg, host["ctx"].tolist()),
            "stages_ms": {"indexer_prefill": round(r["t_idx"], 4), "sparse_prefill": round(r["t_att"], 4)},
            "roofline": r["roofline"],
            "indexer": r["indexer"],
            "peaks": r["peaks"],
            "side_prefill": r["side_prefill"],
            "decode": r["decode"],
            "handoff": r["handoff"],
            "bf16_prefill_attention": r["bf16_prefill_attention"],
            "attention_impl_ab": r["attention_impl_ab"],
            "rope_qkv": r["rope_qkv"],
            "e2e": {"value": r["e2e"], "unit": UNIT, "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"],
                    "note": "each step copies its inputs from pinned host memory (the live rows of q/k/v/idxQ/idxK, "
                            "the norm weights and the lengths; rows at or past a sequence's length are padding no "
                            "kernel reads) and the live rows of O back; two more streams overlap step i+1's input "
                            "copy and step i's output copy with step i's kernels"},
            "cpu_baseline": cpu, "clocks": r["clocks"], "gpu_launches": r["launches"],
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
