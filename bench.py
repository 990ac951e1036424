#!/usr/bin/env python
"""Benchmark of the batched speculative-decoding verify step on GB300.

One step = one verify call (the whole hot path) over one batch of synthetic input.
Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

value      verified draft tokens / s (R per step / kernel time), inputs resident in HBM,
           L2 flushed between steps, CUDA events on the launching stream; under torchrun
           the tokens of all ranks / the slowest rank's time (each rank verifies its own
           batch: requests are independent, no collective in the data path).
e2e        the same metric through the public API with page-locked HOST buffers: every step
           copies the step's inputs host->device, verifies, and reads the outputs back.
roofline   algorithmic bytes per launch / mean step time, against the measured HBM copy
           bandwidth. The bytes are whole rows (logits and mask words of rows 0..a_b, the draw
           row's noise, a rejected draft-model row's q row); the stricter sector-exact count
           (only the 32-byte sectors holding an allowed id on a masked row) is reported beside it.
cpu_baseline  the CPU oracle, single-threaded, on a bounded sample of the same workload; when
           the sample is the whole batch, `parity` compares the last timed step's outputs with
           the oracle's.
per_config the smaller recipes (C0-C3) timed the same way, each with its own parity check.
"""
from __future__ import annotations

import argparse
import dataclasses
import hashlib
import json
import os
import platform
import statistics
import subprocess
import sys
import tempfile
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from speculative_decoding_verification_specdec_gb300 import workloads as W  # noqa: E402

METRIC = "verified draft tokens/s (HBM GB/s and fraction of GB300 peak in roofline)"
UNIT = "tokens/s"
L2_FLUSH_BYTES = 2 * 129 * 1024 * 1024
FALLBACK_HBM_GBS = 6800.0
CSRC = os.path.join(ROOT, "speculative_decoding_verification_specdec_gb300", "csrc")
KERNEL_SRC = os.path.join(CSRC, "specdec_verify.cu")
NGRAM_SRC = os.path.join(CSRC, "specdec_ngram.cu")
SCATTER_SRC = os.path.join(CSRC, "specdec_bitmask.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--config", type=int, default=4, help="workload recipe index (default: the large mixed batch)")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-seconds", type=float, default=15.0, help="budget of the CPU-oracle baseline sample")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-per-config", action="store_true",
                    help="skip the per-recipe lines (C0-C3) of the default large-mixed-batch run")
    ap.add_argument("--ngram", action="store_true",
                    help="time the n-gram proposer (model-free drafter) instead of the verify")
    ap.add_argument("--scatter", action="store_true",
                    help="time the bitmask scatter (compact scheduler-order masks -> batch rows) instead")
    ap.add_argument("--filters", action="store_true",
                    help="verify the random draft-model batch with per-request top-k / top-p instead")
    ap.add_argument("--top-k", type=int, default=None,
                    help="with --filters: this top-k on every request instead of the drawn mix (top-p off unless given)")
    ap.add_argument("--top-p", type=float, default=None,
                    help="with --filters: this top-p on every request instead of the drawn mix (top-k off unless given)")
    ap.add_argument("--requests", type=int, default=0,
                    help="verify only the first N requests of the workload (profiler captures); 0 = all")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def kernel_hash(src: str = KERNEL_SRC) -> str:
    """Hash of a kernel's source file: profiler counters are tied to the code they measured."""
    with open(src, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()[:16]


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def workload_for(cfg: int, rank: int, requests: int = 0, filters: bool = False, top_k=None, top_p=None) -> W.Workload:
    # rank 0 verifies the recipe's own seeded batch; other ranks verify independent batches;
    # requests > 0 keeps the first `requests` requests (smaller cases for profiler captures);
    # filters: the random draft-model batch with per-request top-k / top-p (top_k / top_p: one
    # setting on every request)
    w = W.top_k_top_p_batch(5 + 1000 * rank) if filters else W.config(cfg, seed=cfg + 1000 * rank)
    if filters and (top_k is not None or top_p is not None):
        tk = np.full(w.B, 0 if top_k is None else top_k, np.int32)            # the other one off
        tp = np.full(w.B, 1.0 if top_p is None else top_p, np.float32)
        name = w.name + (f"_topk{top_k}" if top_k is not None else "") + (f"_topp{top_p:g}" if top_p is not None else "")
        w = dataclasses.replace(w, top_k=tk, top_p=tp, name=name)
    if 0 < requests < w.B:
        w = w.subset(range(requests), name=f"{w.name}_first{requests}")
    return w


# ------------------------------------------------------------------------------------------
# algorithmic bytes: what the method must read / write given the accepted lengths
# ------------------------------------------------------------------------------------------

def _sector_bytes(allowed_row: np.ndarray, ids_per_sector: int) -> int:
    """32-byte sectors of a row that hold at least one allowed id."""
    V = allowed_row.size
    pad = (-V) % ids_per_sector
    a = np.concatenate([allowed_row, np.zeros(pad, dtype=bool)]).reshape(-1, ids_per_sector)
    return int(a.any(axis=1).sum()) * 32


def algorithmic_bytes(w: W.Workload, acc: np.ndarray, status: np.ndarray) -> dict:
    """Per-launch bytes the verify must move, given the accepted lengths a_b: for rows 0..a_b the
    mask words and the logits, and for random requests the exponential noise of the draw row plus,
    on a rejected draft-model row, its q row and q(x) of every tested draft; plus the small
    per-request arrays and the outputs. On a row whose bitmask is not all ones only the 32-byte
    sectors holding an allowed id are needed from the logits, noise and q (a forbidden token's
    values cannot change any output). `row_total` counts whole rows instead (the plain
    per-row figure, an upper bound)."""
    es = 2 if w.logits_dtype == W.BF16 else 4
    V, Wd = w.V, w.W
    cu = w.cu_num_draft
    temps = w.temperature
    greedy = ~((temps > 0) & np.isfinite(temps) & (temps >= np.float32(1.17549435e-38)))
    qmode = np.zeros(w.B, dtype=bool)
    if w.draft_probs is not None:
        qmode[:] = True if w.has_q is None else (w.has_q != 0)
    logits = mask = noise = q = small = 0
    row_total = 0

    def sectors(t, ids_per_sector):
        if w.bitmask is None or (w.bitmask[t] == -1).all():
            return None
        return _sector_bytes(W.unpack_mask_rows(w.bitmask[t], V)[0], ids_per_sector)

    for b in range(w.B):
        k = int(cu[b + 1] - cu[b])
        if status[b] & (8 | 16):
            continue
        a = int(acc[b])
        rows = a + 1
        row0 = int(cu[b]) + b
        for j in range(rows):
            sl = sectors(row0 + j, 32 // es)
            logits += V * es if sl is None else sl
            row_total += V * es
        if w.bitmask is not None:
            mask += rows * 4 * Wd
            row_total += rows * 4 * Wd
        sm_ = 4 * 2 + 4 + 4 * k + 4 * (k + 1) + 4      # cu, temperature, ids, out_tokens, out_num_accepted
        small += sm_
        row_total += sm_
        if greedy[b]:
            continue
        small += 4 * min(rows, k)                       # uniforms of the tested drafts
        row_total += 4 * min(rows, k)
        sl = sectors(row0 + a, 8)
        row_bytes = 4 * V if sl is None else sl
        noise += row_bytes
        row_total += 4 * V
        if qmode[b]:
            q += 4 * min(rows, k)
            row_total += 4 * min(rows, k)
            if a < k:
                q += row_bytes
                row_total += 4 * V
    total = logits + mask + noise + q + small + 32
    return {"total": total, "logits": logits, "mask": mask, "noise": noise, "q": q, "small": small,
            "row_total": row_total + 32}


# ------------------------------------------------------------------------------------------
# clocks during the timed region
# ------------------------------------------------------------------------------------------

class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        self.reader = threading.Thread(target=self._read, daemon=True)
        self.reader.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        t0, t1 = (self.t0 or 0) - 0.3, (self.t1 or time.time()) + 0.3
        rows = [l for (ts, l) in self.lines if t0 <= ts <= t1] or [l for (_, l) in self.lines]
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            f = [x.strip() for x in r.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------------------------------
# CPU oracle baseline (test infrastructure; timed here as a reported baseline)
# ------------------------------------------------------------------------------------------

def cpu_oracle_sample(w: W.Workload, budget_s: float):
    import oracle

    oracle.load()
    order = np.arange(w.B)
    # grow the sample until it fills the budget (rough), then time it once
    n = 8
    while True:
        sub = w.subset(order[: min(n, w.B)])
        t0 = time.perf_counter()
        oracle.verify(sub)
        dt = time.perf_counter() - t0
        if dt > budget_s / 4 or n >= w.B:
            break
        n = min(w.B, int(n * max(2.0, (budget_s / 3) / max(dt, 1e-3))))
    sub = w.subset(order[: min(n, w.B)])
    # the whole workload takes less than half the budget: time whole passes until they fill it
    reps = max(1, int((budget_s / 2) / max(dt, 1e-3))) if n >= w.B else 1
    t0 = time.perf_counter()
    for _ in range(reps):
        oracle.verify(sub)
    dt = (time.perf_counter() - t0) / reps
    return sub, dt, reps


def cpu_oracle_threads(sub: W.Workload, threads: int) -> float:
    """The same oracle sample split into `threads` request ranges, one host thread each (the oracle's
    C call releases the interpreter lock); returns the wall time of the parallel pass."""
    import oracle
    from concurrent.futures import ThreadPoolExecutor

    parts = [sub.subset(c) for c in np.array_split(np.arange(sub.B), threads) if len(c)]
    t0 = time.perf_counter()
    with ThreadPoolExecutor(len(parts)) as ex:
        list(ex.map(oracle.verify, parts))
    return time.perf_counter() - t0


def cpu_model() -> str:
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu model")):
                    return line.split(":", 1)[1].strip()
    except OSError:
        pass
    return platform.machine()


def nominal_bytes(w: W.Workload) -> int:
    """The tensors' full sizes: logits + draft probs + bitmask + noise (every row, every id)."""
    es = 2 if w.logits_dtype == W.BF16 else 4
    n = w.T * w.V * es + w.T * w.V * 4
    if w.draft_probs is not None:
        n += w.N * w.V * 4
    if w.bitmask is not None:
        n += w.T * ((w.V + 31) // 32) * 4
    return int(n)


def run_reference(args, world, rank):
    """The oracle as it stands, on the host cores, each step a bounded sample of the workload."""
    if rank != 0:
        return
    import oracle

    w = workload_for(args.config, 0, args.requests, args.filters, args.top_k, args.top_p)
    oracle.load()
    budget_total = 150.0
    per_step = max(0.05, min(5.0, budget_total / max(1, args.steps + args.warmup)))
    # size the per-step sample
    n = 1
    while True:
        sub = w.subset(np.arange(min(n, w.B)))
        t0 = time.perf_counter()
        oracle.verify(sub)
        dt = time.perf_counter() - t0
        if dt >= per_step / 2 or n >= w.B:
            break
        n = min(w.B, n * 2)
    sub = w.subset(np.arange(min(n, w.B)))
    for _ in range(args.warmup):
        oracle.verify(sub)
    times = []
    for _ in range(args.steps):
        t0 = time.perf_counter()
        oracle.verify(sub)
        times.append(time.perf_counter() - t0)
    tot = sum(times)
    value = sub.N * args.steps / tot
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * tot / args.steps,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "requests_per_step": sub.B, "drafts_per_step": sub.N,
                   "note": "CPU oracle (plain C, fp64, single thread) on the first requests of the workload"},
        "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": f"first {sub.B} of {w.B} requests ({sub.N} drafts) per step"},
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


# ------------------------------------------------------------------------------------------
# our arm
# ------------------------------------------------------------------------------------------

def traffic_from_profiles(config_name: str, src: str = KERNEL_SRC):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on this kernel source."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(config_name)
    if not e or e.get("kernel_hash") != kernel_hash(src):
        return None
    return e.get("dram_bytes_per_launch")


def telemetry_summary(tm: np.ndarray, steps: int) -> dict:
    """Per-step drafts / eligible / accepted-through counts by position and the accepted-length
    histogram, trimmed to the longest position with drafts."""
    tm = np.asarray(tm, dtype=np.int64).reshape(4, -1) // max(steps, 1)
    n = int(np.flatnonzero(tm[0]).max()) + 1 if tm[0].any() else 0
    return {"drafts_by_position": tm[0, :n].tolist(), "eligible_by_position": tm[1, :n].tolist(),
            "accepted_through_position": tm[2, :n].tolist(), "accepted_length_histogram": tm[3, :n + 1].tolist()}


def run_ngram(args, world, rank, local):
    """The n-gram proposer on 1024 synthetic histories of 1-8 K tokens (half of them ending inside
    a repeated span): proposals (requests) per second; roofline on the history bytes it must read."""
    import torch

    from speculative_decoding_verification_specdec_gb300 import _native, build

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if rank == 0 and build.needs_rebuild():
        build.build_library()
    _native.load()
    min_n, max_n, k = 2, 5, 8
    hs = W.ngram_histories(7 + 1000 * rank, B=1024 if args.requests <= 0 else args.requests, L=(1024, 8192))
    tokens = torch.from_numpy(hs.tokens).to(dev)
    cu = torch.from_numpy(hs.cu_hist).to(dev)
    B = hs.B
    d = torch.empty((B, k), dtype=torch.int32, device=dev)
    n = torch.empty(B, dtype=torch.int32, device=dev)
    m = torch.empty(B, dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()
    for _ in range(max(3, args.warmup)):
        flush.zero_()
        _native.ngram_propose(tokens, cu, B, min_n, max_n, k, d, n, m, stream=stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler.mark("t0")
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        _native.ngram_propose(tokens, cu, B, min_n, max_n, k, d, n, m, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    clocks = sampler.stop()
    mean_s = sum(ms) / len(ms) / 1e3
    # algorithmic bytes: every token of every history once, the offsets, the outputs
    alg = 4 * int(hs.tokens.size) + 8 * (B + 1) + 4 * B * (k + 2)
    peak, peak_kind = measured_peaks()
    hits = float((m.cpu().numpy() > 0).mean())
    line = {
        "metric": "n-gram proposals/s (requests drafted per second)", "value": B / mean_s, "unit": "proposals/s",
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": hs.name, "B": B, "tokens": int(hs.tokens.size), "min_n": min_n, "max_n": max_n, "k": k,
                   "hit_rate": hits, "l2": "flushed between timed steps (268 MB write)"},
        "roofline": {"bound": "hbm", "achieved": alg / mean_s / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": alg / mean_s / 1e9 / peak, "traffic": traffic_from_profiles(hs.name, NGRAM_SRC),
                     "peak_kind": peak_kind, "kernel": "specdec_ngram_kernel", "algorithmic_bytes_per_launch": alg},
        "gpu_launches": args.steps, "clocks": clocks,
        "kernel_ms": {"median": statistics.median(ms), "min": min(ms), "max": max(ms)},
    }
    print(json.dumps(line), flush=True)


def run_scatter(args, world, rank, local):
    """The bitmask scatter on the large mixed batch's masks (B=1024, V=151936, k~U{1..8}; the masked
    half constrained, in a random scheduler order): rows per second; roofline on the bytes it must
    move (read the constrained rows, write every row)."""
    import torch

    from speculative_decoding_verification_specdec_gb300 import _native, build

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    if rank == 0 and build.needs_rebuild():
        build.build_library()
    _native.load()
    w = workload_for(4, rank, args.requests)
    cu = w.cu_num_draft
    masked = [b for b in range(w.B) if not (w.bitmask[w.row(b, 0)] == -1).all()]
    order = np.random.default_rng(4 + rank).permutation(np.asarray(masked, dtype=np.int32))
    rows = np.concatenate([np.arange(int(cu[b]) + b, int(cu[b + 1]) + b + 1) for b in order])
    compact = torch.from_numpy(np.ascontiguousarray(w.bitmask[rows])).to(dev)
    ids = torch.from_numpy(order).to(dev)
    cut = torch.from_numpy(cu).to(dev)
    out = torch.empty((w.T, w.W), dtype=torch.int32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    sampler = ClockSampler(local)
    sampler.start()

    def step():
        _native.bitmask_scatter(compact, compact.shape[0], ids, ids.numel(), cut, w.B, w.V, out, stream=stream)

    for _ in range(max(3, args.warmup)):
        flush.zero_()
        step()
    torch.cuda.synchronize()
    assert np.array_equal(out.cpu().numpy(), w.bitmask)       # the batch's own masks, unmasked rows all ones
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler.mark("t0")
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    clocks = sampler.stop()
    mean_s = sum(ms) / len(ms) / 1e3
    alg = 4 * w.W * (rows.size + w.T) + 4 * (ids.numel() + w.B + 1)
    peak, peak_kind = measured_peaks()
    line = {
        "metric": "bitmask rows placed per second (batch-order rows written)", "value": w.T / mean_s,
        "unit": "rows/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup, "ms_per_step": mean_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "int32", "data": "synthetic",
        "config": {"workload": f"{w.name}_bitmask_scatter", "B": w.B, "V": w.V, "rows": w.T,
                   "constrained_requests": int(ids.numel()), "compact_rows": int(rows.size),
                   "l2": "flushed between timed steps (268 MB write)"},
        "roofline": {"bound": "hbm", "achieved": alg / mean_s / 1e9, "peak": peak, "unit": "GB/s",
                     "frac": alg / mean_s / 1e9 / peak,
                     "traffic": traffic_from_profiles(f"{w.name}_bitmask_scatter", SCATTER_SRC), "peak_kind": peak_kind,
                     "kernel": "specdec_bitmask_scatter_kernel", "algorithmic_bytes_per_launch": alg},
        "gpu_launches": args.steps, "clocks": clocks,
        "kernel_ms": {"median": statistics.median(ms), "min": min(ms), "max": max(ms)},
    }
    print(json.dumps(line), flush=True)


def time_verify(w, dev_in, out, flush, stream, steps, warmup, pg=None, sampler=None):
    """W untimed warm-up verifies, then `steps` timed ones, each after an L2 flush (outside the
    events), bracketed by a barrier and a synchronize. Returns the per-step kernel times (ms) and
    the outputs of the last step; counters and telemetry are those of the timed steps, summed."""
    import torch

    from speculative_decoding_verification_specdec_gb300 import device

    for _ in range(max(3, warmup)):
        flush.zero_()
        device.verify(w, dev_in, out, stream=stream)
    torch.cuda.synchronize()
    out.counters.zero_()
    if out.telemetry is not None:
        out.telemetry.zero_()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t0")
    for i in range(steps):
        flush.zero_()                      # L2 flush between timed steps (outside the events)
        starts[i].record(stream)
        device.verify(w, dev_in, out, stream=stream)
        ends[i].record(stream)
    torch.cuda.synchronize()
    if sampler:
        sampler.mark("t1")
    if pg:
        pg.barrier()
    return [s_.elapsed_time(e_) for s_, e_ in zip(starts, ends)], out.numpy()


def roofline_fracs(w, res, mean_s, peak):
    """Algorithmic bytes of one launch over the mean step time: whole rows (the headline) and the
    sector-exact count (only the 32-byte sectors holding an allowed id on a masked row)."""
    ab = algorithmic_bytes(w, res["out_num_accepted"], res["status"])
    return ab, ab["row_total"] / mean_s / 1e9, ab["total"] / mean_s / 1e9


def step_outputs(res, steps):
    """The last timed step's outputs with the counters and telemetry of one step."""
    one = {k: res[k] for k in ("out_tokens", "out_num_accepted", "status")}
    one["counters"] = np.asarray(res["counters"], dtype=np.uint64) // np.uint64(steps)
    if res.get("telemetry") is not None:
        one["telemetry"] = np.asarray(res["telemetry"], dtype=np.uint64) // np.uint64(steps)
    return one


def oracle_parity(w, gpu_step):
    """The oracle's outputs for the whole batch against one timed step's outputs (the CPU-baseline
    leg's own oracle run; element by element, with the near-tie exclusions of the parity rules)."""
    import oracle
    from oracle import parity

    rep = parity.compare(w, gpu_step, oracle.verify(w))
    return {"ok": bool(rep.ok), "requests": rep.requests, "excluded_requests": rep.excluded_requests,
            "compared_tokens": rep.compared_tokens, "token_mismatches": len(rep.token_mismatches),
            "accepted_mismatches": len(rep.accepted_mismatches), "counters": rep.counter_mismatch or "exact",
            "telemetry": rep.telemetry_mismatch or "exact"}


def per_config_lines(args, dev, flush, stream, peak, check_parity):
    """The smaller recipes (C0-C3), each timed like the headline workload (fewer steps), with its
    value, kernel median, roofline fractions and, with the CPU leg, parity of its timed outputs."""
    from speculative_decoding_verification_specdec_gb300 import _native, device

    steps = max(1, min(args.steps, 200))
    out_lines = {}
    for cfg in (0, 1, 2, 3):
        w = W.config(cfg)
        dev_in = device.device_tensors(w, dev)
        out = device.alloc_outputs(w, dev, diag=False, telemetry=True)
        ms, res = time_verify(w, dev_in, out, flush, stream, steps, args.warmup)
        mean_s = sum(ms) / len(ms) / 1e3
        ab, rows_gbs, sect_gbs = roofline_fracs(w, res, mean_s, peak)
        shape = _native.launch_config(w.V, 1 if w.logits_dtype == W.BF16 else 0, B=w.B)
        e = {"value": w.N / mean_s, "unit": UNIT, "steps": steps, "kernel_ms_median": statistics.median(ms),
             "ms_per_step": mean_s * 1e3, "frac": rows_gbs / peak, "achieved_gbs": rows_gbs,
             "sector_exact_frac": sect_gbs / peak, "bytes_per_launch": ab["row_total"],
             "kernels_per_step": shape["kernels_with_workspace"]}
        if check_parity:
            e["parity"] = oracle_parity(w, step_outputs(res, steps))
        out_lines[w.name] = e
        del dev_in, out
    return out_lines


def main():
    args = parse()
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    if args.ngram:
        return run_ngram(args, world, rank, local)
    if args.scatter:
        return run_scatter(args, world, rank, local)

    import torch

    from speculative_decoding_verification_specdec_gb300 import _native, build, device

    torch.cuda.set_device(local)
    dev = f"cuda:{local}"
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device(dev))
        pg = dist
    if rank == 0 and build.needs_rebuild():
        build.build_library()
    if pg:
        pg.barrier()
    _native.load()

    w = workload_for(args.config, rank, args.requests, args.filters, args.top_k, args.top_p)
    host = device.host_tensors(w)
    dev_in = device.device_tensors(w, dev, host)
    out = device.alloc_outputs(w, dev, diag=False, telemetry=True)   # per-position counts, every step
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    torch.cuda.synchronize()

    sampler = ClockSampler(local)
    if rank == 0:
        sampler.start()
    kernel_ms, res = time_verify(w, dev_in, out, flush, stream, args.steps, args.warmup, pg=pg, sampler=sampler)
    tot_ms = float(sum(kernel_ms))
    ctr = res["counters"]
    R_per_step = int(ctr[0]) // args.steps
    assert R_per_step == w.N, (R_per_step, w.N)
    if pg:
        t = torch.tensor([tot_ms], dtype=torch.float64, device=dev)
        pg.all_reduce(t, op=pg.ReduceOp.MAX)
        max_ms = float(t.item())
        r = torch.tensor([w.N], dtype=torch.float64, device=dev)
        pg.all_reduce(r)
        R_all = float(r.item())
    else:
        max_ms, R_all = tot_ms, float(w.N)
    value = R_all * args.steps / (max_ms / 1e3)
    clocks = sampler.stop() if rank == 0 else None

    # roofline of the step (schedule + verify kernel)
    mean_s = (tot_ms / args.steps) / 1e3
    peak, peak_kind = measured_peaks()
    ab, achieved_rows, achieved_sect = roofline_fracs(w, res, mean_s, peak)
    traffic = traffic_from_profiles(w.name)

    # e2e through the public API with host buffers
    e2e = None
    if not args.no_e2e:
        pinned = device.host_tensors(w, pin=True)
        out_h = {k: torch.empty(v.shape, dtype=v.dtype).pin_memory()
                 for k, v in (("out_tokens", out.out_tokens), ("out_num_accepted", out.out_num_accepted),
                              ("counters", out.counters), ("status", out.status))}
        h2d = sum(t.numel() * t.element_size() for t in pinned.values() if t is not None)
        d2h = sum(t.numel() * t.element_size() for t in out_h.values())

        def e2e_step():
            for f, t in pinned.items():
                if t is not None:
                    dev_in[f].copy_(t, non_blocking=True)
            device.verify(w, dev_in, out, stream=stream)
            out_h["out_tokens"].copy_(out.out_tokens, non_blocking=True)
            out_h["out_num_accepted"].copy_(out.out_num_accepted, non_blocking=True)
            out_h["counters"].copy_(out.counters, non_blocking=True)
            out_h["status"].copy_(out.status, non_blocking=True)

        for _ in range(2):
            e2e_step()
        torch.cuda.synchronize()
        if pg:
            pg.barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(args.e2e_steps):
            e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = e0.elapsed_time(e1)
        if pg:
            t = torch.tensor([e2e_ms], dtype=torch.float64, device=dev)
            pg.all_reduce(t, op=pg.ReduceOp.MAX)
            e2e_ms = float(t.item())
        e2e = {"value": R_all * args.e2e_steps / (e2e_ms / 1e3), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
               "d2h_bytes_per_step": int(d2h), "ms_per_step": e2e_ms / args.e2e_steps}

    cpu = cpu_all = parity = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        sub, dt, reps = cpu_oracle_sample(w, args.cpu_seconds)
        cpu = {"value": sub.N / dt, "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": (f"first {sub.B} of {w.B} requests ({sub.N} drafts), {reps} pass{'es' if reps > 1 else ''}, "
                          f"{dt * reps:.1f} s"),
               "cpu": cpu_model()}
        nthreads = os.cpu_count() or 1
        dtp = cpu_oracle_threads(sub, nthreads)
        cpu_all = {"value": sub.N / dtp, "unit": UNIT, "cores": nthreads, "kind": "oracle",
                   "sample": f"the same sample split over {nthreads} host threads, {dtp:.2f} s", "cpu": cpu_model()}
        # the oracle's outputs for the whole batch against the last timed step's
        parity = oracle_parity(w, step_outputs(res, args.steps))
    per_config = None
    if rank == 0 and world == 1 and not args.no_per_config and not args.filters and args.requests == 0 \
            and args.config == 4:
        per_config = per_config_lines(args, dev, flush, stream, peak, check_parity=not args.no_cpu_baseline)

    if rank == 0:
        shape = _native.launch_config(w.V, 1 if w.logits_dtype == W.BF16 else 0, B=w.B)
        line = {
            "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": tot_ms / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": w.logits_dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "V": w.V, "drafts_per_step": w.N, "rows": w.T,
                       "l2": "flushed between timed steps (268 MB write)",
                       "launch": {"grid_ctas": (2 * (shape["split_requests"] + (w.B - shape["split_requests"] + 1) // 2)
                                                if shape["split_requests"] else w.B * shape["ctas_per_request"]),
                                  **shape},
                       "per_rank": "independent batch per rank (requests shard with no exchange)"},
            "roofline": {"bound": "hbm", "achieved": achieved_rows, "peak": peak, "unit": "GB/s",
                         "frac": achieved_rows / peak, "traffic": traffic, "peak_kind": peak_kind,
                         "kernel": "specdec_verify_stream_kernel",
                         "time": ("whole step: request-schedule kernel + verify kernel"
                                  if shape["kernels_with_workspace"] == 2 else "verify kernel"),
                         "bytes": ("algorithmic, whole rows: logits and mask words of rows 0..a_b, the draw "
                                   "row's noise, a rejected draft-model row's q row, q(x) of the tested "
                                   "drafts, the per-request arrays and outputs"),
                         "algorithmic_bytes_per_launch": ab["row_total"],
                         "sector_exact_gbs": achieved_sect, "sector_exact_frac": achieved_sect / peak,
                         "sector_exact_bytes": ab,
                         "sector_exact_note": ("stricter count: on a masked row only the 32-byte sectors "
                                               "holding an allowed id")},
            "parity": parity,
            "per_config": per_config,
            "e2e": e2e,
            "cpu_baseline": cpu,
            "cpu_baseline_all_cores": cpu_all,
            "emitted_tokens_per_s": int((res["out_tokens"] >= 0).sum()) / mean_s,
            "mean_acceptance_length": 1.0 + (int(ctr[3]) / args.steps) / max(w.B, 1),
            "nominal": {"bytes_per_launch": nominal_bytes(w), "effective_gbs": nominal_bytes(w) / mean_s / 1e9,
                        "note": "full logits + draft probs + bitmask + noise tensors over the kernel time"},
            "gpu_launches": args.steps * shape["kernels_with_workspace"],
            "clocks": clocks,
            "kernel_ms": {"median": statistics.median(kernel_ms), "min": min(kernel_ms), "max": max(kernel_ms)},
            "counters_per_step": [int(c) // args.steps for c in ctr],
            "telemetry_per_step": telemetry_summary(res["telemetry"], args.steps),
            "kernel_hash": kernel_hash(),
        }
        print(json.dumps(line), flush=True)
    if pg:
        pg.barrier()
        pg.destroy_process_group()


if __name__ == "__main__":
    main()
