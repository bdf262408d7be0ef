#!/usr/bin/env python3
"""Benchmark of one paged-KV decode step (append + GQA decode) on GB300.

Default workload: the Qwen2.5-7B-shaped batch (128 sequences, 28 q / 4 kv
heads, head_dim 128, fp16, lognormal context lengths with median 1024 clipped
to [1, 8192]; seeded synthetic data).  A step is the whole hot path for one
batch: each sequence's new token is appended and each sequence attends over
its context, split contexts merged by log-sum-exp in a second launch.  For
16-bit pools the append runs inside the attention launch (pa_decode_step);
for E4M3 pools, where that is slower, as its own launch first
(pa_cache_append_fp8 + pa_decode_fp8); ``--step`` forces either form.
Between timed steps the L2 is not flushed when the step reads at least 3x
the L2 size (429 MB of K/V against a 129 MB L2 for the default batch);
smaller batches have L2 evicted by reading a 2x-L2 buffer outside the timed
region.

Prints one JSON line.  ``value`` is attended KV tokens/s of the whole job
(sum of context lengths over all ranks / max-over-ranks step time); the line
also carries the decode call's HBM roofline, an end-to-end figure through
pinned host buffers, the fp64 CPU oracle's throughput as a reported baseline,
the number of this library's kernel launches and the SM clocks seen.

``--impl reference`` times the oracle (the only reference that exists for
this path) on the host cores instead, on a bounded sample of the workload.
"""
from __future__ import annotations

import argparse
import gc
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

METRIC = "paged GQA decode: attended KV tokens/s and HBM GB/s (% of GB300 peak)"
UNIT = "tokens/s"
DEFAULT_CONFIG = "qwen2_5_7b"
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers
def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def attended(lens: np.ndarray, window: int = 0) -> np.ndarray:
    """Tokens each sequence attends: all of them, or its last ``window``."""
    L = lens.astype(np.int64)
    return np.minimum(L, window) if window > 0 else L


def algorithmic_bytes(w, lens: np.ndarray, window: int = 0) -> dict:
    """Bytes one decode call must move: K+V of every attended token, q, out,
    the block-table entries and context lengths read (plus page scales for an
    E4M3 pool).  Workspace traffic, the padding rows of each sequence's last
    block and the rows before a sliding window in its first block are
    overhead, not counted."""
    e_kv = 1 if w.kv == "fp8" else 2
    L = lens.astype(np.int64)
    first = np.maximum(L - window, 0) // w.block_size if window > 0 else 0
    nblk = (L + w.block_size - 1) // w.block_size - first
    kv = int(attended(lens, window).sum()) * w.Hkv * 2 * w.D * e_kv
    qo = 2 * w.B * w.Hq * w.D * 2
    meta = int(nblk.sum()) * 4 + w.B * 4
    scales = int(nblk.sum()) * w.Hkv * 2 * 4 if w.kv == "fp8" else 0
    # the fused step also reads this step's K/V rows and writes them to the pools
    append = w.B * w.Hkv * w.D * 2 * (2 + e_kv) + w.B * 8
    # K/V bytes of distinct physical blocks (a shared prefix counted once): the
    # rows of each block attended by any sequence
    tables = w.block_tables.cpu().numpy()
    rows = {}
    for b in range(w.B):
        lo = int(first[b]) if window > 0 else 0
        for j in range(lo, lo + int(nblk[b])):
            blk = int(tables[b, j])
            r0 = max(0, int(L[b]) - window - j * w.block_size) if window > 0 else 0
            n = min(w.block_size, int(L[b]) - j * w.block_size) - min(r0, w.block_size)
            rows[blk] = max(rows.get(blk, 0), n)
    kv_unique = sum(rows.values()) * w.Hkv * 2 * w.D * e_kv
    return {"kv": kv, "q_out": qo, "meta": meta, "scales": scales, "append": append,
            "total": kv + qo + meta + scales, "kv_unique": kv_unique}


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons in the background."""
    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int, period_ms: int = 20):
        self.index = index
        self.period_ms = period_ms
        self.proc = None
        self.file = None
        self.marks = {}

    def start(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", f"-lms={self.period_ms}"],
                stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, ValueError):
            self.proc = None
        time.sleep(0.3)

    def mark(self, name):
        self.marks[name] = time.time()

    def stop(self) -> dict:
        """Stop sampling; the summary of the timed region (marks timed_start / timed_end)."""
        self.rows = []
        if self.proc is None:
            return self.summary()
        time.sleep(0.1)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.file.flush()
        self.file.seek(0)
        for line in self.file.read().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                ts += float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                self.rows.append((ts, float(parts[2]), float(parts[3]), parts[5:]))
            except (ValueError, IndexError):
                continue
        os.unlink(self.file.name)
        return self.summary()

    def summary(self, start="timed_start", end="timed_end", before=None) -> dict:
        """Median SM clock, max clock and throttle reasons seen between two
        marks (falling back to the mark ``before`` .. end, then the whole run,
        when fewer than 3 samples fall inside)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = getattr(self, "rows", [])
        t0, t1 = self.marks.get(start, 0), self.marks.get(end, 1e30)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if len(inside) < 3:
            t0w = self.marks.get(before or "warmup_start", t0)
            inside = [r for r in rows if t0w - 0.05 <= r[0] <= t1 + 0.05]
            window = "warmup+timed"
        if not inside:
            inside, window = rows, "whole run"
        names = ["active", "hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
                 "sw_power_cap"]
        reasons = set()
        for r in inside:
            for n, v in zip(names[1:], r[3][1:]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median([r[1] for r in inside]) if inside else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window}


def oracle_baseline(w, pools, budget_s: float = 10.0, window: int = 0,
                    threads: int = 0) -> dict:
    """The fp64 CPU oracle (as it stands) on a bounded sample of the batch:
    whole passes over a subset of its sequences (their blocks copied to the
    host), repeated to about budget_s.  ``threads`` > 0 runs it on that many
    OpenMP threads (1: one core), else on all host cores."""
    import oracle
    from paged_kv_cache_179_gb300 import workloads as W
    lens = w.context_lens.cpu().numpy()
    att = attended(lens, window)
    tables = w.block_tables.cpu().numpy()
    fp8 = w.kv == "fp8"
    bf16 = w.dtype == "bf16"
    all_threads = oracle.num_threads()
    if threads > 0:
        oracle.set_num_threads(threads)
    try:
        cores = oracle.num_threads()
        order = np.random.default_rng(0).permutation(w.B)

        def host_sample(rows):
            names = ("k_cache", "v_cache", "k_scale", "v_scale") if fp8 else ("k_cache", "v_cache")
            sub_t, sub_l, arrs = W.extract_rows(tables, lens, rows, [pools[n] for n in names])
            q = W.to_numpy16(w.q[torch.as_tensor(np.asarray(rows), device=w.q.device)])
            return q, sub_t, sub_l, arrs

        def run(sample):
            q, sub_t, sub_l, arrs = sample
            if fp8:
                oracle.decode_fp8(q, *arrs, sub_t, sub_l, w.scale, bf16=bf16, window=window)
            else:
                oracle.decode(q, *arrs, sub_t, sub_l, w.scale, bf16=bf16, window=window)

        # calibrate on 4 sequences, then size the sample to about budget_s
        probe = host_sample(order[:4])
        t = time.perf_counter()
        run(probe)
        per_tok = max(time.perf_counter() - t, 1e-3) / max(1, int(att[order[:4]].sum()))
        n, tok = 0, 0
        for b in order:
            if (tok + att[b]) * per_tok > budget_s and n >= 4:
                break
            n += 1
            tok += int(att[b])
        rows = order[:n]
        sample = host_sample(rows)
        reps, t = 0, time.perf_counter()
        while True:
            run(sample)
            reps += 1
            dt = time.perf_counter() - t
            if dt >= budget_s or reps >= 200:
                break
    finally:
        if threads > 0:
            oracle.set_num_threads(all_threads)
    tok = int(att[rows].sum()) * reps
    return {"value": round(tok / dt, 1), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": f"{n} of {w.B} sequences ({int(att[rows].sum())} attended tokens, all "
                      f"{w.Hq} q heads{', E4M3 pool' if fp8 else ''}) x {reps} passes on "
                      f"{cores} thread(s), fp64 two-pass softmax, {dt:.1f} s"}


# ---------------------------------------------------------------- replicas
def replica_seed(seed: int, rank: int) -> int:
    """Each rank draws its own batch: N GPUs run N independent replicas."""
    return seed + rank


def reduce_over_ranks(step_ms: float, e2e_ms: float, tokens: int, world: int, dev):
    """Whole-job figures: the slowest rank's times and the tokens of all ranks."""
    if world <= 1:
        return step_ms, e2e_ms, float(tokens)
    t = torch.tensor([step_ms, e2e_ms], dtype=torch.float64, device=dev)
    n = torch.tensor([float(tokens)], dtype=torch.float64, device=dev)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    torch.distributed.all_reduce(n, op=torch.distributed.ReduceOp.SUM)
    return t[0].item(), t[1].item(), n[0].item()


# ---------------------------------------------------------------- our arm
OTHER_CONFIGS = ("tiny", "smollm2_360m", "qwen2_5_1_5b", "qwen2_5_7b_fp8")
MULTIQUERY_RUNS = (("qwen2_5_7b", 4), ("mqa_32x1", 1))


class ConfigRun:
    """One workload's batch on the device, its decode steps bound once, and
    the device-timed steps: everything a bench line measures except the
    end-to-end leg."""

    def __init__(self, args, name, seed, dev, window=0):
        from paged_kv_cache_179_gb300 import _abi
        from paged_kv_cache_179_gb300 import workloads as W
        from paged_kv_cache_179_gb300.step import DecodeStep

        self.args, self.name, self.dev, self.window = args, name, dev, window
        w = self.w = W.make_workload(name, seed=seed, device=dev)
        self.lens = w.context_lens.cpu().numpy()
        self.tokens = int(attended(self.lens, window).sum())
        if w.kv == "fp8":
            kc = torch.empty(w.k_cache.shape, dtype=torch.uint8, device=dev)
            vc = torch.empty_like(kc)
            ks = torch.empty(w.num_blocks, w.Hkv, dtype=torch.float32, device=dev)
            vs = torch.empty_like(ks)
            _abi.pa_quantize_fp8(w.k_cache, w.v_cache, kc, vc, ks, vs)
            pools = dict(k_cache=kc, v_cache=vc, k_scale=ks, v_scale=vs)
            # the fp16 source pools are not read again (the new rows are in w)
            w.k_cache = w.v_cache = None
            torch.cuda.empty_cache()
        else:
            pools = dict(k_cache=w.k_cache, v_cache=w.v_cache)
        self.pools = pools
        self.out = torch.empty_like(w.q)
        l2 = self.l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
        self.ab = algorithmic_bytes(w, self.lens, window)
        kv_bytes = self.kv_bytes = self.ab["kv"]
        l2_mode = args.l2
        if l2_mode == "auto":
            # Inputs several times larger than L2 stream through it without
            # hits and run back to back.  Smaller pools are replicated (one
            # copy per layer of a model, as a serving step has) and the steps
            # cycle over the copies, so each step's K/V is cold; when that
            # would take more than 16 copies, L2 is evicted before each step by
            # reading a 2x-L2 buffer (a read leaves clean lines, so the timed
            # step pays no write-backs) and steps are timed one by one.
            copies = -(-3 * l2 // max(kv_bytes, 1))
            l2_mode = "none" if kv_bytes >= 3 * l2 else ("rotate" if copies <= 16 else "read")
        copies = max(2, min(16, -(-3 * l2 // max(kv_bytes, 1)))) if l2_mode == "rotate" else 1
        self.l2_mode, self.copies = l2_mode, copies
        self.pool_sets = [pools] + [{k: t.clone() for k, t in pools.items()}
                                    for _ in range(copies - 1)]
        self.back_to_back = l2_mode in ("none", "rotate")
        # the timed steps: nothing between them writes context_lens or
        # block_tables, so the attention launch may start its prologue while
        # the previous step's merge finishes (PA_DECODE_EARLY_PROLOGUE); and
        # the kernels between them write the pools only in each sequence's
        # last block (the previous step's append), so it may also start its
        # first K/V copies then (PA_DECODE_EARLY_COPIES).  Steps that each
        # follow an L2-evicting kernel (not one of ours, which would let the
        # launch start early) gain nothing by it, and launch plainly.
        self.early = args.early_prologue in ("on", "copies") and self.back_to_back
        self.early_copies = self.early and args.early_prologue == "copies"
        self.steps = [DecodeStep(**ps, block_tables=w.block_tables, context_lens=w.context_lens,
                                 max_context_len=w.max_context_len, scale=w.scale,
                                 num_q_heads=w.Hq, split_ctas=args.splits, window=window,
                                 early_prologue=self.early, early_copies=self.early_copies)
                      for ps in self.pool_sets]
        self.step = self.steps[0]
        self.flush_buf = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.int32, device=dev)
        self.stream = torch.cuda.current_stream(dev)
        self.fused = (self.step.prefers_fused if args.step == "auto"
                      else args.step == "fused")
        # decode_kernel + merge_kernel (fused) | append_kernel + decode_kernel + merge_kernel
        self.launches_per_step = 2 if self.fused else 3
        # each copy's step, and its decode alone, bound once (arguments checked
        # and marshalled outside the timed region)
        self.calls = [st.bind(w.q, w.k_new, w.v_new, w.slot_mapping, self.out, fused=self.fused,
                              stream=self.stream) for st in self.steps]
        self.decodes = [_abi.prepare(lambda st=st: st.decode(w.q, self.out), self.stream)
                        for st in self.steps]

    def flush(self):
        if self.l2_mode == "read":
            self.flush_buf.sum(dtype=torch.int64)
        elif self.l2_mode == "write":
            self.flush_buf.add_(1)

    def run_step(self, i=0):
        self.calls[i % self.copies]()

    def _timed(self, fn, K):
        """K calls of fn(i): back to back between two events (an event
        recorded between steps costs the GPU about 2 us, measured, which is
        not the step's), or each after an L2 eviction between its own events."""
        if self.back_to_back:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(self.stream)
            for i in range(K):
                fn(i)
            e1.record(self.stream)
            torch.cuda.synchronize(self.dev)
            return [e0.elapsed_time(e1) / K] * K
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            self.flush()
            ev[i][0].record(self.stream)
            fn(i)
            ev[i][1].record(self.stream)
        torch.cuda.synchronize(self.dev)
        return [a.elapsed_time(b) for a, b in ev]

    def warm(self, warmup):
        from paged_kv_cache_179_gb300 import _abi
        for i in range(max(warmup, self.copies)):
            self.flush()
            self.run_step(i)
        rc, bits = _abi.pa_get_status(self.dev)
        if rc != 0:
            raise RuntimeError(f"{self.name}: device status {rc} bits {bits}")

    def time_steps(self, K):
        self.step_ms = self._timed(self.run_step, K)
        return self.step_ms

    def time_decode(self, K):
        """The dominant kernel (decode_kernel, then merge_kernel): the fused
        step itself, or the decode alone timed the same way."""
        if self.fused:
            self.dec_ms = self.step_ms
        else:
            torch.cuda.synchronize(self.dev)
            self.dec_ms = self._timed(lambda i: self.decodes[i % self.copies](), K)
        return self.dec_ms

    def kernel_bytes(self):
        return self.ab["total"] + (self.ab["append"] if self.fused else 0)

    def check(self):
        from paged_kv_cache_179_gb300 import _abi
        rc, bits = _abi.pa_get_status(self.dev)
        if rc != 0:
            raise RuntimeError(f"{self.name}: device status {rc} bits {bits}")

    def describe_step(self):
        return ("pa_decode_step: append inside the attention launch, then the merge launch"
                if self.fused else "append launch, then attention and merge launches")

    def describe_launch(self):
        if not self.early:
            return "plain launches"
        return ("attention launch with an early prologue (PA_DECODE_EARLY_PROLOGUE: it may "
                "start while the previous step's merge finishes"
                + ("; PA_DECODE_EARLY_COPIES: its first K/V copies, of blocks before each "
                   "sequence's last two, start then too)" if self.early_copies else ")"))

    def decode_us(self):
        d = self.dec_ms
        if self.back_to_back:
            return {"mean": round(statistics.mean(d) * 1e3, 2),
                    "timing": "K decodes back to back between two events"}
        return {"mean": round(statistics.mean(d) * 1e3, 2),
                "median": round(statistics.median(d) * 1e3, 2),
                "p20": round(float(np.percentile(d, 20)) * 1e3, 2),
                "p80": round(float(np.percentile(d, 80)) * 1e3, 2),
                "min": round(min(d) * 1e3, 2),
                "timing": "each decode between its own events, L2 evicted before it"}


def measure_other_config(args, name, dev, clocks, peak):
    """A config other than the headline's: its steps and decode timed as the
    headline's are (same K, warm-up, L2 handling and launch form), with the
    clocks seen during its own timed region."""
    run = ConfigRun(args, name, args.seed, dev)
    run.warm(args.warmup)
    torch.cuda.synchronize(dev)
    clocks.mark(f"{name}:start")
    run.time_steps(args.steps)
    clocks.mark(f"{name}:end")
    run.time_decode(args.steps)
    e2e_ms, h2d, d2h, e2e_mode = measure_e2e(args, run, dev)
    run.check()
    step_s = statistics.mean(run.step_ms) / 1e3
    dec_s = statistics.mean(run.dec_ms) / 1e3
    kb = run.kernel_bytes()
    entry = {
        "workload": describe(run.w, run.tokens), "step": run.describe_step(),
        "ms_per_step": round(step_s * 1e3, 5), "tokens_per_s": round(run.tokens / step_s, 1),
        "dtype": "e4m3->f32" if run.w.kv == "fp8" else run.w.dtype,
        "split_ctas": run.step.split_ctas,
        "l2": describe_l2(run.l2_mode, run.kv_bytes, run.l2, run.copies),
        "launch": run.describe_launch(),
        "decode_us": run.decode_us(),
        "bytes_per_decode": kb, "hbm_gbs": round(kb / dec_s / 1e9, 1),
        "frac_of_peak": round(kb / dec_s / 1e9 / peak, 4),
        "e2e": {"value": round(run.tokens * args.steps / (e2e_ms / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode},
        "gpu_launches": run.launches_per_step * args.steps,
        "clocks_marks": (f"{name}:start", f"{name}:end"),
    }
    if name == "tiny":
        entry["note"] = ("0.03 MB per step: parity case, launch- and latency-bound; its "
                         "fraction of peak is no bandwidth claim")
    cpu = None
    if run.w.kv == "fp8" and not args.no_cpu_baseline:
        cpu = oracle_baseline(run.w, run.pools, args.cpu_budget / 2)
    del run
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    if cpu is not None:
        entry["cpu_baseline"] = cpu
    return entry


def measure_e2e(args, run, dev):
    """End to end through the public API: the step's inputs packed in one
    pinned host buffer and uploaded by one copy, the output copied back.  Back
    to back (large or replicated pools) the steps run as a pipeline (the next
    step's upload and the last step's read-back overlap the current step's
    attention; one slot per pool copy), timed over the K steps; otherwise step
    by step, L2 evicted outside each step's events.  Returns (total ms, bytes
    uploaded per step, bytes read back per step, mode)."""
    from paged_kv_cache_179_gb300.step import DecodeStep, StepPipeline, StepStaging
    w, out, stream, K = run.w, run.out, run.stream, args.steps
    names = ("q", "k_new", "v_new", "slot_mapping", "block_tables", "context_lens")
    specs = {k: (getattr(w, k).shape, getattr(w, k).dtype) for k in names}
    made = []
    fused, copies = run.fused, run.copies

    shared_ws = []

    def make_step(staging):
        ps = run.pool_sets[len(made) % copies]
        made.append(staging)
        # the pipeline orders each step after its upload and after the last
        # read-back of its slot by events; with those between two steps the
        # attention launch starts once the previous merge has completed, early
        # prologue or not (a full dependency, which it does not relax).  The
        # slots' steps run one after another, so they share one workspace.
        st = DecodeStep(**ps, block_tables=staging.dev["block_tables"],
                        context_lens=staging.dev["context_lens"],
                        max_context_len=w.max_context_len, scale=w.scale, num_q_heads=w.Hq,
                        split_ctas=args.splits, window=run.window,
                        early_prologue=run.early, early_copies=run.early_copies,
                        workspace=shared_ws[0] if shared_ws else None)
        shared_ws[:1] = [st.workspace]
        return st
    h2d = d2h = 0
    host_us = None
    if run.back_to_back:
        pipe = StepPipeline(make_step, specs, out.shape, out.dtype, dev, depth=max(2, copies),
                            handshake=args.handshake)
        mode = ("pipelined: uploads and read-backs on two copy streams, overlapping the "
                f"steps ({max(2, copies)} slots), ordered by "
                + ("a device-side handshake (the attention launch waits for its upload's word, "
                   "the read-back for the step's done word; only kernels on the compute stream)"
                   if pipe.uses_device_handshake(fused) else "stream events"))
        for st_ in pipe.stagings:
            for k in names:
                st_.host[k].copy_(getattr(w, k).cpu())
        for _ in range(max(args.warmup, pipe.depth)):
            pipe.submit(fused=fused)
        pipe.finish()
        torch.cuda.synchronize(dev)
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t_host = time.perf_counter()
        for i in range(K):
            _, h2d, d2h = pipe.submit(fused=fused)
        host_us = (time.perf_counter() - t_host) / K * 1e6
        pipe.finish()
        e1.record(stream)
        ev = [(e0, e1)]
    else:
        mode = "step by step: upload, step, read-back, L2 evicted between steps"
        staging = StepStaging(specs, dev)
        for k in names:
            staging.host[k].copy_(getattr(w, k).cpu())
        e2e_step = make_step(staging)
        host_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for _ in range(max(1, args.warmup)):
            e2e_step.run_from_staging(staging, host_out, out, fused=fused)
        torch.cuda.synchronize(dev)
        for i in range(K):
            run.flush()
            ev[i][0].record(stream)
            h2d, d2h = e2e_step.run_from_staging(staging, host_out, out, fused=fused)
            ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    if host_us is not None:
        mode += f"; the host issues a step in {host_us:.1f} us"
    return sum(a.elapsed_time(b) for a, b in ev), h2d, d2h, mode


def run_ours(args, rank, world, dev):
    from paged_kv_cache_179_gb300 import _abi

    _abi.load()
    run = ConfigRun(args, args.config, replica_seed(args.seed, rank), dev, args.window)
    w, out, stream, K = run.w, run.out, run.stream, args.steps

    clocks = ClockSampler(dev.index if dev.index is not None else 0)
    if rank == 0:
        clocks.start()
    clocks.mark("warmup_start")
    run.warm(args.warmup)

    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize(dev)
    clocks.mark("timed_start")
    step_ms = run.time_steps(K)
    total_ms = sum(step_ms)
    clocks.mark("timed_end")
    if world > 1:
        torch.distributed.barrier()

    # for the spread of single steps: each step between its own two events
    # (which add about 2 us each to what they time), after the timed region
    per_ev = []
    if run.back_to_back:
        pe = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            pe[i][0].record(stream)
            run.run_step(i)
            pe[i][1].record(stream)
        torch.cuda.synchronize(dev)
        per_ev = [a.elapsed_time(b) for a, b in pe]

    dec_ms = run.time_decode(K)

    # for reference: the same step as two launches (append, then decode), each
    # timed with its own events (they include the events' own cost)
    sep = []
    for i in range(min(K, 20)):
        a0, a1, a2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        run.flush()
        a0.record(stream)
        run.step.append(w.k_new, w.v_new, w.slot_mapping)
        a1.record(stream)
        run.step.decode(w.q, out)
        a2.record(stream)
        sep.append((a0, a1, a2))
    torch.cuda.synchronize(dev)
    app_ms = [a0.elapsed_time(a1) for a0, a1, _ in sep]
    dec2_ms = [a1.elapsed_time(a2) for _, a1, a2 in sep]

    e2e_ms, h2d, d2h, e2e_mode = measure_e2e(args, run, dev)
    run.check()

    total_ms_max, e2e_ms_max, tokens_all = reduce_over_ranks(total_ms, e2e_ms, run.tokens,
                                                             world, dev)
    if rank != 0:
        clocks.stop()
        return None

    peak, peak_kind = measured_peaks()
    dec_mean_s = statistics.mean(dec_ms) / 1e3
    kernel_bytes = run.kernel_bytes()
    ab = run.ab
    achieved = kernel_bytes / dec_mean_s / 1e9
    value = tokens_all * K / (total_ms_max / 1e3)
    traffic = load_traffic(args.config, run.step.split_ctas)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(total_ms_max / K, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3->f32" if w.kv == "fp8" else w.dtype, "data": "synthetic",
        "config": {
            "workload": describe(w, run.tokens), "step": run.describe_step(),
            "split_ctas": run.step.split_ctas,
            "l2": describe_l2(run.l2_mode, run.kv_bytes, run.l2, run.copies),
            "launch": run.describe_launch(),
            "seed": args.seed, "parallelism": "replicas" if world > 1 else "single GPU",
            **({"window": args.window} if args.window else {}),
        },
        "hbm_gbs": round(achieved, 1), "hbm_frac_of_peak": round(achieved / peak, 4),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": ("decode_kernel with fused append, then merge_kernel (timed "
                                "together: one decode)" if run.fused
                                else "decode_kernel, then merge_kernel (timed together: one decode)"),
                     "bytes_per_launch": kernel_bytes, "peak_source": peak_kind,
                     **({"kv_bytes_unique": ab["kv_unique"],
                         "note": "a shared prefix is read by each sequence attending it and "
                                 "counted each time; kv_bytes_unique counts it once"}
                        if ab["kv_unique"] != ab["kv"] else {})},
        "decode_us": run.decode_us(),
        **({"step_us_own_events": {
            "median": round(statistics.median(per_ev) * 1e3, 2),
            "p20": round(float(np.percentile(per_ev, 20)) * 1e3, 2),
            "p80": round(float(np.percentile(per_ev, 80)) * 1e3, 2),
            "min": round(min(per_ev) * 1e3, 2),
            "note": "each step between its own two events; the events add about 2 us"}}
           if per_ev else {}),
        "as_two_launches_us": {"append": round(statistics.mean(app_ms) * 1e3, 2),
                               "decode": round(statistics.mean(dec2_ms) * 1e3, 2)},
        "e2e": {"value": round(tokens_all * K / (e2e_ms_max / 1e3), 1), "unit": UNIT,
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "mode": e2e_mode},
        "gpu_launches": run.launches_per_step * K,
        "device": {"name": torch.cuda.get_device_name(dev),
                   "sm_count": torch.cuda.get_device_properties(dev).multi_processor_count},
    }
    if not args.no_cpu_baseline:
        line["cpu_baseline"] = oracle_baseline(w, run.pools, args.cpu_budget, args.window)
        if args.config == DEFAULT_CONFIG and world == 1:
            line["cpu_baseline_single_core"] = oracle_baseline(
                w, run.pools, args.cpu_budget / 2, args.window, threads=1)

    # the other configs, one after another, each batch freed before the next
    # is drawn (single-GPU default runs only)
    others = {}
    if args.configs == "all" and world == 1 and args.config == DEFAULT_CONFIG and not args.window:
        del run, w, out
        gc.collect()
        torch.cuda.synchronize(dev)
        torch.cuda.empty_cache()
        line["gpu_launches_all_configs"] = line["gpu_launches"]
        for name in OTHER_CONFIGS:
            others[name] = measure_other_config(args, name, dev, clocks, peak)
            line["gpu_launches_all_configs"] += others[name]["gpu_launches"]
        # several query rows per (sequence, kv head), decode only: 4 draft
        # tokens on the 7B batch (28 rows) and multi-query attention (32
        # heads on one kv head), both on the tensor-core launch
        multi = {}
        for name, n in MULTIQUERY_RUNS:
            sub = argparse.Namespace(**vars(args))
            sub.config, sub.queries = name, n
            clocks.mark(f"{name}:q{n}:start")
            r = run_multiquery(sub, dev)
            clocks.mark(f"{name}:q{n}:end")
            multi[f"{name}:q{n}"] = {
                "workload": r["config"]["workload"], "queries_per_seq": n,
                "metric": r["metric"], "value": r["value"], "unit": r["unit"],
                "decode_us": r["decode_us"], "split_ctas": r["config"]["split_ctas"],
                "l2": r["config"]["l2"], "launch": r["config"]["launch"],
                "roofline": r["roofline"], "gpu_launches": r["gpu_launches"],
                "clocks_marks": (f"{name}:q{n}:start", f"{name}:q{n}:end")}
            line["gpu_launches_all_configs"] += r["gpu_launches"]
            gc.collect()
            torch.cuda.synchronize(dev)
            torch.cuda.empty_cache()
    line["clocks"] = clocks.stop()
    if others:
        for name, e in others.items():
            start, end = e.pop("clocks_marks")
            e["clocks"] = clocks.summary(start, end, before=start)
        line["configs"] = others
        for name, e in multi.items():
            start, end = e.pop("clocks_marks")
            e["clocks"] = clocks.summary(start, end, before=start)
        line["multiquery"] = multi
    return line


def run_copy_blocks(args, dev):
    """``--op copy_blocks``: pa_copy_blocks forking n_pairs random blocks of a
    pool shaped like the config's (distinct destinations, none a source)."""
    from paged_kv_cache_179_gb300 import _abi
    from paged_kv_cache_179_gb300 import workloads as W

    cfg = W.CONFIGS[args.config]
    Hkv, D = cfg["Hkv"], cfg["D"]
    fp8 = cfg["kv"] == "fp8"
    dtype = torch.uint8 if fp8 else W.TORCH_DTYPE[cfg["kv"]]
    n = args.copy_pairs
    NB = 3 * n
    g = torch.Generator().manual_seed(args.seed)
    k = torch.empty(NB, Hkv, 16, D, dtype=dtype, device=dev)
    v = torch.empty_like(k)
    k.view(torch.uint8).random_(0, 256)
    v.view(torch.uint8).random_(0, 256)
    ks = torch.rand(NB, Hkv, device=dev) if fp8 else None
    vs = torch.rand(NB, Hkv, device=dev) if fp8 else None
    perm = torch.randperm(NB, generator=g)
    pairs = torch.stack([perm[n:2 * n], perm[:n]], dim=1).to(torch.int64).to(dev)
    block_bytes = Hkv * 16 * D * k.element_size()
    moved = 2 * n * (2 * block_bytes + (2 * Hkv * 4 if fp8 else 0))   # read + write, K + V
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        _abi.pa_copy_blocks(k, v, pairs, ks, vs)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
    torch.cuda.synchronize(dev)
    for a, b in ev:
        a.record(stream)
        _abi.pa_copy_blocks(k, v, pairs, ks, vs)
        b.record(stream)
    torch.cuda.synchronize(dev)
    rc, bits = _abi.pa_get_status(dev)
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits}")
    ms = [a.elapsed_time(b) for a, b in ev]
    achieved = moved / (statistics.mean(ms) / 1e3) / 1e9
    peak, peak_kind = measured_peaks()
    return {
        "metric": "pa_copy_blocks: bytes moved (read + write) per second", "impl": "ours",
        "value": round(achieved, 1), "unit": "GB/s", "n_gpus": 1, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(statistics.mean(ms), 5),
        "higher_is_better": True, "dtype": "e4m3" if fp8 else cfg["kv"], "data": "synthetic",
        "config": {"workload": f"{n} block pairs of a {NB}-block pool, {Hkv} kv heads, "
                               f"head_dim {D}, {block_bytes} B per block per pool",
                   "l2": "none: the copy moves more than 3x L2 per call" if moved >= 3 * (129 << 20)
                         else "not flushed"},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "copy_blocks_kernel", "bytes_per_launch": moved,
                     "peak_source": peak_kind},
        "copy_us": {"mean": round(statistics.mean(ms) * 1e3, 2),
                    "median": round(statistics.median(ms) * 1e3, 2),
                    "min": round(min(ms) * 1e3, 2)},
        "gpu_launches": args.steps,
    }


def run_multiquery(args, dev):
    """``--op multiquery``: pa_decode with ``--queries`` n query tokens per
    sequence (the verification pass of speculative decoding: the draft
    tokens' K/V are already in the cache), on the config's batch with a
    seeded [B][n][Hq][D] q.  Every KV block is read once for all n queries."""
    from paged_kv_cache_179_gb300 import _abi
    from paged_kv_cache_179_gb300 import workloads as W
    from paged_kv_cache_179_gb300.step import DecodeStep

    w = W.make_workload(args.config, seed=args.seed, device=dev)
    if w.kv == "fp8":
        raise SystemExit("--op multiquery runs on 16-bit pools")
    n = args.queries
    per_pass = n if n * w.group <= 32 else 32 // w.group   # query tokens per launch pair
    passes = -(-n // per_pass)
    lens = w.context_lens.cpu().numpy()
    g = torch.Generator(device=dev).manual_seed(args.seed + 17)
    q = torch.randn(w.B, n, w.Hq, w.D, generator=g, device=dev).to(w.q.dtype)
    out = torch.empty_like(q)
    ab = algorithmic_bytes(w, lens, args.window)
    moved = ab["kv"] + ab["meta"] + n * ab["q_out"]
    l2 = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 128 << 20)
    # as for the decode step: K/V above 3x L2 runs as is, smaller K/V from
    # cycled copies of the pools (up to 16), else L2 is evicted before each
    # step and each step timed between its own events
    copies = 1 if ab["kv"] >= 3 * l2 else -(-3 * l2 // max(ab["kv"], 1))
    back_to_back = copies <= 16
    copies = copies if back_to_back else 1
    early = args.early_prologue in ("on", "copies") and back_to_back   # as for the decode step
    early_copies = early and args.early_prologue == "copies"   # nothing writes the pools here
    pool_sets = [(w.k_cache, w.v_cache)] + [(w.k_cache.clone(), w.v_cache.clone())
                                           for _ in range(copies - 1)]
    steps = [DecodeStep(k_cache=kc, v_cache=vc, block_tables=w.block_tables,
                        context_lens=w.context_lens, max_context_len=w.max_context_len,
                        scale=w.scale, num_q_heads=w.Hq, split_ctas=args.splits,
                        window=args.window, early_prologue=early, early_copies=early_copies,
                        queries_per_seq=n)
             for kc, vc in pool_sets]
    step = steps[0]
    stream = torch.cuda.current_stream(dev)
    calls = [_abi.prepare(lambda st=st: st.decode(q, out), stream) for st in steps]
    flush_buf = torch.ones(max(2 * l2, 64 << 20) // 4, dtype=torch.int32, device=dev)
    for i in range(max(args.warmup, copies)):
        calls[i % copies]()
    torch.cuda.synchronize(dev)
    if back_to_back:
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for i in range(args.steps):
            calls[i % copies]()
        b.record(stream)
        torch.cuda.synchronize(dev)
        ms = [a.elapsed_time(b) / args.steps] * args.steps
    else:
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(args.steps)]
        for a, b in ev:
            flush_buf.sum(dtype=torch.int64)
            a.record(stream)
            calls[0]()
            b.record(stream)
        torch.cuda.synchronize(dev)
        ms = [a.elapsed_time(b) for a, b in ev]
    rc, bits = _abi.pa_get_status(dev)
    if rc != 0:
        raise RuntimeError(f"device status {rc} bits {bits}")
    t = statistics.mean(ms) / 1e3
    achieved = moved / t / 1e9
    peak, peak_kind = measured_peaks()
    att = int(attended(lens, args.window).sum())
    on_tc = w.D == 128 and per_pass * w.group > 16   # the tensor-core launch serves this pass
    return {
        "metric": "multi-token paged decode: attended (query token, KV token) pairs/s",
        "impl": "ours", "value": round(att * n / t, 1), "unit": "pairs/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t * 1e3, 5),
        "higher_is_better": True, "dtype": w.dtype, "data": "synthetic",
        "config": {"workload": describe(w, att), "queries_per_seq": n,
                   "step": ("pa_decode with n query tokens per sequence (decode and merge "
                            f"launches; {passes} pass(es) of {per_pass} token(s), each reading "
                            "the K/V)"),
                   "split_ctas": step.split_ctas,
                   "l2": (describe_l2("rotate" if copies > 1 else "none", ab["kv"], l2, copies)
                          if back_to_back else describe_l2("read", ab["kv"], l2)),
                   "launch": ("plain launches" if not early else
                              "attention launch with an early prologue"
                              + (" and early K/V copies" if early_copies else "")),
                   **({"window": args.window} if args.window else {})},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "traffic": (load_traffic(f"{args.config}:q{n}", step.split_ctas, tc=on_tc)
                                 if passes == 1 and not args.window else None),
                     "kernel": (("decode_tc_kernel (tcgen05: 17-32 query rows per kv head)"
                                 if on_tc else "decode_kernel (general masks)")
                                + ", then merge_kernel"),
                     "bytes_per_launch": moved, "peak_source": peak_kind},
        "decode_us": {"mean": round(t * 1e6, 2),
                      "timing": ("K decodes back to back between two events" if back_to_back
                                 else "each decode between its own events, L2 evicted")},
        "gpu_launches": 2 * passes * args.steps,
    }


def describe_l2(mode, kv_bytes, l2, copies=1):
    if mode == "rotate":
        return (f"not flushed: the steps cycle over {copies} copies of the pools "
                f"({copies * kv_bytes / 1e6:.0f} MB of K/V vs {l2 / 1e6:.0f} MB L2), so each "
                f"step's K/V is cold; steps back to back")
    if mode == "none":
        return (f"not flushed: inputs larger than L2 ({kv_bytes / 1e6:.0f} MB of K/V per step vs "
                f"{l2 / 1e6:.0f} MB L2), tiles fetched with an L2 evict-first policy")
    if mode == "read":
        return f"flushed before every timed step by reading a {2 * l2 / 1e6:.0f} MB buffer"
    return f"flushed before every timed step by writing a {2 * l2 / 1e6:.0f} MB buffer"


def describe(w, tokens):
    return (f"{w.name}: {w.B} seqs, {w.Hq} q / {w.Hkv} kv heads, head_dim {w.D}, block 16, "
            f"{'E4M3 pool, fp16 q' if w.kv == 'fp8' else w.dtype}, "
            f"{tokens} attended tokens (max {w.max_context_len}), {w.num_blocks}-block pool")


_DECODE_SOURCES = ("decode_kernels.cuh", "decode.cu", "pa_ptx.cuh", "pa_launch.h", "pa_e4m3.cuh")
_TC_SOURCES = _DECODE_SOURCES + ("decode_tc.cu", "pa_tc.cuh")


def kernel_sha(tc: bool = False) -> str:
    """sha256 prefix of the sources of the decode launch (decode_kernel and the
    merge), or with ``tc`` of the tensor-core launch as well."""
    import hashlib
    h = hashlib.sha256()
    for name in (_TC_SOURCES if tc else _DECODE_SOURCES):
        with open(os.path.join(ROOT, "paged_kv_cache_179_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(config, splits, tc: bool = False):
    """DRAM bytes per decode call from the committed ncu summary, when it
    matches this workload, CTA split and kernel source (else null)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            t = json.load(f)
        e = t.get(config)
        if e and e.get("split_ctas") == splits and e.get("kernel_sha") == kernel_sha(tc):
            return e.get("bytes_per_launch")
    except (OSError, ValueError):
        pass
    return None


# ------------------------------------------------------------ reference arm
def run_reference(args):
    import oracle
    from paged_kv_cache_179_gb300 import workloads as W
    w = W.make_workload(args.config, seed=args.seed, device="cpu")
    lens = w.context_lens.numpy()
    att = attended(lens, args.window)
    tables = w.block_tables.numpy()
    q, kp, vp = W.to_numpy16(w.q), W.to_numpy16(w.k_cache), W.to_numpy16(w.v_cache)
    bf16 = w.dtype == "bf16"
    kn, vn = W.to_numpy16(w.k_new), W.to_numpy16(w.v_new)
    slots = w.slot_mapping.numpy()
    if w.kv == "fp8":
        kc, ks = oracle.quantize_fp8(kp)
        vc, vs = oracle.quantize_fp8(vp)
    order = np.random.default_rng(0).permutation(w.B)
    # size each step's sample to about args.ref_step_s seconds of host work
    probe = order[:2]
    t = time.perf_counter()
    if w.kv == "fp8":
        oracle.decode_fp8(q, kc, vc, ks, vs, tables, lens, w.scale, window=args.window,
                          rows=probe)
    else:
        oracle.decode(q, kp, vp, tables, lens, w.scale, bf16=bf16, window=args.window, rows=probe)
    per_tok = max(time.perf_counter() - t, 1e-4) / max(1, int(att[probe].sum()))
    n = max(2, min(w.B, int(args.ref_step_s / per_tok / max(1.0, att.mean()))))
    rows = order[:n]
    sample_tokens = int(att[rows].sum())

    def one_step():
        if w.kv == "fp8":
            oracle.cache_append_fp8(kn, vn, kc, vc, ks, vs, slots, 16)
            oracle.decode_fp8(q, kc, vc, ks, vs, tables, lens, w.scale, window=args.window,
                              rows=rows)
        else:
            oracle.cache_append(kn, vn, kp, vp, slots, 16)
            oracle.decode(q, kp, vp, tables, lens, w.scale, bf16=bf16, window=args.window,
                          rows=rows)

    for _ in range(args.warmup):
        one_step()
    t = time.perf_counter()
    for _ in range(args.steps):
        one_step()
    dt = time.perf_counter() - t
    value = sample_tokens * args.steps / dt
    sample = (f"{n} of {w.B} sequences per step ({sample_tokens} attended tokens, all {w.Hq} "
              f"q heads) + the whole batch's append; fp64 oracle")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 1), "unit": UNIT,
        "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(dt / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": describe(w, int(att.sum())), "step": "oracle append + decode",
                   "seed": args.seed, **({"window": args.window} if args.window else {})},
        "cpu_baseline": {"value": round(value, 1), "unit": UNIT, "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 1), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", default=DEFAULT_CONFIG)
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--splits", type=int, default=0,
                    help="CTAs the batch is divided among (0 = two per SM)")
    ap.add_argument("--l2", choices=["auto", "none", "rotate", "read", "write"], default="auto",
                    help="L2 handling between timed steps (auto: none when the K/V read is "
                         ">= 3x L2; else rotate over copies of the pools, >= 3x L2 together, "
                         "when 16 copies suffice; else evict by reading a 2x-L2 buffer)")
    ap.add_argument("--step", choices=["auto", "fused", "two-launch"], default="auto",
                    help="fused: pa_decode_step (append inside the attention launch); two-launch: "
                         "pa_cache_append + pa_decode; auto: the faster for the pool type "
                         "(fused for 16-bit pools, two-launch for E4M3)")
    ap.add_argument("--op", choices=["step", "copy_blocks", "multiquery"], default="step",
                    help="what to time: the decode step (default), pa_copy_blocks alone, or a "
                         "decode with --queries query tokens per sequence")
    ap.add_argument("--queries", type=int, default=2)
    ap.add_argument("--copy-pairs", type=int, default=8192)
    ap.add_argument("--window", type=int, default=0,
                    help="sliding window in tokens (0: each sequence attends its whole context)")
    ap.add_argument("--early-prologue", choices=["copies", "on", "off"], default="copies",
                    help="steps with PA_DECODE_EARLY_PROLOGUE (on), with PA_DECODE_EARLY_COPIES "
                         "as well (copies), or neither (off): the device-timed steps and the "
                         "pipelined end-to-end run")
    ap.add_argument("--configs", choices=["all", "none"], default="all",
                    help="all: the default single-GPU run also times the other four configs "
                         "(tiny, SmolLM2-360M, Qwen2.5-1.5B, E4M3 Qwen2.5-7B) one after another "
                         "and reports them under 'configs', and two batches with several "
                         "query rows per kv head (4 query tokens on the 7B batch, MQA 32 x 1) "
                         "under 'multiquery'")
    ap.add_argument("--handshake", choices=["auto", "device", "events"], default="auto",
                    help="how the pipelined end-to-end steps order their copies: a device-side "
                         "handshake (auto: when the driver offers stream memory operations) or "
                         "stream events")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--ref-step-s", type=float, default=2.0)
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return 0

    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=dev)
    try:
        if args.op == "copy_blocks":
            line = run_copy_blocks(args, dev)
        elif args.op == "multiquery":
            line = run_multiquery(args, dev)
        else:
            line = run_ours(args, rank, world, dev)
        if rank == 0:
            print(json.dumps(line), flush=True)
    finally:
        if world > 1:
            torch.distributed.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
