#!/usr/bin/env python
"""Benchmark of ragged paged attention (librpa) on one GB300 per rank.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload all]
    python bench.py --impl reference ...      # the CPU oracle as the reference arm

By default every one of the five configurations runs in turn:
  tiny_prefill    1 sequence, 256 queries over 256 keys, 4 q / 1 kv heads, D 64,
                  16-token pages in a permuted pool of 32;
  decode          128 sequences x 1 query, KV lengths uniform in [128, 2048],
                  8 q / 1 kv heads, D 256, 128-token pages from a pool of 4096;
  swa_prefill     one 8192-token prompt, window 1024, 32 q / 16 kv heads, D 256;
  causal_prefill  the same without a window;
  mixed           512 decode sequences (KV uniform in [256, 4096]) and 4
                  chunked prefills of 2048 tokens on a prior of U[0, 4096],
                  8 q / 1 kv heads, D 256, even sequences windowed (1024).
The JSON line's headline is the mixed batch; `workloads` holds every
configuration's record.  `--workload NAME` runs one (its line is then that
workload's), also `decode_fp8` and `spec_decode`.

A step is one rpa_forward over the seeded synthetic batch (every kernel of the
hot path for it: split-KV decode + log-sum-exp combine for decode sequences,
prefill for the rest, side by side on disjoint SMs for a mixed batch), with q,
the KV pages and the metadata resident in HBM and the plan built once for the
batch, as a serving step reuses one plan for every layer.  For inputs smaller
than L2, L2 is flushed before every timed step (a 256 MiB write, then a 256 MiB
read so that the written lines' write-back to HBM falls outside the step) and
each step is bracketed by CUDA events on the launching stream.  When one
step's inputs exceed L2 (the decode batch reads 151 MB, the 8k prefills 403 MB,
the mixed batch 914 MB) the timed steps rotate over R disjoint copies of the
inputs instead: no step finds its data in L2, no flush is needed, and one
event pair brackets the K steps (an event record costs about 2-3 us of device
time on these machines).  `flushed_step_ms` reports the flush-and-event-pair-
per-step time beside it; `--flush` makes it the headline.  The K timed steps
are captured into one CUDA graph and replayed once, as a serving loop replays
its step; `--no-graph` enqueues the same loop from Python instead.

Besides `value` (device-timed query tokens/s) each record carries:
  e2e        the same metric through the public API with host buffers: per step
             one pinned host->device copy of q and the metadata, rpa_plan on the
             host metadata, rpa_forward, and the device->host copy of out (the
             KV pages are the device-resident cache), with its parts;
  roofline   the dominant kernel's algorithmic bytes (or flops) per launch over
             its average launch time, measured with library trace events, and
             its DRAM traffic from the committed ncu summary when that was
             taken on the same device source;
  step_roofline  the whole step's work against the roofline at the measured
             peaks: max(flops / tensor peak, bytes / HBM peak) / step time;
  cpu_baseline  the CPU oracle timed on this host's cores on a bounded sample.
With torchrun (N > 1) every rank runs an independent replica (the path has no
exchange step); the timing is the max over ranks.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "attention tokens/s and % roofline (TFLOP/s prefill, HBM GB/s decode) on 1 GB300"
NOMINAL_TFLOPS = 2250.0   # the roofline constants the metric is quoted against
NOMINAL_GBS = 8000.0
FALLBACK_GBS = 6800.0
FALLBACK_TFLOPS = 1900.0
# The five configurations of the benchmark; the mixed batch (the largest, and
# the one where decode and prefill meet) is the headline of the default run.
ALL_WORKLOADS = ["tiny_prefill", "decode", "swa_prefill", "causal_prefill", "mixed"]
HEADLINE = "mixed"


# ----------------------------------------------------------------- workload


def algorithmic_counts(b, part=None):
    """Visible (query, key) pairs, flops and bytes of one step (part =
    "decode" or "prefill": only the sequences with one query, or with more).

    Pairs: for query i of sequence s at pos = L - q_len + i, keys
    max(0, pos - W + 1) .. pos.  FLOPs = 4 * D * Hq * pairs (QK^T and PV).
    Bytes: each visible KV token of each KV head once (K and V), q read once,
    out written once, plus the page-table entries of visible pages and the
    per-sequence metadata.  Counted from the realised lengths.
    """
    esz = 2 if b.dtype == "bf16" else 4
    kv_esz = 1 if getattr(b, "k_fp8", None) is not None else esz   # e4m3 pages: 1 byte
    hq, hkv, d, p = b.num_q_heads, b.num_kv_heads, b.head_dim, b.page_size
    pairs = kv_tokens = pages = 0
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        if ql == 0 or (part == "decode" and ql != 1) or (part == "prefill" and ql == 1):
            continue
        L = int(b.kv_lens[s])
        w = 0 if b.window is None else int(b.window[s])
        pos = np.arange(L - ql, L, dtype=np.int64)
        lo = np.maximum(0, pos - w + 1) if w > 0 else np.zeros_like(pos)
        pairs += int((pos - lo + 1).sum())
        first = int(lo[0])
        kv_tokens += L - first
        pages += (L - 1) // p - first // p + 1
    flops = 4.0 * d * hq * pairs
    meta = (2 * b.num_seqs + 1 + (b.num_seqs if b.window is not None else 0)) * 4
    nq = sum(int(b.cu_q_lens[s + 1] - b.cu_q_lens[s]) for s in range(b.num_seqs)
             if part is None or (part == "decode") == (b.cu_q_lens[s + 1] - b.cu_q_lens[s] == 1))
    scales = 2 * hkv * 4 if kv_esz == 1 else 0
    byts = (kv_tokens * hkv * d * 2 * kv_esz + 2 * nq * hq * d * esz + pages * 4 + meta + scales)
    return dict(pairs=pairs, kv_tokens=kv_tokens, flops=flops, bytes=float(byts))


def new_token_rows(b, db, torch):
    """Device copies of the step's new K/V rows ([total_q, Hkv, D]): the rows
    the pools already hold at the new tokens' positions, so writing them
    back leaves the cache as it was."""
    P = b.page_size
    idx = np.zeros(b.total_q, dtype=np.int64)
    for s in range(b.num_seqs):
        ql = int(b.cu_q_lens[s + 1] - b.cu_q_lens[s])
        L = int(b.kv_lens[s])
        for i in range(ql):
            pos = L - ql + i
            idx[int(b.cu_q_lens[s]) + i] = int(b.page_table[s, pos // P]) * P + pos % P
    ii = torch.from_numpy(idx).cuda()
    flat_k = db.k_pages.reshape(-1, b.num_kv_heads, b.head_dim)
    flat_v = db.v_pages.reshape(-1, b.num_kv_heads, b.head_dim)
    return flat_k[ii].contiguous(), flat_v[ii].contiguous()


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            pk = json.load(f)
    except (OSError, ValueError):
        return dict(hbm_gbs=FALLBACK_GBS, bf16_tflops=FALLBACK_TFLOPS,
                    bf16_tflops_sustained=1700.0, source="fallback")

    def num(*keys):
        for k in keys:
            v = pk.get(k)
            if isinstance(v, (int, float)):
                return float(v)
            if isinstance(v, dict):
                for kk in ("value", "gbs", "tflops", "median", "max"):
                    if isinstance(v.get(kk), (int, float)):
                        return float(v[kk])
        return None

    hbm = num("hbm_gbs", "hbm_copy_gbs", "hbm")
    tf = num("bf16_tflops", "bf16_tflops_burst")
    tfs = num("bf16_tflops_sustained")
    return dict(hbm_gbs=hbm or FALLBACK_GBS, bf16_tflops=tf or FALLBACK_TFLOPS,
                bf16_tflops_sustained=tfs or tf or 1700.0,
                source="measured" if hbm else "fallback")


# A kernel's device source, and for the persistent kernels the planner whose
# schedule (ranges, item order) decides how often they re-read keys.
KERNEL_SOURCES = {
    "decode_split": ["decode.cu", "decode_sched.cuh", "plan.cpp"],
    "decode_combine": ["decode.cu", "decode_sched.cuh", "plan.cpp"],
    "prefill_tc": ["prefill_tc.cu", "plan.cpp"], "prefill_combine": ["prefill_tc.cu", "plan.cpp"],
    "simt": ["simt.cu"], "kv_write": ["kv_write.cu"], "prologue": ["prologue.cu"],
}


def kernel_source_hash(kernel: str):
    """First 16 hex digits of the SHA-256 of a kernel's sources (KERNEL_SOURCES)
    with comments, blank lines and runs of white space removed (so edits of
    comments alone keep it), together with the device headers every kernel
    includes."""
    names = KERNEL_SOURCES.get(kernel)
    if names is None:
        return None
    csrc = os.path.join(ROOT, "ragged_paged_attention_rpa_gb300", "csrc")
    h = hashlib.sha256()
    for fn in names + ["common.cuh", "sm100_ptx.cuh"]:
        text = open(os.path.join(csrc, fn)).read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        text = "\n".join(" ".join(ln.split()) for ln in text.splitlines() if ln.strip())
        h.update(fn.encode() + b"\0" + text.encode() + b"\0")
    return h.hexdigest()[:16]


def profile_traffic(kernel: str, workload):
    """DRAM bytes per launch from a committed ncu summary
    (profiles/<kernel>.<workload>.txt), or None when absent or taken on a
    different version of the kernel's device source."""
    if workload is None:
        return None
    path = os.path.join(ROOT, "profiles", "%s.%s.txt" % (kernel, workload))
    try:
        lines = open(path).read().splitlines()
    except OSError:
        return None
    kv = {}
    for ln in lines:
        if ":" in ln and not ln.startswith(" "):
            k, v = ln.split(":", 1)
            kv[k.strip()] = v.strip()
    if kv.get("source_sha256_16") != kernel_source_hash(kernel):
        return None
    try:
        return float(kv["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples (SM clock, max clock, throttle reasons) while running."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def _read(self):
        for ln in self.proc.stdout:
            self.lines.append(ln.strip())

    def __exit__(self, *exc):
        time.sleep(0.25)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for row in csv.reader(io.StringIO("\n".join(self.lines))):
            if len(row) < 7:
                continue
            try:
                sm.append(float(row[0]))
                mx.append(float(row[1]))
            except ValueError:
                continue
            for name, val in zip(names, row[3:7]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ----------------------------------------------------------------- CPU oracle


def oracle_sample_rows(b, n_tokens, start=0):
    """Rows (all heads) of n_tokens query tokens, cycling through the batch."""
    toks = (start + np.arange(n_tokens)) % b.total_q
    return (toks[:, None] * b.num_q_heads + np.arange(b.num_q_heads)[None, :]).reshape(-1)


def cpu_oracle_rate(b, seconds: float, threads: int):
    """Query tokens/s of the CPU oracle (fp32) on this host: whole query tokens
    (every head) taken round-robin from the batch until `seconds` have passed."""
    import oracle
    oracle.build()
    done = 0
    t0 = time.perf_counter()
    chunk = max(1, min(b.total_q, 64))
    while True:
        rows = oracle_sample_rows(b, chunk, done)
        oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens, b.kv_lens,
                         b.window, b.sm_scale, rows=rows, precision=32, threads=threads)
        done += chunk
        el = time.perf_counter() - t0
        if el >= seconds:
            return done / el, done, el


# ----------------------------------------------------------------- main


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["rpa", "reference"], default="rpa")
    ap.add_argument("--workload", default="all",
                    choices=["all"] + ALL_WORKLOADS + ["decode_fp8", "spec_decode"],
                    help="'all' (default): the five configurations, the mixed batch as the "
                         "headline, every one under `workloads`")
    ap.add_argument("--seed", type=int, default=None)
    ap.add_argument("--cpu-seconds", type=float, default=None,
                    help="CPU-oracle sample length per workload (default 10 s for one "
                         "workload, 4 s each for all)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--e2e-steps", type=int, default=100)
    ap.add_argument("--q-block", type=int, default=int(os.environ.get("RPA_QBLOCK", "0")),
                    help="prefill query block in tokens (default: $RPA_QBLOCK, else chosen)")
    ap.add_argument("--kv-split", type=int, default=int(os.environ.get("RPA_KV_SPLIT", "0")),
                    help="decode range length in tokens (default: $RPA_KV_SPLIT, else chosen)")
    ap.add_argument("--prefill-split", type=int, default=0,
                    help="plan option: 0 choose, -1 never split prefill items, n > 0 parts "
                         "of at most n key tiles")
    ap.add_argument("--decode-sms", type=int, default=0,
                    help="plan option for mixed batches: 0 choose, -1 run decode and prefill "
                         "one after the other, n > 0 decode on n SMs beside the prefill")
    ap.add_argument("--prefill-dynamic", type=int, default=0,
                    help="plan option: 0 prefill CTAs take items as they get free, -1 each "
                         "CTA runs the planner's list")
    ap.add_argument("--prefill-grouping", type=int, default=0,
                    help="plan option: 0 group the prefill list by (sequence, KV head) when "
                         "its K and V outgrow L2, -1 longest first over the whole batch")
    ap.add_argument("--decode-kernel", type=int, default=0,
                    help="plan option: 0 choose, 1 CUDA-core decode kernel, 2 tensor-core "
                         "decode kernel")
    ap.add_argument("--flush", action="store_true",
                    help="flush L2 before every step and time each step with its own "
                         "event pair, even when a step's inputs exceed L2")
    ap.add_argument("--no-graph", action="store_true",
                    help="enqueue the timed steps from Python instead of replaying them "
                         "from a CUDA graph")
    ap.add_argument("--qkv-prologue", action="store_true",
                    help="time rpa_forward_qkv: q/k RMS norm + rotary embedding, v norm and "
                         "the KV write of the new tokens, then attention")
    ap.add_argument("--kv-write", action="store_true",
                    help="time rpa_forward_kv: write the step's new K/V rows into their "
                         "pages, then attend")
    return ap.parse_args()


def make_workload(args, name):
    from ragged_paged_attention_rpa_gb300 import workloads
    fn = workloads.WORKLOADS[name]
    return fn() if args.seed is None else fn(seed=args.seed)


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    pg = None
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo")
        pg = dist
    return world, rank, local, pg


def max_over_ranks(x: float, dist) -> float:
    """The largest value of x over the ranks (x itself without a process group)."""
    if dist is None:
        return float(x)
    import torch
    t = torch.tensor([float(x)], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_value(world: int, tokens: int, steps: int, total_ms: float) -> float:
    """Whole-job query tokens/s: every rank processes `tokens` per step, the
    job takes the slowest rank's time."""
    return world * tokens * steps / (total_ms / 1e3)


def rotation_copies(nbytes: float, l2_bytes: int, flush: bool) -> int:
    """Input copies the timed steps rotate over (0: one copy, L2 flushed
    before every step): when a step reads more than L2, enough copies that a
    step's data were last touched more than 3 x L2 bytes earlier."""
    if flush or nbytes < l2_bytes:
        return 0
    return max(2, math.ceil(3 * l2_bytes / nbytes))


def workload_config(b, counts, l2_bytes, world, flush=False):
    """The `config` object of a workload's line (the same in both arms)."""
    R = rotation_copies(counts["bytes"], l2_bytes, flush)
    l2 = ("no flush: one step reads %.0f MB (> %.0f MB of L2) and the steps rotate over %d "
          "disjoint copies of the inputs (KV pools, page tables, q, out), so a step's data "
          "were last touched %.0f MB earlier; one event pair around the K steps"
          % (counts["bytes"] / 1e6, l2_bytes / 1e6, R, (R - 1) * counts["bytes"] / 1e6)) if R \
        else ("flushed before every timed step (256 MiB write, then a 256 MiB read that "
              "evicts the dirty lines); an event pair around every step")
    return {"workload": b.name, "seed": b.seed, "l2": l2,
            "parallelism": "replicas" if world > 1 else "single GPU"}


def l2_size(torch=None, local=0):
    try:
        if torch is not None and torch.cuda.is_available():
            v = int(getattr(torch.cuda.get_device_properties(local), "L2_cache_size", 0))
            if v:
                return v
    except Exception:  # noqa: BLE001 - a description only
        pass
    return 126 << 20


def run_reference(args, names, world, rank):
    """The reference arm: the CPU oracle, as it stands, on this host's cores.
    Each step runs a bounded sample of the workload: 64 query tokens (every
    head), taken round-robin, the chunking of the cpu_baseline leg, so the
    oracle's threads have work on every core."""
    if rank != 0:
        return
    import oracle
    oracle.build()
    try:
        import torch
    except ImportError:  # pragma: no cover
        torch = None
    cores = len(os.sched_getaffinity(0))
    recs = {}
    for name in names:
        b = make_workload(args, name)
        counts = algorithmic_counts(b)
        per_step = min(b.total_q, 64)
        for w in range(args.warmup):
            rows = oracle_sample_rows(b, per_step, w * per_step)
            oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens, b.kv_lens,
                             b.window, b.sm_scale, rows=rows, precision=32, threads=cores)
        t0 = time.perf_counter()
        for k in range(args.steps):
            rows = oracle_sample_rows(b, per_step, (args.warmup + k) * per_step)
            oracle.attention(b.q, b.k_pages, b.v_pages, b.page_table, b.cu_q_lens, b.kv_lens,
                             b.window, b.sm_scale, rows=rows, precision=32, threads=cores)
        el = time.perf_counter() - t0
        value = args.steps * per_step / el
        sample = ("%d query tokens per step (all %d heads: %d output rows) of the %s batch, "
                  "round-robin, %d steps" % (per_step, b.num_q_heads, per_step * b.num_q_heads,
                                             b.name, args.steps))
        recs[name] = {
            "value": value, "unit": "tokens/s", "ms_per_step": 1e3 * el / args.steps,
            "config": workload_config(b, counts, l2_size(torch), world, args.flush),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores,
                             "kind": "oracle", "sample": sample},
        }
    head = HEADLINE if HEADLINE in recs else names[0]
    r = recs[head]
    line = {
        "impl": "reference", "metric": METRIC, "value": r["value"], "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": r["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": r["config"], "cpu_baseline": r["cpu_baseline"],
        "e2e": {"value": r["value"], "unit": "tokens/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "oracle": "C++ CPU oracle (plain definition, fp32 accumulation, OpenMP over output "
                  "rows)",
    }
    if len(recs) > 1:
        line["workloads"] = recs
    print(json.dumps(line), flush=True)


def bench_one(args, name, world, rank, local, dist, binding, torch, peaks, l2_bytes):
    """Time one workload; returns its record (the fields of a bench line)."""
    b = make_workload(args, name)
    counts = algorithmic_counts(b)
    db = binding.Batch(b)
    fp8 = b.k_fp8 is not None
    plan_kw = dict(q_block=args.q_block, kv_split=args.kv_split,
                   kv_dtype=binding.RPA_DTYPE_FP8_E4M3 if fp8 else 0,
                   prefill_split=args.prefill_split, decode_sms=args.decode_sms,
                   decode_kernel=0 if fp8 else args.decode_kernel,
                   prefill_dynamic=args.prefill_dynamic,
                   prefill_grouping=args.prefill_grouping)
    plan = db.plan(**plan_kw)
    info = plan.info()
    ws = binding.alloc_workspace(plan)
    fp8_dev = ([torch.from_numpy(x).cuda() for x in (b.k_fp8, b.v_fp8, b.k_scale, b.v_scale)]
               if fp8 else None)
    kv_new = None if not args.kv_write else new_token_rows(b, db, torch)
    qkv = None
    if args.qkv_prologue:
        # The projection's q, k, v rows of the step (seeded N(0, 1)), norm
        # weights near 1 and a rotary base of 10^4: the step runs the q/k/v
        # prologue (norms, rotary embedding, KV write) before attention.
        g = torch.Generator(device="cpu").manual_seed(1234)
        D = b.head_dim
        raw0 = tuple(torch.randn(b.total_q, h, D, generator=g).to(torch.bfloat16).cuda()
                     for h in (b.num_q_heads, b.num_kv_heads, b.num_kv_heads))
        qkv = dict(
            raw=[raw0] + [tuple(x.clone() for x in raw0) for _ in range(2)],
            w=[(0.5 + torch.rand(D, generator=g)).cuda() for _ in range(3)])
        qkv["norm"] = binding.qkv_norm(*qkv["w"], eps=1e-6, rope_theta=10000.0)

    # Step inputs.  When one step's inputs exceed L2, the timed steps rotate
    # over R disjoint copies of them (KV pools stacked R times with the page
    # table shifted by r * num_pages, q and out per copy): the data a step
    # reads were last touched R - 1 steps (more than 3 x L2 bytes) earlier,
    # so no L2 flush is needed and one event pair brackets all K steps.
    # Otherwise (or with --flush) there is one copy and L2 is flushed before
    # every step, each step bracketed by its own event pair.
    R = rotation_copies(counts["bytes"], l2_bytes, args.flush)
    N = b.num_pages
    if R:
        rplan = binding.rpa_plan(b.cu_q_lens, b.kv_lens, b.window, b.num_q_heads,
                                 b.num_kv_heads, b.head_dim, b.page_size,
                                 b.max_pages_per_seq, R * N, dtype=db.dtype, **plan_kw)
        pools = [torch.cat([x] * R) for x in
                 ((fp8_dev[0], fp8_dev[1]) if fp8 else (db.k_pages, db.v_pages))]
        copies = [dict(q=db.q if r == 0 else db.q.clone(),
                       out=db.out if r == 0 else torch.empty_like(db.out),
                       pt=torch.where(db.page_table >= 0, db.page_table + r * N,
                                      db.page_table).contiguous())
                  for r in range(R)]
    else:
        rplan, pools = plan, ((fp8_dev[0], fp8_dev[1]) if fp8 else (db.k_pages, db.v_pages))
        copies = [dict(q=db.q, out=db.out, pt=db.page_table)]

    def make_call(r=0):
        # Copy r's call object, bound to the current stream (inside a graph
        # capture: the capture stream).
        c = copies[r]
        if qkv is not None:
            qr, kr, vr = qkv["raw"][r % 3]
            return binding.ForwardQkvCall(qr, kr, vr, qkv["norm"], c["q"], pools[0], pools[1],
                                          c["pt"], db.cu_q_lens, db.kv_lens, db.window,
                                          b.sm_scale, c["out"], rplan, ws)
        if kv_new is not None:
            return binding.ForwardKvCall(c["q"], kv_new[0], kv_new[1], pools[0], pools[1],
                                         c["pt"], db.cu_q_lens, db.kv_lens, db.window,
                                         b.sm_scale, c["out"], rplan, ws)
        if fp8:
            return binding.ForwardFp8Call(c["q"], pools[0], pools[1], fp8_dev[2], fp8_dev[3],
                                          c["pt"], db.cu_q_lens, db.kv_lens, db.window,
                                          b.sm_scale, c["out"], rplan, ws)
        return binding.ForwardCall(c["q"], pools[0], pools[1], c["pt"], db.cu_q_lens,
                                   db.kv_lens, db.window, b.sm_scale, c["out"], rplan, ws)

    flush = torch.empty(256 << 20, dtype=torch.uint8, device="cuda")
    evict = torch.ones(32 << 20, dtype=torch.int64, device="cuda")   # 256 MiB
    stream = torch.cuda.current_stream()
    flushes = [0]

    def flush_l2():
        # A 256 MiB write evicts the step's inputs from L2; a 256 MiB read
        # then evicts the written (dirty) lines, so their write-back to HBM
        # happens here and not inside the next timed step.
        flushes[0] += 1
        flush.fill_(flushes[0] & 0x7F)
        evict.sum()

    def capture(n, events=None, flushed=False):
        # A CUDA graph of n steps (copies in rotation; with `flushed`, an L2
        # flush before each; with `events`, event pair k around step k).
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, capture_error_mode="thread_local"):
            calls = [make_call(r) for r in range(len(copies))]
            for k in range(n):
                if flushed:
                    flush_l2()
                if events is not None:
                    events[k][0].record()
                calls[k % len(calls)]()
                if events is not None:
                    events[k][1].record()
        return g

    # Warm-up (untimed): eager, then from a graph.
    calls = [make_call(r) for r in range(len(copies))]
    for k in range(max(3, args.warmup)):
        if not R:
            flush_l2()
        calls[k % len(calls)]()
    torch.cuda.synchronize()
    if binding.rpa_get_device_error(ws) != 0:
        raise SystemExit("%s: device error word set during warm-up" % name)

    K = args.steps
    use_graph = not args.no_graph
    gpu_index = int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local)).split(",")[0]) \
        if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local

    def timed_per_step_events(n, flushed):
        # n steps, each bracketed by its own event pair (graph or stream).
        evs = [(torch.cuda.Event(enable_timing=True, external=use_graph),
                torch.cuda.Event(enable_timing=True, external=use_graph)) for _ in range(n)]
        g = capture(n, evs, flushed) if use_graph else None
        if g is not None:
            capture(max(3, args.warmup), None, flushed).replay()
        torch.cuda.synchronize()
        return evs, g

    if R:
        graph = capture(K) if use_graph else None
        if graph is not None:
            capture(max(3, args.warmup)).replay()
        e_start = torch.cuda.Event(enable_timing=True)
        e_stop = torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
    else:
        ev, graph = timed_per_step_events(K, flushed=True)
    with ClockSampler(gpu_index) as clocks:
        if dist is not None:
            dist.barrier()
        torch.cuda.synchronize()
        if R:
            # The device sleeps while the host enqueues the steps, so the
            # timed region opens on queued work, not on host launch latency.
            torch.cuda._sleep(int(2e6))
            e_start.record(stream)
            if graph is not None:
                graph.replay()
            else:
                for k in range(K):
                    calls[k % R]()
            e_stop.record(stream)
        elif graph is not None:
            graph.replay()
        else:
            torch.cuda._sleep(int(2e6))
            for k in range(K):
                flush_l2()
                ev[k][0].record(stream)
                calls[0]()
                ev[k][1].record(stream)
        torch.cuda.synchronize()
        if dist is not None:
            dist.barrier()
    if R:
        total_ms = e_start.elapsed_time(e_stop)
        step_ms = None
    else:
        step_ms = [a.elapsed_time(e) for a, e in ev]
        total_ms = float(sum(step_ms))
    total_ms = max_over_ranks(total_ms, dist)
    if binding.rpa_get_device_error(ws) != 0:
        raise SystemExit("%s: device error word set during the timed region" % name)
    if R:
        for c in copies[1:]:
            if not torch.equal(c["out"].view(torch.int16), copies[0]["out"].view(torch.int16)):
                raise SystemExit("%s: input copies gave different outputs" % name)
    del graph

    # For comparison (not the headline): L2 flushed and an event pair around
    # every step.
    flushed_ms = None
    if R and rank == 0:
        nf = min(K, 100)
        evf, gf = timed_per_step_events(nf, flushed=True)
        torch.cuda.synchronize()
        if gf is not None:
            gf.replay()
        else:
            for k in range(nf):
                flush_l2()
                evf[k][0].record(stream)
                calls[k % R]()
                evf[k][1].record(stream)
        torch.cuda.synchronize()
        flushed_ms = statistics.mean(a.elapsed_time(e) for a, e in evf)
        del gf

    # Kernel durations from the library's trace events (a separate pass of the
    # same loop, so the events do not touch the headline timing).  Each
    # kernel's time runs from the previous mark on its own stream.
    n_trace = min(K, 100)
    binding.rpa_trace_begin(8 * n_trace)
    if use_graph:
        gt = capture(n_trace, None, flushed=not R)
        gt.replay()
    else:
        torch.cuda._sleep(int(2e6))
        for k in range(n_trace):
            if not R:
                flush_l2()
            calls[k % len(calls)]()
    torch.cuda.synchronize()
    recs = binding.rpa_trace_end(8 * n_trace)
    per_kernel = {}
    for kname, ms in recs:
        per_kernel.setdefault(kname, []).append(ms)
    launches_per_step = len(recs) / n_trace
    kernels = {k: {"launches_per_step": len(v) / n_trace, "avg_us": 1e3 * statistics.mean(v)}
               for k, v in per_kernel.items()}

    # End to end through the public API with host buffers.
    e2e = run_e2e(args, b, db, plan_kw, flush_l2, binding, torch,
                  fp8_dev if b.k_fp8 is not None else None)

    tokens = b.total_q
    ms_per_step = total_ms / K
    value = job_value(world, tokens, K, total_ms)
    dom = max(kernels, key=lambda k: kernels[k]["avg_us"] * kernels[k]["launches_per_step"])
    dom_us = kernels[dom]["avg_us"]
    # The dominant kernel's own work: the decode sequences' bytes for the
    # decode kernel, the prefill sequences' FLOPs for the prefill kernel.
    if dom == "decode_split":
        dom_counts, decode_heavy = algorithmic_counts(b, "decode"), True
    elif dom == "prefill_tc":
        dom_counts, decode_heavy = algorithmic_counts(b, "prefill"), False
    else:
        dom_counts, decode_heavy = counts, info["num_prefill_seqs"] == 0
    # The bound follows the kernel's arithmetic intensity against the ridge
    # point of the peaks (multi-token decode runs on the tensor-core kernel
    # but stays HBM-bound).
    if not decode_heavy and dom_counts["bytes"] > 0:
        ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
        decode_heavy = dom_counts["flops"] / dom_counts["bytes"] < ridge
    if decode_heavy:
        achieved = dom_counts["bytes"] / (dom_us * 1e-6) / 1e9
        peak = peaks["hbm_gbs"]
        roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
                "frac": achieved / peak}
    else:
        achieved = dom_counts["flops"] / (dom_us * 1e-6) / 1e12
        peak = peaks["bf16_tflops"]
        roof = {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                "frac": achieved / peak}
    roof["kernel"] = dom
    roof["kernel_us"] = dom_us
    if info.get("decode_sms", 0) > 0 and dom in ("decode_split", "prefill_tc"):
        # A mixed batch's grids run side by side: the kernel had only its
        # share of the SMs; its fraction of that share of the peak beside.
        sms = info["decode_sms"] if dom == "decode_split" else info["prefill_sms"]
        share = sms / float(info["decode_sms"] + info["prefill_sms"])
        roof["sm_share"] = share
        roof["frac_of_sm_share"] = roof["frac"] / share
    roof["peak_source"] = "of %s (%s)" % (peaks["source"], "MEASURED_PEAKS.json"
                                          if peaks["source"] == "measured" else
                                          "6.8 TB/s, 1.9 PFLOP/s")
    roof["traffic"] = profile_traffic(dom, name if not (args.kv_write or args.qkv_prologue)
                                      else None)
    step_s = ms_per_step / 1e3
    # The whole step against the roofline of all its work at the measured
    # peaks: max(FLOPs / tensor peak, bytes / HBM peak) over the step time.
    t_roof = max(counts["flops"] / (peaks["bf16_tflops"] * 1e12),
                 counts["bytes"] / (peaks["hbm_gbs"] * 1e9))
    step_roof = {"roofline_us": 1e6 * t_roof, "step_us": 1e6 * step_s, "frac": t_roof / step_s,
                 "bound": "tensor" if counts["flops"] / (peaks["bf16_tflops"] * 1e12) >
                 counts["bytes"] / (peaks["hbm_gbs"] * 1e9) else "hbm"}
    nominal_frac = max(counts["flops"] / (NOMINAL_TFLOPS * 1e12),
                       counts["bytes"] / (NOMINAL_GBS * 1e9)) / step_s

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cores = len(os.sched_getaffinity(0))
        secs = args.cpu_seconds if args.cpu_seconds is not None else \
            (10.0 if args.workload != "all" else 4.0)
        rate, n_tok, el = cpu_oracle_rate(b, secs, cores)
        cpu = {"value": rate, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": "%d query tokens (all %d heads) of the %s batch, 64 per call, "
                         "round-robin, %.1f s" % (n_tok, b.num_q_heads, b.name, el)}

    config = workload_config(b, counts, l2_bytes, world, args.flush)
    method = {
        "launch": "stream (Python loop behind a GPU sleep)" if args.no_graph else
                  "CUDA graph of the K timed steps, replayed once",
        "step": "rpa_forward_qkv (q/k RMS norm + rotary embedding, v norm, KV "
                "write of the new tokens, then attention)" if args.qkv_prologue else
                "rpa_forward_kv (KV-cache write of the new tokens, then attention)"
                if args.kv_write else ("rpa_forward_fp8kv" if fp8 else "rpa_forward"),
        "kv_pages": "e4m3 bytes + fp32 scale per KV head (f16 products, fp32 "
                    "accumulation)" if fp8 else "bf16",
    }
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_per_step,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16" if b.dtype == "bf16" else "f32", "data": "synthetic",
        "config": config,
        "method": method,
        "plan": info,
        "achieved_gbs": counts["bytes"] / step_s / 1e9,
        "achieved_tflops": counts["flops"] / step_s / 1e12,
        "roofline_frac_nominal": nominal_frac,
        "algorithmic": counts,
        "kernels": kernels,
        "roofline": roof,
        "step_roofline": step_roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": int(round(launches_per_step * K)),
        "clocks": clocks.summary(),
        "step_ms_p50": statistics.median(step_ms) if step_ms else None,
        "step_ms_min": min(step_ms) if step_ms else None,
        "flushed_step_ms": flushed_ms,
    }


def main():
    args = parse()
    world, rank, local, dist = dist_setup()
    names = ALL_WORKLOADS if args.workload == "all" else [args.workload]
    if args.impl == "reference":
        run_reference(args, names, world, rank)
        if dist is not None:
            dist.destroy_process_group()
        return

    import torch
    from ragged_paged_attention_rpa_gb300 import binding, build

    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU")
    torch.cuda.set_device(local)
    # Rank 0 builds (a no-op when librpa.so is current); the other ranks wait,
    # so concurrent compilers never write the same object files.
    if rank == 0:
        build.build()
    if dist is not None:
        dist.barrier()
    build.build()
    peaks = load_peaks()
    l2_bytes = l2_size(torch, local)
    recs = {}
    for name in names:
        recs[name] = bench_one(args, name, world, rank, local, dist, binding, torch, peaks,
                               l2_bytes)
        torch.cuda.empty_cache()
    head = HEADLINE if HEADLINE in recs else names[0]
    line = dict(recs[head])
    if len(recs) > 1:
        # Every configuration: its own step time, throughput, dominant
        # kernel's roofline (with the ncu traffic where a summary exists), the
        # whole step's roofline fraction, the CPU oracle and e2e.
        keep = ("value", "unit", "ms_per_step", "config", "method", "plan", "achieved_gbs",
                "achieved_tflops", "algorithmic", "kernels", "roofline", "step_roofline",
                "cpu_baseline", "e2e", "gpu_launches", "clocks", "flushed_step_ms",
                "step_ms_p50")
        line["workloads"] = {n: {k: r[k] for k in keep} for n, r in recs.items()}
        line["gpu_launches_all_workloads"] = sum(r["gpu_launches"] for r in recs.values())
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def run_e2e(args, b, db, plan_kw, flush_l2, binding, torch, fp8_dev=None):
    """End to end through the public API with host buffers, per step: one
    pinned host->device copy of q and the metadata (packed into one buffer),
    rpa_plan on the host metadata, rpa_forward, and the device->host copy of
    out; events around the whole step and between its parts."""
    stream = torch.cuda.current_stream()
    parts = [np.ascontiguousarray(b.q).view(np.uint8).reshape(-1)]
    meta = [b.page_table, b.cu_q_lens, b.kv_lens] + ([b.window] if b.window is not None else [])
    parts += [np.ascontiguousarray(x, dtype=np.int32).view(np.uint8).reshape(-1) for x in meta]
    offs, off = [], 0
    for p in parts:
        offs.append(off)
        off += (p.size + 255) // 256 * 256
    host = torch.zeros(off, dtype=torch.uint8).pin_memory()
    hv = host.numpy()
    for p, o in zip(parts, offs):
        hv[o:o + p.size] = p
    dev = torch.empty(off, dtype=torch.uint8, device="cuda")
    qdt = torch.bfloat16 if b.dtype == "bf16" else torch.float32
    dq = dev[offs[0]:offs[0] + parts[0].size].view(qdt).view(tuple(b.q.shape))
    dmeta = [dev[o:o + p.size].view(torch.int32).view(tuple(np.shape(m)))
             for o, p, m in zip(offs[1:], parts[1:], meta)]
    win_d = dmeta[3] if b.window is not None else None
    hout = torch.empty(tuple(db.out.shape), dtype=db.out.dtype).pin_memory()
    plan0 = binding.rpa_plan(b.cu_q_lens, b.kv_lens, b.window, b.num_q_heads, b.num_kv_heads,
                             b.head_dim, b.page_size, b.max_pages_per_seq, b.num_pages,
                             dtype=db.dtype, **plan_kw)
    ws = binding.alloc_workspace(plan0)
    if fp8_dev:
        call = binding.ForwardFp8Call(dq, fp8_dev[0], fp8_dev[1], fp8_dev[2], fp8_dev[3],
                                      dmeta[0], dmeta[1], dmeta[2], win_d, b.sm_scale, db.out,
                                      plan0, ws)
    else:
        call = binding.ForwardCall(dq, db.k_pages, db.v_pages, dmeta[0], dmeta[1], dmeta[2],
                                   win_d, b.sm_scale, db.out, plan0, ws)
    h2d = int(sum(p.size for p in parts))
    d2h = hout.numel() * hout.element_size()
    n = args.e2e_steps
    t_all, t_h2d, t_fwd, t_d2h, t_plan = [], [], [], [], []
    for k in range(n + 3):
        flush_l2()
        torch.cuda.synchronize()
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(4)]
        ev[0].record(stream)
        dev.copy_(host, non_blocking=True)
        ev[1].record(stream)
        t0 = time.perf_counter()
        plan = binding.rpa_plan(b.cu_q_lens, b.kv_lens, b.window, b.num_q_heads,
                                b.num_kv_heads, b.head_dim, b.page_size,
                                b.max_pages_per_seq, b.num_pages, dtype=db.dtype, **plan_kw)
        t1 = time.perf_counter()
        if plan.workspace_bytes > ws.numel():
            raise RuntimeError("workspace too small for the per-step plan")
        call(plan)
        ev[2].record(stream)
        hout.copy_(db.out, non_blocking=True)
        ev[3].record(stream)
        torch.cuda.synchronize()
        if k >= 3:
            t_all.append(ev[0].elapsed_time(ev[3]))
            t_h2d.append(ev[0].elapsed_time(ev[1]))
            t_fwd.append(ev[1].elapsed_time(ev[2]))
            t_d2h.append(ev[2].elapsed_time(ev[3]))
            t_plan.append(1e3 * (t1 - t0))
    ms = statistics.mean(t_all)
    return {"value": b.total_q / (ms / 1e3), "unit": "tokens/s", "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "breakdown_ms": {"h2d": statistics.mean(t_h2d),
                             "plan_host": statistics.mean(t_plan),
                             "plan_and_forward": statistics.mean(t_fwd),
                             "d2h": statistics.mean(t_d2h)},
            "includes": "one pinned H2D copy of q + metadata, rpa_plan (host, per step), "
                        "rpa_forward, D2H of out; plan_and_forward is the device time from "
                        "the end of the H2D copy to the end of the attention, which holds "
                        "the host's rpa_plan time when that exceeds the copy"}


if __name__ == "__main__":
    main()
