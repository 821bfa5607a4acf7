"""Benchmark: masked varlen attention forward on GB300, one JSON line.

Step = one pass of the whole path over one batch: the range-table fill
(``fill_query_ranges``) and the attention forward (``attn_fwd_varlen``) on the
chunked-prefill workload (8 requests, each a 2048-token chunk after a context
of 0..30000 tokens, 16 q / 8 KV heads, D 256, causal 4096-token window OR-ed
with 1..64 bidirectional ranges per request), inputs resident in HBM, L2
flushed (256 MiB write) between steps.

value  = effective TFLOP/s over unmasked score entries:
         4 * D * Hq * (exact number of visible (query, key) pairs) / step time.
e2e    = the same metric through the public API from pinned HOST tensors, the
         host->device input copies and device->host output copy inside the
         timed region.
roofline: the attention kernel's algorithmic FLOPs per launch / its average
         CUDA-event duration, against the measured bf16 tensor peak.
configs: every other workload of the benchmark set measured in the same run
         (the mm_prefix sliding layer, the D 512 global layer, both mixed
         serving batches with their decode and prefill sub-batches and the
         mixed roofline, the tiny windowed batch) and the range fill at a
         stress size against the HBM roofline.
cpu_baseline: the float64 CPU oracle on a bounded sample of query rows of
         the headline workload, on this host's cores.

``--impl reference`` times that oracle (the only reference implementation
that exists for this path) on the same metric.  Multi-GPU (torchrun): every
rank runs its own replica of the workload on its own GPU (no collective on
the data path); value = all ranks' FLOPs / max-over-ranks time.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import multiprocessing as mp
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "unmasked-attention TFLOP/s (bf16) & % tensor peak; prefill tokens/s"
WORKLOAD = "chunked_prefill_ranges"
WORKLOAD_DESCS = {
    "tiny_window_sinks": ("tiny windowed attention: lengths 37 and 5, ctx 0, 4 q / 2 KV heads, D 64, bf16 N(0,1), "
                          "non-causal symmetric window 8, key-0-bias sinks"),
    "mm_prefix_sliding": ("mm_prefix sliding layer: 4 x 4096-token prefill, ctx 0, 16 q / 8 KV heads, D 256, bf16 "
                          "N(0,1), causal 1024-token window OR 8 bidirectional 256-token ranges per request "
                          "(range table filled on the GPU each step)"),
    "global_causal_d512": ("global layer: 2 x 8192-token prefill, ctx 0, 8 q / 2 KV heads, D 512, bf16 N(0,1), "
                           "pure causal, no ranges, no sinks"),
    "chunked_prefill_ranges": ("chunked prefill with context offset: 8 requests x 2048-token chunk after a context "
                               "U{0..30000}, 16 q / 8 KV heads, D 256, bf16 N(0,1), causal 4096-token window OR "
                               "1-64 bidirectional ranges per request (64-320 tokens, some degenerate, some clipped "
                               "at the chunk) (range table filled on the GPU each step)"),
    "mixed_serving_a": ("mixed serving batch, full-causal layer: 256 decode rows (ctx U{1024..32768}) + 4 prefill "
                        "chunks of 1024 after ctx U{0..16384}, 32 q / 8 KV heads, D 128, bf16 N(0,1), null-logit "
                        "sinks"),
    "mixed_serving_b": ("mixed serving batch, 4096-window layer: 256 decode rows (ctx U{1024..32768}) + 4 prefill "
                        "chunks of 1024 after ctx U{0..16384}, 32 q / 8 KV heads, D 128, bf16 N(0,1), null-logit "
                        "sinks"),
}
WORKLOAD_DESC = WORKLOAD_DESCS[WORKLOAD]
CONFIG_NUMBER = {"tiny_window_sinks": "1", "mm_prefix_sliding": "2", "global_causal_d512": "3",
                 "chunked_prefill_ranges": "4", "mixed_serving_a": "5a", "mixed_serving_b": "5b"}
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
L2_FLUSH_BYTES = 256 << 20


# ----------------------------------------------------------------- helpers
def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def visible_counts_per_row(w, table):
    """Exact visible-key count of every packed query row, from the two closed
    intervals of the mask rule (causal/window base, window-clamped range).
    Measurement accounting only; tests pin it against the oracle's dense mask."""
    cu_q, cu_k = w.cu_seqlens()
    counts = np.zeros(w.total_q, dtype=np.int64)
    wl, wr = w.window_left, w.window_right
    for b in range(w.num_reqs):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        k_len = int(cu_k[b + 1] - cu_k[b])
        ctx = k_len - (q1 - q0)
        p = ctx + np.arange(q1 - q0, dtype=np.int64)
        lo = np.maximum(p - wl, 0) if wl >= 0 else np.zeros_like(p)
        if w.causal:
            hi = p.copy()
        else:
            hi = (p + wr) if wr >= 0 else np.full_like(p, k_len - 1)
        hi = np.minimum(hi, k_len - 1)
        n = np.maximum(hi - lo + 1, 0)
        if table is not None:
            rs = table[q0:q1, 0].astype(np.int64)
            re = table[q0:q1, 1].astype(np.int64)
            rlo = np.maximum(rs, p - wl) if wl >= 0 else rs
            rlo = np.maximum(rlo, 0)
            rhi = np.minimum(re, k_len - 1)
            rn = np.maximum(rhi - rlo + 1, 0)
            ov = np.maximum(np.minimum(hi, rhi) - np.maximum(lo, rlo) + 1, 0)
            ov = np.where((n > 0) & (rn > 0), ov, 0)
            n = n + rn - ov
        counts[q0:q1] = n
    return counts


KERNEL_HEADERS = ("mask.cuh", "mvp_internal.cuh", "ptx.cuh")


def source_hash(path):
    """sha256 (first 16 hex digits) of a kernel's translation unit followed by
    the headers it includes from the same folder, in KERNEL_HEADERS order."""
    h = hashlib.sha256()
    for p in (path,) + tuple(os.path.join(os.path.dirname(path), n) for n in KERNEL_HEADERS):
        with open(p, "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def load_traffic(kernel_src, workload_name):
    """DRAM traffic per launch from the committed ncu summary, or None when
    the counters were taken on another workload or the kernel source changed
    since."""
    path = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(path) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("workload_name") != workload_name or d.get("source_sha256_16") != source_hash(kernel_src):
        return None
    return d.get("bytes_per_launch")


class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled during the timed region."""

    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "20",
                 "-i", str(self.gpu)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self._reader = threading.Thread(target=self._read, daemon=True)
            self._reader.start()
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def mark(self, which):
        setattr(self, which, time.time())

    def stop(self):
        time.sleep(0.1)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = []
        for t, line in self.lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append((t, float(parts[1]), float(parts[2]), parts[5:9]))
            except ValueError:
                continue
        inside = [r for r in rows if self.t0 is not None and self.t0 - 0.05 <= r[0] <= self.t1 + 0.05]
        use = inside if inside else rows
        if not use:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in use for i, v in enumerate(r[3]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in use), "sm_max_mhz": max(r[2] for r in use),
                "reasons": reasons, "samples": len(inside), "samples_total": len(rows)}


# ----------------------------------------------------------------- oracle timing
_W = {}


def _worker_init(w_name):
    """Spawned worker: the workload's shapes and the oracle's range table.
    Inputs are drawn per request on first use (same N(0,1) recipe as the GPU
    run, a per-request generator), so a worker never holds the whole batch."""
    from masked_varlen_prefill_gb300 import workloads
    from oracle import range_table as ort

    w = workloads.workload(w_name)
    cu_q, cu_k = w.cu_seqlens()
    table = None
    if w.ranges is not None:
        table = np.full((w.total_q, 2), -1, dtype=np.int32)
        ort.fill_by_spans(table, ort.ranges_from_padded(w.ranges), cu_q, np.asarray(w.k_lens))
    _W.update(w=w, cu_q=cu_q, cu_k=cu_k, table=table)


def _request_inputs(b):
    import torch

    w = _W["w"]
    if _W.get("req") != b:
        g = torch.Generator().manual_seed(w.seed * 100003 + b)
        ql, kl = w.q_lens[b], w.k_lens[b]
        _W["req"] = b
        _W["qb"] = torch.randn(ql, w.num_heads_q, w.head_dim, generator=g).to(torch.bfloat16).double().numpy()
        _W["kb"] = torch.randn(kl, w.num_heads_kv, w.head_dim, generator=g).to(torch.bfloat16).double().numpy()
        _W["vb"] = torch.randn(kl, w.num_heads_kv, w.head_dim, generator=g).to(torch.bfloat16).double().numpy()
        _W["sk"] = (torch.randn(w.num_heads_q, generator=g).double().numpy() if w.sink_mode else None)
    return _W["qb"], _W["kb"], _W["vb"], _W["sk"]


def _oracle_task(args):
    """One timed oracle call: ``rows`` of request ``b``, every head.  Input
    drawing happens before the clock starts; returns the oracle's seconds."""
    b, rows = args
    from oracle import attention as oatt

    w, cu_q, cu_k, table = _W["w"], _W["cu_q"], _W["cu_k"], _W["table"]
    rows = np.asarray(rows, dtype=np.int64)
    if rows.size == 0:
        return 0.0
    qb, kb, vb, sk = _request_inputs(b)
    q0 = int(cu_q[b])
    ctx = w.k_lens[b] - w.q_lens[b]
    t = time.perf_counter()
    oatt.attend_rows(rows, qb, kb, vb, ctx, w.causal, w.window_left, w.window_right,
                     None if table is None else table[q0 + rows], sk, w.sink_mode, w.scale)
    return time.perf_counter() - t


def oracle_sample_plan(w, rows_per_req):
    """(request, rows) tasks: ``rows_per_req`` random query rows per request in
    chunks of 32 rows."""
    cu_q, _ = w.cu_seqlens()
    rng = np.random.default_rng(7)
    tasks = []
    for b in range(w.num_reqs):
        ql = int(cu_q[b + 1] - cu_q[b])
        rows = np.sort(rng.choice(ql, size=min(rows_per_req, ql), replace=False))
        for chunk in np.array_split(rows, max(1, len(rows) // 32)):
            tasks.append((b, [int(x) for x in chunk]))
    return tasks


def time_oracle(w, counts, rows_per_req, pool, cores):
    """The oracle over the sample: summed oracle seconds across workers, the
    wall time of the parallel run, the sample's FLOPs and rows.  Throughput is
    the sample's FLOPs over the wall time with ``cores`` workers busy."""
    tasks = oracle_sample_plan(w, rows_per_req)
    tasks.sort(key=lambda t: t[0])
    cu_q, _ = w.cu_seqlens()
    vis = sum(int(counts[int(cu_q[b]) + r]) for (b, rows) in tasks for r in rows)
    flops = 4.0 * w.head_dim * w.num_heads_q * vis
    chunk = max(1, math.ceil(len(tasks) / cores))
    secs = pool.map(_oracle_task, tasks, chunksize=chunk)
    cpu_s = float(sum(secs))
    wall = max(cpu_s / cores, max(secs) if secs else 0.0)
    return wall, flops, sum(len(r) for _, r in tasks), cpu_s


def oracle_workers(w, cores):
    """Workers for the oracle pool: one per core, fewer when the host's
    available memory would not hold a float64 copy of the largest request's
    q, K and V (with its temporaries) per worker within a quarter of it."""
    per = 2 * 8 * (max(w.k_lens) * w.num_heads_kv * w.head_dim * 2 + max(w.q_lens) * w.num_heads_q * w.head_dim)
    try:
        avail = os.sysconf("SC_AVPHYS_PAGES") * os.sysconf("SC_PAGE_SIZE")
    except (ValueError, OSError, AttributeError):
        avail = 0
    if avail <= 0:
        return max(1, min(cores, 4))
    return max(1, min(cores, int(0.25 * avail // max(per, 1))))


def make_pool(cores, w_name):
    """Spawned process pool, one single-threaded-BLAS worker per core, each
    holding the workload's inputs; returns once every worker is ready."""
    saved = {v: os.environ.get(v) for v in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS")}
    for var in saved:
        os.environ[var] = "1"
    try:
        pool = mp.get_context("spawn").Pool(cores, initializer=_worker_init, initargs=(w_name,))
    finally:
        for var, val in saved.items():
            if val is None:
                os.environ.pop(var, None)
            else:
                os.environ[var] = val
    pool.map(_oracle_task, [(0, [])] * (4 * cores), chunksize=1)  # wait for every initializer
    return pool


# ----------------------------------------------------------------- distributed
def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value, world):
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([value], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def aggregate(per_rank_flops, max_seconds):
    """Whole-job throughput: all ranks' work over the slowest rank's time."""
    return per_rank_flops / max_seconds / 1e12




# ----------------------------------------------------------------- main arms
def run_reference(args, world, rank):
    from masked_varlen_prefill_gb300 import workloads
    from oracle import range_table as ort

    if rank != 0:
        return 0
    w = workloads.workload(args.workload)
    cu_q, _ = w.cu_seqlens()
    table = None
    if w.ranges is not None:
        table = np.full((w.total_q, 2), -1, dtype=np.int32)
        ort.fill_by_spans(table, ort.ranges_from_padded(w.ranges), cu_q, np.asarray(w.k_lens))
    counts = visible_counts_per_row(w, table)
    cores = oracle_workers(w, os.cpu_count() or 1)
    pool = make_pool(cores, args.workload)
    rows_per_req = 64 if max(w.k_lens) <= 8192 else 32
    for _ in range(args.warmup):
        time_oracle(w, counts, rows_per_req, pool, cores)
    total_t, total_f, nrows = 0.0, 0.0, 0
    for _ in range(args.steps):
        t, f, n, _ = time_oracle(w, counts, rows_per_req, pool, cores)
        total_t += t
        total_f += f
        nrows += n
    pool.close()
    pool.join()
    value = total_f / total_t / 1e12
    sample = (f"{nrows // max(1, args.steps)} query rows per step (up to {rows_per_req} per request, all heads) "
              f"of the {args.workload} workload, float64 dense oracle")
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total_t / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic",
            "config": {"workload": WORKLOAD_DESCS.get(args.workload, args.workload), "parallelism": "replicas"},
            "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))
    return 0


def _leading_decode(w):
    n = 0
    while n < w.num_reqs and w.q_lens[n] == 1:
        n += 1
    return n


class Batch:
    """One workload's inputs resident on the device, and the library calls of
    one step on them: the range-table fill (when the workload has ranges) and
    the attention call, packed, paged or in scan mode.  Decode requests come
    first in every workload, so the call passes their count."""

    def __init__(self, w, dev, paged=0, scan=False):
        import torch

        import masked_varlen_prefill_gb300 as mvp
        from masked_varlen_prefill_gb300 import workloads

        self.mvp, self.torch = mvp, torch
        self.w, self.dev, self.paged_bs, self.scan = w, dev, paged, scan
        self.n_dec = _leading_decode(w)
        self.q, self.k, self.v, self.sinks = workloads.make_tensors(w, device=dev)
        self.cu_q_np, self.cu_k_np = w.cu_seqlens()
        self.cu_q = torch.from_numpy(self.cu_q_np).to(dev)
        self.cu_k = torch.from_numpy(self.cu_k_np).to(dev)
        self.seq_lens = torch.tensor(w.k_lens, dtype=torch.int32, device=dev)
        self.ranges = torch.from_numpy(w.ranges).to(dev) if w.ranges is not None else None
        self.table = torch.empty((w.total_q, 2), dtype=torch.int32, device=dev) if self.ranges is not None else None
        self.covered = torch.empty(1, dtype=torch.int32, device=dev) if self.ranges is not None else None
        self.out = torch.empty_like(self.q)
        self.max_q, self.max_k = max(w.q_lens), max(w.k_lens)
        # workspace: the prefill work queue (header) and the decode split
        # partials; uninitialised, as a serving engine would allocate it once
        nbytes = mvp.attn_workspace_size(self.n_dec, w.num_heads_q, w.head_dim, self.max_k)
        self.ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev) if nbytes else None
        self.pg = None
        if paged:
            kc, vc, bt, sl = workloads.to_paged(self.k, self.v, w.k_lens, paged, seed=w.seed)
            self.pg = dict(k_cache=kc, v_cache=vc, block_table=bt, seq_lens_k=sl)
        self.kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right, sinks=self.sinks,
                       sink_mode=w.sink_mode, scale=w.scale, workspace=self.ws)

    def fill(self):
        if self.ranges is None or self.scan:
            return 0
        self.mvp.fill_query_ranges(self.ranges, self.cu_q, self.seq_lens, self.table, num_tokens=self.w.total_q,
                                   rows_written=self.covered)
        return self.mvp.last_launch_count()

    def attn(self, lo=0, hi=None):
        """Attention over requests [lo, hi) of the batch (default: all)."""
        mvp, w = self.mvp, self.w
        hi = w.num_reqs if hi is None else hi
        nd = max(0, min(self.n_dec, hi) - lo)
        cq, ck = self.cu_q[lo:hi + 1], self.cu_k[lo:hi + 1]
        mq, mk = max(w.q_lens[lo:hi]), max(w.k_lens[lo:hi])
        if self.scan:
            mvp.attn_fwd_varlen_scan(self.q, self.k, self.v, self.out, cq, ck, mq, mk,
                                     None if self.ranges is None else self.ranges[lo:hi], num_decode_reqs=nd,
                                     **self.kw)
        elif self.pg is not None:
            mvp.attn_fwd_paged(self.q, self.pg["k_cache"], self.pg["v_cache"], self.out, cq,
                               self.pg["seq_lens_k"][lo:hi], self.pg["block_table"][lo:hi], self.paged_bs, mq, mk,
                               range_table=self.table, range_covered=self.covered, num_decode_reqs=nd, **self.kw)
        else:
            mvp.attn_fwd_varlen(self.q, self.k, self.v, self.out, cq, ck, mq, mk, range_table=self.table,
                                range_covered=self.covered, num_decode_reqs=nd, **self.kw)
        return mvp.last_launch_count()

    def step(self):
        # nothing between the two calls: the attention kernel may start its
        # setup while the fill kernel runs (programmatic dependent launch)
        n = self.fill()
        return n + self.attn()

    def prepare(self):
        """Fill the table once outside any timed region (scan mode has no fill
        step; its exact visible count still comes from the table, which the
        workloads' non-overlapping ranges make identical to the scan)."""
        if self.ranges is not None:
            self.mvp.fill_query_ranges(self.ranges, self.cu_q, self.seq_lens, self.table,
                                       num_tokens=self.w.total_q, rows_written=self.covered)

    def accounting(self):
        """Exact visible pairs per row (from the GPU-filled table, which the
        tests pin bit-exact) and the library's accounting of the call."""
        w = self.w
        table_np = None if self.table is None else self.table.cpu().numpy()
        counts = visible_counts_per_row(w, table_np)
        covered = self.covered is not None and int(self.covered.item()) != 0
        acct = self.mvp.attn_accounting(self.cu_q_np, w.k_lens, w.num_heads_q, w.num_heads_kv, w.head_dim,
                                        range_table=table_np if covered else None, causal=w.causal,
                                        window_left=w.window_left, window_right=w.window_right)
        flops = 4.0 * w.head_dim * w.num_heads_q * int(counts.sum())
        if acct["exact_flops"] != flops:
            raise RuntimeError("library accounting disagrees with the bench's visible count")
        return counts, acct

    def release(self):
        for name in ("q", "k", "v", "sinks", "out", "ws", "pg", "table", "covered", "ranges"):
            setattr(self, name, None)


def time_calls(fn, reps, flush, stream):
    """Mean seconds of ``fn`` over ``reps`` runs, each bracketed by CUDA events
    on ``stream`` with an L2 flush before it (outside the events)."""
    import torch

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in ev:
        flush.zero_()
        a.record(stream)
        fn()
        b.record(stream)
    torch.cuda.synchronize()
    return sum(a.elapsed_time(b) for a, b in ev) / reps / 1e3


def sub_batches(bt, counts, acct, peaks, flush, stream, reps):
    """Decode-only and prefill-only sub-batches of a mixed batch, or the
    attention call alone: kernel time, achieved rate and fraction of the
    roofline of each side; returns (sub, dec_s, pre_s, dec_bytes, pre_flops)."""
    w, n_dec = bt.w, bt.n_dec
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_b = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    cu_q_l = [int(x) for x in bt.cu_q_np]
    visible = int(counts.sum())
    dec_vis = int(counts[:cu_q_l[n_dec]].sum()) if n_dec else 0
    pre_flops = 4.0 * w.head_dim * w.num_heads_q * (visible - dec_vis)
    if 0 < n_dec < w.num_reqs:
        for _ in range(2):
            time_calls(lambda: bt.attn(0, n_dec), 1, flush, stream)
            time_calls(lambda: bt.attn(n_dec, w.num_reqs), 1, flush, stream)
        dec_s = time_calls(lambda: bt.attn(0, n_dec), reps, flush, stream)
        pre_s = time_calls(lambda: bt.attn(n_dec, w.num_reqs), reps, flush, stream)
    else:
        time_calls(bt.attn, 1, flush, stream)
        attn_s = time_calls(bt.attn, reps, flush, stream)
        dec_s, pre_s = (attn_s, 0.0) if n_dec == w.num_reqs else (0.0, attn_s)
    dec_bytes = dec_vis * w.num_heads_kv * w.head_dim * 2 * 2 + n_dec * w.num_heads_q * w.head_dim * 2 * 2
    sub = {}
    if n_dec:
        sub["decode"] = {"ms": 1e3 * dec_s, "rows": n_dec, "algorithmic_bytes": dec_bytes,
                         "GB_per_s": dec_bytes / dec_s / 1e9, "frac_hbm": dec_bytes / dec_s / 1e9 / peak_b}
    if pre_s > 0:
        sub["prefill"] = {"ms": 1e3 * pre_s, "TFLOP_per_s": pre_flops / pre_s / 1e12,
                          "frac_tensor": pre_flops / pre_s / 1e12 / peak_t,
                          "exact_over_executed_mma": (pre_flops / acct["prefill_mma_flops"]
                                                      if acct["prefill_mma_flops"] else None)}
    return sub, dec_s, pre_s, dec_bytes, pre_flops


def mixed_roofline(step_s, flops, dec_bytes, acct, peaks):
    """The step against max(algorithmic bytes / HBM peak, FLOPs / tensor peak):
    bytes = the decode rows' K/V (once per KV head) and q / out plus the
    prefill rows' compulsory bytes; FLOPs = every visible entry's 4 D Hq."""
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_b = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    nbytes = dec_bytes + acct["prefill_compulsory_bytes"]
    bound = max(nbytes / (peak_b * 1e9), flops / (peak_t * 1e12))
    return {"algorithmic_bytes": nbytes, "flops": flops, "bytes_bound_ms": 1e3 * nbytes / (peak_b * 1e9),
            "flops_bound_ms": 1e3 * flops / (peak_t * 1e12), "bound_ms": 1e3 * bound, "step_ms": 1e3 * step_s,
            "frac": bound / step_s}


def measure_config(name, dev, peaks, flush, stream, reps):
    """One workload of the benchmark set: the whole step (fill + attention)
    timed over ``reps`` L2-flushed runs, its sub-batches, and for mixed
    batches the mixed roofline."""
    import torch

    import masked_varlen_prefill_gb300 as mvp
    from masked_varlen_prefill_gb300 import workloads

    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    w = workloads.workload(name)
    bt = Batch(w, dev)
    for _ in range(3):
        flush.zero_()
        bt.step()
    torch.cuda.synchronize()
    if mvp.get_last_device_error() != 0:
        raise RuntimeError(f"device timeout during {name}")
    counts, acct = bt.accounting()
    visible = int(counts.sum())
    flops = 4.0 * w.head_dim * w.num_heads_q * visible
    step_s = time_calls(bt.step, reps, flush, stream)
    sub, dec_s, pre_s, dec_bytes, pre_flops = sub_batches(bt, counts, acct, peaks, flush, stream, reps)
    if mvp.get_last_device_error() != 0:
        raise RuntimeError(f"device timeout during {name}")
    res = {"config": CONFIG_NUMBER.get(name, name), "workload": WORKLOAD_DESCS.get(name, name),
           "step_ms": 1e3 * step_s, "visible_entries": visible, "TFLOP_per_s": flops / step_s / 1e12,
           "frac_tensor": flops / step_s / 1e12 / peak_t, "tokens_per_s": w.total_q / step_s,
           "sub_batches": sub}
    if 0 < bt.n_dec < w.num_reqs:
        res["mixed_roofline"] = mixed_roofline(step_s, flops, dec_bytes, acct, peaks)
    elif pre_s > 0:
        res["kernel"] = {"ms": 1e3 * pre_s, "TFLOP_per_s": pre_flops / pre_s / 1e12,
                         "frac_tensor": pre_flops / pre_s / 1e12 / peak_t}
    bt.release()
    del bt
    torch.cuda.empty_cache()
    return res


def measure_fill_stress(dev, peaks, flush, stream, reps):
    """The range fill at a stress size (4096 requests x 1024 rows, 64 ranges
    each): algorithmic bytes 8 N (table rows written) + 4 (2 B + 1) (offsets
    and lengths) + 8 B R (ranges read) against the HBM peak."""
    import torch

    import masked_varlen_prefill_gb300 as mvp
    from masked_varlen_prefill_gb300 import workloads

    peak_b = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    ranges_np, q_lens, seq = workloads.fill_stress_case()
    nb, nr = ranges_np.shape[0], ranges_np.shape[1]
    qsl = np.zeros(nb + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    n = int(qsl[-1])
    ranges = torch.from_numpy(ranges_np).to(dev)
    d_qsl = torch.from_numpy(qsl).to(dev)
    d_seq = torch.tensor(seq, dtype=torch.int32, device=dev)
    out = torch.empty((n, 2), dtype=torch.int32, device=dev)
    covered = torch.empty(1, dtype=torch.int32, device=dev)

    def fill():
        mvp.fill_query_ranges(ranges, d_qsl, d_seq, out, num_tokens=n, rows_written=covered)

    time_calls(fill, 3, flush, stream)
    t = time_calls(fill, reps, flush, stream)
    nbytes = 8 * n + 4 * (2 * nb + 1) + 8 * nb * nr
    return {"requests": nb, "rows": n, "ranges_per_request": nr, "algorithmic_bytes": nbytes, "us": 1e6 * t,
            "GB_per_s": nbytes / t / 1e9, "frac_hbm": nbytes / t / 1e9 / peak_b,
            "timing": "CUDA events around the fill call (one kernel plus the 4-byte flag reset), L2 flushed "
                      "between calls"}


def graph_measure(args, w, q, k, v, sinks, flops, flush, stream, dev):
    """The same step through the step-metadata path (StepMetadata: host
    staging, one copy, the table fill) and attention sized for a capacity of
    ``args.graph`` x the batch (requests, rows, q / k length bounds), once
    captured in a CUDA graph and replayed, once launched eagerly.  The staging
    (host) happens before each step's start event; wall times include it."""
    import torch

    import masked_varlen_prefill_gb300 as mvp

    f = float(args.graph)
    cap_r = math.ceil(w.num_reqs * f)
    cap_t = math.ceil(w.total_q * f)
    max_q = math.ceil(max(w.q_lens) * f)
    max_k = math.ceil(max(w.k_lens) * f)
    n_ranges = 0 if w.ranges is None else w.ranges.shape[1]
    meta = mvp.StepMetadata(cap_r, cap_t, n_ranges, dev)
    qsl, _ = w.cu_seqlens()
    k_lens = np.asarray(w.k_lens, np.int32)
    qc = torch.zeros(cap_t, w.num_heads_q, w.head_dim, dtype=q.dtype, device=dev)
    qc[:w.total_q].copy_(q)
    outs = [torch.zeros_like(qc) for _ in range(2)]
    nbytes = mvp.attn_workspace_size(cap_r, w.num_heads_q, w.head_dim, max_k)
    ws = torch.empty(max(nbytes, 16), dtype=torch.uint8, device=dev)
    kw = dict(causal=w.causal, window_left=w.window_left, window_right=w.window_right, sinks=sinks,
              sink_mode=w.sink_mode, scale=w.scale, workspace=ws)

    def attention(o):
        mvp.attn_fwd_varlen(qc, k, v, o, meta.query_start_loc, meta.cu_seqlens_k, max_q, max_k,
                            range_table=meta.range_table if n_ranges else None,
                            range_covered=meta.range_covered if n_ranges else None, **kw)
        return mvp.last_launch_count()

    def stage():
        meta.stage(qsl, k_lens, None, w.ranges)

    stage()
    meta.upload()
    n_attn = attention(outs[1])
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        meta.upload()
        attention(outs[0])
    torch.cuda.synchronize()
    per_step = 1 + n_attn  # the fill kernel + the attention kernels

    def timed(run):
        for _ in range(args.warmup):
            flush.zero_()
            stage()
            run()
        torch.cuda.synchronize()
        ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
              for _ in range(args.steps)]
        wall = 0.0
        for a, b in ev:
            flush.zero_()
            torch.cuda.synchronize()
            t0 = time.perf_counter()
            stage()
            a.record(stream)
            run()
            b.record(stream)
            torch.cuda.synchronize()
            wall += time.perf_counter() - t0
        return sum(a.elapsed_time(b) for a, b in ev) / len(ev), 1e3 * wall / len(ev)

    g_ms, g_wall = timed(g.replay)

    def eager():
        meta.upload()
        attention(outs[1])

    e_ms, e_wall = timed(eager)
    same = bool(torch.equal(outs[0][:w.total_q].view(torch.int16), outs[1][:w.total_q].view(torch.int16)))
    if mvp.get_last_device_error() != 0:
        raise RuntimeError("device timeout during graph replays")
    meta.close()
    return {"capacity_factor": f, "max_reqs": cap_r, "max_tokens": cap_t, "max_q_len": max_q, "max_k_len": max_k,
            "kernels_per_step": per_step, "value": flops / (g_ms / 1e3) / 1e12, "unit": "TFLOP/s",
            "graph_ms_per_step": g_ms, "graph_wall_ms_per_step": g_wall,
            "eager_ms_per_step": e_ms, "eager_wall_ms_per_step": e_wall,
            "out_bitwise_equal_to_eager": same,
            "timing": "device events around the replay (or eager launches); wall clock from before the host "
                      "staging to after a synchronize"}


def e2e_measure(args, bt, flops, stream, world):
    """Every step copies its inputs from pinned host memory and its output
    back, inside the timed region.  Steps are pipelined the way a serving loop
    would run them: two device buffer sets, host->device copies on one
    stream, the fill and attention calls on another, device->host copies on a
    third, so step i + 1's inputs travel while step i computes and step i - 1's
    output returns.  The sequential form (copy, compute, copy on one stream)
    is reported beside it."""
    import torch

    import masked_varlen_prefill_gb300 as mvp

    w, dev, n_dec = bt.w, bt.dev, bt.n_dec
    paged = bt.pg
    max_q, max_k = bt.max_q, bt.max_k
    kv_names = ["k", "v", "cu_k"] if paged is None else ["k_cache", "v_cache", "block_table", "seq_lens_k"]
    kv_dev = [bt.k, bt.v, bt.cu_k] if paged is None else [paged[n] for n in kv_names]
    names = ["q", "cu_q"] + kv_names + (["seq_lens", "ranges"] if bt.ranges is not None else []) + \
        (["sinks"] if bt.sinks is not None else [])
    dev_in = [bt.q, bt.cu_q] + kv_dev + ([bt.seq_lens, bt.ranges] if bt.ranges is not None else []) + \
        ([bt.sinks] if bt.sinks is not None else [])
    host_in = [t.cpu().pin_memory() for t in dev_in]
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = bt.out.numel() * bt.out.element_size()
    sets = []
    for b in range(2):
        d = dict(zip(names, dev_in if b == 0 else [torch.empty_like(t) for t in dev_in]))
        d["out"] = bt.out if b == 0 else torch.empty_like(bt.out)
        d["table"] = bt.table if (b == 0 or bt.table is None) else torch.empty_like(bt.table)
        d["covered"] = bt.covered if (b == 0 or bt.covered is None) else torch.empty_like(bt.covered)
        d["ws"] = bt.ws if (b == 0 or bt.ws is None) else torch.empty_like(bt.ws)
        d["host_out"] = torch.empty(bt.out.shape, dtype=bt.out.dtype, pin_memory=True)
        sets.append(d)

    def compute(d, st):
        kw2 = dict(bt.kw, sinks=d.get("sinks"), workspace=d["ws"])
        if args.scan:
            mvp.attn_fwd_varlen_scan(d["q"], d["k"], d["v"], d["out"], d["cu_q"], d["cu_k"], max_q, max_k,
                                     d.get("ranges"), num_decode_reqs=n_dec, stream=st, **kw2)
            return
        if bt.ranges is not None:
            mvp.fill_query_ranges(d["ranges"], d["cu_q"], d["seq_lens"], d["table"], num_tokens=w.total_q,
                                  rows_written=d["covered"], stream=st)
        if paged is not None:
            mvp.attn_fwd_paged(d["q"], d["k_cache"], d["v_cache"], d["out"], d["cu_q"], d["seq_lens_k"],
                               d["block_table"], args.paged, max_q, max_k, range_table=d["table"],
                               range_covered=d["covered"], num_decode_reqs=n_dec, stream=st, **kw2)
        else:
            mvp.attn_fwd_varlen(d["q"], d["k"], d["v"], d["out"], d["cu_q"], d["cu_k"], max_q, max_k,
                                range_table=d["table"], range_covered=d["covered"], num_decode_reqs=n_dec,
                                stream=st, **kw2)

    s_in, s_cmp, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_done = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def pipelined(n_steps):
        t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        torch.cuda.synchronize()
        t0.record(s_in)
        for i in range(n_steps):
            b = i % 2
            d = sets[b]
            if i >= 2:
                s_in.wait_event(ev_done[b])  # step i - 2 no longer reads these inputs
            with torch.cuda.stream(s_in):
                for n, h in zip(names, host_in):
                    d[n].copy_(h, non_blocking=True)
                ev_in[b].record(s_in)
            s_cmp.wait_event(ev_in[b])
            if i >= 2:
                s_cmp.wait_event(ev_out[b])  # step i - 2's output has left this buffer
            with torch.cuda.stream(s_cmp):
                compute(d, s_cmp)
                ev_done[b].record(s_cmp)
            s_out.wait_event(ev_done[b])
            with torch.cuda.stream(s_out):
                d["host_out"].copy_(d["out"], non_blocking=True)
                ev_out[b].record(s_out)
        t1.record(s_out)
        s_in.wait_event(ev_out[(n_steps - 1) % 2])
        torch.cuda.synchronize()
        return t0.elapsed_time(t1) / 1e3

    def sequential(n_steps):
        d = sets[0]
        ts = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_steps)]
        for a, z in ts:
            a.record(stream)
            for n, h in zip(names, host_in):
                d[n].copy_(h, non_blocking=True)
            compute(d, stream)
            d["host_out"].copy_(d["out"], non_blocking=True)
            z.record(stream)
        torch.cuda.synchronize()
        return sum(a.elapsed_time(z) for a, z in ts) / 1e3

    pipelined(3)
    sequential(2)
    barrier(world)
    e2e_s = reduce_max(pipelined(args.e2e_steps), world)
    seq_s = reduce_max(sequential(args.e2e_steps), world)
    if mvp.get_last_device_error() != 0:
        raise RuntimeError("device timeout during the e2e steps")
    return {"value": aggregate(flops * args.e2e_steps * world, e2e_s), "unit": "TFLOP/s",
            "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": args.e2e_steps,
            "ms_per_step": 1e3 * e2e_s / args.e2e_steps,
            "timing": "pinned host inputs -> device, fill + attention, output -> pinned host, every step; "
                      "steps pipelined over two buffer sets and three streams",
            "sequential": {"value": aggregate(flops * args.e2e_steps * world, seq_s), "unit": "TFLOP/s",
                           "ms_per_step": 1e3 * seq_s / args.e2e_steps}}


def run_gpu(args, world, rank, local):
    import torch

    import masked_varlen_prefill_gb300 as mvp
    from masked_varlen_prefill_gb300 import workloads

    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    mvp.load_library()
    peaks, peak_src = load_peaks()

    w = workloads.scaled_workload(args.workload) if args.scaled else workloads.workload(args.workload)
    # CPU baseline pool first (spawned, rank 0 only)
    pool = None
    cores = oracle_workers(w, os.cpu_count() or 1)
    if rank == 0 and not args.no_cpu_baseline:
        pool = make_pool(cores, args.workload)

    bt = Batch(w, dev, paged=args.paged, scan=args.scan)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)
    if args.scan:
        bt.prepare()
    for _ in range(args.warmup):
        flush.zero_()
        bt.step()
    torch.cuda.synchronize()
    if mvp.get_last_device_error() != 0:
        raise RuntimeError("device timeout during warm-up")

    counts, acct = bt.accounting()
    visible = int(counts.sum())
    flops = 4.0 * w.head_dim * w.num_heads_q * visible
    est = acct["est_attn_qk_flops"] + acct["est_attn_av_flops"]
    accounting = {
        "estimate_flops_pr55624": est, "exact_flops": flops, "executed_mma_flops": acct["prefill_mma_flops"],
        "estimate_over_exact": est / flops if flops else None,
        "exact_prefill_over_executed": (4.0 * w.head_dim * w.num_heads_q * acct["visible_prefill"]
                                        / acct["prefill_mma_flops"]) if acct["prefill_mma_flops"] else None,
        "prefill_items": acct["prefill_items"], "prefill_tiles": acct["prefill_tiles"],
        "prefill_mma_instructions": acct["prefill_mma_instructions"],
        "prefill_compulsory_bytes": acct["prefill_compulsory_bytes"],
        "estimate_decode_kv_bytes_pr55624": acct["est_decode_kv_read_bytes"],
        "exact_decode_kv_bytes": acct["exact_decode_kv_bytes"], "decode_read_bytes": acct["decode_read_bytes"],
        "decode_cta_read_bytes": acct["decode_cta_read_bytes"],
        "source": "mvp_attn_accounting (estimate: vLLM PR #55624 ExecutionContext with the window clamp)"}

    # ------------------------------------------------------------- timed steps
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    sampler = ClockSampler(local)
    sampler.start()
    launches = 0
    barrier(world)
    torch.cuda.synchronize()
    sampler.mark("t0")
    for i in range(args.steps):
        flush.zero_()
        starts[i].record(stream)
        launches += bt.step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    sampler.mark("t1")
    barrier(world)
    sampler.stop()
    if mvp.get_last_device_error() != 0:
        raise RuntimeError("device timeout during timed steps")
    step_ms = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    local_s = sum(step_ms) / 1e3
    max_s = reduce_max(local_s, world)
    value = aggregate(flops * args.steps * world, max_s)
    ms_per_step = 1e3 * max_s / args.steps
    tokens_per_s = w.total_q * args.steps * world / max_s

    # ------------------------------------------------------------- roofline
    peak_t = float(peaks.get("bf16_tflops", FALLBACK_PEAKS["bf16_tflops"]))
    peak_b = float(peaks.get("hbm_gbs", FALLBACK_PEAKS["hbm_gbs"]))
    sub_reps = max(10, args.steps // 2)
    sub, dec_s, pre_s, dec_bytes, pre_flops = sub_batches(bt, counts, acct, peaks, flush, stream, sub_reps)
    kernel_dir = os.path.join(ROOT, "masked_varlen_prefill_gb300", "csrc")
    if pre_s >= dec_s:
        achieved = pre_flops / pre_s / 1e12
        roofline = {"bound": "tensor", "achieved": achieved, "peak": peak_t, "unit": "TFLOP/s",
                    "frac": achieved / peak_t,
                    "traffic": (None if (args.paged or args.scaled or args.scan)
                                else load_traffic(os.path.join(kernel_dir, "attn_prefill.cu"), args.workload)),
                    "kernel": f"attn_prefill_kernel (D={w.head_dim})",
                    "peak_source": f"bf16_tflops (burst) of {peak_src}", "kernel_ms_per_launch": 1e3 * pre_s}
    else:
        achieved = dec_bytes / dec_s / 1e9
        roofline = {"bound": "hbm", "achieved": achieved, "peak": peak_b, "unit": "GB/s",
                    "frac": achieved / peak_b, "traffic": None, "kernel": f"attn_decode_kernel (D={w.head_dim})",
                    "peak_source": f"hbm_gbs of {peak_src}", "kernel_ms_per_launch": 1e3 * dec_s}
    fill_ms = 0.0
    if bt.ranges is not None and not args.scan:
        fill_ms = 1e3 * time_calls(bt.fill, 10, flush, stream)
    roofline["fill_ms_per_launch"] = fill_ms
    mixed = mixed_roofline(max_s / args.steps, flops, dec_bytes, acct, peaks) if 0 < bt.n_dec < w.num_reqs else None

    # ------------------------------------------------------------- e2e (host buffers)
    e2e = None if args.no_e2e else e2e_measure(args, bt, flops, stream, world)

    # ------------------------------------------------------------- graph replays
    graph = None
    if args.graph is not None:
        graph = graph_measure(args, w, bt.q, bt.k, bt.v, bt.sinks, flops, flush, stream, dev)

    # ------------------------------------------------------------- CPU baseline
    cpu_baseline = None
    if pool is not None:
        t_cpu, f_cpu, n_rows, cpu_s = time_oracle(w, counts, args.cpu_rows_per_req, pool, cores)
        pool.close()
        pool.join()  # the workers' exit must not compete with the host side of the GPU timings below
        cpu_baseline = {"value": f_cpu / t_cpu / 1e12, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                        "sample": f"{n_rows} query rows (up to {args.cpu_rows_per_req} per request, all heads) of "
                                  f"the {args.workload} workload, float64 dense oracle, {cpu_s:.1f} core-seconds "
                                  f"over {cores} single-threaded workers"}

    # ------------------------------------------------------------- the other configs
    configs = None
    plain = not (args.scaled or args.paged or args.scan or args.graph is not None)
    if rank == 0 and plain and not args.no_configs:
        bt.release()
        del bt
        torch.cuda.empty_cache()
        reps = max(5, args.steps // 2)
        wanted = set(args.configs.split(",")) if args.configs else None
        configs = {}
        for name in workloads.WORKLOADS:
            if name != args.workload and (wanted is None or name in wanted):
                configs[name] = measure_config(name, dev, peaks, flush, stream, reps)
        if wanted is None or "fill_stress" in wanted:
            configs["fill_stress"] = measure_fill_stress(dev, peaks, flush, stream, reps)
    barrier(world)

    if rank == 0:
        desc = WORKLOAD_DESCS.get(args.workload, args.workload) if not args.scaled else w.name
        line = {"metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
                "config": {"workload": desc, "config_number": CONFIG_NUMBER.get(args.workload),
                           "global_batch": w.num_reqs * world, "seq_len": max(w.q_lens),
                           "kv_layout": (f"paged, {args.paged}-token blocks in a seeded random order"
                                         if args.paged else "packed"),
                           "ranges": ("scan mode: per-request range lists scanned in the kernels, no fill"
                                      if args.scan else "per-row table filled on the GPU each step"),
                           "l2": "flushed between steps (256 MiB write, outside the events)",
                           "parallelism": "replicas" if world > 1 else "single GPU"},
                "pct_tensor_peak": 100.0 * value / peak_t, "tokens_per_s": tokens_per_s,
                "visible_entries_per_step": visible, "sub_batches": sub,
                "roofline": roofline, "cpu_baseline": cpu_baseline, "e2e": e2e, "accounting": accounting,
                "gpu_launches": launches, "clocks": sampler.summary()}
        if mixed is not None:
            line["mixed_roofline"] = mixed
        if configs is not None:
            line["configs"] = configs
        if graph is not None:
            line["graph"] = graph
        print(json.dumps(line))
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD,
                    help="workload name (default: the headline chunked-prefill workload)")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--cpu-rows-per-req", type=int, default=256)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="do not measure the other workloads of the set (the 'configs' object)")
    ap.add_argument("--configs", default=None, metavar="NAMES",
                    help="comma-separated subset of the other workloads (and 'fill_stress') to measure in the "
                         "'configs' object (default: all)")
    ap.add_argument("--scan", action="store_true",
                    help="scan mode: pass the per-request range lists to the attention call instead of filling "
                         "the per-row table (mvp_attn_fwd_varlen_scan)")
    ap.add_argument("--scaled", action="store_true",
                    help="run the small test-size version of the workload (for profiler and accounting checks; "
                         "not a bench line)")
    ap.add_argument("--graph", type=float, default=None, metavar="CAPACITY",
                    help="also run the step through the step-metadata path, captured in a CUDA graph sized for "
                         "CAPACITY x the batch (>= 1), and eagerly; adds a 'graph' object to the line")
    ap.add_argument("--paged", type=int, default=0, metavar="BLOCK",
                    help="run the workload on a paged K/V cache with this block size (blocks in a seeded random "
                         "order; mvp_attn_fwd_paged) instead of packed K/V")
    args = ap.parse_args(argv)
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.scaled:
        args.no_cpu_baseline = True  # the baseline samples the full workload
    if args.scan and (args.paged or args.graph is not None):
        ap.error("--scan takes a packed K/V layout and no --graph")
    if args.graph is not None and (args.graph < 1.0 or args.paged):
        ap.error("--graph takes a capacity factor >= 1 and a packed K/V layout")
    world, rank, local = dist_setup()
    if args.impl == "reference":
        return run_reference(args, world, rank)
    return run_gpu(args, world, rank, local)


if __name__ == "__main__":
    sys.exit(main())
