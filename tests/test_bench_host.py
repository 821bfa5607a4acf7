"""Host-side logic of bench.py (no GPU): accounting, multi-rank aggregation
over gloo, and the reference arm's JSON line."""

import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as tmp

import bench
from masked_varlen_prefill_gb300 import workloads
from oracle import accounting
from oracle import range_table as ort

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _table(w):
    if w.ranges is None:
        return None
    cu_q, _ = w.cu_seqlens()
    t = np.full((max(1, w.total_q), 2), -1, dtype=np.int32)
    ort.fill_by_spans(t, ort.ranges_from_padded(w.ranges), cu_q, np.asarray(w.k_lens))
    return t[:w.total_q]


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_visible_counts_match_oracle_mask(name):
    w = workloads.scaled_workload(name)
    cu_q, cu_k = w.cu_seqlens()
    t = _table(w)
    got = int(bench.visible_counts_per_row(w, t).sum())
    assert got == accounting.visible_entries(cu_q, cu_k, w.causal, w.window_left, w.window_right,
                                             range_table=t)


def test_visible_counts_arbitrary_tables():
    """Caller tables whose range need not hold the row (two disjoint intervals)."""
    rng = np.random.default_rng(3)
    for seed in range(60):
        w = workloads.random_case(seed, max_q=40, max_ctx=60)
        cu_q, cu_k = w.cu_seqlens()
        t = rng.integers(-1, 120, size=(w.total_q, 2)).astype(np.int32)
        per_row = bench.visible_counts_per_row(w, t)
        ref = accounting.visible_entries(cu_q, cu_k, w.causal, w.window_left, w.window_right, range_table=t)
        assert int(per_row.sum()) == ref, seed


def test_full_workload_counts():
    """Full-size mm_prefix workload: exact count, and it stays below the
    per-request tokens * min(context, window) estimate plus the range extras."""
    w = workloads.workload("mm_prefix_sliding")
    t = _table(w)
    n = int(bench.visible_counts_per_row(w, t).sum())
    assert n == accounting.visible_entries(*w.cu_seqlens(), True, w.window_left, 0, range_table=t)
    no_range = int(bench.visible_counts_per_row(w, None).sum())
    assert no_range == 4 * sum(min(i + 1, 1024) for i in range(4096))
    assert no_range < n < no_range + 4 * 8 * 256 * 256


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out_q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    local_seconds = [2.0, 3.0][rank]
    bench.barrier(world)
    mx = bench.reduce_max(local_seconds, world)
    value = bench.aggregate(1e12 * world, mx)
    out_q.put((rank, mx, value))
    dist.destroy_process_group()


def test_multi_rank_max_and_aggregate_gloo():
    ctx = tmp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, mx, value in res:
        assert mx == 3.0  # slowest rank
        assert abs(value - 2.0 / 3.0) < 1e-12  # both ranks' work over the max time


def test_reference_arm_json_line():
    env = dict(os.environ, PYTHONPATH=ROOT)
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3"],
                       cwd=ROOT, capture_output=True, text=True, timeout=900, env=env)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    assert line["impl"] == "reference" and line["unit"] == "TFLOP/s" and line["value"] > 0
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["e2e"]["h2d_bytes_per_step"] == 0 and line["metric"] == bench.METRIC


def test_warmup_floor():
    with pytest.raises(SystemExit):
        bench.main(["--warmup", "2"])
