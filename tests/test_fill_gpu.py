"""Range-table fill kernel vs the oracle: bit-exact (GPU)."""

import json
import os

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import range_table as ort

from .conftest import GOLDEN

pytestmark = pytest.mark.gpu
DEV = "cuda"


def gpu_fill(ranges_padded, q_lens, seq_lens, capacity=None, poison=12345):
    qsl = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    n = int(qsl[-1])
    cap = capacity if capacity is not None else max(1, n) + 3
    out = torch.full((cap, 2), poison, dtype=torch.int32, device=DEV)
    written = torch.full((1,), -7, dtype=torch.int32, device=DEV)
    r = None if ranges_padded is None else torch.from_numpy(np.ascontiguousarray(ranges_padded, dtype=np.int32)).to(DEV)
    mvp.fill_query_ranges(r, torch.from_numpy(qsl).to(DEV), torch.tensor(seq_lens, dtype=torch.int32, device=DEV),
                          out, num_tokens=n, rows_written=written)
    torch.cuda.synchronize()
    return out.cpu().numpy(), int(written.item()), qsl


def oracle_fill(ranges_padded, q_lens, seq_lens):
    qsl = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    out = np.full((max(1, int(qsl[-1])), 2), -1, dtype=np.int32)
    rr = None if ranges_padded is None else ort.ranges_from_padded(ranges_padded)
    n = ort.fill_by_spans(out, rr, qsl, np.asarray(seq_lens))
    return out[: int(qsl[-1])], n


def check(ranges_padded, q_lens, seq_lens):
    got, written, qsl = gpu_fill(ranges_padded, q_lens, seq_lens)
    ref, n = oracle_fill(ranges_padded, q_lens, seq_lens)
    total = int(qsl[-1])
    if n == 0:
        # nothing covered: the kernel writes (-1, -1) everywhere and reports 0
        assert (got[:total] == -1).all()
    else:
        assert np.array_equal(got[:total], ref)
    assert written == n
    assert (got[total:] == 12345).all()  # rows past num_tokens untouched


def test_printed_example():
    with open(os.path.join(GOLDEN, "range_table_example.json")) as f:
        g = json.load(f)
    ranges = workloads.pad_ranges([g["mm_ranges"]["0"], g["mm_ranges"]["1"]])
    got, written, _ = gpu_fill(ranges, g["query_lens"], g["seq_lens"])
    assert written == g["expected_return"]
    assert got[:14].tolist() == g["expected_table"]


@pytest.mark.parametrize("name", ["mm_prefix_sliding", "chunked_prefill_ranges"])
def test_workload_tables(name):
    w = workloads.workload(name)
    check(w.ranges, w.q_lens, w.k_lens)


@pytest.mark.parametrize("seed", range(60))
def test_random(seed):
    rng = np.random.default_rng(seed)
    nb = int(rng.integers(1, 40))
    q_lens = [int(rng.integers(0, 300)) for _ in range(nb)]
    seq = [q + int(rng.integers(0, 1000)) for q in q_lens]
    per_req = []
    for b in range(nb):
        rl, cur = [], int(rng.integers(0, 50))
        for _ in range(int(rng.integers(0, 70))):
            length = int(rng.integers(1, 80))
            e = cur + length - 1 if rng.integers(0, 7) else cur - int(rng.integers(0, 5))
            rl.append((cur, e))
            cur += length + int(rng.integers(1, 30))
        if rng.integers(0, 4) == 0 and rl:  # overlapping list: last listed wins
            rl.append((max(0, seq[b] - q_lens[b] - 5), seq[b] + 3))
        per_req.append(rl)
    check(workloads.pad_ranges(per_req), q_lens, seq)


@pytest.mark.parametrize("nb,nr", [(1024, 2), (1025, 2), (1000, 3), (600, 3), (64, 32)])
def test_many_short_requests(nb, nr):
    """Batches of many 1- to 9-row requests: up to 1024 requests with at most
    2048 range entries between them are read from shared-memory copies, the
    others from global memory (1025 requests; 3000 entries); CTAs span many
    requests, and a request's rows are split between two CTAs."""
    rng = np.random.default_rng(nb * 7 + nr)
    q_lens = [int(rng.integers(1, 10)) for _ in range(nb)]
    seq = [q + int(rng.integers(0, 40)) for q in q_lens]
    per_req = []
    for b in range(nb):
        rl = []
        for _ in range(int(rng.integers(0, nr + 1))):
            s0 = int(rng.integers(0, seq[b] + 2))
            rl.append((s0, s0 + int(rng.integers(-1, 12))))
        per_req.append(rl)
    ranges = workloads.pad_ranges(per_req, min_width=nr)
    assert ranges.shape == (nb, nr, 2)
    check(ranges, q_lens, seq)


def test_no_ranges_and_degenerate_only():
    check(None, [5, 3], [9, 3])
    check(workloads.pad_ranges([[(3, 3), (7, 2)], []]), [5, 3], [9, 3])
    check(workloads.pad_ranges([[(0, 2)]]), [4], [8])  # wholly in the context


def test_reuse_overwrites_stale_rows():
    qsl = torch.tensor([0, 6], dtype=torch.int32, device=DEV)
    seq = torch.tensor([6], dtype=torch.int32, device=DEV)
    out = torch.full((8, 2), 12345, dtype=torch.int32, device=DEV)
    w = torch.zeros(1, dtype=torch.int32, device=DEV)
    for ranges, expect in (([[0, 5]], [[0, 5]] * 6), ([[4, 5]], [[-1, -1]] * 4 + [[4, 5]] * 2)):
        r = torch.tensor([ranges], dtype=torch.int32, device=DEV)
        mvp.fill_query_ranges(r, qsl, seq, out, num_tokens=6, rows_written=w)
        torch.cuda.synchronize()
        assert out[:6].cpu().tolist() == expect and int(w.item()) == 6
    assert (out[6:].cpu() == 12345).all()


def test_capacity_error_writes_nothing():
    qsl = torch.tensor([0, 10], dtype=torch.int32, device=DEV)
    seq = torch.tensor([10], dtype=torch.int32, device=DEV)
    out = torch.full((4, 2), 12345, dtype=torch.int32, device=DEV)
    r = torch.tensor([[[0, 3]]], dtype=torch.int32, device=DEV)
    with pytest.raises(mvp.MvpError) as ei:
        mvp.fill_query_ranges(r, qsl, seq, out, num_tokens=10)
    assert ei.value.status == mvp.MVP_ERR_CAPACITY
    torch.cuda.synchronize()
    assert (out.cpu() == 12345).all()


def test_stress_size():
    """The benchmark's stress size: 4096 requests x 1024 rows, 64 ranges each."""
    rng = np.random.default_rng(7)
    ranges, q_lens, seq = workloads.fill_stress_case()
    nb = len(q_lens)
    got, written, qsl = gpu_fill(ranges, q_lens, seq)
    # bit-exact on a sample of requests (the oracle is slow at this size)
    for b in rng.choice(nb, size=40, replace=False):
        ref, _ = oracle_fill(ranges[b:b + 1], [q_lens[b]], [seq[b]])
        assert np.array_equal(got[qsl[b]:qsl[b + 1]], ref), b
    assert written == int(qsl[-1])
