"""The bounds-checked build against the product build (GPU).

libmvp_debug.so is the same library compiled with MVP_DEBUG_BOUNDS: every
global access whose index comes from the caller's device-side metadata
(packed-row offsets, the range table, the block table of a paged cache) is
checked against its buffer, and an index outside records
MVP_ERR_DEVICE_BOUNDS in that library's device error word instead of reading
or writing out of bounds.  It stands in for a memory checker the pool does
not offer.  Here every kind of call runs through both libraries on the same
inputs: the checked build must report no out-of-bounds index and produce the
same bits (the checks skip nothing on valid inputs, and change no
arithmetic).  Random shapes over every flag combination, the scaled
workloads, paged caches with unused block-table entries, scan mode, the
range fill, and decode rows with and without split partials.
"""

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _both(fn):
    """fn() with the product library, then with the bounds-checked one; the
    checked run must leave its error word clear.  Returns both results."""
    ref = fn()
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == mvp.MVP_OK
    with mvp.bounds_checked():
        got = fn()
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == mvp.MVP_OK, "bounds-checked build: index out of bounds"
    return ref, got


def _same(a, b, what):
    for x, y in zip(a, b):
        if x is None:
            assert y is None
            continue
        if x.dtype == torch.bfloat16:
            assert torch.equal(x.view(torch.int16), y.view(torch.int16)), what
        else:
            assert torch.equal(x, y), what


def _packed(w, **kw):
    q, k, v, sinks = gh.make_inputs(w)

    def run():
        out, lse, table, covered = gh.run_gpu(w, q, k, v, sinks, **kw)
        return out, lse, table, covered

    ref, got = _both(run)
    _same(ref, got, w.name)


@pytest.mark.parametrize("seed", range(12))
def test_random_cases(seed):
    _packed(workloads.random_case(seed))


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_scaled_workloads(name):
    _packed(workloads.scaled_workload(name))


def test_decode_rows_single_split():
    # no workspace: every decode row is one CTA per KV head
    _packed(workloads.scaled_workload("mixed_serving_b"), use_workspace=False)


@pytest.mark.parametrize("block_size", [16, 64])
def test_paged(block_size):
    w = workloads.scaled_workload("chunked_prefill_ranges")
    q, k, v, sinks = gh.make_inputs(w)
    dev = q.device
    # unused block-table entries hold garbage ids, which the kernels must not read
    kc, vc, bt, sl = workloads.to_paged(k, v, w.k_lens, block_size, seed=5, table_fill=-7)
    cu_q, _ = gh.device_meta(w, dev)
    ranges = torch.from_numpy(w.ranges).to(dev)

    def run():
        table = torch.full((w.total_q, 2), 777, dtype=torch.int32, device=dev)
        covered = torch.zeros(1, dtype=torch.int32, device=dev)
        mvp.fill_query_ranges(ranges, cu_q, sl, table, num_tokens=w.total_q, rows_written=covered)
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
        n = mvp.attn_workspace_size(w.num_reqs, w.num_heads_q, w.head_dim, max(w.k_lens))
        ws = torch.empty(max(n, 16), dtype=torch.uint8, device=dev)
        mvp.attn_fwd_paged(q, kc, vc, out, cu_q, sl, bt, block_size, max(w.q_lens), max(w.k_lens), lse=lse,
                           range_table=table, range_covered=covered, causal=w.causal, window_left=w.window_left,
                           window_right=w.window_right, sinks=sinks, sink_mode=w.sink_mode, scale=w.scale,
                           workspace=ws)
        return out, lse, table

    ref, got = _both(run)
    _same(ref, got, f"paged {block_size}")


def test_scan_mode():
    w = workloads.scaled_workload("mm_prefix_sliding")
    q, k, v, sinks = gh.make_inputs(w)
    dev = q.device
    cu_q, cu_k = gh.device_meta(w, dev)
    rg = torch.from_numpy(np.ascontiguousarray(w.ranges, dtype=np.int32)).to(dev)

    def run():
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
        mvp.attn_fwd_varlen_scan(q, k, v, out, cu_q, cu_k, max(w.q_lens), max(w.k_lens), rg, lse=lse,
                                 causal=w.causal, window_left=w.window_left, window_right=w.window_right,
                                 sinks=sinks, sink_mode=w.sink_mode, scale=w.scale)
        return out, lse

    ref, got = _both(run)
    _same(ref, got, "scan")


def test_fill_stress_case():
    ranges, q_lens, seq = workloads.fill_stress_case(seed=3, num_reqs=512, rows=256, num_ranges=32)
    n = int(sum(q_lens))
    dev = torch.device("cuda", 0)
    r = torch.from_numpy(ranges).to(dev)
    c = torch.from_numpy(np.concatenate([[0], np.cumsum(q_lens)]).astype(np.int32)).to(dev)
    s = torch.tensor(seq, dtype=torch.int32, device=dev)

    def run():
        out = torch.full((n, 2), 12345, dtype=torch.int32, device=dev)
        flag = torch.full((1,), -1, dtype=torch.int32, device=dev)
        mvp.fill_query_ranges(r, c, s, out, num_tokens=n, rows_written=flag)
        return out, flag

    ref, got = _both(run)
    _same(ref, got, "fill")
