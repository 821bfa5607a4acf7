"""Attention forward through the C-ABI vs the float64 oracle (GPU).

* scaled versions of every workload, compared element by element;
* random shapes over every flag combination (D 64..512, GQA 1..8, q_len 0/1,
  ragged tails, windows shorter than a tile, ranges longer than the window);
* the full-size workloads in the launch configuration the benchmark times,
  compared on sampled rows that the oracle computes one by one.
"""

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _parity_full(w, use_workspace=True, num_decode_reqs=-1, strict=False):
    q, k, v, sinks = gh.make_inputs(w)
    out, lse, table, covered = gh.run_gpu(w, q, k, v, sinks, use_workspace=use_workspace,
                                          num_decode_reqs=num_decode_reqs)
    ref_table, n = gh.oracle_table(w)
    if ref_table is not None:
        got = table[:w.total_q].cpu().numpy()
        if n:
            assert np.array_equal(got, ref_table), "range table"
        else:
            assert (got == -1).all()
        assert int(covered.item()) == n
    ro, rl = gh.oracle_full(w, q, k, v, sinks, ref_table)
    return gh.compare(out, lse, ro, rl, what=w.name, strict=strict)


@pytest.mark.parametrize("name", workloads.WORKLOADS)
def test_scaled_workloads(name):
    _parity_full(workloads.scaled_workload(name), strict=True)


@pytest.mark.parametrize("seed", range(48))
def test_random_cases(seed):
    _parity_full(workloads.random_case(seed))


@pytest.mark.parametrize("seed", [1033, 1251])
def test_random_cases_near_the_bf16_bound(seed):
    """Two shapes from a sweep of 300 further seeds whose largest error sits
    just above max(1e-2, 2^-8 |ref|) (rows of a few visible keys with a
    null-logit sink, |out| about 2-2.5, the bf16 output one ulp from the
    correctly rounded value): within the two-rounding bound 2^-7 |ref|."""
    _parity_full(workloads.random_case(seed))


@pytest.mark.parametrize("seed", range(6))
def test_random_cases_without_workspace(seed):
    _parity_full(workloads.random_case(100 + seed), use_workspace=False)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("group", [1, 2, 4])
def test_head_dims_and_groups(d, group):
    w = workloads.Workload(f"d{d}g{group}", 7 + d + group, [200, 1, 77, 130], [450, 900, 77, 300],
                           2 * group, 2, d, True, 150, 0, workloads.SINK_NULL_LOGIT, None)
    _parity_full(w)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("sink_mode", [workloads.SINK_NONE, workloads.SINK_NULL_LOGIT])
def test_output_does_not_depend_on_the_lse_request(d, sink_mode):
    """O does not depend on whether the caller asks for the LSE: bit for bit
    the same output with and without an LSE buffer (a prefill request with
    ranges, a decode row and a request of one tile's ragged tail), and the
    oracle's output and LSE within tolerance."""
    w = workloads.Workload(f"nolse_d{d}", 40 + d, [260, 1, 70], [700, 500, 70], 4, 2, d, True, 300, 0, sink_mode,
                           workloads.pad_ranges([[(500, 560)], [], [(2, 30)]]))
    q, k, v, sinks = gh.make_inputs(w)
    out_l, lse, _, _ = gh.run_gpu(w, q, k, v, sinks, with_lse=True)
    out_n, none, _, _ = gh.run_gpu(w, q, k, v, sinks, with_lse=False)
    assert none is None
    assert torch.equal(out_l.view(torch.int16), out_n.view(torch.int16))
    ref_table, _ = gh.oracle_table(w)
    ro, rl = gh.oracle_full(w, q, k, v, sinks, ref_table)
    gh.compare(out_n, lse, ro, rl, what=w.name, strict=False)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
@pytest.mark.parametrize("sink_mode", [workloads.SINK_NONE, workloads.SINK_NULL_LOGIT])
def test_running_max_moves_on_every_tile(d, sink_mode):
    """Scores that rise along the keys by ~12 (log2 units) per 128 keys move
    every row's running max past the lazy-rescale threshold tile after tile,
    so O (and, at D = 128, the row sums the PV MMA accumulates beside it) is
    rescaled on every tile; N(0, 1) inputs almost never do that after the
    first tile.  Full (non-causal) attention over ragged lengths."""
    w = workloads.Workload(f"rising_d{d}", 500 + d, [200, 130], [1200, 700], 4, 2, d, False, -1, -1, sink_mode,
                           None)
    q, k, v, sinks = gh.make_inputs(w)
    slope = 12.0 / (1.4426950408889634 * w.scale * 128)
    _, cu_k = w.cu_seqlens()
    for b in range(w.num_reqs):
        n = int(cu_k[b + 1] - cu_k[b])
        ramp = slope * torch.arange(n, device=k.device, dtype=torch.float32)
        k[cu_k[b]:cu_k[b + 1], :, 0] = ramp[:, None].to(torch.bfloat16)
    q[:, :, 0] = 1.0
    out, lse, _, _ = gh.run_gpu(w, q, k, v, sinks)
    ro, rl = gh.oracle_full(w, q, k, v, sinks, None)
    gh.compare(out, lse, ro, rl, what=w.name, strict=False)


@pytest.mark.parametrize("d,group", [(64, 4), (128, 4), (128, 8), (128, 2), (256, 4)])
@pytest.mark.parametrize("use_workspace", [True, False])
def test_decode_running_max_rises_along_the_keys(d, group, use_workspace):
    """Single-token rows whose scores rise by ~12 (log2 units) per 128 keys:
    a warp's running max passes the lazy-rescale threshold every few steps
    and lags the step maximum by up to the threshold in between, so both the
    rescale and the stale-max paths of the decode kernel run (N(0, 1) scores
    settle after the first tile).  Rows of up to 5000 keys: split over two
    key chunks with the workspace (plus the combine), one without; the
    1-key row has only key 0; the null-logit sink adds one more term."""
    k_lens = [5000, 3000, 700, 4500, 1]
    w = workloads.Workload(f"dec_rising_d{d}_g{group}", 900 + d + group, [1] * len(k_lens), k_lens, 2 * group, 2,
                           d, True, -1, 0, workloads.SINK_NULL_LOGIT, None)
    q, k, v, sinks = gh.make_inputs(w)
    slope = 12.0 / (1.4426950408889634 * w.scale * 128)
    _, cu_k = w.cu_seqlens()
    for b in range(w.num_reqs):
        n = int(cu_k[b + 1] - cu_k[b])
        ramp = slope * torch.arange(n, device=k.device, dtype=torch.float32)
        k[cu_k[b]:cu_k[b + 1], :, 0] = ramp[:, None].to(torch.bfloat16)
    q[:, :, 0] = 1.0
    out, lse, _, _ = gh.run_gpu(w, q, k, v, sinks, use_workspace=use_workspace, num_decode_reqs=w.num_reqs)
    ro, rl = gh.oracle_full(w, q, k, v, sinks, None)
    gh.compare(out, lse, ro, rl, what=w.name, strict=False)


@pytest.mark.parametrize("d", [128, 256])
def test_upper_bound_item_space_with_the_alternating_static_order(d):
    """A windowed batch without ranges runs every item statically, odd rounds
    walking the pairs backwards.  Sized by an upper bound of the query
    lengths (4x), most items have no rows and the scheduler jumps over them
    (to the block's first q tile with rows, or the next request with any);
    zero-row requests sit between the others.  Every item computes the same
    arithmetic whichever pair takes it: the bits must equal the call sized by
    the exact maximum, and both the oracle."""
    q_lens = [300, 0, 700, 1, 0, 520, 64, 0, 900]
    k_lens = [800, 0, 700, 1500, 3, 2000, 64, 9, 4000]
    w = workloads.Workload(f"ubound_d{d}", 70 + d, q_lens, k_lens, 8, 2, d, True, 511, 0,
                           workloads.SINK_NULL_LOGIT, None)
    q, k, v, sinks = gh.make_inputs(w)
    cu_q, cu_k = gh.device_meta(w, q.device)

    def call(max_q):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=q.device)
        mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max_q, max(k_lens), lse=lse, causal=True,
                            window_left=w.window_left, sinks=sinks, sink_mode=w.sink_mode, scale=w.scale)
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0
        return out, lse

    out_e, lse_e = call(max(q_lens))
    out_u, lse_u = call(4 * max(q_lens))
    assert torch.equal(out_e.view(torch.int16), out_u.view(torch.int16))
    assert torch.equal(lse_e, lse_u)
    ro, rl = gh.oracle_full(w, q, k, v, sinks, None)
    gh.compare(out_u, lse_u, ro, rl, what=w.name, strict=False)


def test_key0_bias_with_key0_outside_window():
    # rows beyond the window never see key 0: the bias must not touch them
    w = workloads.Workload("k0", 3, [300], [300], 4, 2, 128, False, 20, 20, workloads.SINK_KEY0_BIAS, None)
    _parity_full(w)


def test_ranges_longer_than_window():
    per = [[(10, 400), (420, 421), (600, 999)]]
    w = workloads.Workload("longrange", 5, [700], [1000], 4, 2, 128, True, 31, 0, workloads.SINK_NONE,
                           workloads.pad_ranges(per))
    _parity_full(w)


def test_empty_and_single_rows():
    w = workloads.Workload("edges", 9, [0, 1, 0, 129, 1], [0, 1, 5, 129, 2000], 8, 2, 128, True, -1, 0,
                           workloads.SINK_NULL_LOGIT, None)
    _parity_full(w)


def test_window_zero_one_key_per_row():
    w = workloads.Workload("w0", 11, [257], [257], 2, 1, 256, True, 0, 0, workloads.SINK_KEY0_BIAS, None)
    _parity_full(w)


@pytest.mark.parametrize("name", ["mixed_serving_a", "mixed_serving_b"])
def test_decode_first_batches(name):
    # decode requests first: each kernel covers only its own requests
    w = workloads.scaled_workload(name)
    n_dec = sum(1 for x in w.q_lens if x == 1)
    assert w.q_lens[:n_dec] == [1] * n_dec
    _parity_full(w, num_decode_reqs=n_dec)
    _parity_full(w, num_decode_reqs=n_dec, use_workspace=False)


def test_prefill_only_and_decode_only_batches():
    w = workloads.scaled_workload("mm_prefix_sliding")
    w.q_lens, w.k_lens = [517, 300, 129], [517, 300, 129]
    w.ranges = w.ranges[[0, 1, 3]]
    _parity_full(w, num_decode_reqs=0)
    d = workloads.Workload("dec", 5, [1] * 7, [1, 2, 700, 5000, 64, 9000, 333], 8, 2, 128, True, 1000, 0,
                           workloads.SINK_KEY0_BIAS, None)
    _parity_full(d, num_decode_reqs=7)
    _parity_full(d, num_decode_reqs=-1)


@pytest.mark.parametrize("sink_mode", [workloads.SINK_NONE, workloads.SINK_KEY0_BIAS, workloads.SINK_NULL_LOGIT])
def test_split_decode_rows(sink_mode):
    """Decode rows longer than one split-KV chunk (4096 keys): 1 to 4 chunks,
    chunk-boundary lengths, a window that starts inside a chunk, ranges, next
    to a prefill request."""
    k_lens = [4096, 4097, 8192, 9001, 12289, 100, 16000, 700]
    q_lens = [1] * 7 + [300]
    ranges = workloads.pad_ranges([[(10, 5000)], [], [(4000, 4200)], [], [(0, 3)], [], [(15000, 15999)],
                                   [(20, 80), (400, 650)]])
    for wl in (-1, 5000):
        w = workloads.Workload(f"split{sink_mode}_{wl}", 88 + sink_mode, q_lens, k_lens, 16, 4, 128, True, wl, 0,
                               sink_mode, ranges)
        _parity_full(w, num_decode_reqs=7)


FULL = ["tiny_window_sinks", "mm_prefix_sliding", "global_causal_d512", "chunked_prefill_ranges",
        "mixed_serving_a", "mixed_serving_b"]


@pytest.mark.parametrize("name", FULL)
def test_full_size_sampled_rows(name):
    """Full-size workload, bench launch configuration (workspace on), sampled
    rows: first/last rows of requests, tile boundaries, random interior rows,
    every decode row of a few requests."""
    w = workloads.workload(name)
    q, k, v, sinks = gh.make_inputs(w)
    n_dec = 0
    while n_dec < w.num_reqs and w.q_lens[n_dec] == 1:
        n_dec += 1
    out, lse, table, covered = gh.run_gpu(w, q, k, v, sinks, num_decode_reqs=n_dec)
    ref_table, n = gh.oracle_table(w)
    if ref_table is not None:
        got = table[:w.total_q].cpu().numpy()
        assert np.array_equal(got, ref_table) if n else (got == -1).all()
    cu_q, _ = w.cu_seqlens()
    rng = np.random.default_rng(1234)
    rows = set()
    for b in range(w.num_reqs):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        if q1 == q0:
            continue
        if q1 - q0 == 1:
            if rng.random() < 0.06:
                rows.add(q0)
            continue
        rows.update([q0, q1 - 1, min(q1 - 1, q0 + 63), min(q1 - 1, q0 + 64), min(q1 - 1, q0 + 127)])
        rows.update(int(x) for x in rng.integers(q0, q1, size=6))
    rows = sorted(rows)
    ro, rl = gh.oracle_rows(w, q, k, v, sinks, ref_table, rows)
    gh.compare(out, lse, ro, rl, rows=rows, what=name, strict=True)
    # every output is finite (no NaN from unwritten rows)
    assert torch.isfinite(out.float()).all()
