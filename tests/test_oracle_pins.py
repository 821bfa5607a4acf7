"""The CPU oracle against what the pages and the mathematics fix (no GPU)."""

import numpy as np
import torch

from oracle import accounting, attention, range_table
from masked_varlen_prefill_gb300 import workloads

from . import oracle_pins as pins


def make_tiny_case(seed, fill):
    w = workloads.random_tiny(seed)
    q, k, v, sinks = workloads.make_tensors(w)
    q, k, v = (x.to(torch.float64).numpy() for x in (q, k, v))
    sinks = None if sinks is None else sinks.numpy().astype(np.float64)
    cu_q, cu_k = w.cu_seqlens()
    table = None
    if w.ranges is not None:
        table = np.full((max(1, w.total_q), 2), -1, dtype=np.int32)
        fill(table, range_table.ranges_from_padded(w.ranges), cu_q, np.asarray(w.k_lens))
        table = table[:w.total_q]
    return w, q, k, v, sinks, table, cu_q, cu_k


def test_causal_formula_matches_tutorial_and_tril():
    pins.check_causal_formula(attention.visible_mask)


def test_range_table_printed_example():
    pins.check_range_example(range_table.fill_by_spans, range_table.scan_keep)
    pins.check_range_example(range_table.fill_by_scan, range_table.scan_keep)


def test_range_lookup_equals_scan_random():
    pins.check_range_lookup_random(range_table.fill_by_spans, range_table.scan_keep)


def test_scan_mode_mask():
    pins.check_scan_mask(attention.visible_mask_scan, attention.visible_mask, range_table.fill_by_spans)


def test_fill_edge_cases():
    pins.check_fill_edge_cases(range_table.fill_by_spans)
    pins.check_fill_edge_cases(range_table.fill_by_scan)


def test_span_fill_agrees_with_scan_fill():
    pins.check_fills_agree(range_table.fill_by_spans, range_table.fill_by_scan)


def test_window_count_exactly_8x():
    pins.check_window_count(accounting.visible_entries, accounting.token_context_product)


def test_rows_sum_to_one():
    pins.check_rows_sum_to_one(attention.attention_forward)


def test_sink_modes_behave_as_described():
    pins.check_sink_modes(attention.attention_forward)


def test_equals_sdpa_special_case():
    pins.check_sdpa(attention.attention_forward)


def test_brute_force_tiny():
    pins.check_brute_force(attention.attention_forward, range_table.fill_by_spans,
                           make_tiny_case, cases=150)


def test_explicit_context_lens():
    pins.check_context_lens(attention.attention_forward, range_table.fill_by_spans, make_tiny_case)


def test_row_subset_equals_full():
    """Computing a subset of rows gives the same rows as the full batch."""
    w = workloads.scaled_workload("chunked_prefill_ranges")
    w.num_heads_q, w.num_heads_kv, w.head_dim = 2, 1, 16
    q, k, v, _ = workloads.make_tensors(w)
    cu_q, cu_k = w.cu_seqlens()
    table = np.full((w.total_q, 2), -1, dtype=np.int32)
    range_table.fill_by_spans(table, range_table.ranges_from_padded(w.ranges), cu_q,
                              np.asarray(w.k_lens))
    full_o, full_l = attention.attention_forward(q, k, v, cu_q, cu_k, True, w.window_left, 0,
                                                 w.scale, range_table=table)
    rows = [0, 5, 255, 256, 300, 511, 512, w.total_q - 1]
    sub_o, sub_l = attention.attention_forward(q, k, v, cu_q, cu_k, True, w.window_left, 0,
                                               w.scale, range_table=table, rows=rows)
    # equal up to BLAS summation order
    assert np.allclose(sub_o[rows], full_o[rows], rtol=0, atol=1e-12)
    assert np.allclose(sub_l[:, rows], full_l[:, rows], rtol=0, atol=1e-12)


def test_workload_recipes():
    """The generators produce what the workload descriptions say."""
    w = workloads.workload("mm_prefix_sliding")
    assert w.ranges.shape == (4, 8, 2)
    for b in range(4):
        r = w.ranges[b]
        assert ((r[:, 1] - r[:, 0]) == 255).all()
        assert (r[:, 0] >= 0).all() and (r[:, 1] < 4096).all()
        assert (r[1:, 0] > r[:-1, 1] + 1).all()  # >= 1 free token between ranges
    w = workloads.workload("chunked_prefill_ranges")
    ctx = w.context_lens()
    assert ((ctx >= 0) & (ctx <= 30000)).all() and w.ranges.shape[1] <= 64
    for b in range(8):
        valid = [(s, e) for s, e in w.ranges[b] if s < e]
        valid.sort()
        for (s0, e0), (s1, e1) in zip(valid, valid[1:]):
            assert s1 > e0 + 1, (b, (s0, e0), (s1, e1))
        assert any(s <= ctx[b] + 2047 < e for s, e in valid)  # clipped at the chunk end
        if ctx[b] > 0:
            assert any(s < ctx[b] <= e for s, e in valid)
        for s, e in valid:
            assert 64 <= e - s + 1 <= 320
    w = workloads.workload("mixed_serving_b")
    assert w.q_lens.count(1) == 256 and w.num_reqs == 260 and w.window_left == 4095


def test_paged_gather_hand_example_and_round_trip():
    """The paged view: key j of request b is row table[b][j // bs] * bs + j % bs.
    A hand-worked table pins the index arithmetic; a generator round trip
    (random block order, garbage in unused entries) must give back the packed
    keys exactly."""
    bs = 2
    k_cache = torch.arange(8 * bs, dtype=torch.float32).reshape(8 * bs, 1, 1)
    table = np.array([[3, 0, -1], [5, 1, 6]], dtype=np.int32)
    k, v, cu = attention.gather_paged(k_cache, k_cache, table, [3, 5], bs)
    # request 0: keys 0,1 in block 3 (rows 6,7), key 2 in block 0 (row 0)
    # request 1: keys 0,1 block 5 (rows 10,11), keys 2,3 block 1 (rows 2,3), key 4 block 6 (row 12)
    assert k[:, 0, 0].tolist() == [6, 7, 0, 10, 11, 2, 3, 12]
    assert cu.tolist() == [0, 3, 8]
    gen = torch.Generator().manual_seed(3)
    lens = [5, 37, 1, 64]
    kp = torch.randn(sum(lens), 2, 8, generator=gen).to(torch.bfloat16)
    vp = torch.randn(sum(lens), 2, 8, generator=gen).to(torch.bfloat16)
    for block in (16, 32):
        kc, vc, bt, sl = workloads.to_paged(kp, vp, lens, block, seed=block, table_fill=99999)
        k2, v2, cu2 = attention.gather_paged(kc, vc, bt.numpy(), sl.numpy(), block)
        assert np.array_equal(k2, kp.to(torch.float64).numpy())
        assert np.array_equal(v2, vp.to(torch.float64).numpy())
        assert cu2.tolist() == [0, 5, 42, 43, 107]
