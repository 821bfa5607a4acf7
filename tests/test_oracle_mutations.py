"""Planted mistakes in copies of the oracle must be caught by the pins.

Each case copies one oracle module's source, applies one plausible mistake
(a wrong sign, a dropped term, a wrong index, an off-by-one range end) and
runs the pin that should catch it.  The real oracle is never modified.
"""

import importlib.util
import os
import types

import numpy as np
import pytest

from oracle import accounting as real_accounting
from oracle import range_table as real_range_table

from . import oracle_pins as pins
from .test_oracle_pins import make_tiny_case

ORACLE = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "oracle")


def _mutant(module_file, old, new, count=1):
    path = os.path.join(ORACLE, module_file)
    src = open(path).read()
    assert src.count(old) >= count, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new, count)
    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = path
    exec(compile(src, path + "<mutant>", "exec"), mod.__dict__)
    return mod


def _window_count_with(att):
    def visible_entries(cu_q, cu_k, causal, wl, wr, context_lens=None, range_table=None):
        total = 0
        for b in range(len(cu_q) - 1):
            ql = int(cu_q[b + 1] - cu_q[b]); kl = int(cu_k[b + 1] - cu_k[b])
            total += int(att.visible_mask(np.arange(ql), kl, kl - ql, causal, wl, wr).sum())
        return total
    pins.check_window_count(visible_entries, real_accounting.token_context_product)


ATTENTION_MUTANTS = [
    # window sign flipped on the causal side
    ("window_sign", "base = base & (j >= p - window_left)", "base = base & (j >= p + window_left)",
     lambda m: _window_count_with(m)),
    # window off by one (keeps W+1 keys)
    ("window_off_by_one", "base = base & (j >= p - window_left)",
     "base = base & (j >= p - window_left - 1)", lambda m: _window_count_with(m)),
    # causal comparison strict (drops the diagonal)
    ("causal_strict", "base = j <= p\n", "base = j < p\n",
     lambda m: pins.check_causal_formula(m.visible_mask)),
    # context offset ignored (the packed-row reading)
    ("ctx_dropped", "p = ctx + i", "p = i", lambda m: pins.check_causal_formula(m.visible_mask)),
    # an explicit context length ignored (always k_len - q_len)
    ("explicit_ctx_ignored",
     "ctx = (k_len - q_len) if context_lens is None else int(np.asarray(context_lens)[b])",
     "ctx = k_len - q_len",
     lambda m: pins.check_context_lens(m.attention_forward, real_range_table.fill_by_spans, make_tiny_case,
                                       cases=10)),
    # range end treated as half-open
    ("range_half_open", "in_range = (start <= j) & (j <= end)", "in_range = (start <= j) & (j < end)",
     lambda m: pins.check_brute_force(m.attention_forward, real_range_table.fill_by_spans,
                                      make_tiny_case, cases=60)),
    # window clamp on the range part dropped
    ("range_unclamped", "in_range = in_range & (j >= p - window_left)", "in_range = in_range",
     lambda m: pins.check_brute_force(m.attention_forward, real_range_table.fill_by_spans,
                                      make_tiny_case, cases=150)),
    # null-logit sink dropped from the denominator
    ("null_sink_dropped", "z = z + np.exp(sinks[h] - safe_max)", "z = z",
     lambda m: pins.check_rows_sum_to_one(m.attention_forward)),
    # key-0 bias with the wrong sign
    ("key0_sign", "s[:, 0] = s[:, 0] + sinks[h]", "s[:, 0] = s[:, 0] - sinks[h]",
     lambda m: pins.check_sink_modes(m.attention_forward)),
    # GQA head map transposed (h % G instead of h // G)
    ("gqa_modulo", "kh = k[:, h // group, :]", "kh = k[:, h % hkv, :]",
     lambda m: pins.check_sdpa(m.attention_forward)),
    # scale applied twice
    ("scale_twice", "s = scale * (q[q_rows, h, :] @ kh.T)", "s = scale * scale * (q[q_rows, h, :] @ kh.T)",
     lambda m: pins.check_sdpa(m.attention_forward)),
    # V transposed against K's head
    ("v_head", "vh = v[:, h // group, :]", "vh = v[:, (h + 1) % hkv, :]",
     lambda m: pins.check_sdpa(m.attention_forward)),
    # LSE without the max shift
    ("lse_shift", "safe_max + np.log(z)", "np.log(z)",
     lambda m: pins.check_sdpa(m.attention_forward)),
    # scan mode: only the first listed range consulted
    ("scan_first_only", "for start, end in req_ranges:", "for start, end in req_ranges[:1]:",
     lambda m: pins.check_scan_mask(m.visible_mask_scan, m.visible_mask, real_range_table.fill_by_spans)),
    # scan mode: the query side of "holds both" dropped
    ("scan_query_unchecked", "keep |= (start <= p) & (p <= end) & (start <= j) & (j <= end)",
     "keep |= (start <= j) & (j <= end)",
     lambda m: pins.check_scan_mask(m.visible_mask_scan, m.visible_mask, real_range_table.fill_by_spans)),
    # scan mode: the window clamp on the range part dropped
    ("scan_unclamped", "keep &= j >= p - window_left", "keep &= True",
     lambda m: pins.check_scan_mask(m.visible_mask_scan, m.visible_mask, real_range_table.fill_by_spans)),
]


@pytest.mark.parametrize("name,old,new,check", ATTENTION_MUTANTS, ids=[m[0] for m in ATTENTION_MUTANTS])
def test_attention_mutant_is_caught(name, old, new, check):
    mutant = _mutant("attention.py", old, new)
    with pytest.raises(AssertionError):
        check(mutant)


RANGE_MUTANTS = [
    ("degenerate_kept", "if start >= end:\n                continue", "if start > end:\n                continue",
     lambda m: pins.check_fill_edge_cases(m.fill_by_spans)),
    ("no_reset", "out[:n_tokens] = NO_RANGE\n", "pass\n",
     lambda m: pins.check_fill_edge_cases(m.fill_by_spans)),
    ("ctx_sign", "ctx = int(seq_lens[b]) - q_len  # absolute", "ctx = q_len - int(seq_lens[b])  # absolute",
     lambda m: pins.check_range_example(m.fill_by_spans, real_range_table.scan_keep)),
    ("clip_exclusive", "hi = min(end - ctx, q_len - 1)", "hi = min(end - ctx - 1, q_len - 1)",
     lambda m: pins.check_range_example(m.fill_by_spans, real_range_table.scan_keep)),
    ("first_wins", "hit = (start, end)  # later", "hit = hit or (start, end)  # later",
     lambda m: pins.check_fills_agree(real_range_table.fill_by_spans, m.fill_by_scan)),
]


@pytest.mark.parametrize("name,old,new,check", RANGE_MUTANTS, ids=[m[0] for m in RANGE_MUTANTS])
def test_range_mutant_is_caught(name, old, new, check):
    mutant = _mutant("range_table.py", old, new)
    with pytest.raises(AssertionError):
        check(mutant)


def test_mutation_harness_runs_real_oracle_clean():
    """The harness itself: an identity 'mutation' passes every check."""
    m = _mutant("attention.py", "import math", "import math")
    pins.check_sdpa(m.attention_forward)
    _window_count_with(m)
