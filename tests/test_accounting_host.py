"""Work accounting (``mvp_attn_accounting``; host only, no GPU needed).

Pins:
* the PR #55624 window clamp: a decode token with 8192 keys of context
  under a 1024-token window costs exactly 1/8 of the unwindowed attn_qk /
  attn_av FLOPs and KV reads, and 512 keys of context cost the same with and
  without the window (the page's test_attention_metrics_sliding_window_flops_bounds);
* the exact visible pairs equal the oracle's dense mask, summed;
* the page's estimate bounds the exact count from above without ranges (its
  risk section's claim) and can fall below it with bidirectional ranges under
  a window (the window clamps a range on the past side only);
* the executed tile work covers every visible pair, and the decode kernel's
  aligned walk covers each row's hull by less than one tile.
"""

import numpy as np
import pytest

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import attention as oatt
from oracle import range_table as ort

# tile shapes of the kernels: keys per prefill tile; per key tile, the
# tcgen05.mma instructions and their FLOPs (D 64: one CTA, M 128; D 128 / 256:
# a CTA pair, M 256; D 512: a CTA pair, M 256, half the value columns per item);
# keys per decode tile
BN = {64: 128, 128: 128, 256: 128, 512: 64}
# (D 128: the PV MMA also sums the rows, 2 x 16 more columns)
INSTR_PER_TILE = {64: 64 // 16 + 128 // 16, 128: 128 // 16 + 128 // 16, 256: 256 // 16 + 128 // 16,
                  512: 512 // 16 + 64 // 16}
FLOPS_PER_TILE = {64: 2 * 128 * 128 * (64 + 64), 128: 2 * 256 * 128 * (128 + 128 + 32),
                  256: 2 * 256 * 128 * (256 + 256), 512: 2 * 256 * 64 * (512 + 256)}
# the opt-in D 512 head-dim split: two CTAs, each M 128 over half the head
# dimension and half the value columns
HEAD_SPLIT_INSTR = 2 * (256 // 16 + 64 // 16)
HEAD_SPLIT_FLOPS = 2 * (2 * 128 * 64 * (256 + 256))
KT = {64: 128, 128: 64, 256: 32, 512: 32}


def _counts(w, table=None, context_lens=None, variant=0):
    cu_q, _ = w.cu_seqlens()
    return mvp.attn_accounting(cu_q, w.k_lens, w.num_heads_q, w.num_heads_kv, w.head_dim,
                               context_lens=context_lens, range_table=table, causal=w.causal,
                               window_left=w.window_left, window_right=w.window_right, variant=variant)


def _table(w):
    if w.ranges is None:
        return None
    cu_q, _ = w.cu_seqlens()
    out = np.full((max(1, w.total_q), 2), 7, dtype=np.int32)
    n = ort.fill_by_spans(out, ort.ranges_from_padded(w.ranges), cu_q, np.asarray(w.k_lens))
    t = out[:w.total_q].copy()
    if n == 0:
        t[:] = -1
    return t


def _dense_visible(w, table):
    cu_q, cu_k = w.cu_seqlens()
    pre = dec = 0
    for b in range(w.num_reqs):
        q0, q1 = int(cu_q[b]), int(cu_q[b + 1])
        kl = int(cu_k[b + 1] - cu_k[b])
        if q1 == q0:
            continue
        m = oatt.visible_mask(np.arange(q1 - q0), kl, kl - (q1 - q0), w.causal, w.window_left, w.window_right,
                              None if table is None else table[q0:q1])
        if q1 - q0 == 1:
            dec += int(m.sum())
        else:
            pre += int(m.sum())
    return pre, dec


def test_page_window_clamp_is_exactly_eightfold():
    for ctx, ratio in [(8192, 8), (512, 1)]:
        args = dict(cu_seqlens_q=[0, 1], seq_lens_k=[ctx], num_heads_q=16, num_heads_kv=16, head_dim=128)
        dense = mvp.attn_accounting(**args, window_left=-1)
        swa = mvp.attn_accounting(**args, window_left=1023)
        assert swa["est_attn_qk_flops"] * ratio == dense["est_attn_qk_flops"]
        assert swa["est_attn_av_flops"] * ratio == dense["est_attn_av_flops"]
        assert swa["est_decode_kv_read_bytes"] * ratio == dense["est_decode_kv_read_bytes"]
        # the formula itself: 2 heads head_dim per token-context product
        assert dense["est_attn_qk_flops"] == 2 * 16 * 128 * ctx
        assert dense["est_decode_kv_read_bytes"] == 2 * 16 * 128 * 2 * ctx
        # exact: the decode row sees min(ctx, window) keys
        assert swa["visible_decode"] == min(ctx, 1024) and dense["visible_decode"] == ctx


@pytest.mark.parametrize("seed", range(24))
def test_exact_visible_equals_dense_oracle_mask(seed):
    w = workloads.random_case(seed)
    table = _table(w)
    c = _counts(w, table)
    pre, dec = _dense_visible(w, table)
    assert (c["visible_prefill"], c["visible_decode"]) == (pre, dec)
    assert c["exact_flops"] == 4.0 * w.head_dim * w.num_heads_q * (pre + dec)


@pytest.mark.parametrize("name", ["mm_prefix_sliding", "chunked_prefill_ranges", "mixed_serving_b",
                                  "global_causal_d512", "tiny_window_sinks"])
def test_scaled_workloads_exact_and_executed(name):
    w = workloads.scaled_workload(name)
    table = _table(w)
    c = _counts(w, table)
    pre, dec = _dense_visible(w, table)
    assert (c["visible_prefill"], c["visible_decode"]) == (pre, dec)
    d = w.head_dim
    # every visible pair of a prefill row is inside a visited tile
    assert c["prefill_mma_flops"] >= 4.0 * d * w.num_heads_q * pre
    assert c["prefill_mma_instructions"] == c["prefill_tiles"] * INSTR_PER_TILE[d]
    assert c["prefill_mma_flops"] == c["prefill_tiles"] * FLOPS_PER_TILE[d]


def test_d512_head_split_accounting():
    w = workloads.scaled_workload("global_causal_d512")
    base = _counts(w)
    split = _counts(w, variant=mvp.VARIANT_D512_HEAD_SPLIT)
    # the same visible pairs; items of 128 rows with every value column (the
    # default's items are 256 rows with half of them); QK is not recomputed
    # per value half, so at most two thirds of the default's MMA work (less
    # where the narrower items skip more causal tiles)
    assert split["visible_prefill"] == base["visible_prefill"]
    assert split["prefill_mma_instructions"] == split["prefill_tiles"] * HEAD_SPLIT_INSTR
    assert split["prefill_mma_flops"] == split["prefill_tiles"] * HEAD_SPLIT_FLOPS
    assert split["prefill_mma_flops"] * 3 <= base["prefill_mma_flops"] * 2


@pytest.mark.parametrize("seed", range(16))
def test_estimate_bounds_exact_without_ranges(seed):
    w = workloads.random_case(100 + seed)
    if not w.causal:
        w.causal, w.window_right = True, 0
    c = _counts(w, None)
    assert c["est_token_context_product"] >= c["visible_prefill"] + c["visible_decode"]


def test_estimate_misses_bidirectional_ranges_under_a_window():
    # 100 prefill tokens, one range over all of them, 10-token causal window:
    # the window clamps the range on the past side only, so row p sees keys
    # max(0, p - 9) .. 99
    w = workloads.Workload("r", 0, [100], [100], 2, 1, 64, True, 9, 0, workloads.SINK_NONE,
                           workloads.pad_ranges([[(0, 99)]]))
    table = _table(w)
    c = _counts(w, table)
    pre, _ = _dense_visible(w, table)
    assert c["visible_prefill"] == pre == sum(100 - max(0, p - 9) for p in range(100))
    assert c["est_token_context_product"] == 100 * 10 < pre


@pytest.mark.parametrize("seed", range(16))
def test_decode_walk_covers_each_hull_by_less_than_a_tile(seed):
    rng = np.random.default_rng(seed)
    d = int(rng.choice([64, 128, 256, 512]))
    n = int(rng.integers(1, 30))
    k = rng.integers(1, 5000, size=n).astype(np.int32)
    wl = int(rng.choice([-1, 0, 31, 1000]))
    c = mvp.attn_accounting(np.arange(n + 1, dtype=np.int32), k, 4, 2, d, window_left=wl)
    hull = np.minimum(k, wl + 1) if wl >= 0 else k  # one decode row per request: keys [k - hull, k)
    assert c["visible_decode"] == int(hull.sum())
    walked = 0
    for kl, h in zip(k.tolist(), hull.tolist()):
        lo = (kl - h) & ~(KT[d] - 1)
        walked += -(-(kl - lo) // KT[d]) * KT[d]
    assert c["decode_keys_walked"] == walked
    assert walked >= hull.sum() and walked < hull.sum() + 2 * KT[d] * n
    assert c["decode_read_bytes"] == walked * 2 * d * 2 * 2 + n * 4 * d * 2


def test_headline_workload_counts():
    w = workloads.workload("mm_prefix_sliding")
    c = _counts(w, _table(w))
    # 4 requests x 32 items of 128 positions x 8 KV heads
    assert c["prefill_items"] == 4 * 32 * 8
    # q and out once (bf16), K and V once: everything of the 4 requests is reached
    assert c["prefill_compulsory_bytes"] == 2 * 16384 * 16 * 256 * 2 + 2 * 16384 * 8 * 256 * 2
    assert c["est_token_context_product"] == 4 * 4096 * 1024


def test_argument_errors():
    with pytest.raises(mvp.MvpError):
        mvp.attn_accounting([1, 2], [3], 2, 1, 64)          # offsets not starting at 0
    with pytest.raises(mvp.MvpError):
        mvp.attn_accounting([0, 5], [3], 2, 1, 64)          # fewer keys than queries
    with pytest.raises(mvp.MvpError):
        mvp.attn_accounting([0, 1], [3], 3, 2, 64)          # heads not a multiple
    with pytest.raises(mvp.MvpError):
        mvp.attn_accounting([0, 1], [3], 2, 1, 96)          # head_dim
    with pytest.raises(mvp.MvpError):
        mvp.attn_accounting([0, 1], [3], 2, 1, 64, window_left=-2)
    with pytest.raises(mvp.MvpError):
        mvp.attn_accounting([0, 1], [3], 2, 1, 64, variant=7)   # unknown variant
    with pytest.raises(mvp.MvpError) as e:
        mvp.attn_accounting([0, 1], [3], 2, 1, 256, variant=mvp.VARIANT_D512_HEAD_SPLIT)
    assert e.value.status == mvp.MVP_ERR_UNSUPPORTED
    lib = mvp.load_library()
    assert lib.mvp_attn_accounting(None, None, None, None, 0, 1, 1, 64, 1, -1, -1, 0, None) == mvp.MVP_ERR_ARG
