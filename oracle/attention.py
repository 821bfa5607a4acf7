"""Oracle: dense masked varlen attention forward in float64 (test infrastructure).

Definitions restated here, each from the page that fixes it:

* Causal with a chunked-prefill offset -- step14_4 "Causal Mask optimisation"
  tutorial, section "broadcast comparison": query ``i`` of a chunk whose first
  token sits at ``start_pos`` may not see key ``j`` iff ``j > start_pos + i``.
  Here ``start_pos`` is the request's context length ``ctx``.
* Sliding window -- vLLM PR #50294 review, "Key source snippets" (the
  ``mask_mod`` and its ``forward()`` wiring): with ``delta = p - j`` the causal
  side keeps ``0 <= delta < 1 + window_left``, i.e. ``j >= p - window_left``.
  A non-causal symmetric window keeps ``|p - j| <= w`` (vLLM PR #49815 review,
  the ``_reference`` test helper), i.e. ``window_left = window_right = w``.
  ``-1`` means the side is unbounded.
* Multimodal-prefix ranges -- PR #50294 ``mask_mod``: a key is also visible
  when it lies in the closed ``[start, end]`` of the query row's range-table
  entry; the window clamps that part on the past side only.  The visible set
  is ``base OR range``.  ``(-1, -1)`` never matches a key ``>= 0``.
* Scan mode -- the request-level range list that PR #50294 keeps for the
  Triton path (``(num_seqs, max_ranges, 2)``, "Implementation breakdown" 2)
  and the old per-score rule its metadata test restates: a key is also
  visible when some valid range (``start < end``) holds both the query
  position and the key, with the same past-side window clamp.
* Scores, sinks, softmax -- PR #49815 review, "Key source snippets": scores are
  ``scale * q.k`` with KV head ``h // G`` (``repeat_interleave`` grouping).
  Key-0-bias mode adds ``sink[h]`` to the logit of key 0 when key 0 is
  visible; null-logit mode adds ``exp(sink[h])`` to the softmax denominator
  only.  Both are in natural-log units.
* LSE is not on the pages; it is defined here as ``ln Z`` of the row's full
  denominator (sink term included).  A row with nothing visible gets output
  0 and LSE ``-inf`` (``sink`` in null-logit mode).

Everything is materialised: the boolean mask ``[rows, k_len]`` by broadcast,
then a dense float64 score matrix per head, then a max-subtracted softmax.
"""

from __future__ import annotations

import math

import numpy as np

SINK_NONE = 0
SINK_KEY0_BIAS = 1
SINK_NULL_LOGIT = 2


def visible_mask(q_rows, k_len, ctx, causal, window_left, window_right, row_ranges=None):
    """Dense boolean mask ``[len(q_rows), k_len]``; True = key visible.

    ``q_rows`` are local query indices ``i`` (absolute position ``ctx + i``);
    ``row_ranges`` is ``[len(q_rows), 2]`` of closed ``(start, end)`` or None.
    """
    i = np.asarray(q_rows, dtype=np.int64).reshape(-1, 1)
    j = np.arange(k_len, dtype=np.int64).reshape(1, -1)
    p = ctx + i
    if causal:
        base = j <= p
    elif window_right >= 0:
        base = j <= p + window_right
    else:
        base = np.ones((i.shape[0], k_len), dtype=bool)
    if window_left >= 0:
        base = base & (j >= p - window_left)
    if row_ranges is None:
        return base
    rr = np.asarray(row_ranges, dtype=np.int64).reshape(-1, 2)
    start = rr[:, 0:1]
    end = rr[:, 1:2]
    in_range = (start <= j) & (j <= end)
    if window_left >= 0:
        in_range = in_range & (j >= p - window_left)
    return base | in_range


def visible_mask_scan(q_rows, k_len, ctx, causal, window_left, window_right, req_ranges):
    """Dense mask of scan mode: ``base OR any(range holds query and key)``.

    ``req_ranges`` is the request's list of closed ``(start, end)``; entries
    with ``start >= end`` are skipped, as the scan skips them.
    """
    base = visible_mask(q_rows, k_len, ctx, causal, window_left, window_right, None)
    i = np.asarray(q_rows, dtype=np.int64).reshape(-1, 1)
    j = np.arange(k_len, dtype=np.int64).reshape(1, -1)
    p = ctx + i
    keep = np.zeros_like(base)
    for start, end in req_ranges:
        if not start < end:
            continue
        keep |= (start <= p) & (p <= end) & (start <= j) & (j <= end)
    if window_left >= 0:
        keep &= j >= p - window_left
    return base | keep


def _as_f64(x):
    """Widen a torch/numpy bf16/fp32 array to float64 exactly."""
    try:
        import torch

        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover - torch is always present here
        pass
    return np.asarray(x, dtype=np.float64)


def attend_rows(q_rows, q, k, v, ctx, causal, window_left, window_right,
                row_ranges, sinks, sink_mode, scale, req_ranges=None):
    """Attention for some query rows of ONE request, every query head.

    q: ``[q_len, Hq, D]``; k: ``[k_len, Hkv, D]``; v: ``[k_len, Hkv, Dv]``
    (float64).  Returns ``out [rows, Hq, Dv]`` and ``lse [Hq, rows]``.
    ``req_ranges`` (the request's range list) selects scan mode instead of
    the per-row ``row_ranges``.
    """
    q_rows = np.asarray(q_rows, dtype=np.int64)
    n_rows = q_rows.shape[0]
    k_len, hkv = k.shape[0], k.shape[1]
    hq = q.shape[1]
    group = hq // hkv
    dv = v.shape[2]
    if req_ranges is not None:
        mask = visible_mask_scan(q_rows, k_len, ctx, causal, window_left, window_right, req_ranges)
    else:
        mask = visible_mask(q_rows, k_len, ctx, causal, window_left, window_right, row_ranges)
    out = np.zeros((n_rows, hq, dv), dtype=np.float64)
    lse = np.full((hq, n_rows), -np.inf, dtype=np.float64)
    for h in range(hq):
        kh = k[:, h // group, :]
        vh = v[:, h // group, :]
        s = scale * (q[q_rows, h, :] @ kh.T)  # [rows, k_len]
        if sink_mode == SINK_KEY0_BIAS and k_len > 0:
            s[:, 0] = s[:, 0] + sinks[h]
        s = np.where(mask, s, -np.inf)
        row_max = s.max(axis=1) if k_len > 0 else np.full(n_rows, -np.inf)
        if sink_mode == SINK_NULL_LOGIT:
            row_max = np.maximum(row_max, sinks[h])
        safe_max = np.where(np.isfinite(row_max), row_max, 0.0)
        e = np.where(mask, np.exp(s - safe_max[:, None]), 0.0)
        z = e.sum(axis=1)
        if sink_mode == SINK_NULL_LOGIT:
            z = z + np.exp(sinks[h] - safe_max)
        with np.errstate(divide="ignore", invalid="ignore"):
            out[:, h, :] = np.where(z[:, None] > 0, (e @ vh) / z[:, None], 0.0)
            lse[h] = np.where(z > 0, safe_max + np.log(z), -np.inf)
    return out, lse


def attention_forward(q, k, v, cu_seqlens_q, cu_seqlens_k, causal, window_left,
                      window_right, scale, context_lens=None, range_table=None,
                      sinks=None, sink_mode=SINK_NONE, rows=None, scan_ranges=None):
    """Whole packed batch (or the packed rows listed in ``rows``).

    q ``[total_q, Hq, D]``, k/v ``[total_k, Hkv, D]`` (any dtype; widened to
    float64); ``range_table`` ``[total_q, 2]`` int or None; ``scan_ranges``
    ``[B, max_ranges, 2]`` (scan mode, instead of a table) or None.  Returns
    ``out [total_q, Hq, Dv]`` and ``lse [Hq, total_q]`` in float64.  With
    ``rows`` given, only those packed rows are computed; the others stay 0 /
    NaN and callers compare only the requested rows.
    """
    q = _as_f64(q)
    k = _as_f64(k)
    v = _as_f64(v)
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    sinks = None if sinks is None else _as_f64(sinks).reshape(-1)
    table = None if range_table is None else np.asarray(range_table, dtype=np.int64)
    total_q, hq, _ = q.shape
    out = np.zeros((total_q, hq, v.shape[2]), dtype=np.float64)
    lse = np.full((hq, total_q), np.nan, dtype=np.float64)
    wanted = None if rows is None else np.asarray(sorted(set(int(r) for r in rows)))
    for b in range(len(cu_q) - 1):
        q0, q1 = cu_q[b], cu_q[b + 1]
        k0, k1 = cu_k[b], cu_k[b + 1]
        q_len, k_len = q1 - q0, k1 - k0
        if q_len <= 0:
            continue
        ctx = (k_len - q_len) if context_lens is None else int(np.asarray(context_lens)[b])
        if wanted is None:
            local = np.arange(q_len)
        else:
            sel = wanted[(wanted >= q0) & (wanted < q1)]
            if sel.size == 0:
                continue
            local = sel - q0
        rr = None if table is None else table[q0 + local]
        req = None if scan_ranges is None else [(int(s_), int(e_)) for s_, e_ in np.asarray(scan_ranges)[b]]
        o, l = attend_rows(local, q[q0:q1], k[k0:k1], v[k0:k1], ctx, causal,
                           window_left, window_right, rr, sinks, sink_mode, scale, req_ranges=req)
        out[q0 + local] = o
        lse[:, q0 + local] = l
    return out, lse


def gather_paged(k_cache, v_cache, block_table, seq_lens, block_size):
    """Packed ``(k, v, cu_seqlens_k)`` from a paged cache (float64 oracle view).

    The paged layout of vLLM's paged attention, which the FA4 pages run their
    masks on: key ``j`` of request ``b`` is row
    ``block_table[b][j // block_size] * block_size + j % block_size`` of
    ``k_cache`` / ``v_cache`` (``[num_blocks * block_size, Hkv, D]``).  The
    paged forward pass is the packed forward pass of these gathered keys.
    """
    kc = np.asarray(_as_f64(k_cache))
    vc = np.asarray(_as_f64(v_cache))
    bt = np.asarray(block_table)
    rows = []
    for b, n in enumerate(np.asarray(seq_lens).tolist()):
        for j in range(int(n)):
            rows.append(int(bt[b, j // block_size]) * block_size + j % block_size)
    idx = np.asarray(rows, dtype=np.int64)
    cu = np.zeros(len(seq_lens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(seq_lens, dtype=np.int64))
    return kc[idx], vc[idx], cu


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
