"""Oracle: the per-query-row multimodal-prefix range table (test infrastructure).

Source: vLLM PR #50294 review ("FA4 mm_prefix range scan -> O(1) table
lookup", prhub.com.cn), sections "Implementation breakdown" step 1 and "Key
source snippets" (``fill_mm_prefix_query_ranges`` and the metadata test
``test_matches_range_scan_semantics_with_context_offset``).

What the table is.  Row ``t`` of an ``(num_actual_tokens, 2)`` int32 table
belongs to packed query token ``t``.  It holds the absolute ``[start, end]``
(both ends inclusive, as every comparison on that page is written) of the
bidirectional range of that token's request that contains the token's absolute
position, or ``(-1, -1)`` when no range does.  A query token of request ``b``
with local index ``i`` sits at absolute position ``ctx_b + i`` where
``ctx_b = seq_len_b - query_len_b``.

Two independent constructions are given:

* :func:`fill_by_spans` follows the page's fill procedure: for every request
  turn each valid range (``start < end``) into the span of local query rows it
  covers, clipped to the scheduled chunk; drop ranges that clip to nothing;
  if any span survives, reset rows ``[0, N)`` to ``-1`` and write the spans in
  list order; return ``N`` if something was written, else ``0`` with the
  caller's buffer untouched.
* :func:`fill_by_scan` is the brute-force reading: every row scans all of its
  request's ranges in list order and keeps the last valid range whose closed
  interval contains the row's absolute position.  This is the O(max_ranges)
  per-row work that the page says the old kernel did per score.

Both return the page's return value (``N`` or ``0``).
"""

from __future__ import annotations

import numpy as np

NO_RANGE = -1


def ranges_from_padded(ranges: np.ndarray) -> dict[int, list[tuple[int, int]]]:
    """Turn a padded ``[B, max_ranges, 2]`` array into the page's dict form.

    Padding entries are ordinary degenerate ranges (``start >= end``); they are
    kept, because both fills skip them exactly as they skip any degenerate
    range, so dropping them here would hide a bug in that skip.
    """
    ranges = np.asarray(ranges)
    out: dict[int, list[tuple[int, int]]] = {}
    for b in range(ranges.shape[0]):
        out[b] = [(int(s), int(e)) for s, e in ranges[b]]
    return out


def fill_by_spans(out: np.ndarray, req_ranges, query_start_loc, seq_lens) -> int:
    """Fill ``out`` the way the PR #50294 helper does; return rows written.

    ``out`` is the caller's ``(capacity, 2)`` int32 staging buffer.  Raises
    ``ValueError`` when the scheduled tokens do not fit (the page asserts).
    """
    if req_ranges is None:
        return 0
    qsl = [int(x) for x in np.asarray(query_start_loc).reshape(-1)]
    n_tokens = qsl[-1]
    if n_tokens <= 0:
        return 0
    if n_tokens > out.shape[0]:
        raise ValueError(f"staging buffer holds {out.shape[0]} rows, need {n_tokens}")

    # Resolve every range to a clipped span of packed rows before touching
    # the buffer: a batch whose ranges all fall outside the scheduled chunk
    # must leave the buffer as it was.
    spans = []
    for b, ranges in req_ranges.items():
        if not ranges:
            continue
        first_row = qsl[b]
        q_len = qsl[b + 1] - first_row
        if q_len <= 0:
            continue
        ctx = int(seq_lens[b]) - q_len  # absolute position of local row 0
        for start, end in ranges:
            if start >= end:
                continue  # degenerate ranges are skipped
            lo = max(start - ctx, 0)
            hi = min(end - ctx, q_len - 1)
            if lo > hi:
                continue  # wholly outside the scheduled chunk
            spans.append((first_row + lo, first_row + hi + 1, start, end))
    if not spans:
        return 0

    # The buffer is reused across steps: every scheduled row is reset first
    # so that no stale range survives outside this step's spans.
    out[:n_tokens] = NO_RANGE
    for row_lo, row_hi, start, end in spans:
        out[row_lo:row_hi, 0] = start
        out[row_lo:row_hi, 1] = end
    return n_tokens


def fill_by_scan(out: np.ndarray, req_ranges, query_start_loc, seq_lens) -> int:
    """Brute-force table: per row, scan the request's ranges in list order.

    The rows are resolved into a private table first.  If at least one row got
    a range, rows ``[0, N)`` of ``out`` are overwritten with it and ``N`` is
    returned; otherwise ``out`` is left as it was and ``0`` is returned, which
    is the page's contract for a batch with no covered query token.
    """
    qsl = [int(x) for x in np.asarray(query_start_loc).reshape(-1)]
    n_tokens = qsl[-1]
    if req_ranges is None or n_tokens <= 0:
        return 0
    if n_tokens > out.shape[0]:
        raise ValueError(f"staging buffer holds {out.shape[0]} rows, need {n_tokens}")
    table = np.full((n_tokens, 2), NO_RANGE, dtype=np.int64)
    covered = False
    for b in range(len(qsl) - 1):
        q_len = qsl[b + 1] - qsl[b]
        ctx = int(seq_lens[b]) - q_len
        ranges = req_ranges.get(b, []) if isinstance(req_ranges, dict) else req_ranges[b]
        for i in range(q_len):
            q_abs = ctx + i
            hit = None
            for start, end in ranges:
                if start < end and start <= q_abs <= end:
                    hit = (start, end)  # later ranges win, as later spans overwrite
            if hit is not None:
                table[qsl[b] + i] = hit
                covered = True
    if not covered:
        return 0
    out[:n_tokens] = table.astype(out.dtype)
    return n_tokens


def scan_keep(req_ranges_b, q_abs: int, kv_idx: int) -> bool:
    """The old per-score test: some valid range holds both query and key."""
    return any(s < e and s <= q_abs <= e and s <= kv_idx <= e for s, e in req_ranges_b)
