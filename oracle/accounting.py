"""Oracle: score-entry accounting (test infrastructure).

* :func:`visible_entries` counts the True entries of the dense mask of
  :mod:`oracle.attention`, request by request.  This is the exact number of
  score entries a masked attention has to compute per query head; the
  effective-FLOP figure is ``4 * D * Hq * visible_entries`` (one multiply-add
  for ``q.k`` and one for ``p*v`` per entry and head dimension).
* :func:`token_context_product` restates the per-request estimate of vLLM
  PR #55624 ("Support Sliding Window Attention ... in MFU/MBU estimation"),
  section "Key source snippets" (``ExecutionContext``): the sum over requests
  of ``num_tokens * min(context_len, sliding_window)``, or of
  ``num_tokens * context_len`` when there is no window.  The page's own
  risk section calls it an upper bound (it ignores the prefill triangle); it is
  kept here to pin the exact count against it.
"""

from __future__ import annotations

import numpy as np

from .attention import visible_mask


def visible_entries(cu_seqlens_q, cu_seqlens_k, causal, window_left, window_right,
                    context_lens=None, range_table=None, row_chunk=4096) -> int:
    """Exact number of visible (query row, key) pairs over the packed batch."""
    cu_q = [int(x) for x in np.asarray(cu_seqlens_q).reshape(-1)]
    cu_k = [int(x) for x in np.asarray(cu_seqlens_k).reshape(-1)]
    table = None if range_table is None else np.asarray(range_table, dtype=np.int64)
    total = 0
    for b in range(len(cu_q) - 1):
        q_len = cu_q[b + 1] - cu_q[b]
        k_len = cu_k[b + 1] - cu_k[b]
        ctx = (k_len - q_len) if context_lens is None else int(np.asarray(context_lens)[b])
        for r0 in range(0, q_len, row_chunk):
            rows = np.arange(r0, min(q_len, r0 + row_chunk))
            rr = None if table is None else table[cu_q[b] + rows]
            total += int(visible_mask(rows, k_len, ctx, causal, window_left,
                                      window_right, rr).sum())
    return total


def token_context_product(requests, sliding_window=None) -> int:
    """``sum(num_tokens * min(context_len, window))`` over ``requests``.

    ``requests`` is a list of ``(num_tokens, context_len)``; with no window the
    plain product is summed.
    """
    if sliding_window is None:
        return sum(n * c for n, c in requests)
    return sum(n * min(c, sliding_window) for n, c in requests)
