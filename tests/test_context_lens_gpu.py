"""An explicit ``context_lens`` through the C-ABI vs the float64 oracle (GPU).

The spec signature passes each request's context length; the query at
local index i then sits at absolute position ``ctx + i`` (step14_4 "Causal
Mask optimisation" tutorial, *Solution*: key j is masked iff
``j > start_pos + i``; vLLM PR #50294 review, the metadata test with a context
offset).  Covered here, each compared element by element with
``oracle.attention.attention_forward(..., context_lens=...)``:

* ``context_lens`` equal to ``k_len - q_len`` on a decode-first batch with
  ranges (one holding a decode row), a window and null-logit sinks, through
  the packed, paged and scan entry points, with and without workspace;
* a ``context_lens`` that differs from ``k_len - q_len`` (queries that end
  before the last key), causal and symmetric-window masks: it alone defines
  the positions;
* a sub-batch passed as slices of the offset arrays, which then start at a
  non-zero row, next to rows the call must not touch.
"""

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import attention as oatt
from oracle import range_table as ort

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu

# decode requests first (vLLM's order), then prefill chunks after a context
Q_LENS = [1, 1, 1, 1, 1, 1, 300, 129, 77, 260]
K_LENS = [900, 5000, 4100, 70, 8300, 1, 700, 129, 2000, 3000]
RANGES = [[(100, 400)], [(4990, 5100)], [], [(0, 3), (10, 69)], [(20, 300), (8290, 8310)], [],
          [(410, 420), (500, 650)], [(3, 60)], [(1930, 1999), (2000, 2000)], [(2700, 2950)]]
N_DEC = 6


def _workload(name, seed, head_dim, causal, wl, wr, ctx=None):
    w = workloads.Workload(name, seed, list(Q_LENS), list(K_LENS), 8, 2, head_dim, causal, wl, wr,
                           workloads.SINK_NULL_LOGIT, workloads.pad_ranges(RANGES))
    ctx = w.context_lens() if ctx is None else np.asarray(ctx, dtype=np.int32)
    return w, ctx


def _oracle_table(w, ctx):
    """The page's fill with the caller's positions: the fill takes key lengths,
    from which it derives the context, so it gets ctx + q_len."""
    cu_q, _ = w.cu_seqlens()
    out = np.full((w.total_q, 2), 12345, dtype=np.int32)
    n = ort.fill_by_spans(out, ort.ranges_from_padded(w.ranges), cu_q, np.asarray(ctx) + np.asarray(w.q_lens))
    if n == 0:
        out[:] = -1
    return out, n


def _gpu_table(w, ctx, dev):
    cu_q, _ = gh.device_meta(w, dev)
    table = torch.full((w.total_q, 2), 777, dtype=torch.int32, device=dev)
    covered = torch.full((1,), -5, dtype=torch.int32, device=dev)
    fill_lens = torch.from_numpy((np.asarray(ctx) + np.asarray(w.q_lens)).astype(np.int32)).to(dev)
    mvp.fill_query_ranges(torch.from_numpy(w.ranges).to(dev), cu_q, fill_lens, table, num_tokens=w.total_q,
                          rows_written=covered)
    return table, covered


def _workspace(w, n_dec, dev):
    nbytes = mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))
    return torch.empty(nbytes, dtype=torch.uint8, device=dev) if nbytes else None


def _run(entry, w, ctx, q, k, v, sinks, use_workspace, n_dec):
    dev = q.device
    cu_q, cu_k = gh.device_meta(w, dev)
    d_ctx = torch.from_numpy(np.ascontiguousarray(ctx, dtype=np.int32)).to(dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
    ws = _workspace(w, n_dec, dev) if use_workspace else None
    kw = dict(lse=lse, context_lens=d_ctx, causal=w.causal, window_left=w.window_left,
              window_right=w.window_right, sinks=sinks, sink_mode=w.sink_mode, scale=w.scale, workspace=ws,
              num_decode_reqs=n_dec)
    max_q, max_k = max(w.q_lens), max(w.k_lens)
    if entry == "scan":
        rg = torch.from_numpy(w.ranges).to(dev)
        mvp.attn_fwd_varlen_scan(q, k, v, out, cu_q, cu_k, max_q, max_k, rg, **kw)
    else:
        table, covered = _gpu_table(w, ctx, dev)
        ref_table, n = _oracle_table(w, ctx)
        assert np.array_equal(table.cpu().numpy(), ref_table), "range table with explicit positions"
        assert int(covered.item()) == n
        if entry == "packed":
            mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max_q, max_k, range_table=table,
                                range_covered=covered, **kw)
        else:
            kc, vc, bt, sl = workloads.to_paged(k, v, w.k_lens, 64, seed=w.seed)
            mvp.attn_fwd_paged(q, kc, vc, out, cu_q, sl, bt, 64, max_q, max_k, range_table=table,
                               range_covered=covered, **kw)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    return out, lse


def _oracle(w, ctx, q, k, v, sinks, scan):
    cu_q, cu_k = w.cu_seqlens()
    if scan:
        return oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), cu_q, cu_k, w.causal, w.window_left,
                                      w.window_right, w.scale, context_lens=ctx, sinks=sinks.cpu(),
                                      sink_mode=w.sink_mode, scan_ranges=w.ranges)
    ref_table, _ = _oracle_table(w, ctx)
    return oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), cu_q, cu_k, w.causal, w.window_left, w.window_right,
                                  w.scale, context_lens=ctx, range_table=ref_table, sinks=sinks.cpu(),
                                  sink_mode=w.sink_mode)


@pytest.mark.parametrize("entry", ["packed", "paged", "scan"])
@pytest.mark.parametrize("use_workspace", [True, False])
def test_context_equal_to_derived(entry, use_workspace):
    w, ctx = _workload(f"ctx_{entry}", 31, 128, True, 1000, 0)
    q, k, v, sinks = gh.make_inputs(w)
    out, lse = _run(entry, w, ctx, q, k, v, sinks, use_workspace, N_DEC)
    ro, rl = _oracle(w, ctx, q, k, v, sinks, entry == "scan")
    gh.compare(out, lse, ro, rl, what=f"explicit context_lens ({entry})", strict=False)


@pytest.mark.parametrize("head_dim", [64, 128, 256, 512])
@pytest.mark.parametrize("causal", [True, False])
def test_context_defines_positions(head_dim, causal):
    """Queries that end before the request's last key: with an explicit
    context the position of local row i is ctx + i, whatever k_len is."""
    _, derived = _workload("tmp", 0, head_dim, causal, -1, -1)
    ctx = derived.copy()
    ctx[[0, 1, 4]] -= np.array([37, 2100, 4000])   # decode rows placed earlier
    ctx[6] -= 150                                   # a prefill chunk ending 150 keys early
    ctx[9] = 0                                      # a chunk read as a fresh prompt
    wl, wr = (700, 0) if causal else (200, 90)
    w, ctx = _workload(f"ctxpos_d{head_dim}_{int(causal)}", 41 + head_dim, head_dim, causal, wl, wr, ctx)
    q, k, v, sinks = gh.make_inputs(w)
    for entry in ("packed", "scan"):
        out, lse = _run(entry, w, ctx, q, k, v, sinks, True, N_DEC)
        ro, rl = _oracle(w, ctx, q, k, v, sinks, entry == "scan")
        gh.compare(out, lse, ro, rl, what=f"positions from context_lens ({entry}, D {head_dim})", strict=False)


def test_sub_batch_slice_with_nonzero_offsets():
    """Requests [3, 8) of the batch as slices of cu_seqlens / context_lens
    (their first offset is not 0) with the whole batch's table; rows outside
    the slice stay untouched."""
    w, ctx = _workload("ctx_slice", 53, 128, True, 1500, 0)
    q, k, v, sinks = gh.make_inputs(w)
    dev = q.device
    cu_q_np, cu_k_np = w.cu_seqlens()
    cu_q, cu_k = gh.device_meta(w, dev)
    table, covered = _gpu_table(w, ctx, dev)
    lo, hi = 3, 8
    n_dec = N_DEC - lo  # requests 3..5 are the slice's decode rows
    d_ctx = torch.from_numpy(ctx).to(dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
    sub = workloads.Workload("sub", 0, w.q_lens[lo:hi], w.k_lens[lo:hi], w.num_heads_q, w.num_heads_kv,
                             w.head_dim, True, w.window_left, 0, w.sink_mode, None)
    ws = _workspace(sub, n_dec, dev)
    mvp.attn_fwd_varlen(q, k, v, out, cu_q[lo:hi + 1], cu_k[lo:hi + 1], max(w.q_lens[lo:hi]),
                        max(w.k_lens[lo:hi]), lse=lse, context_lens=d_ctx[lo:hi], range_table=table,
                        range_covered=covered, causal=True, window_left=w.window_left, sinks=sinks,
                        sink_mode=w.sink_mode, scale=w.scale, workspace=ws, num_decode_reqs=n_dec)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    ref_table, _ = _oracle_table(w, ctx)
    ro, rl = oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), cu_q_np[lo:hi + 1], cu_k_np[lo:hi + 1], True,
                                    w.window_left, 0, w.scale, context_lens=ctx[lo:hi], range_table=ref_table,
                                    sinks=sinks.cpu(), sink_mode=w.sink_mode)
    r0, r1 = int(cu_q_np[lo]), int(cu_q_np[hi])
    gh.compare(out[r0:r1], lse[:, r0:r1], ro[r0:r1], rl[:, r0:r1], what="sub-batch slice", strict=False)
    # rows of the other requests were not written
    assert torch.isnan(out[:r0].float()).all() and torch.isnan(out[r1:].float()).all()
    assert torch.isnan(lse[:, :r0]).all() and torch.isnan(lse[:, r1:]).all()
