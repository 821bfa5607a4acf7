"""Mixed batches: the decode kernel beside the prefill kernel (GPU).

A decode-first batch (num_decode_reqs >= 1 followed by longer requests) runs
its decode kernel on the library's second stream while the prefill kernel
holds a share of the SMs (mvp_attn_options.mixed_prefill_sms).  Every work
item and every decode split computes the same arithmetic whichever CTA runs
it, so the results must equal the serial launch order (mixed_prefill_sms =
-1) bit for bit at any share, eagerly and replayed from a CUDA graph, and the
float64 oracle within the tolerances; later work on the caller's stream must
see the decode rows' results (the join).
"""

import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _batch(name="mixed_serving_b"):
    w = workloads.scaled_workload(name)
    n_dec = 0
    while n_dec < w.num_reqs and w.q_lens[n_dec] == 1:
        n_dec += 1
    assert 0 < n_dec < w.num_reqs
    return w, n_dec


def _call(w, n_dec, q, k, v, sinks, share, ws, out=None, lse=None, stream=None, cu=None):
    cu_q, cu_k = gh.device_meta(w, q.device) if cu is None else cu
    out = torch.full_like(q, float("nan")) if out is None else out
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=q.device) if lse is None else lse
    mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max(w.q_lens), max(w.k_lens), lse=lse, causal=w.causal,
                        window_left=w.window_left, window_right=w.window_right, sinks=sinks, sink_mode=w.sink_mode,
                        scale=w.scale, workspace=ws, num_decode_reqs=n_dec, mixed_prefill_sms=share, stream=stream)
    return out, lse


def _workspace(w, n_dec, dev):
    return torch.empty(max(16, mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))),
                       dtype=torch.uint8, device=dev)


@pytest.mark.parametrize("name", ["mixed_serving_a", "mixed_serving_b"])
def test_any_share_equals_serial_order(name):
    w, n_dec = _batch(name)
    q, k, v, sinks = gh.make_inputs(w)
    ws = _workspace(w, n_dec, q.device)
    ref_o, ref_l = _call(w, n_dec, q, k, v, sinks, -1, ws)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    n_sms = torch.cuda.get_device_properties(q.device).multi_processor_count
    for share in (0, 2, 24, 77, n_sms - 2, n_sms + 100):
        out, lse = _call(w, n_dec, q, k, v, sinks, share, ws)
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16)), f"share {share}: output bits differ"
        assert torch.equal(lse, ref_l), f"share {share}: lse differs"
    ro, rl = gh.oracle_full(w, q, k, v, sinks, None)
    gh.compare(ref_o, ref_l, ro, rl, what=f"{name} mixed", strict=True)


def test_join_orders_later_work_on_the_callers_stream():
    """A copy enqueued on the caller's stream right after the call sees the
    decode rows, which the side stream wrote."""
    w, n_dec = _batch("mixed_serving_a")
    q, k, v, sinks = gh.make_inputs(w)
    ws = _workspace(w, n_dec, q.device)
    ref_o, _ = _call(w, n_dec, q, k, v, sinks, -1, ws)
    torch.cuda.synchronize()
    s = torch.cuda.Stream(q.device)
    with torch.cuda.stream(s):
        for _ in range(3):
            out = torch.full_like(q, float("nan"))
            _call(w, n_dec, q, k, v, sinks, 0, ws, out=out, stream=s)
            snap = out[:n_dec].clone()  # ordered after the call on s only
        s.synchronize()
    assert torch.equal(snap.view(torch.int16), ref_o[:n_dec].view(torch.int16))


def test_graph_capture_of_the_fork_and_join():
    w, n_dec = _batch("mixed_serving_b")
    q, k, v, sinks = gh.make_inputs(w)
    ws = _workspace(w, n_dec, q.device)
    ref_o, ref_l = _call(w, n_dec, q, k, v, sinks, -1, ws)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=q.device)
    cu = gh.device_meta(w, q.device)  # (no host copies inside the capture)
    _call(w, n_dec, q, k, v, sinks, 0, ws, out=out, lse=lse, cu=cu)  # eager first (per-device setup)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        _call(w, n_dec, q, k, v, sinks, 0, ws, out=out, lse=lse, cu=cu)
    for _ in range(3):
        out.fill_(float("nan"))
        g.replay()
        torch.cuda.synchronize()
        assert torch.equal(out.view(torch.int16), ref_o.view(torch.int16))
        assert torch.equal(lse, ref_l)
    assert mvp.get_last_device_error() == 0
