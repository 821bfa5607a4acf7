"""Bounded device waits: a withheld arrival ends in a reported timeout (GPU).

Every mbarrier wait in the kernels is bounded; on expiry the waiting thread
records a code in the library's device error word, raises its CTA's abort
flag, and the CTA drains its copies and MMAs, frees its tensor memory and
returns, so the context stays usable (vLLM PR #50294 review, *Risks and
impact* item 2: a broken assumption should fail loudly instead of corrupting
results silently).  Here the wait is made to run out on purpose in the
accepted way: the test asks (mvp_attn_fwd_varlen_ext, fault option) for one
softmax warp of the first prefill CTA to withhold its "probabilities ready"
arrival, with a 20 ms wait budget.  Checked: the call returns, the stream
completes, mvp_get_last_device_error reports MVP_ERR_DEVICE_TIMEOUT once, and
the next ordinary call on the same context matches the float64 oracle (it
could not even allocate tensor memory if the aborted CTAs had kept theirs).
"""

import time

import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu

LIMIT_US = 20000


def _case(head_dim):
    # one decode row, two prefill requests with ranges, a window and sinks
    return workloads.Workload(f"timeout_d{head_dim}", 61 + head_dim, [1, 300, 129], [700, 900, 129], 4, 2,
                              head_dim, True, 200, 0, workloads.SINK_NULL_LOGIT,
                              workloads.pad_ranges([[], [(640, 700), (720, 800)], [(3, 60)]]))


def _parity(w, q, k, v, sinks, **ext):
    out, lse, _, _ = gh.run_gpu(w, q, k, v, sinks, **ext)
    ref_table, _ = gh.oracle_table(w)
    ro, rl = gh.oracle_full(w, q, k, v, sinks, ref_table)
    gh.compare(out, lse, ro, rl, what=w.name, strict=False)


@pytest.mark.parametrize("head_dim", [64, 128, 256, 512])
def test_withheld_arrival_times_out_and_context_recovers(head_dim):
    w = _case(head_dim)
    q, k, v, sinks = gh.make_inputs(w)
    assert mvp.get_last_device_error() == mvp.MVP_OK
    cu_q, cu_k = gh.device_meta(w, q.device)
    out = torch.zeros_like(q)
    t0 = time.monotonic()
    # the launch itself succeeds; the failure is on the device
    mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max(w.q_lens), max(w.k_lens), causal=True,
                        window_left=w.window_left, sinks=sinks, sink_mode=w.sink_mode, scale=w.scale,
                        wait_limit_us=LIMIT_US, fault=mvp.FAULT_WITHHOLD_PROBS)
    torch.cuda.synchronize()
    elapsed = time.monotonic() - t0
    assert mvp.get_last_device_error() == mvp.MVP_ERR_DEVICE_TIMEOUT
    assert mvp.get_last_device_error() == mvp.MVP_OK  # read once, then clear
    # a handful of budgets (the expiring wait, then the waits it releases),
    # not the one-second default
    assert elapsed < 5.0, elapsed
    # the context is healthy: the same batch, default options, is correct
    _parity(w, q, k, v, sinks)


def test_short_budget_without_fault_is_not_a_timeout():
    w = _case(128)
    q, k, v, sinks = gh.make_inputs(w)
    _parity(w, q, k, v, sinks, wait_limit_us=LIMIT_US)
