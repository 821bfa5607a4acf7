"""The allocation-free entry point, called through the C ABI.

mvp_attn_fwd_varlen_static_ws serves callers that cannot allocate device
memory where they run attention (their free memory is committed to a KV-cache
pool, or a host framework owns the allocator), so they cannot hand the
split-KV workspace to mvp_attn_fwd_varlen.  It keeps the partial results in a
fixed array inside the library.  These tests check that it returns what the
workspace-taking entry point returns, on two calls in a row (the second call
finds the first call's partials and work-queue words still in the array;
the decode-heavy batch is also compared with the float64 oracle):
a decode-heavy batch, the full mixed serving batch (256 long decode rows,
which the array holds with fewer splits than a full workspace would give),
and an unwindowed prefill batch large enough to use the work queue kept in
the array's header; and that a batch whose decode rows need more than the
array for a single split is refused before anything runs.

The file is named so that pytest collects it last.
"""

import ctypes

import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _args(q, k, v, out, lse, cu_q, cu_k, w, n_dec):
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return [p(q), p(k), p(v), p(out), p(lse), p(cu_q), p(cu_k), None, w.num_reqs, w.total_q, w.total_k,
            max(w.q_lens), max(w.k_lens), n_dec, w.num_heads_q, w.num_heads_kv, w.head_dim, None, None,
            int(w.causal), w.window_left, w.window_right]


def _sig(lib):
    vp, i, f = ctypes.c_void_p, ctypes.c_int, ctypes.c_float
    fn = lib.mvp_attn_fwd_varlen_static_ws
    fn.restype = i
    fn.argtypes = [vp] * 8 + [i] * 9 + [vp, vp, i, i, i, vp, i, f, vp]
    lib.mvp_static_scratch_bytes.restype = ctypes.c_size_t
    return fn


def test_static_scratch_matches_workspace_entry_point():
    lib = mvp.load_library()
    fn = _sig(lib)
    scratch = lib.mvp_static_scratch_bytes()
    assert scratch == 16 << 20
    # 24 decode rows with long contexts (several splits each) + 2 prefill chunks,
    # decode requests first; null-logit sinks, 4096-key causal window
    w = workloads.Workload("noalloc", 77, [1] * 24 + [300, 129],
                           [9000 + 731 * i for i in range(24)] + [2300, 129], 16, 4, 128, True, 4095, 0,
                           workloads.SINK_NULL_LOGIT, None)
    n_dec = 24
    need = mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))
    assert 0 < need <= scratch
    dev = torch.device("cuda", 0)
    q, k, v, sinks = workloads.make_tensors(w, device=dev)
    cu_q_np, cu_k_np = w.cu_seqlens()
    cu_q = torch.from_numpy(cu_q_np).to(dev)
    cu_k = torch.from_numpy(cu_k_np).to(dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)

    # reference: the workspace-taking entry point
    ref_out = torch.empty_like(q)
    ref_lse = torch.empty((w.num_heads_q, w.total_q), device=dev)
    ws = torch.empty(need, dtype=torch.uint8, device=dev)
    mvp.attn_fwd_varlen(q, k, v, ref_out, cu_q, cu_k, max(w.q_lens), max(w.k_lens), lse=ref_lse,
                        causal=w.causal, window_left=w.window_left, sinks=sinks, sink_mode=w.sink_mode,
                        scale=w.scale, workspace=ws, num_decode_reqs=n_dec)
    torch.cuda.synchronize()
    ref_o = ref_out.float().cpu().numpy()
    ref_l = ref_lse.cpu().numpy()

    for call in range(2):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
        st = fn(*_args(q, k, v, out, lse, cu_q, cu_k, w, n_dec), ctypes.c_void_p(sinks.data_ptr()),
                w.sink_mode, ctypes.c_float(w.scale), stream)
        assert st == mvp.MVP_OK, st
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0
        gh.compare(out, lse, ref_o, ref_l, what=f"static-scratch call {call}", strict=True)
    # and directly against the float64 oracle
    ro, rl = gh.oracle_full(w, q, k, v, sinks, None)
    gh.compare(out, lse, ro, rl, what="static scratch vs oracle", strict=True)


def _static_call(fn, w, q, k, v, sinks, cu_q, cu_k, n_dec, stream):
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=q.device)
    sp = None if sinks is None else ctypes.c_void_p(sinks.data_ptr())
    st = fn(*_args(q, k, v, out, lse, cu_q, cu_k, w, n_dec), sp, w.sink_mode, ctypes.c_float(w.scale), stream)
    assert st == mvp.MVP_OK, st
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    return out, lse


def _workspace_call(w, q, k, v, sinks, cu_q, cu_k, n_dec):
    out = torch.empty_like(q)
    lse = torch.empty((w.num_heads_q, w.total_q), device=q.device)
    need = mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))
    ws = torch.empty(need, dtype=torch.uint8, device=q.device)
    mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max(w.q_lens), max(w.k_lens), lse=lse, causal=w.causal,
                        window_left=w.window_left, window_right=w.window_right, sinks=sinks,
                        sink_mode=w.sink_mode, scale=w.scale, workspace=ws, num_decode_reqs=n_dec)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    return out, lse


def _device_inputs(w):
    dev = torch.device("cuda", 0)
    q, k, v, sinks = workloads.make_tensors(w, device=dev)
    cu_q_np, cu_k_np = w.cu_seqlens()
    n_dec = 0
    while n_dec < w.num_reqs and w.q_lens[n_dec] == 1:
        n_dec += 1
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    return q, k, v, sinks, torch.from_numpy(cu_q_np).to(dev), torch.from_numpy(cu_k_np).to(dev), n_dec, stream


def test_static_scratch_full_mixed_serving_batch():
    """256 decode rows of up to 32768 keys (32 q heads, D 128) next to four
    prefill chunks: one split of partials is 4.3 MB, so the 16 MiB array
    holds three where a full workspace gives eight; the results agree within
    the tolerance (the splits only regroup fp32 partial sums)."""
    lib = mvp.load_library()
    fn = _sig(lib)
    w = workloads.workload("mixed_serving_a")
    q, k, v, sinks, cu_q, cu_k, n_dec, stream = _device_inputs(w)
    assert n_dec == 256
    assert mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens)) > lib.mvp_static_scratch_bytes()
    ref_out, ref_lse = _workspace_call(w, q, k, v, sinks, cu_q, cu_k, n_dec)
    ref_o, ref_l = ref_out.float().cpu().numpy(), ref_lse.cpu().numpy()
    for call in range(2):
        out, lse = _static_call(fn, w, q, k, v, sinks, cu_q, cu_k, n_dec, stream)
        gh.compare(out, lse, ref_o, ref_l, what=f"static scratch, mixed batch, call {call}", strict=True)


def test_static_scratch_work_queue_words():
    """No window and 512 prefill items (more than two per CTA pair), so the
    prefill kernel claims its last round from the work-queue words at the
    start of the array; the second call finds the first call's words there.
    The split count is the same as with a workspace, so the bits agree."""
    lib = mvp.load_library()
    fn = _sig(lib)
    w = workloads.Workload("noalloc_queue", 79, [1] * 8 + [2048, 1900, 2048, 1500],
                           [5000 + 977 * i for i in range(8)] + [2048, 3000, 2600, 1500], 16, 4, 128, True, -1,
                           0, workloads.SINK_KEY0_BIAS, None)
    q, k, v, sinks, cu_q, cu_k, n_dec, stream = _device_inputs(w)
    ref_out, ref_lse = _workspace_call(w, q, k, v, sinks, cu_q, cu_k, n_dec)
    for call in range(2):
        out, lse = _static_call(fn, w, q, k, v, sinks, cu_q, cu_k, n_dec, stream)
        assert torch.equal(out.view(torch.int16), ref_out.view(torch.int16)), f"call {call}: output bits differ"
        assert torch.equal(lse, ref_lse), f"call {call}: lse differs"


def test_static_scratch_rejects_oversized_batch():
    lib = mvp.load_library()
    fn = _sig(lib)
    # 512 decode rows x 64 heads x (256 + 2) floats is 33.8 MB for a single
    # split, more than the 16 MiB array; the call must refuse before touching
    # any pointer
    w = workloads.Workload("big", 1, [1] * 512, [60000] * 512, 64, 8, 256, True, -1, 0, 0, None)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    ptr = ctypes.c_void_p(dummy.data_ptr())
    args = [ptr] * 7 + [None, w.num_reqs, 512, 512 * 60000, 1, 60000, 512, 64, 8, 256, None, None, 1, -1, 0]
    st = fn(*args, None, 0, ctypes.c_float(0.1), None)
    assert st == mvp.MVP_ERR_CAPACITY
