"""The allocation-free entry point, called through the C ABI.

mvp_attn_fwd_varlen_static_ws serves callers that cannot allocate device
memory where they run attention (their free memory is committed to a KV-cache
pool, or a host framework owns the allocator), so they cannot hand the
split-KV workspace to mvp_attn_fwd_varlen.  It keeps the partial results in a
fixed array inside the library.  This test checks that it returns what the
workspace-taking entry point returns, on two calls in a row (the second call
finds the first call's partials still in the array), and that a batch too
large for the array is refused before anything runs.

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


def test_static_scratch_rejects_oversized_batch():
    lib = mvp.load_library()
    fn = _sig(lib)
    # 512 decode rows x 64 heads x D 256 x many splits needs far more than 16 MiB;
    # the call must refuse before touching any pointer
    w = workloads.Workload("big", 1, [1] * 512, [60000] * 512, 64, 8, 256, True, -1, 0, 0, None)
    dummy = torch.empty(16, dtype=torch.uint8, device="cuda")
    ptr = ctypes.c_void_p(dummy.data_ptr())
    args = [ptr] * 7 + [None, w.num_reqs, 512, 512 * 60000, 1, 60000, 512, 64, 8, 256, None, None, 1, -1, 0]
    st = fn(*args, None, 0, ctypes.c_float(0.1), None)
    assert st == mvp.MVP_ERR_CAPACITY
