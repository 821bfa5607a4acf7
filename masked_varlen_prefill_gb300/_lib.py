"""ctypes binding of ``lib/libmvp.so``: argument marshalling only."""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

MVP_OK = 0
MVP_ERR_ARG = -1
MVP_ERR_CAPACITY = -2
MVP_ERR_UNSUPPORTED = -3
MVP_ERR_CUDA = -4
MVP_ERR_DEVICE_TIMEOUT = -5
MVP_ERR_DEVICE_BOUNDS = -6

SINK_NONE = 0
SINK_KEY0_BIAS = 1
SINK_NULL_LOGIT = 2

VARIANT_DEFAULT = 0
VARIANT_D512_HEAD_SPLIT = 1
FAULT_NONE = 0
FAULT_WITHHOLD_PROBS = 1

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "lib", "libmvp.so")
# The bounds-checked build of the same library (include/mvp.h,
# MVP_ERR_DEVICE_BOUNDS): for tests, selected per thread by bounds_checked().
_DEBUG_LIB_PATH = os.path.join(_HERE, "lib", "libmvp_debug.so")
_lib = None
_debug_lib = None
_lock = threading.Lock()
_local = threading.local()

_vp = ctypes.c_void_p
_i = ctypes.c_int
_f = ctypes.c_float
_sz = ctypes.c_size_t

class AttnCounts(ctypes.Structure):
    """``mvp_attn_counts`` (include/mvp.h)."""

    _fields_ = [("est_token_context_product", ctypes.c_double), ("est_attn_qk_flops", ctypes.c_double),
                ("est_attn_av_flops", ctypes.c_double), ("est_decode_kv_read_bytes", ctypes.c_double),
                ("visible_prefill", ctypes.c_longlong), ("visible_decode", ctypes.c_longlong),
                ("exact_flops", ctypes.c_double), ("exact_decode_kv_bytes", ctypes.c_double),
                ("prefill_items", ctypes.c_longlong), ("prefill_tiles", ctypes.c_longlong),
                ("prefill_mma_instructions", ctypes.c_longlong), ("prefill_mma_flops", ctypes.c_double),
                ("prefill_compulsory_bytes", ctypes.c_double), ("decode_keys_walked", ctypes.c_longlong),
                ("decode_read_bytes", ctypes.c_double), ("decode_cta_read_bytes", ctypes.c_double)]


class AttnOptions(ctypes.Structure):
    """``mvp_attn_options`` (include/mvp.h)."""

    _fields_ = [("variant", ctypes.c_int), ("wait_limit_us", ctypes.c_uint), ("fault", ctypes.c_int),
                ("mixed_prefill_sms", ctypes.c_int)]


_SIGNATURES = {
    "mvp_fill_query_ranges": (_i, [_vp, _i, _i, _vp, _vp, _i, _vp, _i, _vp, _vp]),
    "mvp_attn_workspace_size": (_sz, [_i, _i, _i, _i]),
    "mvp_attn_fwd_varlen": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                 _vp, _vp, _i, _i, _i, _vp, _i, _f, _vp, _sz, _vp]),
    "mvp_attn_fwd_varlen_ext": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                     _vp, _vp, _i, _i, _i, _vp, _i, _f, _vp, _sz, _vp, ctypes.POINTER(AttnOptions)]),
    "mvp_attn_fwd_paged": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _vp, _i, _i, _i, _i, _i, _i, _i,
                                _i, _vp, _vp, _i, _i, _i, _vp, _i, _f, _vp, _sz, _vp]),
    "mvp_attn_fwd_varlen_static_ws": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i,
                                           _i, _i, _vp, _vp, _i, _i, _i, _vp, _i, _f, _vp]),
    "mvp_static_scratch_bytes": (_sz, []),
    "mvp_get_last_device_error": (_i, [_vp]),
    "mvp_status_str": (ctypes.c_char_p, [_i]),
    "mvp_last_launch_count": (_i, []),
    "mvp_meta_block_bytes": (_sz, [_i, _i]),
    "mvp_meta_offsets": (_i, [_i, _i, ctypes.POINTER(_sz)]),
    "mvp_meta_pack": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp]),
    "mvp_meta_create": (_i, [_i, _i, _i, _vp, _vp, _vp, ctypes.POINTER(_vp)]),
    "mvp_meta_destroy": (_i, [_vp]),
    "mvp_meta_stage": (_i, [_vp, _vp, _vp, _vp, _vp, _i, _i]),
    "mvp_meta_upload": (_i, [_vp, _vp]),
    "mvp_attn_fwd_varlen_scan": (_i, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _i,
                                      _vp, _i, _i, _i, _i, _vp, _i, _f, _vp, _sz, _vp]),
    "mvp_attn_accounting": (_i, [_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, ctypes.POINTER(AttnCounts)]),
}


class MvpError(RuntimeError):
    def __init__(self, fn, status):
        self.status = status
        msg = load_library().mvp_status_str(status).decode()
        super().__init__(f"{fn} failed: {msg} ({status})")


def library_path(debug_bounds: bool = False) -> str:
    return _DEBUG_LIB_PATH if debug_bounds else _LIB_PATH


def _open(path):
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with `python -m masked_varlen_prefill_gb300._build` "
            "(there is no CPU fallback)")
    lib = ctypes.CDLL(path)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    return lib


def load_library(debug_bounds: bool | None = None):
    """Load the C-ABI library; raise if it has not been built.  debug_bounds:
    the bounds-checked build instead (default: the one bounds_checked()
    selected for this thread, else the product library)."""
    global _lib, _debug_lib
    if debug_bounds is None:
        debug_bounds = getattr(_local, "debug_bounds", False)
    if debug_bounds:
        if _debug_lib is None:
            with _lock:
                if _debug_lib is None:
                    _debug_lib = _open(_DEBUG_LIB_PATH)
        return _debug_lib
    if _lib is not None:
        return _lib
    with _lock:
        if _lib is None:
            _lib = _open(_LIB_PATH)
    return _lib


class bounds_checked:
    """Context manager: every call of this binding made on this thread inside
    it goes to the bounds-checked library (its own device error word; read
    it with get_last_device_error() inside the block)."""

    def __enter__(self):
        self._prev = getattr(_local, "debug_bounds", False)
        _local.debug_bounds = True
        return load_library(True)

    def __exit__(self, *exc):
        _local.debug_bounds = self._prev
        return False


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _check_cuda(name, t, dtype, device):
    if t is None:
        return
    if not t.is_cuda or t.device != device:
        raise ValueError(f"{name} must be a CUDA tensor on {device}")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def fill_query_ranges(ranges, query_start_loc, seq_lens, out, num_tokens, rows_written=None, stream=None):
    """Per-row range table (see ``mvp_fill_query_ranges`` in include/mvp.h).

    ranges int32 [B, R, 2] (or None), query_start_loc int32 [B+1], seq_lens
    int32 [B], out int32 [capacity, 2], rows_written int32 [1] or None;
    num_tokens is a host int (== query_start_loc[-1]).
    """
    lib = load_library()
    dev = out.device
    for n, t in (("ranges", ranges), ("query_start_loc", query_start_loc), ("seq_lens", seq_lens),
                 ("out", out), ("rows_written", rows_written)):
        _check_cuda(n, t, torch.int32, dev)
    num_reqs = seq_lens.shape[0]
    max_ranges = 0 if ranges is None else ranges.shape[1]
    if ranges is not None and (ranges.dim() != 3 or ranges.shape[0] != num_reqs or ranges.shape[2] != 2):
        raise ValueError("ranges must be [num_reqs, max_ranges, 2]")
    st = lib.mvp_fill_query_ranges(_ptr(ranges), num_reqs, max_ranges, _ptr(query_start_loc), _ptr(seq_lens),
                                   int(num_tokens), _ptr(out), out.shape[0], _ptr(rows_written),
                                   _stream(stream, dev))
    if st != MVP_OK:
        raise MvpError("mvp_fill_query_ranges", st)


def attn_workspace_size(num_reqs, num_heads_q, head_dim, max_k_len) -> int:
    return int(load_library().mvp_attn_workspace_size(num_reqs, num_heads_q, head_dim, max_k_len))


def attn_fwd_varlen(q, k, v, out, cu_seqlens_q, cu_seqlens_k, max_q_len, max_k_len, *, lse=None,
                    context_lens=None, range_table=None, range_covered=None, causal=True, window_left=-1,
                    window_right=-1, sinks=None, sink_mode=SINK_NONE, scale=None, workspace=None,
                    num_decode_reqs=-1, stream=None, variant=VARIANT_DEFAULT, wait_limit_us=0,
                    fault=FAULT_NONE, mixed_prefill_sms=0):
    """Masked varlen attention forward (see ``mvp_attn_fwd_varlen``).

    q [total_q, Hq, D], k/v [total_k, Hkv, D] bf16; out like q; lse fp32
    [Hq, total_q] or None; cu_seqlens int32 [B+1]; the rest as in the header.
    ``variant`` / ``wait_limit_us`` / ``fault`` / ``mixed_prefill_sms`` other
    than their defaults go through ``mvp_attn_fwd_varlen_ext`` with those
    options.
    """
    lib = load_library()
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_cuda(n, t, torch.bfloat16, dev)
    for n, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("context_lens", context_lens),
                 ("range_table", range_table), ("range_covered", range_covered)):
        _check_cuda(n, t, torch.int32, dev)
    _check_cuda("lse", lse, torch.float32, dev)
    _check_cuda("sinks", sinks, torch.float32, dev)
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("q/out must be [total_q, Hq, D] and k/v [total_k, Hkv, D]")
    total_q, hq, d = q.shape
    total_k, hkv, dk = k.shape
    if dk != d:
        raise ValueError("q and k head_dim differ")
    num_reqs = cu_seqlens_q.shape[0] - 1
    if scale is None:
        scale = d ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    args = [_ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            _ptr(context_lens), num_reqs, total_q, total_k, int(max_q_len), int(max_k_len), int(num_decode_reqs),
            hq, hkv, d, _ptr(range_table), _ptr(range_covered), int(bool(causal)), int(window_left),
            int(window_right), _ptr(sinks), int(sink_mode), float(scale), _ptr(workspace), ws_bytes,
            _stream(stream, dev)]
    if variant == VARIANT_DEFAULT and wait_limit_us == 0 and fault == FAULT_NONE and mixed_prefill_sms == 0:
        name, st = "mvp_attn_fwd_varlen", lib.mvp_attn_fwd_varlen(*args)
    else:
        opts = AttnOptions(int(variant), int(wait_limit_us), int(fault), int(mixed_prefill_sms))
        name, st = "mvp_attn_fwd_varlen_ext", lib.mvp_attn_fwd_varlen_ext(*args, ctypes.byref(opts))
    if st != MVP_OK:
        raise MvpError(name, st)


def attn_fwd_varlen_scan(q, k, v, out, cu_seqlens_q, cu_seqlens_k, max_q_len, max_k_len, ranges, *, lse=None,
                         context_lens=None, causal=True, window_left=-1, window_right=-1, sinks=None,
                         sink_mode=SINK_NONE, scale=None, workspace=None, num_decode_reqs=-1, stream=None):
    """Scan-mode attention (``mvp_attn_fwd_varlen_scan``): the request-level
    range list ``ranges`` int32 [B, max_ranges, 2] instead of a range table."""
    lib = load_library()
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_cuda(n, t, torch.bfloat16, dev)
    for n, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("context_lens", context_lens),
                 ("ranges", ranges)):
        _check_cuda(n, t, torch.int32, dev)
    _check_cuda("lse", lse, torch.float32, dev)
    _check_cuda("sinks", sinks, torch.float32, dev)
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if q.dim() != 3 or k.dim() != 3 or v.shape != k.shape or out.shape != q.shape:
        raise ValueError("q/out must be [total_q, Hq, D] and k/v [total_k, Hkv, D]")
    total_q, hq, d = q.shape
    total_k, hkv, dk = k.shape
    if dk != d:
        raise ValueError("q and k head_dim differ")
    num_reqs = cu_seqlens_q.shape[0] - 1
    if ranges is not None and (ranges.dim() != 3 or ranges.shape[0] != num_reqs or ranges.shape[2] != 2):
        raise ValueError("ranges must be [num_reqs, max_ranges, 2]")
    max_ranges = 0 if ranges is None else ranges.shape[1]
    if scale is None:
        scale = d ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.mvp_attn_fwd_varlen_scan(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        _ptr(context_lens), num_reqs, total_q, total_k, int(max_q_len), int(max_k_len), int(num_decode_reqs),
        hq, hkv, d, _ptr(ranges), max_ranges, int(bool(causal)), int(window_left), int(window_right),
        _ptr(sinks), int(sink_mode), float(scale), _ptr(workspace), ws_bytes, _stream(stream, dev))
    if st != MVP_OK:
        raise MvpError("mvp_attn_fwd_varlen_scan", st)


def attn_fwd_paged(q, k_cache, v_cache, out, cu_seqlens_q, seq_lens_k, block_table, block_size, max_q_len,
                   max_k_len, *, lse=None, context_lens=None, range_table=None, range_covered=None, causal=True,
                   window_left=-1, window_right=-1, sinks=None, sink_mode=SINK_NONE, scale=None, workspace=None,
                   num_decode_reqs=-1, stream=None):
    """Masked varlen attention over a paged K/V cache (see
    ``mvp_attn_fwd_paged``): k_cache/v_cache [num_blocks * block_size, Hkv,
    D] (or [num_blocks, block_size, Hkv, D]) bf16, block_table int32 [B,
    max_blocks_per_seq], seq_lens_k int32 [B]; the rest as ``attn_fwd_varlen``."""
    lib = load_library()
    dev = q.device
    if k_cache.dim() == 4:
        k_cache = k_cache.reshape(-1, k_cache.shape[2], k_cache.shape[3])
        v_cache = v_cache.reshape(-1, v_cache.shape[2], v_cache.shape[3])
    for n, t in (("q", q), ("k_cache", k_cache), ("v_cache", v_cache), ("out", out)):
        _check_cuda(n, t, torch.bfloat16, dev)
    for n, t in (("cu_seqlens_q", cu_seqlens_q), ("seq_lens_k", seq_lens_k), ("block_table", block_table),
                 ("context_lens", context_lens), ("range_table", range_table), ("range_covered", range_covered)):
        _check_cuda(n, t, torch.int32, dev)
    _check_cuda("lse", lse, torch.float32, dev)
    _check_cuda("sinks", sinks, torch.float32, dev)
    if workspace is not None and (not workspace.is_cuda or not workspace.is_contiguous()):
        raise ValueError("workspace must be a contiguous CUDA tensor")
    if q.dim() != 3 or k_cache.dim() != 3 or v_cache.shape != k_cache.shape or out.shape != q.shape:
        raise ValueError("q/out must be [total_q, Hq, D] and the caches [num_blocks * block_size, Hkv, D]")
    if block_table is None or block_table.dim() != 2 or seq_lens_k is None:
        raise ValueError("block_table must be [B, max_blocks_per_seq] and seq_lens_k [B]")
    total_q, hq, d = q.shape
    rows, hkv, dk = k_cache.shape
    if dk != d:
        raise ValueError("q and the caches differ in head_dim")
    if rows % int(block_size) != 0:
        raise ValueError("cache rows must be a multiple of block_size")
    if scale is None:
        scale = d ** -0.5
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = lib.mvp_attn_fwd_paged(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(seq_lens_k),
        _ptr(block_table), int(block_size), block_table.shape[1], rows // int(block_size), _ptr(context_lens),
        cu_seqlens_q.shape[0] - 1, total_q, int(max_q_len), int(max_k_len), int(num_decode_reqs), hq, hkv, d,
        _ptr(range_table), _ptr(range_covered), int(bool(causal)), int(window_left), int(window_right),
        _ptr(sinks), int(sink_mode), float(scale), _ptr(workspace), ws_bytes, _stream(stream, dev))
    if st != MVP_OK:
        raise MvpError("mvp_attn_fwd_paged", st)


def attn_fwd_varlen_static_ws(q, k, v, out, cu_seqlens_q, cu_seqlens_k, max_q_len, max_k_len, *, lse=None,
                              context_lens=None, range_table=None, range_covered=None, causal=True,
                              window_left=-1, window_right=-1, sinks=None, sink_mode=SINK_NONE, scale=None,
                              num_decode_reqs=-1, stream=None):
    """Like ``attn_fwd_varlen`` but without a workspace argument, for callers
    that cannot allocate device memory at the call site: the split-KV partials
    use the library's fixed scratch array (``mvp_attn_fwd_varlen_static_ws``
    in include/mvp.h; calls that overlap on the GPU race on it)."""
    lib = load_library()
    dev = q.device
    for n, t in (("q", q), ("k", k), ("v", v), ("out", out)):
        _check_cuda(n, t, torch.bfloat16, dev)
    for n, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k), ("context_lens", context_lens),
                 ("range_table", range_table), ("range_covered", range_covered)):
        _check_cuda(n, t, torch.int32, dev)
    _check_cuda("lse", lse, torch.float32, dev)
    _check_cuda("sinks", sinks, torch.float32, dev)
    total_q, hq, d = q.shape
    total_k, hkv, _ = k.shape
    if scale is None:
        scale = d ** -0.5
    st = lib.mvp_attn_fwd_varlen_static_ws(
        _ptr(q), _ptr(k), _ptr(v), _ptr(out), _ptr(lse), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
        _ptr(context_lens), cu_seqlens_q.shape[0] - 1, total_q, total_k, int(max_q_len), int(max_k_len),
        int(num_decode_reqs), hq, hkv, d, _ptr(range_table), _ptr(range_covered), int(bool(causal)),
        int(window_left), int(window_right), _ptr(sinks), int(sink_mode), float(scale), _stream(stream, dev))
    if st != MVP_OK:
        raise MvpError("mvp_attn_fwd_varlen_static_ws", st)


def attn_fwd_varlen_host(q, k, v, cu_seqlens_q, cu_seqlens_k, max_q_len, max_k_len, *, device_buffers,
                         want_lse=False, **kw):
    """End-to-end call from HOST tensors: copy inputs into the given device
    buffers, run ``attn_fwd_varlen`` and copy the output back to a pinned host
    tensor.  ``device_buffers`` is a dict with preallocated 'q','k','v','out'
    (and 'lse', 'cu_q', 'cu_k', plus any other device inputs already named in
    ``kw``).  Returns the host output (and host lse)."""
    dq, dk, dv, dout = (device_buffers[n] for n in ("q", "k", "v", "out"))
    dq.copy_(q, non_blocking=True)
    dk.copy_(k, non_blocking=True)
    dv.copy_(v, non_blocking=True)
    dcu_q = device_buffers["cu_q"]
    dcu_k = device_buffers["cu_k"]
    dcu_q.copy_(cu_seqlens_q, non_blocking=True)
    dcu_k.copy_(cu_seqlens_k, non_blocking=True)
    lse = device_buffers.get("lse") if want_lse else None
    attn_fwd_varlen(dq, dk, dv, dout, dcu_q, dcu_k, max_q_len, max_k_len, lse=lse, **kw)
    host_out = device_buffers["host_out"]
    host_out.copy_(dout, non_blocking=True)
    if lse is not None:
        device_buffers["host_lse"].copy_(lse, non_blocking=True)
    return host_out


def get_last_device_error(stream=None) -> int:
    """Synchronise and return (and clear) the library's device error status."""
    lib = load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    return int(lib.mvp_get_last_device_error(_stream(stream, dev)))


def last_launch_count() -> int:
    return int(load_library().mvp_last_launch_count())


# ------------------------------------------------------------ step metadata
def _host_i32(a, name, shape=None):
    """Contiguous host int32 numpy array (or None) and its pointer."""
    if a is None:
        return None, None
    if isinstance(a, torch.Tensor):
        if a.is_cuda:
            raise ValueError(f"{name} must be a host array")
        a = a.numpy()
    a = np.ascontiguousarray(np.asarray(a, dtype=np.int32))
    if shape is not None and a.shape != shape:
        raise ValueError(f"{name} must have shape {shape}, got {a.shape}")
    return a, ctypes.c_void_p(a.ctypes.data)


def _meta_args(query_start_loc, seq_lens_k, seq_lens_bound, ranges):
    qsl, p_qsl = _host_i32(query_start_loc, "query_start_loc")
    if qsl is None or qsl.ndim != 1 or qsl.shape[0] < 1:
        raise ValueError("query_start_loc must be a 1-D host array of num_reqs + 1 offsets")
    n = qsl.shape[0] - 1
    sk, p_sk = _host_i32(seq_lens_k, "seq_lens_k", (n,))
    sb, p_sb = _host_i32(seq_lens_bound, "seq_lens_bound", (n,))
    rg, p_rg = _host_i32(ranges, "ranges")
    if rg is not None and (rg.ndim != 3 or rg.shape[0] != n or rg.shape[2] != 2):
        raise ValueError("ranges must be [num_reqs, num_ranges, 2]")
    keep = (qsl, sk, sb, rg)  # the arrays must outlive the call
    return keep, (p_qsl, p_sk, p_sb, p_rg, n, 0 if rg is None else rg.shape[1])


def meta_block_layout(max_reqs, max_ranges):
    """(bytes, element offsets of query_start_loc, seq_lens_k, cu_seqlens_k,
    seq_lens_bound, ranges) of a metadata block (``mvp_meta_offsets``)."""
    lib = load_library()
    nbytes = int(lib.mvp_meta_block_bytes(max_reqs, max_ranges))
    offs = (_sz * 5)()
    st = lib.mvp_meta_offsets(max_reqs, max_ranges, offs)
    if st != MVP_OK:
        raise MvpError("mvp_meta_offsets", st)
    return nbytes, tuple(int(x) for x in offs)


def meta_pack(query_start_loc, seq_lens_k, seq_lens_bound, ranges, max_reqs, max_tokens, max_ranges):
    """Padded metadata block of one batch (``mvp_meta_pack``; host only, no
    GPU needed).  Returns an int32 numpy array."""
    lib = load_library()
    nbytes, _ = meta_block_layout(max_reqs, max_ranges)
    block = np.zeros(nbytes // 4, dtype=np.int32)
    keep, (p_qsl, p_sk, p_sb, p_rg, n, nr) = _meta_args(query_start_loc, seq_lens_k, seq_lens_bound, ranges)
    st = lib.mvp_meta_pack(p_qsl, p_sk, p_sb, p_rg, n, nr, max_reqs, max_tokens, max_ranges,
                           ctypes.c_void_p(block.ctypes.data))
    del keep
    if st != MVP_OK:
        raise MvpError("mvp_meta_pack", st)
    return block


class StepMetadata:
    """Persistent step metadata for CUDA-graph replays (``mvp_meta_*``).

    Owns the device block, the range table and the covered flag as torch
    tensors whose addresses never change; ``stage`` packs a batch on the host
    into the library's pinned staging block, ``upload`` enqueues the copy and
    the table fill on a stream (capturable).  The views ``query_start_loc``,
    ``seq_lens_k``, ``cu_seqlens_k``, ``range_table`` and ``range_covered``
    are what an attention call captured with them reads."""

    def __init__(self, max_reqs, max_tokens, max_ranges, device=None):
        lib = load_library()
        device = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
        self.max_reqs, self.max_tokens, self.max_ranges = int(max_reqs), int(max_tokens), int(max_ranges)
        nbytes, offs = meta_block_layout(self.max_reqs, self.max_ranges)
        if nbytes == 0:
            raise ValueError("capacity out of range")
        self.device = device
        self.block = torch.zeros(nbytes // 4, dtype=torch.int32, device=device)
        self.range_table = torch.full((self.max_tokens, 2), -1, dtype=torch.int32, device=device)
        self.range_covered = torch.zeros(1, dtype=torch.int32, device=device)
        r = self.max_reqs
        self.query_start_loc = self.block[offs[0]:offs[0] + r + 1]
        self.seq_lens_k = self.block[offs[1]:offs[1] + r]
        self.cu_seqlens_k = self.block[offs[2]:offs[2] + r + 1]
        self.seq_lens_bound = self.block[offs[3]:offs[3] + r]
        self.ranges = self.block[offs[4]:offs[4] + r * self.max_ranges * 2].view(r, self.max_ranges, 2)
        handle = _vp()
        with torch.cuda.device(device):
            st = lib.mvp_meta_create(self.max_reqs, self.max_tokens, self.max_ranges, _ptr(self.block),
                                     _ptr(self.range_table), _ptr(self.range_covered), ctypes.byref(handle))
        if st != MVP_OK:
            raise MvpError("mvp_meta_create", st)
        self._lib = lib  # the handle belongs to the library that made it
        self._handle = handle

    def stage(self, query_start_loc, seq_lens_k, seq_lens_bound=None, ranges=None):
        """Pack one batch (host arrays) into the staging block."""
        keep, (p_qsl, p_sk, p_sb, p_rg, n, nr) = _meta_args(query_start_loc, seq_lens_k, seq_lens_bound, ranges)
        st = self._lib.mvp_meta_stage(self._handle, p_qsl, p_sk, p_sb, p_rg, n, nr)
        del keep
        if st != MVP_OK:
            raise MvpError("mvp_meta_stage", st)

    def upload(self, stream=None):
        """Copy the staged block to the device and fill the range table."""
        st = self._lib.mvp_meta_upload(self._handle, _stream(stream, self.device))
        if st != MVP_OK:
            raise MvpError("mvp_meta_upload", st)

    def close(self):
        if getattr(self, "_handle", None) is not None and self._handle.value is not None:
            self._lib.mvp_meta_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def attn_accounting(cu_seqlens_q, seq_lens_k, num_heads_q, num_heads_kv, head_dim, *, context_lens=None,
                    range_table=None, causal=True, window_left=-1, window_right=-1, variant=0) -> dict:
    """Work accounting of one attention call from host arrays
    (``mvp_attn_accounting``): the PR #55624 estimate, the exact mask and the
    kernels' executed work, as a dict.  No GPU needed."""
    keep = []

    def arr(a, name, shape=None):
        x, ptr = _host_i32(a, name, shape)
        keep.append(x)
        return ptr

    cu = np.ascontiguousarray(np.asarray(cu_seqlens_q, dtype=np.int32))
    n = cu.shape[0] - 1
    p_cu = arr(cu, "cu_seqlens_q")
    p_sk = arr(seq_lens_k, "seq_lens_k", (n,))
    p_cl = arr(context_lens, "context_lens", (n,))
    tbl = None if range_table is None else np.asarray(range_table)
    if tbl is not None and (tbl.ndim != 2 or tbl.shape[1] != 2 or tbl.shape[0] < int(cu[-1])):
        raise ValueError("range_table must be [>= total_q, 2]")
    p_tb = arr(tbl, "range_table")
    out = AttnCounts()
    st = load_library().mvp_attn_accounting(p_cu, p_sk, p_cl, p_tb, n, num_heads_q, num_heads_kv, head_dim,
                                            int(bool(causal)), window_left, window_right, int(variant),
                                            ctypes.byref(out))
    del keep
    if st != MVP_OK:
        raise MvpError("mvp_attn_accounting", st)
    return {name: getattr(out, name) for name, _ in AttnCounts._fields_}

