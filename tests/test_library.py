"""The C-ABI library: it loads, exports what include/mvp.h declares, and
rejects bad arguments on the host before touching a GPU (no GPU needed)."""

import ctypes
import os
import re

import pytest

import masked_varlen_prefill_gb300 as mvp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for f in os.listdir(os.path.join(ROOT, "include")):
        if f.endswith(".h"):
            src = open(os.path.join(ROOT, "include", f)).read()
            names.update(re.findall(r"\b(mvp_\w+)\s*\(", src))
    return sorted(names)


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(mvp.library_path()):
        from masked_varlen_prefill_gb300 import _build

        _build.build()
    return mvp.load_library()


def test_exports_every_declared_symbol(lib):
    names = _declared()
    assert "mvp_fill_query_ranges" in names and "mvp_attn_fwd_varlen" in names
    for n in names:
        assert hasattr(lib, n), n


def test_bounds_checked_build_exports_the_same_symbols(lib):
    """libmvp_debug.so (MVP_DEBUG_BOUNDS) is the same library with device
    bounds checks: every declared entry point, and its own status string."""
    dbg = mvp.load_library(debug_bounds=True)
    assert dbg is not lib
    for n in _declared():
        assert hasattr(dbg, n), n
    assert dbg.mvp_status_str(mvp.MVP_ERR_DEVICE_BOUNDS).decode() != "unknown status"
    with mvp.bounds_checked() as d:
        assert d is dbg and mvp.load_library() is dbg
    assert mvp.load_library() is lib


def test_status_strings(lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert lib.mvp_status_str(code).decode() != "unknown status"
    assert lib.mvp_status_str(99).decode() == "unknown status"


def _attn(lib, **over):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, out=1 << 20, lse=None, cu_q=1 << 20, cu_k=1 << 20, ctx=None,
                num_reqs=1, total_q=4, total_k=4, max_q=4, max_k=4, ndec=-1, hq=4, hkv=2, d=128, table=None,
                covered=None, causal=1, wl=-1, wr=-1, sinks=None, sink_mode=0, scale=0.1, ws=None, ws_bytes=0,
                stream=None)
    args.update(over)
    return lib.mvp_attn_fwd_varlen(*[args[k] for k in (
        "q", "k", "v", "out", "lse", "cu_q", "cu_k", "ctx", "num_reqs", "total_q", "total_k", "max_q", "max_k", "ndec",
        "hq", "hkv", "d", "table", "covered", "causal", "wl", "wr", "sinks", "sink_mode", "scale", "ws",
        "ws_bytes", "stream")])


def test_argument_errors_return_before_any_launch(lib):
    # None of these reach a CUDA call: validation runs first on the host.
    assert _attn(lib, d=96) == mvp.MVP_ERR_UNSUPPORTED
    assert _attn(lib, hq=3, hkv=2) == mvp.MVP_ERR_ARG
    assert _attn(lib, num_reqs=0) == mvp.MVP_ERR_ARG
    assert _attn(lib, sink_mode=1, sinks=None) == mvp.MVP_ERR_ARG
    assert _attn(lib, sink_mode=3) == mvp.MVP_ERR_ARG
    assert _attn(lib, wl=-2) == mvp.MVP_ERR_ARG
    assert _attn(lib, causal=2) == mvp.MVP_ERR_ARG
    assert _attn(lib, q=None) == mvp.MVP_ERR_ARG
    assert _attn(lib, q=(1 << 20) + 8) == mvp.MVP_ERR_UNSUPPORTED  # not 16-byte aligned
    assert _attn(lib, total_k=0) == mvp.MVP_ERR_ARG
    assert _attn(lib, scale=float("nan")) == mvp.MVP_ERR_ARG
    assert _attn(lib, scale=0.0) == mvp.MVP_ERR_ARG
    assert _attn(lib, scale=-0.5) == mvp.MVP_ERR_ARG
    assert _attn(lib, ndec=2) == mvp.MVP_ERR_ARG  # more decode requests than requests
    assert _attn(lib, ndec=-2) == mvp.MVP_ERR_ARG
    assert _attn(lib, total_q=0) == mvp.MVP_OK  # nothing to do


def _attn_ext(lib, variant=0, wait_limit_us=0, fault=0, **over):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, out=1 << 20, lse=None, cu_q=1 << 20, cu_k=1 << 20, ctx=None,
                num_reqs=1, total_q=4, total_k=4, max_q=4, max_k=4, ndec=-1, hq=4, hkv=2, d=128, table=None,
                covered=None, causal=1, wl=-1, wr=-1, sinks=None, sink_mode=0, scale=0.1, ws=None, ws_bytes=0,
                stream=None)
    args.update(over)
    opts = mvp.AttnOptions(variant, wait_limit_us, fault)
    return lib.mvp_attn_fwd_varlen_ext(*[args[k] for k in (
        "q", "k", "v", "out", "lse", "cu_q", "cu_k", "ctx", "num_reqs", "total_q", "total_k", "max_q", "max_k", "ndec",
        "hq", "hkv", "d", "table", "covered", "causal", "wl", "wr", "sinks", "sink_mode", "scale", "ws",
        "ws_bytes", "stream")], ctypes.byref(opts))


def test_ext_option_errors_return_before_any_launch(lib):
    assert _attn_ext(lib, variant=7) == mvp.MVP_ERR_ARG
    assert _attn_ext(lib, variant=-1) == mvp.MVP_ERR_ARG
    assert _attn_ext(lib, variant=mvp.VARIANT_D512_HEAD_SPLIT, d=128) == mvp.MVP_ERR_UNSUPPORTED
    assert _attn_ext(lib, fault=9) == mvp.MVP_ERR_ARG
    # the plain argument checks apply as well
    assert _attn_ext(lib, d=96) == mvp.MVP_ERR_UNSUPPORTED
    assert _attn_ext(lib, hq=3, hkv=2) == mvp.MVP_ERR_ARG
    assert _attn_ext(lib, total_q=0) == mvp.MVP_OK


def _paged(lib, **over):
    args = dict(q=1 << 20, kc=1 << 20, vc=1 << 20, out=1 << 20, lse=None, cu_q=1 << 20, seq_k=1 << 20,
                bt=1 << 20, bs=16, max_blocks=4, num_blocks=8, ctx=None, num_reqs=1, total_q=4, max_q=4, max_k=64,
                ndec=-1, hq=4, hkv=2, d=128, table=None, covered=None, causal=1, wl=-1, wr=-1, sinks=None,
                sink_mode=0, scale=0.1, ws=None, ws_bytes=0, stream=None)
    args.update(over)
    return lib.mvp_attn_fwd_paged(*[args[k] for k in (
        "q", "kc", "vc", "out", "lse", "cu_q", "seq_k", "bt", "bs", "max_blocks", "num_blocks", "ctx", "num_reqs",
        "total_q", "max_q", "max_k", "ndec", "hq", "hkv", "d", "table", "covered", "causal", "wl", "wr", "sinks",
        "sink_mode", "scale", "ws", "ws_bytes", "stream")])


def test_paged_argument_errors(lib):
    # Host validation of the block layout, before any CUDA call.
    assert _paged(lib, bs=8) == mvp.MVP_ERR_ARG  # below 16
    assert _paged(lib, bs=48) == mvp.MVP_ERR_ARG  # not a power of two
    assert _paged(lib, bs=512) == mvp.MVP_ERR_ARG  # above 256
    assert _paged(lib, max_blocks=3) == mvp.MVP_ERR_ARG  # 3 x 16 < max_k_len 64
    assert _paged(lib, bt=None) == mvp.MVP_ERR_ARG
    assert _paged(lib, seq_k=None) == mvp.MVP_ERR_ARG
    assert _paged(lib, num_blocks=0) == mvp.MVP_ERR_ARG
    assert _paged(lib, kc=(1 << 20) + 8) == mvp.MVP_ERR_UNSUPPORTED  # not 16-byte aligned
    assert _paged(lib, d=96) == mvp.MVP_ERR_UNSUPPORTED
    assert _paged(lib, total_q=0) == mvp.MVP_OK  # nothing to do


def _scan(lib, **over):
    args = dict(q=1 << 20, k=1 << 20, v=1 << 20, out=1 << 20, lse=None, cu_q=1 << 20, cu_k=1 << 20, ctx=None,
                num_reqs=1, total_q=4, total_k=64, max_q=4, max_k=64, ndec=-1, hq=4, hkv=2, d=128,
                ranges=1 << 20, max_ranges=2, causal=1, wl=-1, wr=-1, sinks=None, sink_mode=0, scale=0.1, ws=None,
                ws_bytes=0, stream=None)
    args.update(over)
    return lib.mvp_attn_fwd_varlen_scan(*[args[k] for k in (
        "q", "k", "v", "out", "lse", "cu_q", "cu_k", "ctx", "num_reqs", "total_q", "total_k", "max_q", "max_k",
        "ndec", "hq", "hkv", "d", "ranges", "max_ranges", "causal", "wl", "wr", "sinks", "sink_mode", "scale", "ws",
        "ws_bytes", "stream")])


def test_scan_argument_errors(lib):
    assert _scan(lib, ranges=None) == mvp.MVP_ERR_ARG           # max_ranges > 0 without ranges
    assert _scan(lib, max_ranges=-1) == mvp.MVP_ERR_ARG
    assert _scan(lib, max_ranges=4097) == mvp.MVP_ERR_ARG
    assert _scan(lib, ranges=(1 << 20) + 4) == mvp.MVP_ERR_UNSUPPORTED  # not 8-byte aligned
    assert _scan(lib, d=96) == mvp.MVP_ERR_UNSUPPORTED
    assert _scan(lib, total_q=0) == mvp.MVP_OK


def test_fill_argument_errors(lib):
    f = lib.mvp_fill_query_ranges
    assert f(None, 1, 1, 1 << 20, 1 << 20, 10, 1 << 20, 4, None, None) == mvp.MVP_ERR_ARG  # ranges null
    assert f(1 << 20, 1, 1, 1 << 20, 1 << 20, 10, 1 << 20, 4, None, None) == mvp.MVP_ERR_CAPACITY
    assert f(1 << 20, 1, 1, None, 1 << 20, 10, 1 << 20, 40, None, None) == mvp.MVP_ERR_ARG
    assert f(1 << 20, -1, 1, 1 << 20, 1 << 20, 10, 1 << 20, 40, None, None) == mvp.MVP_ERR_ARG


def test_workspace_size(lib):
    # a 256-byte header (the prefill work queue), then the decode partials
    assert mvp.attn_workspace_size(4, 16, 256, 1000) == 256  # one split: header only
    assert mvp.attn_workspace_size(0, 16, 256, 100000) == 256  # no decode rows
    n = mvp.attn_workspace_size(260, 32, 128, 32769)  # 4096-key split chunks: 9
    assert n == 256 + 260 * 32 * 9 * 130 * 4
    assert mvp.attn_workspace_size(-1, 16, 256, 1000) == 0
    assert mvp.attn_workspace_size(4, 0, 256, 1000) == 0


def test_binding_has_no_cpu_path():
    """The product modules never import the oracle."""
    pkg = os.path.join(ROOT, "masked_varlen_prefill_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h", ".cpp")):
                src = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f
