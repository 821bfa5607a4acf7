"""Scan mode (``mvp_attn_fwd_varlen_scan``) through the C-ABI (GPU).

With non-overlapping ranges (every workload and random case here; some
degenerate) scan mode must give the bits of fill + table mode.  With
overlapping ranges it follows the scan's union, checked against the float64
oracle's scan mask (``oracle.attention.visible_mask_scan``).
"""

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import attention as oatt

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _run_scan(w, q, k, v, sinks, ranges, use_workspace=True, num_decode_reqs=-1):
    dev = q.device
    cu_q, cu_k = gh.device_meta(w, dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
    ws = None
    if use_workspace:
        n_dec = w.num_reqs if num_decode_reqs < 0 else num_decode_reqs
        nbytes = mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    rg = None if ranges is None else torch.from_numpy(np.ascontiguousarray(ranges, dtype=np.int32)).to(dev)
    mvp.attn_fwd_varlen_scan(q, k, v, out, cu_q, cu_k, max(max(w.q_lens), 1), max(max(w.k_lens), 1), rg, lse=lse,
                             causal=w.causal, window_left=w.window_left, window_right=w.window_right, sinks=sinks,
                             sink_mode=w.sink_mode, scale=w.scale, workspace=ws, num_decode_reqs=num_decode_reqs)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    return out, lse


def _bitwise_vs_table(w, **kw):
    q, k, v, sinks = gh.make_inputs(w)
    out_t, lse_t, _, _ = gh.run_gpu(w, q, k, v, sinks, **kw)
    out_s, lse_s = _run_scan(w, q, k, v, sinks, w.ranges, **kw)
    assert torch.equal(out_s.view(torch.int16), out_t.view(torch.int16)), f"{w.name}: scan != table output"
    assert torch.equal(lse_s, lse_t), f"{w.name}: scan != table lse"
    return q, k, v, sinks, out_s, lse_s


@pytest.mark.parametrize("name", ["mm_prefix_sliding", "chunked_prefill_ranges"])
def test_scaled_workloads_scan_equals_table(name):
    w = workloads.scaled_workload(name)
    q, k, v, sinks, out_s, lse_s = _bitwise_vs_table(w)
    cu_q, cu_k = w.cu_seqlens()
    ro, rl = oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), cu_q, cu_k, w.causal, w.window_left, w.window_right,
                                    w.scale, sinks=None if sinks is None else sinks.cpu(), sink_mode=w.sink_mode,
                                    scan_ranges=w.ranges)
    gh.compare(out_s, lse_s, ro, rl, what=f"{w.name} scan")


@pytest.mark.parametrize("seed", range(16))
def test_random_cases_scan_equals_table(seed):
    w = workloads.random_case(700 + seed)
    if w.ranges is None:
        w.ranges = workloads.pad_ranges([[(0, 3), (10, 40)] for _ in range(w.num_reqs)])
    _bitwise_vs_table(w, use_workspace=seed % 3 != 0)


@pytest.mark.parametrize("seed", range(8))
def test_overlapping_ranges_follow_the_scan(seed):
    rng = np.random.default_rng(seed)
    d = [64, 128, 256, 512][seed % 4]
    q_lens = [int(rng.integers(2, 300)), 1, int(rng.integers(2, 200))]
    k_lens = [q_lens[0] + int(rng.integers(0, 300)), int(rng.integers(50, 700)), q_lens[2]]
    per_req = []
    for kl in k_lens:
        rl = []
        for _ in range(int(rng.integers(1, 6))):
            s = int(rng.integers(0, kl))
            rl.append((s, s + int(rng.integers(-3, kl // 2 + 2))))
        per_req.append(rl)
    per_req[1].append((0, k_lens[1] + 4))  # the decode row sits inside a range
    w = workloads.Workload(f"overlap{seed}", 900 + seed, q_lens, k_lens, 4, 2, d, True,
                           int(rng.choice([-1, 31, 100])), 0, int(rng.integers(0, 3)), workloads.pad_ranges(per_req))
    q, k, v, sinks = gh.make_inputs(w)
    out_s, lse_s = _run_scan(w, q, k, v, sinks, w.ranges)
    cu_q, cu_k = w.cu_seqlens()
    ro, rl = oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), cu_q, cu_k, w.causal, w.window_left, w.window_right,
                                    w.scale, sinks=None if sinks is None else sinks.cpu(), sink_mode=w.sink_mode,
                                    scan_ranges=w.ranges)
    gh.compare(out_s, lse_s, ro, rl, what=f"{w.name} scan", strict=False)


def test_decode_first_scan():
    w = workloads.scaled_workload("mixed_serving_b")
    w.ranges = workloads.pad_ranges([[(0, kl + 3)] if i % 2 else [(5, 60)] for i, kl in enumerate(w.k_lens)])
    n_dec = sum(1 for x in w.q_lens if x == 1)
    _bitwise_vs_table(w, num_decode_reqs=n_dec)
