"""Attention over a paged K/V cache through the C-ABI (GPU).

The same logical keys and values are laid out in a cache whose blocks are
taken in a seeded random order (``workloads.to_paged``), with garbage in the
block-table entries a request does not use.  The paged call must give the
packed call's output bit for bit, and the float64 oracle (run on the keys
gathered back from the cache by ``oracle.attention.gather_paged``) within the
tolerances of the packed tests.
"""

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import attention as oatt

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu


def _run_paged(w, q, k, v, sinks, block_size, table, covered, use_workspace=True, num_decode_reqs=-1,
               table_fill=-1, seed=0):
    dev = q.device
    kc, vc, bt, sl = workloads.to_paged(k, v, w.k_lens, block_size, seed=seed, table_fill=table_fill)
    cu_q, _ = gh.device_meta(w, dev)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev)
    ws = None
    if use_workspace:
        n_dec = w.num_reqs if num_decode_reqs < 0 else num_decode_reqs
        nbytes = mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    mvp.attn_fwd_paged(q, kc, vc, out, cu_q, sl, bt, block_size, max(max(w.q_lens), 1), max(max(w.k_lens), 1),
                       lse=lse, range_table=table, range_covered=covered, causal=w.causal,
                       window_left=w.window_left, window_right=w.window_right, sinks=sinks, sink_mode=w.sink_mode,
                       scale=w.scale, workspace=ws, num_decode_reqs=num_decode_reqs)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    return out, lse, (kc, vc, bt, sl)


def _paged_parity(w, block_size, num_decode_reqs=-1, table_fill=-1, use_workspace=True, strict=False):
    q, k, v, sinks = gh.make_inputs(w)
    out_p, lse_p, table, covered = gh.run_gpu(w, q, k, v, sinks, use_workspace=use_workspace,
                                              num_decode_reqs=num_decode_reqs)
    out_g, lse_g, (kc, vc, bt, sl) = _run_paged(w, q, k, v, sinks, block_size, table, covered,
                                               use_workspace=use_workspace, num_decode_reqs=num_decode_reqs,
                                               table_fill=table_fill, seed=w.seed + block_size)
    # same logical keys, same arithmetic: identical bits
    assert torch.equal(out_g.view(torch.int16), out_p.view(torch.int16)), f"{w.name}: paged != packed output"
    assert torch.equal(lse_g, lse_p) or torch.allclose(lse_g, lse_p, rtol=0, atol=0, equal_nan=True)
    # and the oracle on the keys read back through the block table
    ref_table, _ = gh.oracle_table(w)
    kg, vg, cu_k = oatt.gather_paged(kc.cpu(), vc.cpu(), bt.cpu().numpy(), sl.cpu().numpy(), block_size)
    cu_q, _ = w.cu_seqlens()
    ro, rl = oatt.attention_forward(q.cpu(), kg, vg, cu_q, cu_k, w.causal, w.window_left, w.window_right,
                                    w.scale, range_table=ref_table, sinks=None if sinks is None else sinks.cpu(),
                                    sink_mode=w.sink_mode)
    return gh.compare(out_g, lse_g, ro, rl, what=f"{w.name} paged bs={block_size}", strict=strict)


@pytest.mark.parametrize("name", ["mm_prefix_sliding", "chunked_prefill_ranges", "mixed_serving_b",
                                  "global_causal_d512", "tiny_window_sinks"])
@pytest.mark.parametrize("block_size", [16, 64, 256])
def test_scaled_workloads_paged(name, block_size):
    _paged_parity(workloads.scaled_workload(name), block_size, strict=True)


@pytest.mark.parametrize("seed", range(12))
def test_random_cases_paged(seed):
    w = workloads.random_case(500 + seed)
    bs = [16, 32, 64, 128, 256][seed % 5]
    _paged_parity(w, bs, table_fill=[-1, 0, 2_000_000_000][seed % 3], use_workspace=seed % 4 != 3)


@pytest.mark.parametrize("d", [64, 128, 256, 512])
def test_head_dims_paged(d):
    w = workloads.Workload(f"paged_d{d}", 40 + d, [200, 1, 77, 130], [450, 900, 77, 300], 4, 2, d, True, 150, 0,
                           workloads.SINK_NULL_LOGIT, None)
    _paged_parity(w, 32)


def test_decode_first_paged():
    w = workloads.scaled_workload("mixed_serving_a")
    n_dec = 0
    while n_dec < w.num_reqs and w.q_lens[n_dec] == 1:
        n_dec += 1
    _paged_parity(w, 16, num_decode_reqs=n_dec, strict=True)
