"""The prefill work queue in the workspace header through the C-ABI (GPU).

With a workspace the prefill kernel's CTAs take the last round of items
from a tagged counter in its first 256 bytes instead of the static stride
(batches of fewer than two rounds, and masks with a window shorter than the
longest key run, keep the static stride, so the queue cases here have at
least two rounds and no such window; the windowed ones check that the
workspace changes nothing).  Every item is
computed the same way whichever CTA takes it, so the output must be the
static-stride output bit for bit: from an uninitialised workspace, from words
left by earlier calls or planted stale values, over item spaces that are
mostly empty (the skip-ahead), for single CTAs, pairs and the head-dim split
cluster, over paged caches, and across back-to-back CUDA-graph replays (a
replay can carry the previous replay's tag, so each launch's last CTA resets
the counter).  A 256-byte workspace holds only the header, so
decode rows run unsplit as without workspace and the whole output compares.
"""

import numpy as np
import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu

HEADER = 256


def _call(w, q, k, v, sinks, table, covered, ws, max_q=None, out=None, lse=None, cu=None, variant=0):
    cu_q, cu_k = gh.device_meta(w, q.device) if cu is None else cu
    out = torch.full_like(q, float("nan")) if out is None else out
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=q.device) if lse is None else lse
    mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max_q or max(max(w.q_lens), 1), max(max(w.k_lens), 1), lse=lse,
                        range_table=table, range_covered=covered, causal=w.causal, window_left=w.window_left,
                        window_right=w.window_right, sinks=sinks, sink_mode=w.sink_mode, scale=w.scale,
                        workspace=ws, variant=variant)
    return out, lse


def _check_equal(a, b, what):
    assert torch.equal(a[0].view(torch.int16), b[0].view(torch.int16)), f"{what}: output differs from static"
    assert torch.equal(a[1].nan_to_num(posinf=1e30, neginf=-1e30), b[1].nan_to_num(posinf=1e30, neginf=-1e30)), \
        f"{what}: lse differs from static"


def _static_and_queue(w, ws_fill=None, max_q=None, repeats=1, variant=0):
    q, k, v, sinks = gh.make_inputs(w)
    _, _, table, covered = gh.run_gpu(w, q, k, v, sinks, use_workspace=False)
    ref = _call(w, q, k, v, sinks, table, covered, None, max_q=max_q, variant=variant)
    ws = torch.empty(HEADER, dtype=torch.uint8, device=q.device)
    if ws_fill is not None:
        ws.view(torch.int64)[:] = ws_fill
    for r in range(repeats):
        got = _call(w, q, k, v, sinks, table, covered, ws, max_q=max_q, variant=variant)
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0
        _check_equal(got, ref, f"{w.name} call {r}")
    return q, k, v, sinks, table, covered, ref


@pytest.mark.parametrize("name", ["mm_prefix_sliding", "chunked_prefill_ranges", "mixed_serving_a",
                                  "mixed_serving_b", "global_causal_d512"])
def test_full_workloads(name):
    _static_and_queue(workloads.workload(name), repeats=3)


def _many_items_case(seed):
    """A random batch of 24-40 requests (every mask, sink and range option
    of the random cases) with enough work items for two rounds."""
    rng = np.random.default_rng(5000 + seed)
    d = [64, 128, 256, 512][seed % 4]
    group = int(rng.choice([1, 2, 4] if d == 512 else [1, 2, 4, 8]))
    hkv = 4
    n = int(rng.integers(24, 41))
    q_lens = [0 if rng.integers(0, 8) == 0 else (1 if rng.integers(0, 6) == 0 else int(rng.integers(2, 700)))
              for _ in range(n)]
    q_lens[0] = max(q_lens[0], 5)
    k_lens = [ql + (int(rng.integers(0, 2000)) if rng.integers(0, 2) else 0) for ql in q_lens]
    causal = bool(rng.integers(0, 3) > 0)
    ranges = None
    if rng.integers(0, 2):
        per_req = []
        for kl in k_lens:
            rl, cur = [], int(rng.integers(0, max(1, kl // 2 + 1)))
            for _ in range(int(rng.integers(0, 5))):
                length = int(rng.integers(1, 200))
                rl.append((cur, cur + length - 1))
                cur += length + int(rng.integers(1, 40))
            per_req.append(rl)
        ranges = workloads.pad_ranges(per_req)
    return workloads.Workload(f"many{seed}", 6000 + seed, q_lens, k_lens, hkv * group, hkv, d, causal,
                              -1 if seed % 2 == 0 else int(rng.choice([-1, 63, 400])),
                              -1 if causal else int(rng.choice([-1, 77])),
                              int(rng.integers(0, 3)), ranges)


@pytest.mark.parametrize("seed", range(8))
def test_many_request_batches(seed):
    _static_and_queue(_many_items_case(seed), repeats=2)


# stale words a workspace may hold: zeros, all ones, a tag with the counter
# far past any item, a tag with the counter at 0, arbitrary bits
STALE = [0, -1, (0x1234 << 32) | 0x7fffff00, 0x7ffffffe << 32, 0x5a5a5a5a5a5a5a5a]


@pytest.mark.parametrize("word", STALE)
def test_stale_queue_words(word):
    _static_and_queue(workloads.workload("global_causal_d512"), ws_fill=word)


def test_mostly_empty_item_space():
    """A capacity-sized grid (max_q_len far above the batch's) over a batch
    of empty, decode and short prefill requests: most claimed items have no
    rows and the queue skips past them."""
    q_lens = [0, 1, 0, 200, 1, 0, 0, 37, 0, 1] * 6
    k_lens = [5, 300, 0, 900, 64, 0, 3, 37, 1, 2000] * 6
    w = workloads.Workload("sparse_items", 4242, q_lens, k_lens, 8, 2, 128, True, -1, 0, workloads.SINK_NULL_LOGIT,
                           None)
    _static_and_queue(w, max_q=8192, repeats=2)


def test_head_split_cluster():
    _static_and_queue(workloads.workload("global_causal_d512"), repeats=2, variant=mvp.VARIANT_D512_HEAD_SPLIT)


def test_paged():
    w = workloads.workload("global_causal_d512")
    q, k, v, sinks = gh.make_inputs(w)
    _, _, table, covered = gh.run_gpu(w, q, k, v, sinks, use_workspace=False)
    kc, vc, bt, sl = workloads.to_paged(k, v, w.k_lens, 16, seed=5)
    cu_q, _ = gh.device_meta(w, q.device)
    res = []
    for ws in (None, torch.empty(HEADER, dtype=torch.uint8, device=q.device)):
        out = torch.full_like(q, float("nan"))
        lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=q.device)
        mvp.attn_fwd_paged(q, kc, vc, out, cu_q, sl, bt, 16, max(w.q_lens), max(w.k_lens), lse=lse,
                           range_table=table, range_covered=covered, causal=w.causal, window_left=w.window_left,
                           window_right=w.window_right, sinks=sinks, sink_mode=w.sink_mode, scale=w.scale,
                           workspace=ws)
        res.append((out, lse))
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    _check_equal(res[1], res[0], "paged")


def test_back_to_back_graph_replays():
    """Replays of one captured call with nothing in between: each must start
    from item 0 whatever tag the previous replay left."""
    w = workloads.workload("global_causal_d512")
    q, k, v, sinks = gh.make_inputs(w)
    _, _, table, covered = gh.run_gpu(w, q, k, v, sinks, use_workspace=False)
    ws = torch.empty(HEADER, dtype=torch.uint8, device=q.device)
    qg = q.clone()
    out = torch.zeros_like(q)
    lse = torch.zeros(w.num_heads_q, w.total_q, device=q.device)
    cu = gh.device_meta(w, q.device)  # (no host copies inside the capture)
    _call(w, qg, k, v, sinks, table, covered, ws, out=out, lse=lse, cu=cu)  # eager first (library state)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        _call(w, qg, k, v, sinks, table, covered, ws, out=out, lse=lse, cu=cu)
    torch.cuda.synchronize()
    gen = torch.Generator(device=q.device)
    for r in range(4):
        gen.manual_seed(77 + r)
        qg.copy_(torch.randn(q.shape, generator=gen, device=q.device).to(q.dtype))
        out.fill_(float("nan"))
        lse.fill_(float("nan"))
        graph.replay()
        ref = _call(w, qg, k, v, sinks, table, covered, None)
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0
        _check_equal((out, lse), ref, f"replay {r}")


def test_header_only_workspace_leaves_decode_unsplit():
    """256 bytes: queue only, no split partials (decode rows as without
    workspace).  A full-size workspace also splits the long decode rows,
    which rounds differently: its prefill rows must still be identical and its
    decode rows within the parity tolerance of the unsplit ones."""
    w = workloads.workload("mixed_serving_a")
    q, k, v, sinks, table, covered, ref = _static_and_queue(w)
    n_dec = sum(1 for x in w.q_lens if x == 1)
    nbytes = mvp.attn_workspace_size(w.num_reqs, w.num_heads_q, w.head_dim, max(w.k_lens))
    assert nbytes > HEADER
    ws = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    out, lse = _call(w, q, k, v, sinks, table, covered, ws)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    # prefill rows: identical; decode rows: within the parity tolerances of the unsplit result
    cu_q, _ = w.cu_seqlens()
    pre = np.concatenate([np.arange(cu_q[b], cu_q[b + 1]) for b in range(w.num_reqs) if w.q_lens[b] > 1])
    dec = np.asarray([cu_q[b] for b in range(w.num_reqs) if w.q_lens[b] == 1])
    assert n_dec == len(dec) > 0
    pre_t, dec_t = torch.from_numpy(pre).to(q.device), torch.from_numpy(dec).to(q.device)
    assert torch.equal(out[pre_t].view(torch.int16), ref[0][pre_t].view(torch.int16))
    diff = (out[dec_t].float() - ref[0][dec_t].float()).abs().max().item()
    assert diff <= gh.OUT_ATOL, diff
