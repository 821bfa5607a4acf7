"""Step metadata and CUDA-graph replays through the C-ABI (GPU).

A ``StepMetadata`` (``mvp_meta_*``) is sized for a capacity; each batch is
staged on the host, then ONE captured graph (metadata upload + range-table
fill + attention over the capacity) is replayed.  Checks:

* the range table the upload leaves on the device equals the oracle's fill
  (``oracle.range_table.fill_by_spans`` on the same seq_lens bound) bit for
  bit on the batch's rows, and (-1, -1) on the padding rows;
* decode rows staged with an optimistic seq_lens upper bound stay outside
  every range (the invariant of the persistent-buffer design);
* a replay gives the bits of an eager call with the same (capacity)
  arguments, and the float64 oracle within the packed tests' tolerances;
* a batch without ranges staged after one with ranges leaves no stale
  table rows behind (buffer reuse).
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

HQ, HKV, D = 8, 2, 128
WINDOW_LEFT = 255
MAX_REQS, MAX_TOKENS, MAX_RANGES = 8, 1024, 6
MAX_KEYS = 6144  # packed key rows of the persistent K / V buffers
MAX_K_LEN = 1400


def _batch(seed, n_dec, n_pre, with_ranges=True, bound_slack=8):
    """Host metadata of one batch: decode requests first, then prefill chunks
    (context 0..400) with ranges inside [0, k_len), one straddling the chunk
    end.  Decode requests get prompt-side ranges and a seq_lens bound up to
    bound_slack above the true length."""
    rng = np.random.default_rng(seed)
    q_lens, k_lens, bound, per_req = [], [], [], []
    for _ in range(n_dec):
        kl = int(rng.integers(40, 1000))
        q_lens.append(1)
        k_lens.append(kl)
        bound.append(kl + int(rng.integers(0, bound_slack + 1)))
        s = int(rng.integers(0, kl // 2))
        per_req.append([(s, min(s + int(rng.integers(1, 60)), kl - 2))])
    for _ in range(n_pre):
        ql = int(rng.integers(2, 240))
        kl = ql + int(rng.integers(0, 400))
        q_lens.append(ql)
        k_lens.append(kl)
        bound.append(kl)
        rl, cur = [], int(rng.integers(0, max(1, kl // 3)))
        for _ in range(int(rng.integers(0, 4))):
            length = int(rng.integers(2, 120))
            rl.append((cur, cur + length - 1))
            cur += length + int(rng.integers(1, 30))
        rl.append((kl - int(rng.integers(1, ql + 1)), kl + 50))  # straddles the chunk end
        per_req.append(rl)
    qsl = np.zeros(len(q_lens) + 1, dtype=np.int32)
    qsl[1:] = np.cumsum(q_lens)
    ranges = workloads.pad_ranges(per_req) if with_ranges else None
    assert qsl[-1] <= MAX_TOKENS and sum(k_lens) <= MAX_KEYS and max(k_lens) <= MAX_K_LEN
    return qsl, np.asarray(k_lens, np.int32), np.asarray(bound, np.int32), ranges


def _oracle_table(qsl, bound, ranges):
    n = int(qsl[-1])
    out = np.full((max(1, n), 2), 4242, dtype=np.int32)
    if ranges is None:
        return np.full((n, 2), -1, np.int32), 0
    written = ort.fill_by_spans(out, ort.ranges_from_padded(ranges), qsl, bound)
    table = out[:n].copy()
    if written == 0:
        table[:] = -1
    return table, written


class _Graphed:
    """Persistent buffers + one graph: upload, fill and attention at capacity."""

    def __init__(self, dev, sinks):
        self.meta = mvp.StepMetadata(MAX_REQS, MAX_TOKENS, MAX_RANGES, dev)
        self.q = torch.zeros(MAX_TOKENS, HQ, D, dtype=torch.bfloat16, device=dev)
        self.k = torch.zeros(MAX_KEYS, HKV, D, dtype=torch.bfloat16, device=dev)
        self.v = torch.zeros_like(self.k)
        self.out = torch.zeros_like(self.q)
        self.lse = torch.zeros(HQ, MAX_TOKENS, device=dev)
        nbytes = mvp.attn_workspace_size(MAX_REQS, HQ, D, MAX_K_LEN)
        self.ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
        self.sinks = sinks
        self.graph = None

    def attention(self, out, lse):
        mvp.attn_fwd_varlen(self.q, self.k, self.v, out, self.meta.query_start_loc, self.meta.cu_seqlens_k,
                            MAX_TOKENS, MAX_K_LEN, lse=lse, range_table=self.meta.range_table,
                            range_covered=self.meta.range_covered, causal=True, window_left=WINDOW_LEFT,
                            sinks=self.sinks, sink_mode=mvp.SINK_NULL_LOGIT, scale=D ** -0.5,
                            workspace=self.ws)

    def capture(self):
        # eager first: the library's per-device state is set up outside capture
        self.meta.upload()
        self.attention(self.out, self.lse)
        torch.cuda.synchronize()
        self.graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.graph):
            self.meta.upload()
            self.attention(self.out, self.lse)
        torch.cuda.synchronize()

    def run(self, qsl, k_lens, bound, ranges, q, k, v):
        n_q, n_k = q.shape[0], k.shape[0]
        self.q[:n_q].copy_(q)
        self.k[:n_k].copy_(k)
        self.v[:n_k].copy_(v)
        self.meta.stage(qsl, k_lens, bound, ranges)
        self.graph.replay()
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0


def _inputs(qsl, k_lens, seed, dev):
    gen = torch.Generator(device=dev)
    gen.manual_seed(seed)
    q = torch.randn(int(qsl[-1]), HQ, D, generator=gen, device=dev).to(torch.bfloat16)
    k = torch.randn(int(k_lens.sum()), HKV, D, generator=gen, device=dev).to(torch.bfloat16)
    v = torch.randn(int(k_lens.sum()), HKV, D, generator=gen, device=dev).to(torch.bfloat16)
    return q, k, v


def test_graph_replays_match_eager_and_oracle():
    dev = torch.device("cuda")
    sinks = torch.randn(HQ, generator=torch.Generator(device=dev).manual_seed(5), device=dev)
    g = _Graphed(dev, sinks)
    g.capture()
    batches = [(11, 2, 3, True), (12, 5, 1, True), (13, 0, 2, False), (14, 3, 0, True), (15, 1, 4, True)]
    for seed, n_dec, n_pre, with_ranges in batches:
        qsl, k_lens, bound, ranges = _batch(seed, n_dec, n_pre, with_ranges)
        q, k, v = _inputs(qsl, k_lens, seed, dev)
        g.run(qsl, k_lens, bound, ranges, q, k, v)
        n = int(qsl[-1])
        # 1. the table on the device: the oracle's fill on the bound, then -1 padding
        ref_table, written = _oracle_table(qsl, bound, ranges)
        got_table = g.meta.range_table.cpu().numpy()
        assert np.array_equal(got_table[:n], ref_table), f"batch {seed}: range table"
        assert (got_table[n:] == -1).all(), f"batch {seed}: padding rows"
        assert (int(g.meta.range_covered.item()) != 0) == (written != 0)
        # 2. decode rows (staged with an upper bound) lie outside every range
        assert (got_table[qsl[:n_dec]] == -1).all(), f"batch {seed}: decode row inside a range"
        # 3. the replay's bits equal an eager call with the same arguments
        out_e = torch.full_like(g.out, float("nan"))
        lse_e = torch.full_like(g.lse, float("nan"))
        g.attention(out_e, lse_e)
        torch.cuda.synchronize()
        assert torch.equal(g.out[:n].view(torch.int16), out_e[:n].view(torch.int16)), f"batch {seed}: out"
        assert torch.equal(g.lse[:, :n], lse_e[:, :n]), f"batch {seed}: lse"
        # 4. and the float64 oracle on the exact key lengths
        cu_k = np.zeros(len(k_lens) + 1, np.int32)
        cu_k[1:] = np.cumsum(k_lens)
        ro, rl = oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), qsl, cu_k, True, WINDOW_LEFT, -1, D ** -0.5,
                                        range_table=ref_table if written else None, sinks=sinks.cpu(),
                                        sink_mode=mvp.SINK_NULL_LOGIT)
        gh.compare(g.out[:n], g.lse[:, :n], ro, rl, what=f"graph batch {seed}")
    g.meta.close()


def test_graph_replay_paged():
    """The same graph over a paged cache: block table and seq_lens_k from
    persistent buffers; equals the packed oracle on the gathered keys."""
    dev = torch.device("cuda")
    bs, max_blocks = 64, (MAX_K_LEN + 63) // 64
    meta = mvp.StepMetadata(MAX_REQS, MAX_TOKENS, MAX_RANGES, dev)
    n_cache_blocks = MAX_REQS * max_blocks + 4
    kc = torch.zeros(n_cache_blocks * bs, HKV, D, dtype=torch.bfloat16, device=dev)
    vc = torch.zeros_like(kc)
    table = torch.zeros(MAX_REQS, max_blocks, dtype=torch.int32, device=dev)
    qb = torch.zeros(MAX_TOKENS, HQ, D, dtype=torch.bfloat16, device=dev)
    out = torch.zeros_like(qb)
    nbytes = mvp.attn_workspace_size(MAX_REQS, HQ, D, MAX_K_LEN)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)

    def attention(o):
        mvp.attn_fwd_paged(qb, kc, vc, o, meta.query_start_loc, meta.seq_lens_k, table, bs, MAX_TOKENS,
                           MAX_K_LEN, range_table=meta.range_table, range_covered=meta.range_covered,
                           causal=True, window_left=WINDOW_LEFT, scale=D ** -0.5, workspace=ws)

    meta.upload()
    attention(out)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        meta.upload()
        attention(out)
    torch.cuda.synchronize()
    for seed, n_dec, n_pre in [(21, 2, 2), (22, 4, 1), (23, 0, 3)]:
        qsl, k_lens, bound, ranges = _batch(seed, n_dec, n_pre)
        q, k, v = _inputs(qsl, k_lens, seed, dev)
        kc_b, vc_b, bt_b, _ = workloads.to_paged(k, v, list(k_lens), bs, seed=seed)
        kc[:kc_b.shape[0]].copy_(kc_b)
        vc[:vc_b.shape[0]].copy_(vc_b)
        table.zero_()
        table[:bt_b.shape[0], :min(max_blocks, bt_b.shape[1])].copy_(bt_b[:, :max_blocks])
        qb[:q.shape[0]].copy_(q)
        meta.stage(qsl, k_lens, bound, ranges)
        graph.replay()
        torch.cuda.synchronize()
        assert mvp.get_last_device_error() == 0
        n = int(qsl[-1])
        ref_table, written = _oracle_table(qsl, bound, ranges)
        cu_k = np.zeros(len(k_lens) + 1, np.int32)
        cu_k[1:] = np.cumsum(k_lens)
        ro, rl = oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), qsl, cu_k, True, WINDOW_LEFT, -1, D ** -0.5,
                                        range_table=ref_table if written else None)
        gh.compare(out[:n], None, ro, rl, what=f"paged graph batch {seed}")
    meta.close()


def test_stage_reuse_leaves_no_stale_rows():
    dev = torch.device("cuda")
    meta = mvp.StepMetadata(MAX_REQS, MAX_TOKENS, MAX_RANGES, dev)
    qsl, k_lens, bound, ranges = _batch(31, 1, 4, True)
    meta.stage(qsl, k_lens, bound, ranges)
    meta.upload()
    torch.cuda.synchronize()
    assert int(meta.range_covered.item()) != 0
    assert (meta.range_table.cpu().numpy()[: int(qsl[-1])] >= 0).any()
    qsl2, k2, b2, _ = _batch(32, 2, 1, False)
    meta.stage(qsl2, k2, b2, None)
    meta.upload()
    torch.cuda.synchronize()
    assert int(meta.range_covered.item()) == 0
    assert (meta.range_table.cpu().numpy() == -1).all()
    blk = meta.block.cpu().numpy()
    _, offs = mvp.meta_block_layout(MAX_REQS, MAX_RANGES)
    assert (blk[offs[4]:] == 0).all(), "ranges of the earlier batch left in the block"
    assert np.array_equal(blk[offs[0]:offs[0] + len(qsl2)], qsl2)
    meta.close()


def test_empty_stage_writes_an_all_padding_table():
    dev = torch.device("cuda")
    meta = mvp.StepMetadata(2, 64, 1, dev)
    meta.stage(np.zeros(1, np.int32), np.zeros(0, np.int32))
    meta.upload()
    torch.cuda.synchronize()
    assert (meta.range_table.cpu().numpy() == -1).all()
    assert int(meta.range_covered.item()) == 0
    assert (meta.query_start_loc.cpu().numpy() == 0).all()
    meta.close()


def test_stage_waits_for_the_copy_in_flight():
    """Stage a new batch right after a replay was launched (no synchronize):
    the staging call waits for the replay's copy, so the replay reads the
    first batch and the next replay the second."""
    dev = torch.device("cuda")
    sinks = torch.randn(HQ, generator=torch.Generator(device=dev).manual_seed(6), device=dev)
    g = _Graphed(dev, sinks)
    g.capture()
    b1 = _batch(41, 2, 2)
    b2 = _batch(42, 1, 3)
    q1, k1, v1 = _inputs(b1[0], b1[1], 41, dev)
    n1 = int(b1[0][-1])
    g.q[:n1].copy_(q1)
    g.k[:k1.shape[0]].copy_(k1)
    g.v[:v1.shape[0]].copy_(v1)
    g.meta.stage(*b1)
    g.graph.replay()
    out1 = g.out.clone()  # stream-ordered after the first replay
    g.meta.stage(*b2)     # waits for the first replay's metadata copy only
    q2, k2, v2 = _inputs(b2[0], b2[1], 42, dev)
    n2 = int(b2[0][-1])
    g.q[:n2].copy_(q2)
    g.k[:k2.shape[0]].copy_(k2)
    g.v[:v2.shape[0]].copy_(v2)
    g.graph.replay()
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    for (qsl, k_lens, bound, ranges), q, k, v, out, n in [(b1, q1, k1, v1, out1, n1), (b2, q2, k2, v2, g.out, n2)]:
        ref_table, written = _oracle_table(qsl, bound, ranges)
        cu_k = np.zeros(len(k_lens) + 1, np.int32)
        cu_k[1:] = np.cumsum(k_lens)
        ro, rl = oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), qsl, cu_k, True, WINDOW_LEFT, -1, D ** -0.5,
                                        range_table=ref_table if written else None, sinks=sinks.cpu(),
                                        sink_mode=mvp.SINK_NULL_LOGIT)
        gh.compare(out[:n], None, ro, rl, what="in-flight staging")
    g.meta.close()
