"""Seeded synthetic inputs for masked varlen prefill attention.

This module only draws inputs: lengths, range lists and N(0, 1) tensors.  It
holds none of the attention or range-table arithmetic, so both the GPU path
and the CPU oracle can be fed from it.

The five workloads follow the serving shapes the source pages discuss:

1. ``tiny_window_sinks``   -- vLLM PR #49815 (MiMo window attention): lengths
   37 and 5, 4 q heads / 2 KV heads, D 64, symmetric window 8, key-0-bias
   sinks.
2. ``mm_prefix_sliding``   -- vLLM PR #50294 (Gemma4 sliding layer, D 256):
   4 x 4096-token prefills, 16/8 heads, causal 1024-token window, 8
   bidirectional ranges of 256 tokens per request.
3. ``global_causal_d512``  -- Gemma4 global layer (D 512): 2 x 8192, 8/2
   heads, pure causal.
4. ``chunked_prefill_ranges`` -- 8 chunks of 2048 tokens after a context of
   0..30000, 16/8 heads, D 256, causal 4096 window, 1..64 ranges per request
   (some degenerate, some straddling the context start or the chunk end).
5. ``mixed_serving``       -- 256 decode rows (context 1024..32768) + 4
   prefill chunks of 1024 over contexts 0..16384, 32/8 heads, D 128,
   null-logit sinks; variant ``a`` full causal, ``b`` 4096 window.

Window convention: a W-token causal window is ``window_left = W - 1``,
``window_right = 0`` (the key at distance W-1 is the oldest one kept); a
symmetric window ``|i - j| <= w`` is ``window_left = window_right = w``.
Ranges are closed ``(start, end)``; a range of L tokens is ``(s, s + L - 1)``.
"""

from __future__ import annotations

import dataclasses
import math
from typing import Optional

import numpy as np
import torch

SINK_NONE = 0
SINK_KEY0_BIAS = 1
SINK_NULL_LOGIT = 2


@dataclasses.dataclass
class Workload:
    name: str
    seed: int
    q_lens: list
    k_lens: list
    num_heads_q: int
    num_heads_kv: int
    head_dim: int
    causal: bool
    window_left: int
    window_right: int
    sink_mode: int
    ranges: Optional[np.ndarray]  # int32 [B, max_ranges, 2] closed ranges, or None
    scale: float = 0.0

    def __post_init__(self):
        if self.scale == 0.0:
            self.scale = 1.0 / math.sqrt(self.head_dim)

    @property
    def num_reqs(self):
        return len(self.q_lens)

    @property
    def total_q(self):
        return int(sum(self.q_lens))

    @property
    def total_k(self):
        return int(sum(self.k_lens))

    def cu_seqlens(self):
        cu_q = np.zeros(self.num_reqs + 1, dtype=np.int32)
        cu_k = np.zeros(self.num_reqs + 1, dtype=np.int32)
        cu_q[1:] = np.cumsum(self.q_lens)
        cu_k[1:] = np.cumsum(self.k_lens)
        return cu_q, cu_k

    def context_lens(self):
        return np.asarray(self.k_lens, dtype=np.int32) - np.asarray(self.q_lens, dtype=np.int32)


def _bf16_normal(shape, gen, device):
    return torch.randn(*shape, generator=gen, device=device, dtype=torch.float32).to(torch.bfloat16)


def make_tensors(w: Workload, device="cpu"):
    """Draw q, k, v (bf16 ~ N(0,1)) and sinks (fp32 ~ N(0,1)) for ``w``.

    The generator lives on ``device`` and is seeded with ``w.seed``; q, k, v,
    sinks are drawn in that order.
    """
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    q = _bf16_normal((w.total_q, w.num_heads_q, w.head_dim), gen, device)
    k = _bf16_normal((w.total_k, w.num_heads_kv, w.head_dim), gen, device)
    v = _bf16_normal((w.total_k, w.num_heads_kv, w.head_dim), gen, device)
    sinks = None
    if w.sink_mode != SINK_NONE:
        sinks = torch.randn(w.num_heads_q, generator=gen, device=device, dtype=torch.float32)
    return q, k, v, sinks


def pad_ranges(per_req, min_width=1):
    """List of per-request range lists -> int32 ``[B, width, 2]``, padding (0, 0)."""
    width = max([min_width] + [len(r) for r in per_req])
    arr = np.zeros((len(per_req), width, 2), dtype=np.int32)
    for b, rl in enumerate(per_req):
        for r, (s, e) in enumerate(rl):
            arr[b, r] = (s, e)
    return arr


def _spaced_ranges(rng, n, length, span):
    """``n`` closed ranges of ``length`` tokens inside ``[0, span)``, sorted,
    with at least one free token between neighbours, offsets uniform."""
    slack = span - n * length - (n - 1)
    assert slack >= 0
    u = np.sort(rng.integers(0, slack + 1, size=n))
    starts = u + np.arange(n) * (length + 1)
    return [(int(s), int(s + length - 1)) for s in starts]


def _chunk_ranges(rng, ctx, chunk):
    """Range list of the chunked-prefill workload for one request.

    Anchors: one range straddling the chunk end ``ctx + chunk`` (so it gets
    clipped) and, when ``ctx > 0``, one straddling ``ctx`` (so its context part
    is clipped).  The remaining ranges are laid out from a cursor drawn in
    ``[max(0, ctx - 1024), ctx]`` with lengths 64..320 and gaps 1..64, jumping
    over the anchors.  About one in eight non-anchor ranges is made degenerate
    (``end == start`` or ``end < start``).
    """
    n = int(rng.integers(1, 65))
    anchors = []
    length = int(rng.integers(64, 321))
    back = int(rng.integers(1, length))
    anchors.append((ctx + chunk - back, ctx + chunk - back + length - 1))
    if ctx > 0:
        length = int(rng.integers(64, 321))
        back = int(rng.integers(1, min(ctx, length - 1) + 1))
        anchors.append((ctx - back, ctx - back + length - 1))
    anchors.sort()
    out = list(anchors)
    cursor = int(rng.integers(max(0, ctx - 1024), ctx + 1))
    placed = len(anchors)
    guard = 0
    while placed < n and guard < 10000:
        guard += 1
        length = int(rng.integers(64, 321))
        s, e = cursor, cursor + length - 1
        clash = [a for a in anchors if not (e + 1 < a[0] or s > a[1] + 1)]
        if clash:
            cursor = max(a[1] for a in clash) + int(rng.integers(2, 66))
            continue
        if rng.integers(0, 8) == 0:
            e = s if rng.integers(0, 2) == 0 else s - int(rng.integers(1, 17))
        out.append((s, e))
        placed += 1
        cursor = cursor + length + int(rng.integers(1, 65))
    out.sort(key=lambda r: r[0])
    return out


def workload(name: str) -> Workload:
    """The named full-size workload (see module docstring)."""
    if name == "tiny_window_sinks":
        return Workload(name, 0, [37, 5], [37, 5], 4, 2, 64, False, 8, 8, SINK_KEY0_BIAS, None,
                        scale=1.0 / 8.0)
    if name == "mm_prefix_sliding":
        rng = np.random.default_rng(1)
        per_req = [_spaced_ranges(rng, 8, 256, 4096) for _ in range(4)]
        return Workload(name, 1, [4096] * 4, [4096] * 4, 16, 8, 256, True, 1023, 0, SINK_NONE,
                        pad_ranges(per_req))
    if name == "global_causal_d512":
        return Workload(name, 2, [8192] * 2, [8192] * 2, 8, 2, 512, True, -1, -1, SINK_NONE, None)
    if name == "chunked_prefill_ranges":
        rng = np.random.default_rng(3)
        ctxs = [int(c) for c in rng.integers(0, 30001, size=8)]
        per_req = [_chunk_ranges(rng, c, 2048) for c in ctxs]
        return Workload(name, 3, [2048] * 8, [c + 2048 for c in ctxs], 16, 8, 256, True, 4095, 0,
                        SINK_NONE, pad_ranges(per_req))
    if name in ("mixed_serving_a", "mixed_serving_b"):
        rng = np.random.default_rng(4)
        dec_ctx = [int(c) for c in rng.integers(1024, 32769, size=256)]
        pre_ctx = [int(c) for c in rng.integers(0, 16385, size=4)]
        q_lens = [1] * 256 + [1024] * 4
        k_lens = [c + 1 for c in dec_ctx] + [c + 1024 for c in pre_ctx]
        wl = -1 if name.endswith("a") else 4095
        return Workload(name, 4, q_lens, k_lens, 32, 8, 128, True, wl, 0, SINK_NULL_LOGIT, None)
    if name == "decode_profile":
        # profiler-sized slice of the mixed serving batch: its first 32 decode
        # rows (same context draw), 4096-token window, ~0.5 GB of K/V
        rng = np.random.default_rng(4)
        dec_ctx = [int(c) for c in rng.integers(1024, 32769, size=256)][:32]
        return Workload(name, 4, [1] * 32, [c + 1 for c in dec_ctx], 32, 8, 128, True, 4095, 0, SINK_NULL_LOGIT,
                        None)
    if name == "prefill_d128_profile":
        # profiler-sized slice of the mixed serving batch: its 4 prefill chunks
        # of 1024 tokens (same context draw), 4096-token window
        rng = np.random.default_rng(4)
        rng.integers(1024, 32769, size=256)
        pre_ctx = [int(c) for c in rng.integers(0, 16385, size=4)]
        return Workload(name, 4, [1024] * 4, [c + 1024 for c in pre_ctx], 32, 8, 128, True, 4095, 0,
                        SINK_NULL_LOGIT, None)
    raise KeyError(name)


# Small slices of the mixed serving batch for profiler captures (a few hundred
# MB on the device); not part of the benchmark set.
PROFILE_WORKLOADS = ["decode_profile", "prefill_d128_profile"]

WORKLOADS = ["tiny_window_sinks", "mm_prefix_sliding", "global_causal_d512",
             "chunked_prefill_ranges", "mixed_serving_a", "mixed_serving_b"]


def fill_stress_case(seed: int = 99, num_reqs: int = 4096, rows: int = 1024, num_ranges: int = 64):
    """Range-fill stress input: ``num_reqs`` requests of ``rows`` query rows
    after a context drawn from 0..2047, each with ``num_ranges`` closed ranges
    of 8..39 tokens separated by 1..9 free tokens from a start in 0..199 (so
    about half the rows hold a range).  Returns (ranges int32 [B, R, 2],
    q_lens, seq_lens) as lists / arrays.  Input drawing only."""
    rng = np.random.default_rng(seed)
    seq = rows + rng.integers(0, 2048, size=num_reqs)
    start0 = rng.integers(0, 200, size=num_reqs)
    length = rng.integers(8, 40, size=(num_reqs, num_ranges))
    gap = rng.integers(1, 10, size=(num_reqs, num_ranges))
    step = length + gap
    starts = start0[:, None] + np.concatenate([np.zeros((num_reqs, 1), np.int64), np.cumsum(step, axis=1)[:, :-1]],
                                              axis=1)
    ranges = np.stack([starts, starts + length - 1], axis=2).astype(np.int32)
    return ranges, [rows] * num_reqs, [int(x) for x in seq]


def to_paged(k, v, k_lens, block_size: int, seed: int = 0, spare_blocks: int = 3, table_fill: int = -1):
    """Lay packed keys/values out in a paged cache (input generation only).

    k, v: [total_k, Hkv, D] packed by request (k_lens[b] rows each).  Returns
    (k_cache, v_cache, block_table, seq_lens): the caches are [num_blocks *
    block_size, Hkv, D] (random bf16 in the unused slots of a small cache,
    zeros in a large one), request b's keys
    occupy ceil(k_lens[b] / block_size) blocks drawn in a seeded random order
    from num_blocks = needed + spare_blocks, block_table is int32 [B,
    max_blocks + 1] with unused entries set to ``table_fill``, seq_lens int32
    [B].  Tensors live on k's device.
    """
    gen = np.random.default_rng(seed)
    lens = np.asarray([int(n) for n in k_lens], dtype=np.int64)
    need = (lens + block_size - 1) // block_size
    num_blocks = int(need.sum()) + spare_blocks
    perm = gen.permutation(num_blocks).astype(np.int64)
    max_blocks = max(int(need.max()) if len(need) else 1, 1) + 1
    table = np.full((len(lens), max_blocks), table_fill, dtype=np.int32)
    first = np.concatenate([[0], np.cumsum(need)[:-1]]) if len(need) else np.zeros(0, dtype=np.int64)
    rows = []
    for b in range(len(lens)):
        ids = perm[first[b]: first[b] + need[b]]
        table[b, :need[b]] = ids
        j = np.arange(lens[b], dtype=np.int64)
        rows.append(ids[j // block_size] * block_size + j % block_size)
    dev = k.device
    idx = torch.from_numpy(np.concatenate(rows) if rows else np.zeros(0, dtype=np.int64)).to(dev)
    hkv, d = k.shape[1], k.shape[2]
    n_rows = num_blocks * block_size
    if n_rows * hkv * d <= (1 << 24):  # small caches: random filler in the unused slots
        tg = torch.Generator(device="cpu").manual_seed(seed)
        k_cache = torch.randn(n_rows, hkv, d, generator=tg).to(torch.bfloat16).to(dev)
        v_cache = torch.randn(n_rows, hkv, d, generator=tg).to(torch.bfloat16).to(dev)
    else:
        k_cache = torch.zeros(n_rows, hkv, d, dtype=torch.bfloat16, device=dev)
        v_cache = torch.zeros(n_rows, hkv, d, dtype=torch.bfloat16, device=dev)
    k_cache[idx] = k
    v_cache[idx] = v
    return (k_cache, v_cache, torch.from_numpy(table).to(dev),
            torch.tensor([int(n) for n in k_lens], dtype=torch.int32, device=dev))


def scaled_workload(name: str, seed: int = 100) -> Workload:
    """Small versions of the workloads: same head layout, D, mask kind and
    sink mode, sequence lengths cut so the float64 oracle finishes in seconds
    while still spanning several 128-row / 128-key tiles and ragged tails."""
    rng = np.random.default_rng(seed)
    if name == "tiny_window_sinks":
        return workload(name)
    if name == "mm_prefix_sliding":
        q_lens = [517, 300, 1, 129]
        per_req = []
        for ql in q_lens:
            n = min(5, max(1, ql // 60))
            per_req.append(_spaced_ranges(rng, n, min(40, ql // n - 1) if ql > 5 else 1, ql) if ql > 8 else [])
        return Workload(name + "_small", seed, q_lens, list(q_lens), 4, 2, 256, True, 127, 0,
                        SINK_NONE, pad_ranges(per_req))
    if name == "global_causal_d512":
        return Workload(name + "_small", seed, [333, 64], [333, 64], 4, 1, 512, True, -1, -1,
                        SINK_NONE, None)
    if name == "chunked_prefill_ranges":
        ctxs = [0, 700, 1500]
        per_req = [_chunk_ranges(rng, c, 256) for c in ctxs]
        # keep range lengths compatible with the short chunk: clip anything huge
        return Workload(name + "_small", seed, [256, 256, 200], [256, 956, 1700], 4, 2, 256, True,
                        383, 0, SINK_NONE, pad_ranges(per_req))
    if name in ("mixed_serving_a", "mixed_serving_b"):
        dec_ctx = [int(c) for c in rng.integers(100, 3000, size=6)]
        q_lens = [1] * 6 + [200, 131]
        k_lens = [c + 1 for c in dec_ctx] + [200 + 900, 131]
        wl = -1 if name.endswith("a") else 511
        return Workload(name + "_small", seed, q_lens, k_lens, 8, 2, 128, True, wl, 0,
                        SINK_NULL_LOGIT, None)
    raise KeyError(name)


def random_tiny(seed: int) -> Workload:
    """A random tiny case over every flag combination (brute-force checks)."""
    rng = np.random.default_rng(seed)
    b = int(rng.integers(1, 4))
    q_lens, k_lens = [], []
    for _ in range(b):
        ql = int(rng.integers(0, 9))
        ctx = int(rng.integers(0, 7))
        q_lens.append(ql)
        k_lens.append(ql + ctx)
    hkv = int(rng.choice([1, 2]))
    hq = hkv * int(rng.choice([1, 2, 3]))
    d = int(rng.choice([4, 8]))
    causal = bool(rng.integers(0, 2))
    wl = int(rng.choice([-1, 0, 1, 3]))
    wr = int(rng.choice([-1, 0, 2])) if not causal else 0
    mode = int(rng.integers(0, 3))
    per_req = []
    for ql, kl in zip(q_lens, k_lens):
        rl = []
        cur = int(rng.integers(0, 3))
        for _ in range(int(rng.integers(0, 3))):
            length = int(rng.integers(1, 4))
            s = cur
            e = s + length - 1 if rng.integers(0, 5) else s - int(rng.integers(0, 2))
            rl.append((s, e))
            cur = s + length + int(rng.integers(1, 3))
        per_req.append(rl)
    ranges = pad_ranges(per_req) if rng.integers(0, 2) else None
    return Workload(f"tiny{seed}", seed, q_lens, k_lens, hq, hkv, d, causal, wl, wr, mode, ranges,
                    scale=float(rng.choice([0.5, 1.0 / math.sqrt(d)])))


def random_case(seed: int, max_q: int = 300, max_ctx: int = 600) -> Workload:
    """A random case of a shape the GPU kernels support (D 64..512, GQA
    groups 1..8), covering every mask / sink flag combination, q_len 0 and 1
    members, ragged lengths and ranges longer than the window."""
    rng = np.random.default_rng(10_000 + seed)
    d = int(rng.choice([64, 128, 256, 512]))
    hkv = int(rng.choice([1, 2]))
    group = int(rng.choice([1, 2, 3, 4, 8]))
    if d == 512:
        group = min(group, 4)
    b = int(rng.integers(1, 5))
    q_lens, k_lens = [], []
    for _ in range(b):
        kind = rng.integers(0, 6)
        ql = 0 if kind == 0 else (1 if kind == 1 else int(rng.integers(2, max_q + 1)))
        ctx = int(rng.integers(0, max_ctx + 1)) if rng.integers(0, 2) else 0
        q_lens.append(ql)
        k_lens.append(ql + ctx)
    if sum(q_lens) == 0:
        q_lens[0] = 5
        k_lens[0] += 5
    causal = bool(rng.integers(0, 3) > 0)
    wl = int(rng.choice([-1, 0, 7, 63, 130, 400]))
    wr = int(rng.choice([-1, 0, 5, 77])) if not causal else 0
    mode = int(rng.integers(0, 3))
    ranges = None
    if rng.integers(0, 2):
        per_req = []
        for ql, kl in zip(q_lens, k_lens):
            rl, cur = [], int(rng.integers(0, max(1, kl // 2 + 1)))
            for _ in range(int(rng.integers(0, 6))):
                length = int(rng.integers(1, 200))
                e = cur + length - 1
                if rng.integers(0, 8) == 0:
                    e = cur - int(rng.integers(0, 3))
                rl.append((cur, e))
                cur = cur + length + int(rng.integers(1, 40))
            per_req.append(rl)
        ranges = pad_ranges(per_req)
    return Workload(f"rand{seed}", 20_000 + seed, q_lens, k_lens, hkv * group, hkv, d, causal, wl, wr,
                    mode, ranges, scale=float(rng.choice([1.0 / math.sqrt(d), 0.05])))
