"""Checks that pin the CPU oracle to facts fixed outside it.

Every ``check_*`` takes the oracle pieces it exercises as arguments, so the
same check runs against the real oracle (``test_oracle_pins.py``, must pass)
and against copies of the oracle with a planted mistake
(``test_oracle_mutations.py``, must fail).  Each raises ``AssertionError`` on
a mismatch.

What pins what:

* printed values -- the 4x4 causal picture (step14_4 tutorial), the range
  example with context offset (vLLM PR #50294 review), the exact-8x window
  clamp (vLLM PR #55624 report);
* library routines -- ``torch.tril``, ``torch.nn.functional.
  scaled_dot_product_attention`` and ``torch.logsumexp`` on CPU;
* closed forms -- rows sum to one, a single visible key against a null logit
  is a sigmoid;
* brute force -- element-by-element loops on tiny inputs.
"""

from __future__ import annotations

import json
import math
import os

import numpy as np
import torch

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden_json(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- causal mask
def check_causal_formula(visible_mask):
    # The printed 4x4 picture.
    blocks, cur = {}, None
    with open(os.path.join(GOLDEN, "causal_mask_4x4.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if line in ("allow", "causal_mask"):
                cur = line
                blocks[cur] = []
                continue
            blocks[cur].append([c == "T" for c in line.split()])
    allow = np.array(blocks["allow"])
    got = visible_mask(np.arange(4), 4, 0, True, -1, -1)
    assert np.array_equal(got, allow), "4x4 causal picture"
    assert np.array_equal(~got, np.array(blocks["causal_mask"])), "4x4 mask picture"

    # tril slice and the per-row loop construction, with a start_pos offset.
    for total, start_pos in [(4, 0), (7, 3), (9, 8), (12, 5)]:
        seq = total - start_pos
        tril = torch.tril(torch.ones(total, total, dtype=torch.bool))[start_pos:start_pos + seq]
        got = visible_mask(np.arange(seq), total, start_pos, True, -1, -1)
        assert np.array_equal(got, tril.numpy()), ("tril", total, start_pos)
        loop = np.zeros((seq, total), dtype=bool)
        for i in range(seq):
            loop[i, :start_pos + i + 1] = True
        assert np.array_equal(got, loop), ("loop", total, start_pos)


# ---------------------------------------------------------------- range table
def check_range_example(fill, scan_keep):
    g = _golden_json("range_table_example.json")
    mm = {int(k): [tuple(r) for r in v] for k, v in g["mm_ranges"].items()}
    qsl = np.array([0] + list(np.cumsum(g["query_lens"])), dtype=np.int32)
    out = np.full((64, 2), g["poison"], dtype=np.int32)
    n = fill(out, mm, qsl, np.array(g["seq_lens"], dtype=np.int32))
    assert n == g["expected_return"], n
    assert out[:n].tolist() == g["expected_table"], out[:n].tolist()
    assert (out[n:] == g["poison"]).all()
    # The O(1) lookup equals the old any()-scan for every (request, q, k).
    for b, ql in enumerate(g["query_lens"]):
        ctx = g["seq_lens"][b] - ql
        for i in range(ql):
            rs, re = out[qsl[b] + i]
            for kv in range(g["seq_lens"][b]):
                assert (rs <= kv <= re) == scan_keep(mm[b], ctx + i, kv), (b, i, kv)


def _random_nonoverlap(rng, span):
    """Non-overlapping closed ranges with gaps >= 1, some degenerate."""
    out, cur = [], int(rng.integers(0, 4))
    while cur < span and len(out) < 6:
        length = int(rng.integers(1, 6))
        s, e = cur, cur + length - 1
        r = rng.integers(0, 6)
        if r == 0:
            e = s
        elif r == 1:
            e = s - int(rng.integers(1, 3))
        out.append((s, e))
        cur = cur + length + int(rng.integers(1, 4))
    return out


def check_range_lookup_random(fill, scan_keep, cases=1500, seed=7):
    rng = np.random.default_rng(seed)
    for _ in range(cases):
        nb = int(rng.integers(1, 4))
        qlens = [int(rng.integers(0, 7)) for _ in range(nb)]
        seqs = [q + int(rng.integers(0, 6)) for q in qlens]
        mm = {b: _random_nonoverlap(rng, seqs[b] + 3) for b in range(nb)}
        qsl = np.array([0] + list(np.cumsum(qlens)), dtype=np.int32)
        out = np.full((max(1, int(qsl[-1])) + 2, 2), 12345, dtype=np.int32)
        n = fill(out, mm, qsl, np.array(seqs, dtype=np.int32))
        any_cover = False
        for b in range(nb):
            ctx = seqs[b] - qlens[b]
            for i in range(qlens[b]):
                if n:
                    rs, re = out[qsl[b] + i]
                else:
                    rs, re = -1, -1
                covered_row = any(s < e and s <= ctx + i <= e for s, e in mm[b])
                any_cover |= covered_row
                for kv in range(seqs[b]):
                    assert (rs <= kv <= re) == scan_keep(mm[b], ctx + i, kv), (mm, b, i, kv)
        assert n == (int(qsl[-1]) if any_cover else 0), (n, any_cover)


def check_scan_mask(visible_mask_scan, visible_mask, fill, cases=600, seed=13):
    """Scan mode against element-by-element loops of its definition (base
    rule OR some valid range holds query and key, past-side window clamp),
    with overlapping and degenerate ranges; and, for non-overlapping ranges,
    against the table mask of the same batch (the page's O(1) equivalence).
    Includes the page's printed example."""
    rng = np.random.default_rng(seed)
    g = _golden_json("range_table_example.json")
    printed = (g["query_lens"], g["seq_lens"], {int(k): [tuple(r) for r in v] for k, v in g["mm_ranges"].items()})
    for case in range(cases + 1):
        if case == 0:
            qlens, seqs, mm = printed
            causal, wl, wr = True, -1, -1
            overlap = False
        else:
            nb = int(rng.integers(1, 4))
            qlens = [int(rng.integers(1, 7)) for _ in range(nb)]
            seqs = [q + int(rng.integers(0, 6)) for q in qlens]
            overlap = bool(rng.integers(0, 2))
            if overlap:
                mm = {b: [(int(rng.integers(0, seqs[b] + 2)), int(rng.integers(-1, seqs[b] + 3)))
                          for _ in range(int(rng.integers(0, 5)))] for b in range(nb)}
            else:
                mm = {b: _random_nonoverlap(rng, seqs[b] + 3) for b in range(nb)}
            causal = bool(rng.integers(0, 2))
            wl = int(rng.choice([-1, 0, 1, 3]))
            wr = 0 if causal else int(rng.choice([-1, 0, 2]))
        qsl = np.array([0] + list(np.cumsum(qlens)), dtype=np.int32)
        table = np.full((max(1, int(qsl[-1])), 2), -1, dtype=np.int32)
        n = fill(table, mm, qsl, np.array(seqs, dtype=np.int32))
        for b in range(len(qlens)):
            ctx = seqs[b] - qlens[b]
            got = visible_mask_scan(np.arange(qlens[b]), seqs[b], ctx, causal, wl, wr, mm[b])
            for i in range(qlens[b]):
                p = ctx + i
                for j in range(seqs[b]):
                    base = (j <= p) if causal else (wr < 0 or j <= p + wr)
                    base = base and (wl < 0 or j >= p - wl)
                    rng_keep = any(s < e and s <= p <= e and s <= j <= e for s, e in mm[b])
                    rng_keep = rng_keep and (wl < 0 or j >= p - wl)
                    assert got[i, j] == (base or rng_keep), (case, b, i, j)
            if not overlap:
                rows = table[qsl[b]:qsl[b + 1]] if n else np.full((qlens[b], 2), -1, dtype=np.int32)
                ref = visible_mask(np.arange(qlens[b]), seqs[b], ctx, causal, wl, wr, rows)
                assert np.array_equal(got, ref), (case, b)


def check_fill_edge_cases(fill):
    P = 12345

    def run(mm, qlens, seqs, cap=32):
        qsl = np.array([0] + list(np.cumsum(qlens)), dtype=np.int32)
        out = np.full((cap, 2), P, dtype=np.int32)
        n = fill(out, mm, qsl, np.array(seqs, dtype=np.int32))
        return n, out

    # degenerate ranges are skipped (start == end and start > end)
    n, out = run({0: [(2, 2), (5, 3), (6, 7)]}, [8], [8])
    assert n == 8 and out[:8].tolist() == [[-1, -1]] * 6 + [[6, 7]] * 2
    # clipping at both ends of the scheduled chunk (ctx 4, rows are q_abs 4..7)
    n, out = run({0: [(2, 5), (7, 20)]}, [4], [8])
    assert n == 4 and out[:4].tolist() == [[2, 5], [2, 5], [-1, -1], [7, 20]]
    # a range wholly inside the context is dropped; nothing covered -> 0, untouched
    n, out = run({0: [(0, 3)]}, [4], [8])
    assert n == 0 and (out == P).all()
    # no ranges at all
    n, out = run(None, [4], [8])
    assert n == 0 and (out == P).all()
    n, out = run({}, [4], [8])
    assert n == 0 and (out == P).all()
    # zero scheduled tokens
    n, out = run({0: [(0, 3)]}, [0], [3])
    assert n == 0 and (out == P).all()
    # reuse: stale rows from a previous step are overwritten with -1
    qsl = np.array([0, 6], dtype=np.int32)
    out = np.full((8, 2), P, dtype=np.int32)
    assert fill(out, {0: [(0, 5)]}, qsl, np.array([6], dtype=np.int32)) == 6
    assert fill(out, {0: [(4, 5)]}, qsl, np.array([6], dtype=np.int32)) == 6
    assert out[:6].tolist() == [[-1, -1]] * 4 + [[4, 5]] * 2 and (out[6:] == P).all()
    # request with q_len 0 between others: produces no rows
    n, out = run({0: [(0, 1)], 1: [(0, 9)], 2: [(1, 2)]}, [2, 0, 3], [2, 4, 3])
    assert n == 5 and out[:5].tolist() == [[0, 1], [0, 1], [-1, -1], [1, 2], [1, 2]]
    # capacity overflow is an error
    try:
        run({0: [(0, 1)]}, [40], [40], cap=32)
    except ValueError:
        pass
    else:
        raise AssertionError("capacity overflow not reported")


def check_fills_agree(fill_a, fill_b, cases=800, seed=11):
    rng = np.random.default_rng(seed)
    for _ in range(cases):
        nb = int(rng.integers(1, 5))
        qlens = [int(rng.integers(0, 9)) for _ in range(nb)]
        seqs = [q + int(rng.integers(0, 9)) for q in qlens]
        mm = {b: _random_nonoverlap(rng, seqs[b] + 4) for b in range(nb)}
        # also overlapping lists: the last listed covering range must win
        if rng.integers(0, 3) == 0:
            mm[0] = mm[0] + [(0, seqs[0] + 2)] + [(1, 2)]
        qsl = np.array([0] + list(np.cumsum(qlens)), dtype=np.int32)
        a = np.full((int(qsl[-1]) + 1, 2), 777, dtype=np.int32)
        c = a.copy()
        na = fill_a(a, mm, qsl, np.array(seqs, dtype=np.int32))
        nb_ = fill_b(c, mm, qsl, np.array(seqs, dtype=np.int32))
        assert na == nb_ and np.array_equal(a, c), (mm, qlens, seqs)


# ---------------------------------------------------------------- accounting
def check_window_count(visible_entries, token_context_product):
    g = _golden_json("swa_window_clamp.json")
    w = g["window"]
    for case in g["cases"]:
        n, ctx = case["num_tokens"], case["context_len"]
        # a decode token at the end of ctx keys: q_len 1, k_len ctx
        cu_q = np.array([0, n]); cu_k = np.array([0, ctx])
        dense = visible_entries(cu_q, cu_k, True, -1, -1)
        windowed = visible_entries(cu_q, cu_k, True, w - 1, 0)
        assert dense == case["ratio_dense_over_window"] * windowed, (dense, windowed)
        assert windowed == token_context_product([(n, ctx)], w)
        assert dense == token_context_product([(n, ctx)])
    # a prefill chunk: exact count = triangle, page's estimate is an upper bound
    cu_q = np.array([0, 100]); cu_k = np.array([0, 100])
    assert visible_entries(cu_q, cu_k, True, -1, -1) == 100 * 101 // 2
    assert visible_entries(cu_q, cu_k, True, 9, 0) == sum(min(i + 1, 10) for i in range(100))


# ---------------------------------------------------------------- attention
def _t(x):
    return torch.as_tensor(np.asarray(x))


def check_rows_sum_to_one(attention_forward, seed=3):
    rng = np.random.default_rng(seed)
    cu = np.array([0, 9, 20]); hq, hkv, d = 4, 2, 8
    q = rng.standard_normal((20, hq, d)); k = rng.standard_normal((20, hkv, d))
    v = np.ones((20, hkv, d))
    sinks = rng.standard_normal(hq)
    for mode in (0, 1, 2):
        out, lse = attention_forward(q, k, v, cu, cu, True, 3, 0, 0.4, sinks=sinks, sink_mode=mode)
        if mode == 2:
            expect = 1.0 - np.exp(sinks[None, :] - lse.T)  # [rows, heads]
            assert np.allclose(out, expect[:, :, None], atol=1e-12), mode
        else:
            assert np.allclose(out, 1.0, atol=1e-12), mode


def check_sink_modes(attention_forward, seed=5):
    rng = np.random.default_rng(seed)
    n, hq, d = 6, 2, 4
    cu = np.array([0, n])
    q = rng.standard_normal((n, hq, d)); k = rng.standard_normal((n, hq, d))
    v = rng.standard_normal((n, hq, d)); sinks = np.array([0.7, -1.3])
    # one visible key per row (causal, window_left 0): row i sees key i
    o1, _ = attention_forward(q, k, v, cu, cu, True, 0, 0, 0.5, sinks=sinks, sink_mode=1)
    assert np.allclose(o1, v, atol=1e-12)  # key-0 bias cannot change a lone key
    o2, _ = attention_forward(q, k, v, cu, cu, True, 0, 0, 0.5, sinks=sinks, sink_mode=2)
    for h in range(hq):
        s = 0.5 * np.einsum("nd,nd->n", q[:, h], k[:, h])
        sig = 1.0 / (1.0 + np.exp(-(s - sinks[h])))
        assert np.allclose(o2[:, h], v[:, h] * sig[:, None], atol=1e-12), h
    # the neutral sink of each mode gives plain attention: a zero bias on key
    # 0, a null logit at -inf (exp -> 0 in the denominator)
    o0, l0 = attention_forward(q, k, v, cu, cu, True, 2, 0, 0.5)
    for mode, neutral in ((1, 0.0), (2, -1e30)):
        om, lm = attention_forward(q, k, v, cu, cu, True, 2, 0, 0.5,
                                   sinks=np.array([neutral, neutral]), sink_mode=mode)
        assert np.allclose(om, o0, atol=1e-12) and np.allclose(lm, l0, atol=1e-12), mode
    # a key-0 bias of -inf removes key 0 instead: rows 1, 2 then equal plain
    # attention with window_left 2 over keys >= 1 only
    om, _ = attention_forward(q, k, v, cu, cu, True, 2, 0, 0.5,
                              sinks=np.array([-1e30, -1e30]), sink_mode=1)
    o_nokey0, _ = attention_forward(q[1:], k[1:], v[1:], np.array([0, n - 1]),
                                    np.array([0, n - 1]), True, 2, 0, 0.5)
    assert np.allclose(om[1:3], o_nokey0[0:2], atol=1e-12)
    # key-0 bias only touches rows whose window still holds key 0 (rows 0..2)
    ob, _ = attention_forward(q, k, v, cu, cu, True, 2, 0, 0.5, sinks=sinks, sink_mode=1)
    assert np.allclose(ob[3:], o0[3:], atol=1e-12)
    assert not np.allclose(ob[1:3], o0[1:3], atol=1e-6)
    # and it raises key 0's weight: with a large positive sink rows 0..2 -> v_0
    ob, _ = attention_forward(q, k, v, cu, cu, True, 2, 0, 0.5, sinks=np.array([60.0, 60.0]),
                              sink_mode=1)
    assert np.allclose(ob[:3], np.broadcast_to(v[0], (3, hq, d)), atol=1e-9)


def check_sdpa(attention_forward, seed=9):
    """No ranges, no window, no sink, ctx 0: equals CPU SDPA (float64)."""
    g = torch.Generator().manual_seed(seed)
    for hq, hkv, causal in [(2, 2, True), (4, 2, True), (6, 3, False), (4, 1, True)]:
        lens = [13, 1, 7]
        cu = np.array([0] + list(np.cumsum(lens)))
        d = 8
        q = torch.randn(cu[-1], hq, d, generator=g, dtype=torch.float64)
        k = torch.randn(cu[-1], hkv, d, generator=g, dtype=torch.float64)
        v = torch.randn(cu[-1], hkv, d, generator=g, dtype=torch.float64)
        out, lse = attention_forward(q, k, v, cu, cu, causal, -1, -1, 0.3)
        for b in range(len(lens)):
            s0, s1 = cu[b], cu[b + 1]
            qb = q[s0:s1].transpose(0, 1)
            kb = k[s0:s1].transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
            vb = v[s0:s1].transpose(0, 1).repeat_interleave(hq // hkv, dim=0)
            ref = torch.nn.functional.scaled_dot_product_attention(qb, kb, vb, is_causal=causal,
                                                                   scale=0.3)
            assert np.allclose(out[s0:s1], ref.transpose(0, 1).numpy(), atol=1e-10), (hq, hkv, b)
            sc = 0.3 * qb @ kb.transpose(1, 2)
            if causal:
                sc = sc.masked_fill(~torch.tril(torch.ones(s1 - s0, s1 - s0, dtype=torch.bool)),
                                    float("-inf"))
            assert np.allclose(lse[:, s0:s1], torch.logsumexp(sc, dim=-1).numpy(), atol=1e-10)


def brute_force(q, k, v, cu_q, cu_k, causal, wl, wr, scale, ctxs, table, sinks, mode):
    """Element-by-element definition with Python loops only (tiny inputs)."""
    total_q, hq, d = q.shape
    hkv = k.shape[1]
    out = [[[0.0] * d for _ in range(hq)] for _ in range(total_q)]
    lse = [[float("-inf")] * total_q for _ in range(hq)]
    for b in range(len(cu_q) - 1):
        for i in range(cu_q[b + 1] - cu_q[b]):
            t = cu_q[b] + i
            p = ctxs[b] + i
            k_len = cu_k[b + 1] - cu_k[b]
            vis = []
            for j in range(k_len):
                if causal:
                    ok = j <= p
                else:
                    ok = wr < 0 or j <= p + wr
                if wl >= 0 and j < p - wl:
                    ok = False
                mm = False
                if table is not None:
                    rs, re = int(table[t][0]), int(table[t][1])
                    mm = rs <= j <= re and (wl < 0 or j >= p - wl)
                vis.append(ok or mm)
            for h in range(hq):
                kh = h // (hq // hkv)
                logits = {}
                for j in range(k_len):
                    if not vis[j]:
                        continue
                    s = 0.0
                    for x in range(d):
                        s += float(q[t][h][x]) * float(k[cu_k[b] + j][kh][x])
                    s *= scale
                    if mode == 1 and j == 0:
                        s += float(sinks[h])
                    logits[j] = s
                terms = list(logits.values()) + ([float(sinks[h])] if mode == 2 else [])
                if not terms:
                    continue
                m = max(terms)
                z = sum(math.exp(x - m) for x in terms)
                lse[h][t] = m + math.log(z)
                for x in range(d):
                    acc = 0.0
                    for j, s in logits.items():
                        acc += math.exp(s - m) * float(v[cu_k[b] + j][kh][x])
                    out[t][h][x] = acc / z
    return np.array(out).reshape(total_q, hq, d), np.array(lse).reshape(hq, total_q)


def check_brute_force(attention_forward, fill, make_case, cases=120):
    for seed in range(cases):
        w, q, k, v, sinks, table, cu_q, cu_k = make_case(seed, fill)
        ctxs = [kl - ql for ql, kl in zip(w.q_lens, w.k_lens)]
        out, lse = attention_forward(q, k, v, cu_q, cu_k, w.causal, w.window_left,
                                     w.window_right, w.scale, range_table=table,
                                     sinks=sinks, sink_mode=w.sink_mode)
        ref_o, ref_l = brute_force(q, k, v, list(cu_q), list(cu_k), w.causal, w.window_left,
                                   w.window_right, w.scale, ctxs, table, sinks, w.sink_mode)
        assert np.allclose(out, ref_o, atol=1e-10), seed
        both_inf = np.isneginf(lse) & np.isneginf(ref_l)
        assert np.allclose(np.where(both_inf, 0, lse), np.where(both_inf, 0, ref_l), atol=1e-10), seed


def check_context_lens(attention_forward, fill, make_case, cases=40, seed=17):
    """An explicit context length defines the query positions (step14_4
    tutorial, *Solution*: key j is masked iff j > start_pos + i).

    * Passing ctx = k_len - q_len explicitly changes nothing.
    * Any other ctx matches the element-by-element definition with p = ctx + i.
    * Truncation: a causal row at position p never sees a key past p, so with
      ctx' < k_len - q_len the result equals the same call on the request's
      first ctx' + q_len keys with the context derived from them.
    """
    rng = np.random.default_rng(seed)
    for c in range(cases):
        w, q, k, v, sinks, table, cu_q, cu_k = make_case(c, fill)
        derived = np.asarray(w.k_lens) - np.asarray(w.q_lens)
        kw = dict(range_table=table, sinks=sinks, sink_mode=w.sink_mode)
        o_none, l_none = attention_forward(q, k, v, cu_q, cu_k, w.causal, w.window_left, w.window_right, w.scale,
                                           **kw)
        o_exp, l_exp = attention_forward(q, k, v, cu_q, cu_k, w.causal, w.window_left, w.window_right, w.scale,
                                         context_lens=derived, **kw)
        assert np.array_equal(o_none, o_exp) and np.array_equal(l_none, l_exp, equal_nan=True), c
        # shifted positions against the definition (table rows are taken as given)
        ctx = np.array([int(rng.integers(0, d + 1)) for d in derived])
        out, lse = attention_forward(q, k, v, cu_q, cu_k, w.causal, w.window_left, w.window_right, w.scale,
                                     context_lens=ctx, **kw)
        ref_o, ref_l = brute_force(q, k, v, list(cu_q), list(cu_k), w.causal, w.window_left, w.window_right,
                                   w.scale, list(ctx), table, sinks, w.sink_mode)
        assert np.allclose(out, ref_o, atol=1e-10), c
        both_inf = np.isneginf(lse) & np.isneginf(ref_l)
        assert np.allclose(np.where(both_inf, 0, lse), np.where(both_inf, 0, ref_l), atol=1e-10), c
        # truncation invariant (causal, no range part)
        keep = [np.arange(cu_k[b], cu_k[b] + ctx[b] + w.q_lens[b]) for b in range(w.num_reqs)]
        idx = np.concatenate(keep) if keep else np.zeros(0, dtype=np.int64)
        cu_t = np.zeros(w.num_reqs + 1, dtype=np.int64)
        cu_t[1:] = np.cumsum(ctx + np.asarray(w.q_lens))
        o_c, l_c = attention_forward(q, k, v, cu_q, cu_k, True, w.window_left, 0, w.scale, context_lens=ctx,
                                     sinks=sinks, sink_mode=w.sink_mode)
        o_t, l_t = attention_forward(q, k[idx], v[idx], cu_q, cu_t, True, w.window_left, 0, w.scale,
                                     sinks=sinks, sink_mode=w.sink_mode)
        assert np.allclose(o_c, o_t, atol=1e-12), c
        both_inf = np.isneginf(l_c) & np.isneginf(l_t)
        assert np.allclose(np.where(both_inf, 0, l_c), np.where(both_inf, 0, l_t), atol=1e-12, equal_nan=True), c
