"""Shared plumbing for the GPU parity tests: run a workload through the C-ABI
library and through the CPU oracle, and compare.

Tolerances (float64 oracle vs the GPU's bf16 output): out max-abs <= 1e-2;
lse |diff| / max(|lse|, 1) <= 1e-3; range table bit-exact.
"""

from __future__ import annotations

import numpy as np
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import attention as oatt
from oracle import range_table as ort

OUT_ATOL = 1e-2
LSE_RTOL = 1e-3
# bf16 keeps 8 significant bits (unit roundoff u = 2^-8): a correctly
# rounded bf16 output can differ from the exact value by half an ulp, up to
# u |x| (just above a power of two), and rounding the probabilities to bf16
# for the P.V product perturbs each weight by up to u as well, which can move
# the output by about as much again (a row with a few visible keys and a
# null-logit sink has no cancellation).  Together 2u |x| = 2^-7 |x|: for
# |out| above 1.28 that exceeds 1e-2 however the kernel computes, so shapes
# that produce such outputs (a few visible keys per row) use
# max(1e-2, 2^-7 |ref|).
BF16_REL = 2.0 ** -7


def device_meta(w, dev):
    cu_q, cu_k = w.cu_seqlens()
    return (torch.from_numpy(cu_q).to(dev), torch.from_numpy(cu_k).to(dev))


def oracle_table(w):
    """Oracle range table [total_q, 2] (rows with no range: -1) and its
    return value, or (None, 0) when the workload has no ranges."""
    if w.ranges is None:
        return None, 0
    cu_q, _ = w.cu_seqlens()
    out = np.full((max(1, w.total_q), 2), 12345, dtype=np.int32)
    n = ort.fill_by_spans(out, ort.ranges_from_padded(w.ranges), cu_q, np.asarray(w.k_lens))
    table = out[:w.total_q].copy()
    if n == 0:
        table[:] = -1
    return table, n


def run_gpu(w, q, k, v, sinks, use_workspace=True, with_lse=True, dev="cuda", num_decode_reqs=-1, **ext):
    """Fill the range table (if any) and run attention on the GPU.  ``ext``:
    further keywords of ``attn_fwd_varlen`` (variant, wait_limit_us)."""
    cu_q, cu_k = device_meta(w, dev)
    table = covered = None
    if w.ranges is not None:
        ranges = torch.from_numpy(w.ranges).to(dev)
        table = torch.full((max(1, w.total_q), 2), 777, dtype=torch.int32, device=dev)
        covered = torch.full((1,), -5, dtype=torch.int32, device=dev)
        mvp.fill_query_ranges(ranges, cu_q, cu_k.diff().to(torch.int32).contiguous(), table,
                              num_tokens=w.total_q, rows_written=covered)
    out = torch.full_like(q, float("nan"))
    lse = torch.full((w.num_heads_q, w.total_q), float("nan"), device=dev) if with_lse else None
    ws = None
    if use_workspace:
        n_dec = w.num_reqs if num_decode_reqs < 0 else num_decode_reqs
        nbytes = mvp.attn_workspace_size(n_dec, w.num_heads_q, w.head_dim, max(w.k_lens))
        if nbytes:
            ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    mvp.attn_fwd_varlen(q, k, v, out, cu_q, cu_k, max(max(w.q_lens), 1), max(max(w.k_lens), 1), lse=lse,
                        range_table=table, range_covered=covered, causal=w.causal,
                        window_left=w.window_left, window_right=w.window_right, sinks=sinks,
                        sink_mode=w.sink_mode, scale=w.scale, workspace=ws, num_decode_reqs=num_decode_reqs, **ext)
    torch.cuda.synchronize()
    assert mvp.get_last_device_error() == 0
    return out, lse, table, covered


def oracle_full(w, q, k, v, sinks, table):
    cu_q, cu_k = w.cu_seqlens()
    return oatt.attention_forward(q.cpu(), k.cpu(), v.cpu(), cu_q, cu_k, w.causal, w.window_left,
                                  w.window_right, w.scale, range_table=table,
                                  sinks=None if sinks is None else sinks.cpu(), sink_mode=w.sink_mode)


def oracle_rows(w, q, k, v, sinks, table, rows):
    """Oracle for selected packed rows, one request slice at a time (keeps
    float64 copies small at full workload sizes)."""
    cu_q, cu_k = w.cu_seqlens()
    rows = np.asarray(sorted(set(int(r) for r in rows)))
    out = {}
    lse = {}
    sk = None if sinks is None else sinks.detach().cpu().double().numpy()
    for b in range(w.num_reqs):
        sel = rows[(rows >= cu_q[b]) & (rows < cu_q[b + 1])]
        if sel.size == 0:
            continue
        q0, k0, k1 = cu_q[b], cu_k[b], cu_k[b + 1]
        local = sel - q0
        qb = q[q0 + local].detach().cpu().double().numpy()
        kb = k[k0:k1].detach().cpu().double().numpy()
        vb = v[k0:k1].detach().cpu().double().numpy()
        ctx = (k1 - k0) - (cu_q[b + 1] - q0)
        rr = None if table is None else table[sel]
        o, l = _attend_selected(local, qb, kb, vb, ctx, w, rr, sk)
        for i, r in enumerate(sel):
            out[int(r)] = o[i]
            lse[int(r)] = l[:, i]
    return out, lse


def _attend_selected(local, qb, kb, vb, ctx, w, rr, sk):
    """attend_rows with q rows given as a compact array but positions taken
    from their true local indices."""
    q_full = np.zeros((int(local.max()) + 1, qb.shape[1], qb.shape[2]))
    q_full[local] = qb
    return oatt.attend_rows(local, q_full, kb, vb, ctx, w.causal, w.window_left, w.window_right, rr, sk,
                            w.sink_mode, w.scale)


def compare(out_gpu, lse_gpu, out_ref, lse_ref, rows=None, what="", strict=True):
    """Assert the tolerances; returns (max_abs_out, max_rel_lse).

    strict: out max-abs <= 1e-2 everywhere (the workload shapes).  Otherwise
    each element may also use the bf16 bound 2^-7 |ref| when that is larger."""
    og = out_gpu.float().cpu().numpy()
    lg = None if lse_gpu is None else lse_gpu.cpu().numpy()
    where = ""

    def excess(got, ref):
        tol = OUT_ATOL if strict else np.maximum(OUT_ATOL, BF16_REL * np.abs(ref))
        return np.abs(got - ref) / tol * OUT_ATOL  # error rescaled to the 1e-2 scale

    if rows is None:
        err_o = excess(og, out_ref).max() if og.size else 0.0
        if og.size:
            idx = np.unravel_index(int(np.argmax(excess(og, out_ref))), og.shape)
            where = f" at (row, head, dim)={tuple(int(i) for i in idx)} gpu={og[idx]:.5f} ref={out_ref[idx]:.5f}"
        assert np.isfinite(og).all(), f"{what}: non-finite output"
        if lg is not None:
            finite = np.isfinite(lse_ref)
            assert (np.isneginf(lg) == np.isneginf(lse_ref)).all(), f"{what}: -inf lse mismatch"
            rel = np.abs(lg[finite] - lse_ref[finite]) / np.maximum(np.abs(lse_ref[finite]), 1.0)
            err_l = rel.max() if rel.size else 0.0
        else:
            err_l = 0.0
    else:
        err_o, err_l = 0.0, 0.0
        for r in out_ref:
            assert np.isfinite(og[r]).all(), f"{what}: non-finite output row {r}"
            e = float(excess(og[r], out_ref[r]).max())
            if e > err_o:
                idx = np.unravel_index(int(np.argmax(excess(og[r], out_ref[r]))), og[r].shape)
                where = f" at row {r} (head, dim)={tuple(int(i) for i in idx)} gpu={og[r][idx]:.5f} ref={out_ref[r][idx]:.5f}"
            err_o = max(err_o, e)
            if lg is not None:
                ref = lse_ref[r]
                got = lg[:, r]
                assert (np.isneginf(got) == np.isneginf(ref)).all(), f"{what}: -inf lse mismatch row {r}"
                f = np.isfinite(ref)
                if f.any():
                    err_l = max(err_l, float((np.abs(got[f] - ref[f]) / np.maximum(np.abs(ref[f]), 1.0)).max()))
    kind = "max-abs" if strict else "scaled error (1e-2 or 2^-7|ref|)"
    assert err_o <= OUT_ATOL, f"{what}: out {kind} {err_o:.3e} > {OUT_ATOL}{where}"
    assert err_l <= LSE_RTOL, f"{what}: lse rel {err_l:.3e} > {LSE_RTOL}"
    return err_o, err_l


def make_inputs(w, dev="cuda"):
    return workloads.make_tensors(w, device=dev)
