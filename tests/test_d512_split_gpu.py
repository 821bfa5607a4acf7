"""The D = 512 head-dim split (the head-split variant of mvp_attn_fwd_varlen_ext) through the C-ABI (GPU).

Two CTAs of a cluster share an item's 128 rows: each multiplies its half of
the head dimension into partial scores, the halves are summed through
distributed shared memory every tile, and each CTA keeps its half of the 512
value columns of O in TMEM.  The sum of two partial products rounds
differently from one accumulation, so the check is the float64 oracle at the
packed tests' tolerances (and the default variant within the same bound),
with ranges, sinks and decode rows.  The variant is selected per call.
"""

import pytest
import torch

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads

from . import gpu_helpers as gh

pytestmark = pytest.mark.gpu

SPLIT = dict(variant=mvp.VARIANT_D512_HEAD_SPLIT)


def _parity(w, strict=True):
    q, k, v, sinks = gh.make_inputs(w)
    out, lse, table, _ = gh.run_gpu(w, q, k, v, sinks, **SPLIT)
    ref_table, _ = gh.oracle_table(w)
    ro, rl = gh.oracle_full(w, q, k, v, sinks, ref_table)
    gh.compare(out, lse, ro, rl, what=f"{w.name} head split", strict=strict)
    return q, k, v, sinks, out


def test_scaled_global_causal():
    _parity(workloads.scaled_workload("global_causal_d512"))


@pytest.mark.parametrize("sink_mode", [workloads.SINK_NONE, workloads.SINK_KEY0_BIAS, workloads.SINK_NULL_LOGIT])
def test_masks_ranges_sinks_decode(sink_mode):
    w = workloads.Workload(f"split_s{sink_mode}", 77 + sink_mode, [300, 1, 129, 1, 64], [700, 900, 129, 40, 500],
                           8, 2, 512, True, 200, 0, sink_mode,
                           workloads.pad_ranges([[(10, 90), (400, 650)], [(0, 5)], [(3, 60)], [], [(450, 499)]]))
    _parity(w, strict=False)


@pytest.mark.parametrize("seed", range(4))
def test_random_cases(seed):
    w = workloads.random_case(seed)
    w.head_dim = 512
    w.num_heads_q = w.num_heads_kv * min(w.num_heads_q // w.num_heads_kv, 4)
    w.scale = 512 ** -0.5
    _parity(w, strict=False)


def test_other_head_dims_refused():
    w = workloads.scaled_workload("mm_prefix_sliding")
    q, k, v, sinks = gh.make_inputs(w)
    with pytest.raises(mvp.MvpError) as e:
        gh.run_gpu(w, q, k, v, sinks, **SPLIT)
    assert e.value.status == mvp.MVP_ERR_UNSUPPORTED


def test_close_to_default_variant():
    w = workloads.scaled_workload("global_causal_d512")
    q, k, v, sinks = gh.make_inputs(w)
    out_d, _, _, _ = gh.run_gpu(w, q, k, v, sinks)
    out_s, _, _, _ = gh.run_gpu(w, q, k, v, sinks, **SPLIT)
    diff = (out_s.float() - out_d.float()).abs().max().item()
    assert diff <= 2 * gh.OUT_ATOL, diff
    assert mvp.get_last_device_error() == 0
    assert torch.isfinite(out_s.float()).all()
