"""CPU oracle for masked varlen prefill attention -- TEST INFRASTRUCTURE ONLY.

This package is a plain, slow, deliberately unoptimised restatement of what the
GPU library computes.  It exists so that the CUDA path can be checked against
something written independently of it:

* ``range_table``  -- the per-query-row multimodal-prefix range table, built two
  ways: the span-and-clip fill described in the vLLM PR #50294 review ("FA4
  mm_prefix range scan -> O(1) table lookup"), and the O(max_ranges) per-row
  scan that the same page describes as the old in-kernel behaviour.
* ``attention``    -- the dense visibility mask built by broadcast comparison
  (step14_4 "Causal Mask optimisation" tutorial) OR-ed with the range part
  (PR #50294 mask_mod), and a dense float64 softmax attention with the two sink
  modes of vLLM PR #49815 (MiMo window attention sinks).
* ``accounting``   -- exact visible-score counts from the dense mask, and the
  per-request ``num_tokens * min(context_len, window)`` estimate of vLLM
  PR #55624 (SWA-aware MFU accounting).

Rules this package keeps:

* It imports nothing from the GPU package and the GPU package imports nothing
  from it.  Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
  CPU-baseline / reference arms may use it.
* Floating point is float64 (inputs are bf16 values widened exactly).
* No blocking, fusion or reordering beyond the definitions: the mask is
  materialised, the softmax is dense, the range table is filled by the printed
  algorithm's steps and by a brute-force scan.
"""

from . import accounting, attention, range_table  # noqa: F401
