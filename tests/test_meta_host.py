"""Host logic of the step-metadata block (``mvp_meta_pack``; no GPU needed).

The block packs one batch padded to a capacity.  Checked here: the layout,
a hand-worked block, the padding (requests with no rows, keys or ranges),
that the padded arrays make the oracle fill the same table as the batch
itself, and that every argument error leaves the block untouched.
"""

import ctypes

import numpy as np
import pytest

import masked_varlen_prefill_gb300 as mvp
from masked_varlen_prefill_gb300 import workloads
from oracle import range_table as ort


def test_layout():
    nbytes, offs = mvp.meta_block_layout(4, 3)
    assert offs == (0, 5, 9, 14, 18)  # qsl[5], seq_k[4], cu_k[5], bound[4], ranges (8-byte aligned)
    assert nbytes == 4 * (18 + 4 * 3 * 2)
    for r, m in [(1, 0), (7, 5), (255, 64), (65535, 1)]:
        nbytes, offs = mvp.meta_block_layout(r, m)
        assert offs[4] % 2 == 0 and nbytes % 8 == 0
        assert offs[1] - offs[0] == r + 1 and offs[2] - offs[1] == r and offs[3] - offs[2] == r + 1
        assert nbytes // 4 >= offs[4] + r * m * 2
    lib = mvp.load_library()
    assert lib.mvp_meta_block_bytes(0, 1) == 0 and lib.mvp_meta_block_bytes(1, -1) == 0
    assert lib.mvp_meta_block_bytes(65536, 1) == 0 and lib.mvp_meta_block_bytes(1, 4097) == 0


def test_hand_worked_block():
    ranges = np.array([[[0, 2], [5, 8]], [[1, 1], [0, 0]]], np.int32)
    blk = mvp.meta_pack([0, 3, 4], [10, 5], [10, 9], ranges, max_reqs=4, max_tokens=16, max_ranges=3)
    want = [0, 3, 4, 4, 4,            # query_start_loc, padded with the batch's row count
            10, 5, 0, 0,              # seq_lens_k, padding requests have no keys
            0, 10, 15, 15, 15,        # cu_seqlens_k
            10, 9, 0, 0,              # seq_lens_bound
            0, 2, 5, 8, 0, 0,         # ranges of request 0 (third slot empty)
            1, 1, 0, 0, 0, 0,         # request 1
            0, 0, 0, 0, 0, 0,
            0, 0, 0, 0, 0, 0]
    assert blk.tolist() == want


def _random_batch(rng, max_reqs, max_tokens, max_ranges):
    n = int(rng.integers(0, max_reqs + 1))
    q = rng.integers(0, max(1, max_tokens // max(n, 1)) + 1, size=n)
    while q.sum() > max_tokens:
        q[np.argmax(q)] -= 1
    qsl = np.zeros(n + 1, np.int32)
    qsl[1:] = np.cumsum(q)
    k = (q + rng.integers(0, 50, size=n)).astype(np.int32)
    bound = (k + (q == 1) * rng.integers(0, 5, size=n)).astype(np.int32)
    nr = int(rng.integers(0, max_ranges + 1))
    per_req = []
    for b in range(n):
        rl, cur = [], int(rng.integers(0, 10))
        for _ in range(nr):
            ln = int(rng.integers(1, 12))
            e = cur + ln - 1 if rng.integers(0, 6) else cur - 1  # some degenerate
            rl.append((cur, e))
            cur += ln + int(rng.integers(1, 4))
        per_req.append(rl)
    ranges = workloads.pad_ranges(per_req, min_width=nr)[:, :nr] if n and nr else None
    return qsl, k, bound, ranges


@pytest.mark.parametrize("seed", range(20))
def test_random_blocks_and_padding(seed):
    rng = np.random.default_rng(seed)
    max_reqs, max_tokens, max_ranges = int(rng.integers(1, 9)), int(rng.integers(1, 200)), int(rng.integers(0, 5))
    qsl, k, bound, ranges = _random_batch(rng, max_reqs, max_tokens, max_ranges)
    n = len(qsl) - 1
    blk = mvp.meta_pack(qsl, k, bound, ranges, max_reqs, max_tokens, max_ranges)
    _, o = mvp.meta_block_layout(max_reqs, max_ranges)
    b_qsl = blk[o[0]:o[0] + max_reqs + 1]
    b_k = blk[o[1]:o[1] + max_reqs]
    b_cuk = blk[o[2]:o[2] + max_reqs + 1]
    b_bd = blk[o[3]:o[3] + max_reqs]
    b_rg = blk[o[4]:o[4] + max_reqs * max_ranges * 2].reshape(max_reqs, max_ranges, 2)
    assert np.array_equal(b_qsl[:n + 1], qsl) and (b_qsl[n + 1:] == qsl[-1]).all()
    assert np.array_equal(b_k[:n], k) and (b_k[n:] == 0).all()
    assert b_cuk[0] == 0 and np.array_equal(np.diff(b_cuk), b_k)
    assert np.array_equal(b_bd[:n], bound) and (b_bd[n:] == 0).all()
    nr = 0 if ranges is None else ranges.shape[1]
    if nr:
        assert np.array_equal(b_rg[:n, :nr], ranges)
    assert (b_rg[n:] == 0).all() and (b_rg[:, nr:] == 0).all()
    # The padded arrays describe the same batch: the oracle fills the same
    # table from them as from the batch itself.
    if ranges is not None and qsl[-1] > 0:
        t1 = np.full((qsl[-1], 2), 99, np.int32)
        t2 = np.full((qsl[-1], 2), 99, np.int32)
        w1 = ort.fill_by_scan(t1, ort.ranges_from_padded(ranges), qsl, bound)
        w2 = ort.fill_by_scan(t2, ort.ranges_from_padded(b_rg), b_qsl, b_bd)
        assert w1 == w2 and np.array_equal(t1, t2)


def test_bound_defaults_to_seq_lens_k_and_keys_may_be_omitted():
    a = mvp.meta_pack([0, 2, 3], [5, 4], None, None, 3, 8, 0)
    b = mvp.meta_pack([0, 2, 3], [5, 4], [5, 4], None, 3, 8, 0)
    assert np.array_equal(a, b)
    c = mvp.meta_pack([0, 2, 3], None, [5, 4], None, 3, 8, 0)
    _, o = mvp.meta_block_layout(3, 0)
    assert (c[o[1]:o[3]] == 0).all() and c[o[3]:o[3] + 2].tolist() == [5, 4]


def _raw_pack(qsl, k, bound, ranges, n, nr, max_reqs, max_tokens, max_ranges):
    lib = mvp.load_library()
    nbytes = lib.mvp_meta_block_bytes(max_reqs, max_ranges)
    blk = np.full(nbytes // 4, 0x5A5A, np.int32)
    arrs = [None if a is None else np.ascontiguousarray(a, dtype=np.int32) for a in (qsl, k, bound, ranges)]
    ptrs = [None if a is None else ctypes.c_void_p(a.ctypes.data) for a in arrs]
    st = lib.mvp_meta_pack(*ptrs, n, nr, max_reqs, max_tokens, max_ranges, ctypes.c_void_p(blk.ctypes.data))
    return st, blk


@pytest.mark.parametrize("case,status", [
    (dict(qsl=[1, 3], k=[5], n=1), mvp.MVP_ERR_ARG),                 # does not start at 0
    (dict(qsl=[0, 3, 2], k=[5, 5], n=2), mvp.MVP_ERR_ARG),           # decreasing
    (dict(qsl=[0, 3], k=[2], n=1), mvp.MVP_ERR_ARG),                 # fewer keys than queries
    (dict(qsl=[0, 3], k=[5], bound=[2], n=1), mvp.MVP_ERR_ARG),      # bound below the query count
    (dict(qsl=None, k=[5], n=1), mvp.MVP_ERR_ARG),
    (dict(qsl=[0, 3], k=None, n=1), mvp.MVP_ERR_ARG),                # neither lengths nor bound
    (dict(qsl=[0, 1, 2, 3, 4, 5], k=[1] * 5, n=5), mvp.MVP_ERR_CAPACITY),   # more requests than max_reqs
    (dict(qsl=[0, 40], k=[40], n=1), mvp.MVP_ERR_CAPACITY),          # more rows than max_tokens
    (dict(qsl=[0, 3], k=[5], ranges=np.zeros((1, 3, 2)), nr=3, n=1), mvp.MVP_ERR_CAPACITY),  # ranges > max
])
def test_pack_errors_leave_block_untouched(case, status):
    st, blk = _raw_pack(case.get("qsl"), case.get("k"), case.get("bound"), case.get("ranges"), case["n"],
                        case.get("nr", 0), 4, 32, 2)
    assert st == status
    assert (blk == 0x5A5A).all()


def test_pack_rejects_key_total_past_int_max():
    st, blk = _raw_pack([0, 1, 2], [2**31 - 100, 200], None, None, 2, 0, 4, 32, 0)
    assert st == mvp.MVP_ERR_ARG and (blk == 0x5A5A).all()


def test_bad_capacity():
    lib = mvp.load_library()
    blk = np.zeros(64, np.int32)
    assert lib.mvp_meta_pack(None, None, None, None, 0, 0, 0, 8, 0, ctypes.c_void_p(blk.ctypes.data)) == mvp.MVP_ERR_ARG
    assert lib.mvp_meta_pack(None, None, None, None, 0, 0, 2, 0, 0, ctypes.c_void_p(blk.ctypes.data)) == mvp.MVP_ERR_ARG
    assert lib.mvp_meta_pack(None, None, None, None, 0, 0, 2, 8, 0, None) == mvp.MVP_ERR_ARG
    handle = ctypes.c_void_p()
    assert lib.mvp_meta_create(0, 8, 0, None, None, None, ctypes.byref(handle)) == mvp.MVP_ERR_ARG
    assert lib.mvp_meta_create(2, 8, 0, None, None, None, ctypes.byref(handle)) == mvp.MVP_ERR_ARG
    assert lib.mvp_meta_destroy(None) == mvp.MVP_OK
