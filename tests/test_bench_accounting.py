"""bench.py's algorithmic bytes and FLOPs, checked by counting on tiny batches."""
from __future__ import annotations

import numpy as np

import bench
import workloads


def _count(b):
    """Visible (query row, key) pairs per query head, by enumeration."""
    pairs = 0
    for lq, lkv in zip(b.qo_lens(), b.kv_lens()):
        for t in range(int(lq)):
            last = lkv - lq + t if b.causal else lkv - 1
            pairs += max(0, min(int(lkv), int(last) + 1))
    return pairs


def test_decode_bytes_and_flops():
    b = workloads.make_batch("acct", "bf16", [1, 1, 1], [5, 17, 40], 8, 2, 4, 0, 1)
    nbytes, formula, exact = bench.algorithmic(b)
    kv_tokens = 5 + 17 + 40
    assert nbytes == kv_tokens * 2 * 128 * 2 * 2 + 3 * 8 * (128 * 2 * 2 + 4)
    assert exact == formula == 4 * 128 * 8 * _count(b)


def test_causal_prefill_flops():
    b = workloads.make_batch("acct", "bf16", [3, 5, 2], [7, 5, 9], 4, 2, 4, 1, 2)
    _, formula, exact = bench.algorithmic(b)
    assert exact == 4 * 128 * 4 * _count(b)
    assert formula == 4 * 128 * 4 * float((np.array([3, 5, 2]) * np.array([7, 5, 9])).sum()) / 2


def test_mla_bytes_and_flops():
    b = workloads.make_mla_batch("acct", [5, 0, 70], 16, 8, 3, pool_pages=12)
    nbytes, flops = bench.mla_algorithmic(b)
    pages = 1 + 0 + 9
    assert nbytes == 75 * (512 + 64) * 2 + pages * 4 + 3 * 16 * (576 * 2 + 512 * 2 + 4)
    assert flops == 75 * 16 * (2 * 576 + 2 * 512)


def test_mix_decode_part_is_the_decode_requests():
    """The mix's decode part: requests 8.. re-based as a batch of their own
    hold exactly the decode requests' pages, lengths and query rows, and
    their bytes are the mix's bytes minus the prefill requests'."""
    b = workloads.continuous_batch(n_prefill=3, n_decode=7, chunk=16, prefix_max=40, kv_max=300)
    qo, kvp, kvi, lpl, start = bench.tail_requests(b, 3)
    assert start == 3 * 16 and qo[0] == 0 and np.array_equal(np.diff(qo), np.ones(7))
    assert kvp[0] == 0 and kvp[-1] == kvi.size
    for r in range(7):
        orig = b.kv_indices[b.kv_indptr[3 + r]:b.kv_indptr[4 + r]]
        assert np.array_equal(kvi[kvp[r]:kvp[r + 1]], orig)
    assert np.array_equal(lpl, b.last_page_len[3:])
    d = workloads.PagedBatch("d", b.dtype, qo, kvp, kvi, lpl, 32, 8, 16, 1, b.sm_scale, b.q[start:], b.k, b.v)
    assert np.array_equal(d.kv_lens(), b.kv_lens()[3:])
    head = workloads.PagedBatch("h", b.dtype, b.qo_indptr[:4], b.kv_indptr[:4], b.kv_indices, b.last_page_len[:3],
                                32, 8, 16, 1, b.sm_scale, b.q, b.k, b.v)
    assert bench.algorithmic(d)[0] + bench.algorithmic(head)[0] == bench.algorithmic(b)[0]
