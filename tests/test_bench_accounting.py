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
