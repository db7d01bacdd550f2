"""The MLA decode planner (C++, through the C ABI) against its Python
restatement in oracle/plan_ref.py, byte for byte, plus the properties every
plan must have and the host-side argument checks."""
from __future__ import annotations

import numpy as np
import pytest

from oracle import plan_ref
from serving_attention_gb300 import mla
import workloads

HEADER = plan_ref.MLA_HEADER_INTS


def _plan(b, pairs=8, heads=128, **kw):
    cfg = mla.make_config(pairs, **kw)
    st, img, info = mla.plan_host(cfg, b.kv_indptr, b.kv_indices, b.last_page_len, heads, b.page_size, b.num_pages)
    assert st == 0, st
    return cfg, img, info


def _ref(b, cfg, heads=128):
    return plan_ref.mla_make_plan(b.kv_indptr, b.last_page_len, b.page_size, heads, cfg.num_pairs, cfg.min_chunk)


@pytest.mark.parametrize("seed,batch,kv_max,page,pairs,min_chunk", [
    (1, 7, 3000, 64, 4, 256), (2, 64, 32768, 64, 74, 512), (3, 1, 100000, 16, 76, 512),
    (4, 40, 700, 32, 76, 64), (5, 9, 5000, 8, 3, 128), (6, 300, 200, 64, 76, 512),
    (7, 3, 90, 16, 76, 256), (8, 120, 20000, 64, 1, 256), (9, 17, 64, 64, 5, 64),
])
def test_matches_restatement(seed, batch, kv_max, page, pairs, min_chunk):
    b = workloads.random_mla_batch(seed, batch=batch, kv_max=kv_max, num_heads=4, page_size=page)
    cfg, img, info = _plan(b, pairs, min_chunk=min_chunk)
    ref = _ref(b, cfg)
    assert np.array_equal(img, ref)
    assert info.num_units == img[1] and info.num_merge == img[10] and info.num_parts == img[14]


def test_length_mix_workload_plan():
    b = workloads.mla_decode(batch=64)
    cfg, img, info = _plan(b, 74)
    assert np.array_equal(img, _ref(b, cfg))


def _units(img):
    off, n = img[7], img[1]
    return img[off:off + 4 * n].reshape(n, 4)


@pytest.mark.parametrize("seed", [11, 12, 13])
def test_every_token_once_and_blocks_aligned(seed):
    b = workloads.random_mla_batch(seed, batch=50, kv_max=9000, num_heads=4, page_size=64)
    _, img, info = _plan(b, 20, min_chunk=256)
    units = _units(img)
    lens = b.kv_lens()
    covered = {r: [] for r in range(b.batch)}
    for bb, k0, k1, part in units:
        assert k0 % 64 == 0 and 0 <= k0 < k1 <= lens[bb]
        covered[int(bb)].append((int(k0), int(k1), int(part)))
    slots = set()
    for r in range(b.batch):
        segs = sorted(covered[r])
        assert sum(k1 - k0 for k0, k1, _ in segs) == lens[r]
        assert all(segs[i][1] == segs[i + 1][0] for i in range(len(segs) - 1))
        if len(segs) == 1:
            assert segs[0][2] == -1
        for _, _, part in segs if len(segs) > 1 else []:
            assert part not in slots
            slots.add(part)
    assert slots == set(range(info.num_parts))
    # pair ranges tile the unit list
    off, P = img[6], img[2]
    ptr = img[off:off + P + 1]
    assert ptr[0] == 0 and ptr[-1] == info.num_units and np.all(np.diff(ptr) >= 0)


def test_empty_requests_get_a_merge_entry():
    b = workloads.make_mla_batch("empty", [0, 100, 0], 4, 16, 3, pool_pages=10)
    _, img, info = _plan(b, 2)
    off = img[9]
    merge = img[off:off + 4 * info.num_merge].reshape(-1, 4)
    assert sorted(merge[:, 0].tolist()) == [0, 2] and np.all(merge[:, 2] == 0)
    assert np.array_equal(img, _ref(b, mla.make_config(2)))


def _pair_costs(img):
    units = _units(img)
    off, P = img[6], img[2]
    ptr = img[off:off + P + 1]
    return np.array([(units[ptr[p]:ptr[p + 1], 2] - units[ptr[p]:ptr[p + 1], 1] + plan_ref.MLA_UNIT_COST_TOKENS).sum() for p in range(P)])


@pytest.mark.parametrize("pairs", [74, 76])
def test_split_is_balanced(pairs):
    """The length mix: the busiest pair within 5 % of the mean (dealing
    fixed chunks longest-first left it 24 % above), and no piece shorter than
    min_chunk except a request's last."""
    b = workloads.mla_decode(batch=64)
    _, img, _ = _plan(b, pairs)
    cost = _pair_costs(img)
    assert cost.max() <= 1.05 * cost.mean()
    lens = b.kv_lens()
    for bb, k0, k1, _ in _units(img):
        assert k1 - k0 >= 256 or k1 == lens[bb]


@pytest.mark.parametrize("seed", [31, 32, 33, 34])
def test_split_balance_random(seed):
    b = workloads.random_mla_batch(seed, batch=int(np.random.default_rng(seed).integers(1, 200)), kv_max=40000,
                                   num_heads=4, page_size=64)
    _, img, info = _plan(b, 76)
    cost = _pair_costs(img)
    used = cost[cost > 0]
    assert cost.max() <= used.mean() + 2 * (plan_ref.MLA_UNIT_COST_TOKENS + 256) + 64


def test_rejects():
    b = workloads.random_mla_batch(21, batch=4, kv_max=300, num_heads=4, page_size=16)
    cfg = mla.make_config(4)
    args = (b.kv_indptr, b.kv_indices, b.last_page_len)
    assert mla.plan_host(cfg, *args, 129, 16)[0] == 2            # too many heads
    assert mla.plan_host(cfg, *args, 128, 4)[0] == 2             # page size 4
    bad = b.last_page_len.copy()
    bad[0] = 17
    assert mla.plan_host(cfg, b.kv_indptr, b.kv_indices, bad, 128, 16)[0] == 1
    assert mla.plan_host(cfg, *args, 128, 16, num_pages=1)[0] == 1   # page id out of range
    assert mla.plan_host(mla.make_config(4, max_batch=2), *args, 128, 16)[0] == 3
    long = workloads.make_mla_batch("long", [3000], 4, 16, 22)   # cut over the 4 pairs: 4 partial states
    assert mla.plan_host(mla.make_config(4, min_chunk=64, max_parts=1), long.kv_indptr, long.kv_indices,
                         long.last_page_len, 128, 16)[0] == 3
    assert mla.plan_host(mla.make_config(4, min_chunk=100), *args, 128, 16)[0] == 1   # not a multiple of 64


def test_library_exports_mla_entry_points():
    lib = mla.load()
    for name in mla.EXPORTS:
        assert hasattr(lib, name)
