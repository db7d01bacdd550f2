"""The host planner (C++, through the C ABI, no GPU) against the independent
Python re-derivation of the same rule, byte for byte, plus the invariants the
rule promises (coverage, no empty work, LPT balance, determinism)."""
from __future__ import annotations

import numpy as np
import pytest

import serving_attention_gb300 as fi
import workloads
from oracle import plan_ref

HEADER = 32


def _cfg(num_ctas=148, **kw):
    c = fi.make_plan_config(num_ctas, **kw)
    return c, c.as_dict()


def _plan_both(cfg, cfgd, qo, kvp, kvi, lpl, hq, hkv, page, causal, num_pages):
    st_c, ws_c, info_c = fi.plan_host(cfg, qo, kvp, kvi, lpl, hq, hkv, 128, page, causal, num_pages)
    st_p, ws_p, info_p = plan_ref.make_plan(cfgd, qo, kvp, kvi, lpl, hq, hkv, 128, page, causal, num_pages)
    assert st_c == st_p, (st_c, st_p)
    if st_c == 0:
        assert np.array_equal(ws_c, ws_p), np.nonzero(ws_c != ws_p)[0][:10]
        got = info_c.as_dict()
        for k, v in info_p.items():
            assert got[k] == v, (k, got[k], v)
    return st_c, ws_c, info_c


def _random_lengths(rng, batch, page):
    qo = rng.choice([1, 1, 1, 2, 4, 5, 17, 40, 130, 300], size=batch)
    kv = rng.integers(0, 3000, size=batch)
    kv[rng.random(batch) < 0.1] = 0
    return qo, kv


@pytest.mark.parametrize("seed", range(40))
def test_plan_matches_reference_random(seed):
    rng = np.random.default_rng(seed)
    batch = int(rng.integers(1, 40))
    page = int(rng.choice([1, 2, 4, 16, 32, 128]))
    hkv = int(rng.choice([1, 2, 8]))
    group = int(rng.choice([1, 2, 4, 8, 16]))
    causal = int(rng.integers(0, 2))
    qo, kv = _random_lengths(rng, batch, page)
    kvp, lpl = workloads._pages_for(kv, page)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    nnz = int(kvp[-1])
    kvi = rng.permutation(nnz + 5)[:nnz].astype(np.int32)
    cfg, cfgd = _cfg(num_ctas=int(rng.choice([1, 7, 148, 152])), split_factor=int(rng.integers(1, 6)),
                     decode_min_chunk=int(rng.choice([64, 256])), prefill_min_chunk=int(rng.choice([128, 1024])))
    st, ws, info = _plan_both(cfg, cfgd, qop, kvp, kvi, lpl, hkv * group, hkv, page, causal, nnz + 5)
    assert st == 0
    _check_invariants(ws, qop, kv, hkv * group, hkv, causal, cfgd)


def _items(ws, off_items, n_items):
    """The plan's work items, [item, field]: the first 8 fields, and per item
    its KV-head count (1, or H of a multi-head unit); the request's copy that
    follows the 8 fields is checked against the request table."""
    full = ws[off_items:off_items + plan_ref.ITEM_INTS * n_items].reshape(-1, plan_ref.ITEM_INTS)
    off_req = ws[10]
    req = ws[off_req:off_req + 4 * ws[4]].reshape(-1, 4)
    assert np.array_equal(full[:, 8:12], req[full[:, 0]]) and np.all(full[:, 13:] == 0)
    assert np.all(np.isin(full[:, 12], (0, 2, 4, 8)))
    return full[:, :8], np.maximum(full[:, 12], 1)


def _per_head(items, heads, G):
    """Items with every multi-head item split into one item per KV head, in
    one-head numbering: head hk + h holds rows 0..G of the unit's rows
    h*G .. h*G + G - 1, so its partial rows start at part + h*G."""
    out = []
    for it, H in zip(items, heads):
        b, hk, r0, r1, k0, k1, part, merge = (int(x) for x in it)
        if H == 1:
            out.append((b, hk, r0, r1, k0, k1, part, merge))
            continue
        assert (r0, r1) == (0, H * G) and H * G == plan_ref.MH_ROWS and hk % H == 0
        for h in range(H):
            out.append((b, hk + h, 0, G, k0, k1, part + h * G if part >= 0 else -1, merge))
    return np.array(out, dtype=np.int64).reshape(-1, 8)


def _check_invariants(ws, qop, kv, hq, hkv, causal, cfgd):
    G = hq // hkv
    n_items, n_merge, C = ws[1], ws[2], ws[3]
    off_cta, off_items, off_merge, off_cnt, off_req = ws[6], ws[7], ws[8], ws[9], ws[10]
    cta = ws[off_cta:off_cta + C + 1]
    assert cta[0] == 0 and cta[-1] == n_items and np.all(np.diff(cta) >= 0)
    items, heads = _items(ws, off_items, n_items)
    assert np.all(ws[off_cnt:off_cnt + n_merge] == 0)
    req = ws[off_req:off_req + 4 * (len(qop) - 1)].reshape(-1, 4)
    assert np.array_equal(req[:, 3], kv)
    # multi-head items: one query token of a decode-class request
    for it in items[heads > 1]:
        assert qop[it[0] + 1] - qop[it[0]] == 1
    # coverage: per (b, hk) the row ranges tile [0, R); per unit the chunks tile [0, kv_eff)
    by_unit = {}
    for it, H in zip(items, heads):
        b, hk, r0, r1, k0, k1, part, merge = (int(x) for x in it)
        by_unit.setdefault((b, hk, r0, r1, int(H)), []).append((k0, k1, part, merge))
    rows_of = {}  # (b, hk) -> [(r0, r1) in one-head numbering]
    for (b, hk, r0, r1, H) in by_unit:
        for h in range(H):
            rows_of.setdefault((b, hk + h), []).append((r0, r1) if H == 1 else (0, G))
    for b in range(len(qop) - 1):
        R = int(qop[b + 1] - qop[b]) * G
        for hk in range(hkv):
            units = sorted(rows_of.get((b, hk), []))
            if R == 0:
                assert not units
                continue
            assert units[0][0] == 0 and units[-1][1] == R
            assert all(units[i][1] == units[i + 1][0] for i in range(len(units) - 1))
    for (b, hk, r0, r1, H), chunks in by_unit.items():
        chunks = sorted(chunks)
        lq, lkv = int(qop[b + 1] - qop[b]), int(kv[b])
        t_last = 0 if H > 1 else (r1 - 1) // G
        need = min(lkv, max(0, lkv - lq + t_last + 1)) if causal else lkv
        assert chunks[0][0] == 0 and chunks[-1][1] == need
        assert all(chunks[i][1] == chunks[i + 1][0] for i in range(len(chunks) - 1))
        if need > 0:
            assert all(k1 > k0 for (k0, k1, _, _) in chunks), "empty chunk in a non-empty unit"
        else:
            assert len(chunks) == 1
        if len(chunks) > 1:
            m = chunks[0][3]
            assert m >= 0 and all(c[3] == m for c in chunks)
            mu = ws[off_merge + 8 * m: off_merge + 8 * m + 8]
            assert tuple(mu[:4]) == (b, hk, r0, r1) and mu[4] == len(chunks)
            # merged after the run exactly when the unit is of the prefill class
            assert mu[6] == (1 if lq * G > 16 else 0) and mu[7] == 0
            parts = [c[2] for c in chunks]
            assert parts == [mu[5] + i * (r1 - r0) for i in range(len(chunks))]
        else:
            assert chunks[0][2] == -1 and chunks[0][3] == -1
    # LPT bound: max CTA load <= mean load + largest item
    w = {16: cfgd["decode_cost_weight"], plan_ref.TILE_PREFILL: cfgd["prefill_cost_weight"]}
    cost = []
    for it, H in zip(items, heads):
        R = int(qop[it[0] + 1] - qop[it[0]]) * G
        cost.append(((int(it[5]) - int(it[4])) * int(H) + plan_ref.ITEM_COST_TOKENS)
                    * w[16 if R <= 16 else plan_ref.TILE_PREFILL])
    cost = np.array(cost, dtype=np.int64)
    loads = np.array([cost[cta[c]:cta[c + 1]].sum() for c in range(C)])
    if cost.size:
        assert loads.max() <= cost.sum() / C + cost.max()


def _visible(lkv, lq, t, causal, window, sink):
    """Keys query token t may see under the mask reading (brute force)."""
    q_pos = lkv - lq + t
    return {j for j in range(lkv) if (not causal or j <= q_pos) and (window < 0 or j >= q_pos - window or j < sink)}


def _check_variant_coverage(ws, qop, kv, hq, hkv, causal, page, window, sink):
    """Every key a row can see lies in one of its unit's chunks; chunks are
    disjoint, start on the class granule and none is invisible to all rows."""
    G = hq // hkv
    n_items, off_items = ws[1], ws[7]
    items = _per_head(*_items(ws, off_items, n_items), G)
    by_unit = {}
    for it in items:
        b, hk, r0, r1, k0, k1 = (int(x) for x in it[:6])
        by_unit.setdefault((b, hk, r0, r1), []).append((k0, k1))
    for (b, hk, r0, r1), chunks in by_unit.items():
        lq, lkv = int(qop[b + 1] - qop[b]), int(kv[b])
        gran = max(page, 64) if lq * G <= 16 else max(page, 128)
        need = set()
        for t in range(r0 // G, (r1 - 1) // G + 1):
            need |= _visible(lkv, lq, t, causal, window, sink)
        chunks = sorted(chunks)
        covered = set()
        for k0, k1 in chunks:
            if k1 == k0:
                assert len(chunks) == 1 and not need
                continue
            assert k0 % gran == 0, (k0, gran)
            span = set(range(k0, k1))
            assert not (span & covered) and span & need, (b, hk, r0, k0, k1)
            covered |= span
        assert need <= covered


@pytest.mark.parametrize("seed", range(24))
def test_plan_with_window_and_sink_matches_reference(seed):
    rng = np.random.default_rng(100 + seed)
    batch = int(rng.integers(1, 24))
    page = int(rng.choice([1, 4, 16, 64]))
    hkv = int(rng.choice([1, 2, 8]))
    group = int(rng.choice([1, 4, 8]))
    causal = int(rng.integers(0, 2))
    qo, kv = _random_lengths(rng, batch, page)
    kvp, lpl = workloads._pages_for(kv, page)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    nnz = int(kvp[-1])
    kvi = rng.permutation(nnz + 2)[:nnz].astype(np.int32)
    window = int(rng.choice([-1, 0, 5, 127, 300, 1000, 4096]))
    sink = int(rng.choice([0, 0, 4, 64, 700]))
    cap = float(rng.choice([0.0, 30.0]))
    cfg, cfgd = _cfg(num_ctas=int(rng.choice([1, 7, 152])), split_factor=int(rng.integers(1, 6)),
                     decode_min_chunk=int(rng.choice([64, 256])), prefill_min_chunk=int(rng.choice([128, 1024])),
                     window_left=window, sink_tokens=sink, logits_soft_cap=cap)
    st, ws, info = _plan_both(cfg, cfgd, qop, kvp, kvi, lpl, hkv * group, hkv, page, causal, nnz + 2)
    assert st == 0
    assert info.variant == (1 if cap > 0 else 0) | (2 if window >= 0 else 0)
    assert tuple(ws[16:19]) == (window, sink, int(np.array([cap], np.float32).view(np.int32)[0]))
    _check_variant_coverage(ws, qop, kv, hkv * group, hkv, causal, page, window, sink)


def test_window_skips_chunks():
    """A 4096-token window on the long decode requests plans far less KV than the full attention."""
    qo, kv = np.ones(64, np.int64), workloads.llama8b_decode_lengths(np.random.default_rng(2000))
    kvp, lpl = workloads._pages_for(kv, 16)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    kvi = np.arange(int(kvp[-1]), dtype=np.int32)

    def planned_kv(**kw):
        cfg, _ = _cfg(num_ctas=152, **kw)
        st, ws, _ = fi.plan_host(cfg, qop, kvp, kvi, lpl, 32, 8, 128, 16, 0)
        assert st == 0
        items, heads = _items(ws, ws[7], ws[1])
        return int(((items[:, 5] - items[:, 4]) * heads).sum())

    full = planned_kv()
    windowed = planned_kv(window_left=4096, sink_tokens=4)
    expect = int(sum(min(k, 4096 + 1 + 64) for k in kv)) * 8  # window + the granule it rounds to, per KV head
    assert windowed <= expect + 64 * 8 * 64 and windowed < full / 2


@pytest.mark.parametrize("seed", range(6))
def test_plan_with_rope_matches_reference(seed):
    rng = np.random.default_rng(200 + seed)
    batch = int(rng.integers(1, 12))
    page = int(rng.choice([1, 16]))
    kv = rng.integers(1, 3000, size=batch)
    qo = np.minimum(kv, rng.choice([1, 1, 7, 300], size=batch))  # RoPE needs Lq <= Lkv
    kvp, lpl = workloads._pages_for(kv, page)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    nnz = int(kvp[-1])
    kvi = rng.permutation(nnz).astype(np.int32)
    cfg, cfgd = _cfg(num_ctas=152, rope_max_positions=4096, rope_theta=float(rng.choice([1e4, 5e5])),
                     rope_scale=float(rng.choice([1.0, 8.0])), window_left=int(rng.choice([-1, 500])))
    st, ws, info = _plan_both(cfg, cfgd, qop, kvp, kvi, lpl, 32, 8, 16 if page == 16 else 1, 1, nnz)
    assert st == 0 and info.variant & 4
    assert ws[19] == 4096 and ws[22] * 4 == (plan_ref.int_workspace_ints(cfgd) * 4 + 255) // 256 * 256
    assert fi.int_workspace_bytes(cfg) == ws[22] * 4 + 4096 * 64 * 8
    small, _ = _cfg(num_ctas=152, rope_max_positions=3)
    assert fi.int_workspace_bytes(small) == (plan_ref.int_workspace_ints(small.as_dict()) * 4 + 255) // 256 * 256 + 16 * 64 * 8


@pytest.mark.parametrize("case", ["long", "lq_gt_lkv", "theta", "scale", "negative"])
def test_plan_rejects_bad_rope(case):
    kv = np.array([100, 3000]) if case == "long" else np.array([100, 10])
    qo = np.array([1, 20]) if case == "lq_gt_lkv" else np.array([1, 2])
    kvp, lpl = workloads._pages_for(kv, 16)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    kw = dict(rope_max_positions=2048)
    if case == "theta":
        kw["rope_theta"] = 0.0
    elif case == "scale":
        kw["rope_scale"] = -1.0
    elif case == "negative":
        kw["rope_max_positions"] = -5
    cfg, cfgd = _cfg(**kw)
    kvi = np.arange(int(kvp[-1]), dtype=np.int32)
    st, ws, _ = fi.plan_host(cfg, qop, kvp, kvi, lpl, 8, 2, 128, 16, 1)
    assert st == 1 and ws is None
    st_p, _, _ = plan_ref.make_plan(cfgd, qop, kvp, kvi, lpl, 8, 2, 128, 16, 1, 0)
    assert st_p == 1


@pytest.mark.parametrize("field,value", [("window_left", -2), ("sink_tokens", -1), ("logits_soft_cap", -1.0),
                                         ("logits_soft_cap", float("inf")), ("logits_soft_cap", float("nan"))])
def test_plan_rejects_bad_variant(field, value):
    qo = np.array([0, 1], np.int32)
    kvp = np.array([0, 1], np.int32)
    cfg, cfgd = _cfg(**{field: value})
    st, ws, _ = fi.plan_host(cfg, qo, kvp, np.array([0], np.int32), np.array([3], np.int32), 8, 2, 128, 16, 0)
    assert st == 1 and ws is None
    st_p, _, _ = plan_ref.make_plan(cfgd, qo, kvp, np.array([0], np.int32), np.array([3], np.int32), 8, 2, 128, 16,
                                    0, 1)
    assert st_p == 1


@pytest.mark.parametrize("name", ["tiny_decode", "llama8b_decode", "ragged_prefill", "continuous_batch"])
def test_plan_matches_reference_workloads(name):
    rng_lengths = {
        "tiny_decode": lambda: (np.ones(4, np.int64), np.random.default_rng(1000).integers(1, 513, size=4), 8, 2, 16, 0),
        "llama8b_decode": lambda: (np.ones(64, np.int64),
                                   workloads.llama8b_decode_lengths(np.random.default_rng(2000)), 32, 8, 16, 0),
        "ragged_prefill": lambda: (*workloads.ragged_prefill_lengths(np.random.default_rng(3000)), 32, 8, 16, 1),
        "continuous_batch": lambda: (*workloads.continuous_batch_lengths(np.random.default_rng(5000)), 32, 8, 16, 1),
    }
    qo, kv, hq, hkv, page, causal = rng_lengths[name]()
    kvp, lpl = workloads._pages_for(np.asarray(kv), page)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    nnz = int(kvp[-1])
    kvi = np.random.default_rng(7).permutation(nnz).astype(np.int32)
    cfg, cfgd = _cfg(num_ctas=152)
    st, ws, info = _plan_both(cfg, cfgd, qop, kvp, kvi, lpl, hq, hkv, page, causal, nnz)
    assert st == 0
    _check_invariants(ws, qop, np.asarray(kv), hq, hkv, causal, cfgd)


def test_plan_is_deterministic():
    rng = np.random.default_rng(9)
    qo, kv = _random_lengths(rng, 30, 16)
    kvp, lpl = workloads._pages_for(kv, 16)
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    kvi = np.arange(int(kvp[-1]), dtype=np.int32)
    cfg, _ = _cfg()
    a = fi.plan_host(cfg, qop, kvp, kvi, lpl, 32, 8, 128, 16, 1)[1]
    b = fi.plan_host(cfg, qop, kvp, kvi, lpl, 32, 8, 128, 16, 1)[1]
    assert np.array_equal(a, b)


@pytest.mark.parametrize("case,status", [
    ("head_dim", 2), ("page_size", 2), ("heads", 2), ("group", 2), ("indptr", 1), ("lpl", 1), ("index", 1),
    ("capacity", 3), ("causal", 1),
])
def test_plan_rejects(case, status):
    qo = np.array([0, 1, 3], np.int32)
    kvp = np.array([0, 2, 3], np.int32)
    kvi = np.array([0, 1, 2], np.int32)
    lpl = np.array([5, 16], np.int32)
    args = dict(hq=8, hkv=2, d=128, page=16, causal=0, num_pages=3)
    cfg, cfgd = _cfg()
    if case == "head_dim":
        args["d"] = 64
    elif case == "page_size":
        args["page"] = 12
    elif case == "heads":
        args["hq"] = 7
    elif case == "group":
        args["hq"], args["hkv"] = 34, 1
    elif case == "indptr":
        qo = np.array([0, 3, 1], np.int32)
    elif case == "lpl":
        lpl = np.array([0, 16], np.int32)
    elif case == "index":
        kvi = np.array([0, 1, 3], np.int32)
    elif case == "capacity":
        cfg, cfgd = _cfg(max_items=1)
    elif case == "causal":
        args["causal"] = 2
    st, ws, _ = fi.plan_host(cfg, qo, kvp, kvi, lpl, args["hq"], args["hkv"], args["d"], args["page"],
                             args["causal"], args["num_pages"])
    assert st == status and ws is None
    st_p, _, _ = plan_ref.make_plan(cfgd, qo, kvp, kvi, lpl, args["hq"], args["hkv"], args["d"], args["page"],
                                    args["causal"], args["num_pages"])
    assert st_p == status


def test_default_capacity_holds_every_workload():
    """The default config's capacities hold all five workloads (10 draws of the mix)."""
    cfg, cfgd = _cfg(num_ctas=152)
    cases = [workloads.continuous_batch_lengths(np.random.default_rng(5000 + r)) + (1,) for r in range(10)]
    cases.append(workloads.ragged_prefill_lengths(np.random.default_rng(3000)) + (1,))
    cases.append((np.ones(64, np.int64), workloads.llama8b_decode_lengths(np.random.default_rng(2000)), 0))
    for qo, kv, causal in cases:
        kvp, lpl = workloads._pages_for(np.asarray(kv), 16)
        qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
        st, ws, info = fi.plan_host(cfg, qop, kvp, np.zeros(int(kvp[-1]), np.int32), lpl, 32, 8, 128, 16, causal)
        assert st == 0, st


# ---------------------------------------------------------------- two-level (cascade) plans


def _cascade_both(cfg, cfgd, shared, own, hq, hkv, causal, num_pages=0, shared_num_pages=0):
    """shared / own: (qo_indptr, kv_indptr, kv_indices, last_page_len, page_size)."""
    sqo, skvp, skvi, slpl, sp = shared
    qo, kvp, kvi, lpl, p = own
    st_c, ws_c, info_c = fi.plan_cascade_host(cfg, sqo, skvp, skvi, slpl, sp, qo, kvp, kvi, lpl, hq, hkv, 128, p,
                                              causal, num_pages, shared_num_pages)
    st_p, ws_p, info_p = plan_ref.make_cascade_plan(cfgd, sqo, skvp, skvi, slpl, sp, shared_num_pages, qo, kvp, kvi,
                                                    lpl, hq, hkv, 128, p, causal, num_pages)
    assert st_c == st_p, (st_c, st_p)
    if st_c == 0:
        assert np.array_equal(ws_c, ws_p), np.nonzero(ws_c != ws_p)[0][:10]
        got = info_c.as_dict()
        for k, v in info_p.items():
            assert got[k] == v, (k, got[k], v)
    return st_c, ws_c, info_c


def _random_cascade(rng):
    nblk = int(rng.integers(1, 5))
    sizes = rng.integers(1, 6, size=nblk)
    B = int(sizes.sum())
    qo = rng.choice([0, 1, 1, 2, 3, 9, 40, 70], size=B)
    causal = int(rng.integers(0, 2))
    kv = rng.integers(0, 2500, size=B)
    if causal:
        kv = np.maximum(kv, qo)
    page, spage = int(rng.choice([1, 2, 16])), int(rng.choice([1, 8, 16, 64]))
    skv = rng.integers(0, 9000, size=nblk)
    skv[rng.random(nblk) < 0.2] = 0
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    first = np.concatenate([[0], np.cumsum(sizes)])
    sqo = qop[first].astype(np.int32)
    kvp, lpl = workloads._pages_for(kv, page)
    skvp, slpl = workloads._pages_for(skv, spage)
    kvi = rng.permutation(int(kvp[-1]) + 3)[:int(kvp[-1])].astype(np.int32)
    skvi = rng.permutation(int(skvp[-1]) + 3)[:int(skvp[-1])].astype(np.int32)
    return (sqo, skvp, skvi, slpl, spage), (qop, kvp, kvi, lpl, page), causal, kv, skv


def _check_cascade_invariants(ws, shared, own, kv, skv, hq, hkv, causal):
    """Every unit writes partial states and none merges in the run; every row
    of every request is in exactly one merge entry of at most 16 rows, whose
    two part lists are exactly the partial rows its block's chunks and its
    own chunks wrote for that row; those chunks tile the visible keys."""
    G = hq // hkv
    S = len(shared[0]) - 1
    n_items, n_merge, C = ws[1], ws[2], ws[3]
    assert n_merge == 0 and ws[26] == S
    off_items, off_req, off_cas, n_cas = ws[7], ws[10], ws[27], ws[28]
    items = _per_head(*_items(ws, off_items, n_items), G)
    reqs = ws[off_req:off_req + 4 * ws[4]].reshape(-1, 4)
    ents = ws[off_cas:off_cas + 12 * n_cas].reshape(-1, 12)
    assert ws[31] == (ents[:, 3] - ents[:, 2]).max()  # the merge launch's row tasks per entry
    assert np.all(items[:, 6] >= 0) and np.all(items[:, 7] == -1)
    parts = {}  # (b, hk, row) -> [(kv0, kv1, partial row)]
    for b, hk, r0, r1, k0, k1, part, _ in items:
        for r in range(r0, r1):
            parts.setdefault((b, hk, r), []).append((k0, k1, part + r - r0))
    qo = np.diff(own[0])
    seen = set()
    for b, hk, r0, r1, n0, b0, s0, n1, b1, s1, z0, z1 in ents:
        assert 0 < r1 - r0 <= 16 and z0 == z1 == 0 and b >= S
        blk = int(np.searchsorted(shared[0], reqs[b][0], side="right") - 1)
        for r in range(r0, r1):
            assert (b, hk, r) not in seen
            seen.add((b, hk, r))
            sr = (reqs[b][0] - reqs[blk][0]) * G + r
            mine = sorted(parts[(b, hk, r)])
            theirs = sorted(parts[(blk, hk, sr)])
            assert [p for _, _, p in theirs] == [b0 + c * s0 + r - r0 for c in range(n0)]
            assert [p for _, _, p in mine] == [b1 + c * s1 + r - r0 for c in range(n1)]
            # the chunks tile the visible keys: all of the block's, the own causal range
            t = r // G
            hi = min(kv[b - S], kv[b - S] - qo[b - S] + t + 1) if causal else kv[b - S]
            for chunks, end in ((theirs, skv[blk]), (mine, hi)):
                ks = [(k0, k1) for k0, k1, _ in chunks if k1 > k0]
                assert sum(k1 - k0 for k0, k1 in ks) >= end
                covered = np.zeros(max(end, 1), bool)
                for k0, k1 in ks:
                    covered[k0:min(k1, end)] = True
                assert end == 0 or covered[:end].all()
    want = {(S + r, hk, row) for r in range(len(qo)) for hk in range(hkv) for row in range(qo[r] * G)}
    assert seen == want


@pytest.mark.parametrize("seed", range(24))
def test_cascade_plan_matches_reference_random(seed):
    rng = np.random.default_rng(700 + seed)
    shared, own, causal, kv, skv = _random_cascade(rng)
    hkv = int(rng.choice([1, 2, 8]))
    group = int(rng.choice([1, 4, 8]))
    cfg, cfgd = _cfg(num_ctas=int(rng.choice([1, 9, 152])), split_factor=int(rng.integers(1, 4)),
                     decode_min_chunk=int(rng.choice([64, 256])), prefill_min_chunk=int(rng.choice([128, 1024])))
    st, ws, info = _cascade_both(cfg, cfgd, shared, own, hkv * group, hkv, causal,
                                 num_pages=int(own[1][-1]) + 3, shared_num_pages=int(shared[1][-1]) + 3)
    assert st == 0
    assert info.num_shared == len(shared[0]) - 1 and info.num_merge_units == 0
    _check_cascade_invariants(ws, shared, own, kv, skv, hkv * group, hkv, causal)


def test_cascade_plan_of_the_shared_prefix_workload():
    """The parallel-generation case: one block holding the 8192-token dense
    prefix (pages of 16) for 64 branches of one query each, suffixes at page 1."""
    rng = np.random.default_rng(4000)
    suf = rng.integers(64, 513, size=64)
    kvp, lpl = workloads._pages_for(suf, 1)
    qop = np.arange(65, dtype=np.int32)
    shared = (np.array([0, 64], np.int32), np.array([0, 512], np.int32), np.arange(512, dtype=np.int32),
              np.array([16], np.int32), 16)
    own = (qop, kvp, rng.permutation(int(kvp[-1])).astype(np.int32), lpl, 1)
    cfg, cfgd = _cfg(num_ctas=152)
    st, ws, info = _cascade_both(cfg, cfgd, shared, own, 32, 8, 0)
    assert st == 0 and info.prefill_caches == 2  # the block's 256-row units read the shared cache on tensor cores
    _check_cascade_invariants(ws, shared, own, suf, np.array([8192]), 32, 8, 0)
    # every suffix unit takes all 8 KV heads of its branch (32 rows: G = 4)
    items, heads = _items(ws, ws[7], ws[1])
    own_items = items[:, 0] >= 1
    assert np.all(heads[own_items] == 8) and np.all(heads[~own_items] == 1)
    assert np.all(items[own_items, 1] == 0) and np.all(items[own_items, 3] == 32)


@pytest.mark.parametrize("group,hkv,heads", [(4, 8, 8), (8, 4, 4), (16, 2, 2), (4, 4, 1), (2, 8, 1), (8, 2, 1)])
def test_multi_head_units_of_a_page_1_decode(group, hkv, heads):
    """One-token requests on pages of 1 form units of 32 / G KV heads when G
    is a multiple of 4 and those heads tile Hkv; a longer request, another
    page size or a RoPE plan keeps one head per unit."""
    rng = np.random.default_rng(4100 + group)
    kv = rng.integers(1, 2000, size=12)
    qo = np.ones(12, np.int64)
    qo[3] = 3  # a three-token request keeps one head per unit
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    for page, rope in ((1, 0), (2, 0), (1, 4096)):
        kvp, lpl = workloads._pages_for(kv, page)
        nnz = int(kvp[-1])
        kvi = rng.permutation(nnz).astype(np.int32)
        cfg, cfgd = _cfg(num_ctas=152, rope_max_positions=rope)
        st, ws, _ = _plan_both(cfg, cfgd, qop, kvp, kvi, lpl, hkv * group, hkv, page, 1, nnz)
        assert st == 0
        _check_invariants(ws, qop, kv, hkv * group, hkv, 1, cfgd)
        items, h = _items(ws, ws[7], ws[1])
        want = heads if (page == 1 and rope == 0) else 1
        assert np.all(h[items[:, 0] == 3] == 1)
        assert np.all(h[items[:, 0] != 3] == want)


@pytest.mark.parametrize("case,status", [
    ("straddle", 1), ("cover", 1), ("causal_short", 1), ("window", 2), ("rope", 2), ("shared_page", 2),
    ("no_blocks", 1), ("shared_index", 1), ("capacity", 3),
])
def test_cascade_plan_rejects(case, status):
    qo = np.array([0, 2, 3, 5], np.int32)
    kvp = np.array([0, 1, 2, 3], np.int32)
    lpl = np.array([16, 5, 16], np.int32)
    kvi = np.array([0, 1, 2], np.int32)
    sqo = np.array([0, 3, 5], np.int32)
    skvp = np.array([0, 2, 3], np.int32)
    skvi = np.array([2, 0, 1], np.int32)
    slpl = np.array([8, 8], np.int32)
    sp, causal, kw = 8, 1, {}
    if case == "straddle":
        sqo = np.array([0, 1, 5], np.int32)  # request 0's rows [0, 2) cross block boundary 1
    elif case == "cover":
        sqo = np.array([0, 3, 4], np.int32)  # the blocks stop before the last row
    elif case == "causal_short":
        lpl = np.array([1, 5, 16], np.int32)  # request 0: 2 queries, 1 own key
    elif case == "window":
        kw = dict(window_left=64)
    elif case == "rope":
        kw = dict(rope_max_positions=4096)
    elif case == "shared_page":
        sp = 12
    elif case == "no_blocks":
        sqo, skvp, skvi, slpl = np.array([0], np.int32), np.array([0], np.int32), skvi[:0], slpl[:0]
    elif case == "shared_index":
        skvi = np.array([2, 0, 7], np.int32)
    elif case == "capacity":
        kw = dict(max_merge_units=1)
    cfg, cfgd = _cfg(**kw)
    st, ws, _ = _cascade_both(cfg, cfgd, (sqo, skvp, skvi, slpl, sp), (qo, kvp, kvi, lpl, 16), 8, 2, causal,
                              num_pages=3, shared_num_pages=3)
    assert st == status and ws is None


@pytest.mark.parametrize("num_ctas,page", [(152, 16), (60, 16), (152, 1)])
def test_decode_chunk_counts_the_ctas_prefill_items_leave(num_ctas, page):
    """Decode chunks are sized over the CTAs the prefill-class items leave
    free when those take at most half the CTAs (48 of 152 here; 48 of 60 is
    more than half, so all 60 count), and a multi-head unit's chunk is the
    one-head chunk over its heads, rounded up to the granule."""
    rng = np.random.default_rng(4300 + num_ctas + page)
    hkv, group = 8, 4
    kv = np.concatenate([[3000, 3000], rng.integers(100, 5000, size=40)])
    qo = np.concatenate([[64, 64], np.ones(40, np.int64)])  # two 256-row requests, 40 one-token ones
    qop = np.concatenate([[0], np.cumsum(qo)]).astype(np.int32)
    kvp, lpl = workloads._pages_for(kv, page)
    nnz = int(kvp[-1])
    kvi = rng.permutation(nnz).astype(np.int32)
    cfg, cfgd = _cfg(num_ctas=num_ctas)
    st, ws, info = _plan_both(cfg, cfgd, qop, kvp, kvi, lpl, hkv * group, hkv, page, 0, nnz)
    assert st == 0
    _check_invariants(ws, qop, kv, hkv * group, hkv, 0, cfgd)
    assert info.chunk_prefill == 1024
    n_pre = 2 * hkv * 3  # per KV head, 3000 keys in chunks of 1024
    free = num_ctas - n_pre if 2 * n_pre <= num_ctas else num_ctas
    total_dec = int(kv[2:].sum()) * hkv
    gran = max(page, 64)
    want = -(-max(256, -(-total_dec // free)) // gran) * gran
    assert info.chunk_decode == want
    items, heads = _items(ws, ws[7], ws[1])
    dec = items[items[:, 0] >= 2]
    lens = dec[:, 5] - dec[:, 4]
    if page == 1:  # 8 heads per unit: chunks of ceil(want / 8) rounded up to 64 keys
        assert np.all(heads[items[:, 0] >= 2] == 8)
        want = -(-(-(-want // 8)) // 64) * 64
    assert lens.max() == min(want, kv[2:].max())
