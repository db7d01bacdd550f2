"""Pins of the fp64 oracle against things other than itself (no GPU needed).

* storage decoding against numpy / torch (library routines);
* the result against torch's scaled_dot_product_attention in fp64 (a library
  routine) with GQA by repeat_interleave and the bottom-right causal mask as
  an explicit boolean matrix, and LSE against torch.logsumexp;
* closed forms: one key, identical keys, zero query, a dominant key, one-hot
  values (weights are exactly the output and sum to 1);
* invariants: physical page permutation, page size 1 vs 16, splitting the keys
  and merging the two states, the merge identity / commutativity;
* edge cases: requests without pages, causal rows that see no key.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import oracle_problem


def _bits16(dtype) -> torch.Tensor:
    return torch.arange(-32768, 32768, dtype=torch.int32).to(torch.int16).view(dtype)


def test_fp16_decode_matches_numpy():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    want = bits.view(np.float16).astype(np.float64)
    got = np.array([oracle.decode_fp16(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def test_bf16_decode_matches_torch():
    t = _bits16(torch.bfloat16)
    want = t.to(torch.float64).numpy()
    bits = t.view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.decode_bf16(int(b)) for b in bits])
    nan = np.isnan(want)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan], want[~nan])


def _logical_kv(b: workloads.PagedBatch, r: int):
    """K, V of request r as [Lkv, Hkv, d] float64, gathered by page-table indexing."""
    pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
    lkv = int(b.kv_lens()[r])
    k = b.k.double()[torch.as_tensor(pages, dtype=torch.long)].reshape(-1, b.num_kv_heads, 128)[:lkv]
    v = b.v.double()[torch.as_tensor(pages, dtype=torch.long)].reshape(-1, b.num_kv_heads, 128)[:lkv]
    return k, v


def _sdpa_reference(b: workloads.PagedBatch):
    """torch SDPA (fp64) per request; rows with no visible key are left NaN."""
    G = b.num_qo_heads // b.num_kv_heads
    o = np.full((b.total_qo, b.num_qo_heads, 128), np.nan)
    lse = np.full((b.total_qo, b.num_qo_heads), np.nan)
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        lq = q1 - q0
        if lq == 0:
            continue
        k, v = _logical_kv(b, r)
        lkv = k.shape[0]
        if lkv == 0:
            continue
        q = b.q.double()[q0:q1].permute(1, 0, 2).unsqueeze(0)               # [1, Hq, Lq, d]
        kk = k.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)     # [1, Hq, Lkv, d]
        vv = v.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        t = torch.arange(lq).unsqueeze(1)
        j = torch.arange(lkv).unsqueeze(0)
        mask = (j <= lkv - lq + t) if b.causal else torch.ones(lq, lkv, dtype=torch.bool)
        out = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=b.sm_scale)
        scores = torch.matmul(q, kk.transpose(-1, -2)) * b.sm_scale
        scores = scores.masked_fill(~mask, float("-inf"))
        ls = torch.logsumexp(scores, dim=-1)                                  # [1, Hq, Lq]
        seen = mask.any(dim=1)
        for ti in range(lq):
            if seen[ti]:
                o[q0 + ti] = out[0, :, ti].numpy()
                lse[q0 + ti] = ls[0, :, ti].numpy()
    return o, lse


@pytest.mark.parametrize("seed,page,group,causal,dtype", [
    (1, 1, 1, 0, "bf16"), (2, 3, 2, 1, "fp16"), (3, 16, 4, 0, "bf16"), (4, 16, 4, 1, "bf16"),
    (5, 2, 2, 0, "fp16"), (6, 16, 1, 1, "fp16"), (7, 5, 4, 1, "bf16"), (8, 1, 4, 1, "bf16"),
])
def test_matches_sdpa(seed, page, group, causal, dtype):
    hkv = 2
    b = workloads.random_batch(seed, batch=3, qo_max=7, kv_max=40, num_qo_heads=hkv * group, num_kv_heads=hkv,
                               page_size=page, causal=causal, dtype=dtype, kv_min=1)
    o, lse = oracle.attention(oracle_problem(b))
    o_ref, lse_ref = _sdpa_reference(b)
    seen = ~np.isnan(lse_ref)
    assert seen.any()
    np.testing.assert_allclose(o[seen], o_ref[seen], rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[seen], lse_ref[seen], rtol=0, atol=1e-12)
    assert np.all(np.isneginf(lse[~seen]))


def _batch(kv_lens, qo_lens, page=4, group=2, causal=0, seed=11, dtype="bf16"):
    return workloads.make_batch("t", dtype, qo_lens, kv_lens, 2 * group, 2, page, causal, seed, pool_pages=None)


def test_single_key_gives_its_value():
    b = _batch([1, 1], [2, 1], page=4)
    o, lse = oracle.attention(oracle_problem(b))
    G = 2
    for r in range(2):
        k, v = _logical_kv(b, r)
        for t in range(int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])):
            for h in range(b.num_qo_heads):
                assert np.array_equal(o[t, h], v[0, h // G].numpy())
                s = b.sm_scale * float(np.dot(b.q[t, h].double().numpy(), k[0, h // G].numpy()))
                assert abs(lse[t, h] - s) < 1e-12


@pytest.mark.parametrize("causal", [0, 1])
def test_identical_keys_average_values(causal):
    b = _batch([37, 9], [5, 3], page=4, causal=causal)
    with torch.no_grad():
        b.k.copy_(b.k[b.kv_indices[0], 0].expand_as(b.k))  # every key of the pool is the same row
    o, lse = oracle.attention(oracle_problem(b))
    G = 2
    for r in range(2):
        k, v = _logical_kv(b, r)
        lq, lkv = int(b.qo_lens()[r]), int(b.kv_lens()[r])
        for ti in range(lq):
            t = int(b.qo_indptr[r]) + ti
            n = min(lkv, lkv - lq + ti + 1) if causal else lkv
            for h in range(b.num_qo_heads):
                s = b.sm_scale * float(np.dot(b.q[t, h].double().numpy(), k[0, h // G].numpy()))
                assert abs(lse[t, h] - (s + math.log(n))) < 1e-12
                np.testing.assert_allclose(o[t, h], v[:n, h // G].mean(0).numpy(), rtol=0, atol=1e-12)


def test_zero_query_counts_visible_keys():
    b = _batch([20, 6, 13], [4, 6, 1], page=2, causal=1)
    with torch.no_grad():
        b.q.zero_()
    o, lse = oracle.attention(oracle_problem(b))
    for r in range(3):
        _, v = _logical_kv(b, r)
        lq, lkv = int(b.qo_lens()[r]), int(b.kv_lens()[r])
        for ti in range(lq):
            t = int(b.qo_indptr[r]) + ti
            n = lkv - lq + ti + 1  # bottom-right aligned causal mask
            for h in range(b.num_qo_heads):
                assert abs(lse[t, h] - math.log(n)) < 1e-13
                np.testing.assert_allclose(o[t, h], v[:n, h // 2].mean(0).numpy(), rtol=0, atol=1e-12)


def test_dominant_key_selects_its_value():
    b = _batch([30], [1], page=16, group=1)
    pages = b.kv_indices
    star = 17
    with torch.no_grad():
        qv = b.q[0].float()
        b.k[pages[star // 16], star % 16] = (qv / qv.norm(dim=-1, keepdim=True) * 200).to(b.k.dtype)
    o, lse = oracle.attention(oracle_problem(b))
    _, v = _logical_kv(b, 0)
    for h in range(b.num_qo_heads):
        np.testing.assert_allclose(o[0, h], v[star, h].numpy(), rtol=0, atol=1e-10)


def test_one_hot_values_are_softmax_weights():
    b = _batch([100, 128], [3, 2], page=8, group=2, causal=1)
    with torch.no_grad():
        for r in range(2):
            pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
            for j in range(int(b.kv_lens()[r])):
                row = torch.zeros(128)
                row[j] = 1.0
                b.v[pages[j // 8], j % 8] = row.to(b.v.dtype)
    o, lse = oracle.attention(oracle_problem(b))
    for r in range(2):
        k, _ = _logical_kv(b, r)
        lq, lkv = int(b.qo_lens()[r]), int(b.kv_lens()[r])
        for ti in range(lq):
            t = int(b.qo_indptr[r]) + ti
            n = lkv - lq + ti + 1
            for h in range(b.num_qo_heads):
                w = o[t, h]
                assert abs(w.sum() - 1.0) < 1e-12
                assert np.all(w[n:] == 0.0)
                s = b.sm_scale * (k[:n, h // 2].numpy() @ b.q[t, h].double().numpy())
                np.testing.assert_allclose(np.log(w[:n]) - np.log(w[0]), s - s[0], rtol=0, atol=1e-10)
                np.testing.assert_allclose(lse[t, h], s[0] - np.log(w[0]), rtol=0, atol=1e-12)


def test_page_permutation_is_bit_identical():
    b = workloads.random_batch(21, batch=3, qo_max=3, kv_max=60, num_qo_heads=8, num_kv_heads=2, page_size=4,
                               causal=1, kv_min=1)
    o1, l1 = oracle.attention(oracle_problem(b))
    perm = np.random.default_rng(5).permutation(b.num_pages)
    inv = np.argsort(perm)
    with torch.no_grad():
        k2 = b.k[torch.as_tensor(inv)].clone()   # new page p holds old page inv[p]
        v2 = b.v[torch.as_tensor(inv)].clone()
    b2 = workloads.PagedBatch(b.name, b.dtype, b.qo_indptr, b.kv_indptr, perm[b.kv_indices].astype(np.int32),
                              b.last_page_len, b.num_qo_heads, b.num_kv_heads, b.page_size, b.causal, b.sm_scale,
                              b.q, k2, v2, k2, v2)
    o2, l2 = oracle.attention(oracle_problem(b2))
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def test_page_size_layouts_agree():
    b16 = workloads.random_batch(31, batch=2, qo_max=4, kv_max=70, num_qo_heads=4, num_kv_heads=2, page_size=16,
                                 causal=1, kv_min=5)
    o16, l16 = oracle.attention(oracle_problem(b16))
    # the same logical sequences on pages of one token
    ks, vs, ind = [], [], [0]
    for r in range(b16.batch):
        k, v = _logical_kv(b16, r)
        ks.append(k)
        vs.append(v)
        ind.append(ind[-1] + k.shape[0])
    k1 = torch.cat(ks).unsqueeze(1).to(b16.k.dtype)
    v1 = torch.cat(vs).unsqueeze(1).to(b16.v.dtype)
    n = k1.shape[0]
    b1 = workloads.PagedBatch("p1", b16.dtype, b16.qo_indptr, np.array(ind, np.int32), np.arange(n, dtype=np.int32),
                              np.ones(b16.batch, np.int32), b16.num_qo_heads, b16.num_kv_heads, 1, b16.causal,
                              b16.sm_scale, b16.q, k1, v1, k1, v1)
    o1, l1 = oracle.attention(oracle_problem(b1))
    assert np.array_equal(o16, o1) and np.array_equal(l16, l1)


def test_split_and_merge_equals_whole():
    b = workloads.random_batch(41, batch=3, qo_max=2, kv_max=90, num_qo_heads=8, num_kv_heads=2, page_size=4,
                               causal=0, kv_min=9)
    o, lse = oracle.attention(oracle_problem(b))
    # split every request's pages after its first `cut` pages
    cuts = [1, 2, 1]
    pre_ind, suf_ind, pre_ptr, suf_ptr, pre_lpl = [], [], [0], [0], []
    for r in range(b.batch):
        pages = list(b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]])
        pre_ind += pages[:cuts[r]]
        suf_ind += pages[cuts[r]:]
        pre_ptr.append(len(pre_ind))
        suf_ptr.append(len(suf_ind))
        pre_lpl.append(4)
    mk = lambda ptr, ind, lpl: workloads.PagedBatch("s", b.dtype, b.qo_indptr, np.array(ptr, np.int32),
                                                    np.array(ind, np.int32), np.array(lpl, np.int32),
                                                    b.num_qo_heads, b.num_kv_heads, 4, 0, b.sm_scale, b.q, b.k,
                                                    b.v, b.k_base, b.v_base)
    oa, la = oracle.attention(oracle_problem(mk(pre_ptr, pre_ind, pre_lpl)))
    ob, lb = oracle.attention(oracle_problem(mk(suf_ptr, suf_ind, b.last_page_len)))
    om, lm = oracle.merge_states(oa, la, ob, lb)
    np.testing.assert_allclose(om, o, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lm, lse, rtol=0, atol=1e-12)
    om2, lm2 = oracle.merge_states(ob, lb, oa, la)
    np.testing.assert_allclose(om2, om, rtol=0, atol=1e-15)
    np.testing.assert_allclose(lm2, lm, rtol=0, atol=1e-15)


def test_merge_identity_and_empty():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((5, 128))
    s = rng.standard_normal(5)
    ninf = np.full(5, -np.inf)
    om, sm = oracle.merge_states(o, s, np.zeros_like(o), ninf)
    assert np.array_equal(om, o) and np.array_equal(sm, s)
    om, sm = oracle.merge_states(np.zeros_like(o), ninf, o, s)
    assert np.array_equal(om, o) and np.array_equal(sm, s)
    om, sm = oracle.merge_states(o, ninf, o, ninf)
    assert np.all(om == 0) and np.all(np.isneginf(sm))
    # associativity on three random states
    o3 = rng.standard_normal((3, 5, 128))
    s3 = rng.standard_normal((3, 5)) * 3
    a1, b1 = oracle.merge_states(*oracle.merge_states(o3[0], s3[0], o3[1], s3[1]), o3[2], s3[2])
    a2, b2 = oracle.merge_states(o3[0], s3[0], *oracle.merge_states(o3[1], s3[1], o3[2], s3[2]))
    np.testing.assert_allclose(a1, a2, atol=1e-13)
    np.testing.assert_allclose(b1, b2, atol=1e-13)
    np.testing.assert_allclose(b1, np.log(np.exp(s3).sum(0)), atol=1e-13)


def test_empty_requests_and_blind_rows():
    b = _batch([0, 5, 2], [2, 1, 4], page=4, causal=1)
    o, lse = oracle.attention(oracle_problem(b))
    # request 0 has no pages: every row is empty
    assert np.all(np.isneginf(lse[0:2])) and np.all(o[0:2] == 0)
    # request 2: Lq 4 > Lkv 2, rows t = 0, 1 see nothing, rows 2, 3 see 1, 2 keys
    r2 = slice(int(b.qo_indptr[2]), int(b.qo_indptr[3]))
    assert np.all(np.isneginf(lse[r2][:2])) and np.all(o[r2][:2] == 0)
    assert np.all(np.isfinite(lse[r2][2:]))


def test_shared_prefix_composition_matches_flat():
    d = workloads.shared_prefix(prefix_len=64, branches=5, suffix_lo=3, suffix_hi=9)
    op, lp = oracle.attention(oracle_problem(d["prefix"]))
    os_, ls = oracle.attention(oracle_problem(d["suffix"]))
    of, lf = oracle.attention(oracle_problem(d["flat"]))
    om, lm = oracle.merge_states(op, lp, os_, ls)
    np.testing.assert_allclose(om, of, rtol=0, atol=1e-10)
    np.testing.assert_allclose(lm, lf, rtol=0, atol=1e-10)


def test_select_matches_all():
    b = workloads.random_batch(51, batch=4, qo_max=5, kv_max=50, num_qo_heads=8, num_kv_heads=2, page_size=16,
                               causal=1, kv_min=1)
    p = oracle_problem(b)
    o, lse = oracle.attention(p)
    rows = np.arange(b.total_qo).repeat(2)
    heads = np.tile([0, 7], b.total_qo)
    os_, ls = oracle.attention_select(p, rows, heads)
    assert np.array_equal(os_, o[rows, heads]) and np.array_equal(ls, lse[rows, heads])


@pytest.mark.parametrize("seed,causal,page,spage,group", [(61, 0, 1, 16, 4), (62, 1, 4, 8, 2), (63, 1, 16, 1, 1),
                                                         (64, 0, 2, 4, 8)])
def test_two_level_attention_is_attention_over_the_concatenation(seed, causal, page, spage, group):
    """The two-level (cascade) reading: each row's shared-block keys, all
    visible, merged by LSE with its own keys under the bottom-right causal
    mask, equals attention over block ++ own keys under the bottom-right
    causal mask (own keys >= queries), to 1e-10."""
    d = workloads.cascade_batch(seed, [3, 1, 2], 4, 30, 40, 2 * group, 2, page, spage, causal, kv_min=0)
    so, sl = oracle.attention(oracle_problem(d["shared"]))
    oo, ol = oracle.attention(oracle_problem(d["own"]))
    fo, fl = oracle.attention(oracle_problem(d["flat"]))
    mo, ml = oracle.merge_states(so, sl, oo, ol)
    np.testing.assert_allclose(mo, fo, rtol=0, atol=1e-10)
    fin = np.isfinite(fl)
    assert np.array_equal(np.isfinite(ml), fin)
    np.testing.assert_allclose(ml[fin], fl[fin], rtol=0, atol=1e-10)
