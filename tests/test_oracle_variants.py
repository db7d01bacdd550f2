"""Pins of the oracle's mask and logit variants against things other than itself.

Readings (the pages name the variants without formulas: FlashInfer 0.6 wiki
page, section "Blackwell (SM100/SM103) 전용 경로 / CuTe-DSL GQA Decode 커널";
FlashInfer paper summary, section "2. 유연한 어텐션 변형 지원"):
  sliding window W: query token t at q_pos = Lkv - Lq + t also needs
    j >= q_pos - W;
  attention sink S: keys j < S ignore the window (not the causal bound);
  logits soft-cap c: the logit is c * tanh(scale * q.k / c).

Pins:
* window and sink against torch's scaled_dot_product_attention (fp64, a
  library routine) with the mask as an explicit boolean matrix;
* window and sink against the plain oracle run on a second problem that holds
  only the visible keys, gathered into a page-1 table (bit-identical: same
  keys, same order);
* special cases: a window wider than the sequence changes nothing; a zero
  window without sink gives each causal row its own value;
* soft-cap: a huge cap reduces to plain attention; torch fp64 softmax of the
  capped logits; saturated logits give the closed-form weights
  1 / (1 + exp(-2c)) and exp(-2c) / (1 + exp(-2c)).
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

import oracle
import workloads
from helpers import ORACLE_DTYPE, oracle_problem


def _logical_kv(b: workloads.PagedBatch, r: int):
    pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
    lkv = int(b.kv_lens()[r])
    idx = torch.as_tensor(pages, dtype=torch.long)
    k = b.k.double()[idx].reshape(-1, b.num_kv_heads, 128)[:lkv]
    v = b.v.double()[idx].reshape(-1, b.num_kv_heads, 128)[:lkv]
    return k, v


def _torch_reference(b, window_left=-1, sink=0, cap=0.0):
    """fp64 torch per request: explicit mask, SDPA (no cap) or softmax of capped logits."""
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
        q = b.q.double()[q0:q1].permute(1, 0, 2).unsqueeze(0)
        kk = k.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        vv = v.permute(1, 0, 2).repeat_interleave(G, dim=0).unsqueeze(0)
        t = torch.arange(lq).unsqueeze(1)
        j = torch.arange(lkv).unsqueeze(0)
        q_pos = lkv - lq + t
        mask = (j <= q_pos) if b.causal else torch.ones(lq, lkv, dtype=torch.bool)
        if window_left >= 0:
            mask = mask & ((j >= q_pos - window_left) | (j < sink))
        scores = torch.matmul(q, kk.transpose(-1, -2)) * b.sm_scale
        if cap > 0:
            scores = cap * torch.tanh(scores / cap)
            w = torch.softmax(scores.masked_fill(~mask, float("-inf")), dim=-1)
            out = torch.matmul(w, vv)
        else:
            out = torch.nn.functional.scaled_dot_product_attention(q, kk, vv, attn_mask=mask, scale=b.sm_scale)
        ls = torch.logsumexp(scores.masked_fill(~mask, float("-inf")), dim=-1)
        seen = mask.any(dim=1)
        for ti in range(lq):
            if seen[ti]:
                o[q0 + ti] = out[0, :, ti].numpy()
                lse[q0 + ti] = ls[0, :, ti].numpy()
    return o, lse


def _check(o, lse, o_ref, lse_ref, atol=1e-12):
    seen = ~np.isnan(lse_ref)
    assert seen.any()
    np.testing.assert_allclose(o[seen], o_ref[seen], rtol=0, atol=atol)
    np.testing.assert_allclose(lse[seen], lse_ref[seen], rtol=0, atol=atol)
    assert np.all(np.isneginf(lse[~seen])) and np.all(o[~seen] == 0)


@pytest.mark.parametrize("seed,causal,qo_max,window,sink", [
    (21, 1, 1, 0, 0), (22, 1, 1, 5, 0), (23, 1, 1, 5, 3), (24, 1, 6, 4, 2), (25, 0, 5, 3, 0),
    (26, 0, 1, 7, 4), (27, 1, 9, 0, 1), (28, 1, 4, 1000, 0), (29, 0, 3, 2, 40),
])
def test_window_and_sink_match_sdpa_mask(seed, causal, qo_max, window, sink):
    b = workloads.random_batch(seed, batch=4, qo_max=qo_max, kv_max=40, num_qo_heads=4, num_kv_heads=2,
                               page_size=4, causal=causal, kv_min=1)
    o, lse = oracle.attention(oracle_problem(b, window_left=window, sink_tokens=sink))
    _check(o, lse, *_torch_reference(b, window, sink))


def _visible_keys(lkv, lq, t, causal, window, sink):
    q_pos = lkv - lq + t
    hi = min(lkv, q_pos + 1) if causal else lkv
    keys = set(range(0, max(0, min(sink, hi))))
    if window >= 0:
        keys |= set(range(max(0, q_pos - window), max(0, hi)))
    else:
        keys |= set(range(0, max(0, hi)))
    return sorted(keys)


@pytest.mark.parametrize("causal,window,sink", [(1, 6, 0), (1, 6, 3), (0, 2, 5), (1, 0, 2)])
def test_window_equals_plain_attention_over_gathered_keys(causal, window, sink):
    """Each query row against a page-1 table that lists only its visible keys."""
    b = workloads.random_batch(31 + window + sink, batch=3, qo_max=5, kv_max=30, num_qo_heads=4, num_kv_heads=2,
                               page_size=4, causal=causal, kv_min=1)
    o, lse = oracle.attention(oracle_problem(b, window_left=window, sink_tokens=sink))
    q_all, k_all, v_all = workloads.host_views(b)
    lkvs = b.kv_lens()
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        pages = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        for t in range(q1 - q0):
            keys = _visible_keys(int(lkvs[r]), q1 - q0, t, causal, window, sink)
            if not keys:
                assert np.all(np.isneginf(lse[q0 + t]))
                continue
            # slot (page, offset) of each visible key, as a page-1 view of the same storage
            phys = [int(pages[j // b.page_size]) * b.page_size + j % b.page_size for j in keys]
            k1 = k_all.reshape(-1, 1, *k_all.shape[2:])
            v1 = v_all.reshape(-1, 1, *v_all.shape[2:])
            n = len(keys)
            prob = oracle.Problem(np.array([0, 1], np.int32), np.array([0, n], np.int32), np.array(phys, np.int32),
                                  np.array([1], np.int32), b.num_qo_heads, b.num_kv_heads, 1, 0, b.sm_scale,
                                  ORACLE_DTYPE[b.dtype], q_all[q0 + t:q0 + t + 1], k1, v1)
            o1, l1 = oracle.attention(prob)
            assert np.array_equal(o1[0], o[q0 + t]) and np.array_equal(l1[0], lse[q0 + t])


def test_wide_window_changes_nothing():
    b = workloads.random_batch(41, batch=4, qo_max=6, kv_max=50, num_qo_heads=4, num_kv_heads=2, page_size=8,
                               causal=1, kv_min=1)
    o0, l0 = oracle.attention(oracle_problem(b))
    o1, l1 = oracle.attention(oracle_problem(b, window_left=int(b.kv_lens().max()) + 1, sink_tokens=3))
    assert np.array_equal(o0, o1) and np.array_equal(l0, l1)


def test_zero_window_sees_only_its_own_position():
    b = workloads.random_batch(42, batch=3, qo_max=5, kv_max=20, num_qo_heads=4, num_kv_heads=2, page_size=4,
                               causal=1, kv_min=6, qo_min=1)
    o, lse = oracle.attention(oracle_problem(b, window_left=0))
    lkvs, G = b.kv_lens(), 2
    for r in range(b.batch):
        q0, q1 = int(b.qo_indptr[r]), int(b.qo_indptr[r + 1])
        k, v = _logical_kv(b, r)
        for t in range(q1 - q0):
            j = int(lkvs[r]) - (q1 - q0) + t
            for h in range(b.num_qo_heads):
                assert np.array_equal(o[q0 + t, h], v[j, h // G].numpy())
                s = b.sm_scale * float(np.dot(b.q[q0 + t, h].double().numpy(), k[j, h // G].numpy()))
                assert math.isclose(lse[q0 + t, h], s, rel_tol=0, abs_tol=1e-12)


def test_huge_cap_is_plain_attention():
    b = workloads.random_batch(51, batch=3, qo_max=4, kv_max=30, num_qo_heads=4, num_kv_heads=2, page_size=4,
                               causal=1, kv_min=1)
    o0, l0 = oracle.attention(oracle_problem(b))
    o1, l1 = oracle.attention(oracle_problem(b, logits_soft_cap=1e9))
    seen = ~np.isneginf(l0)
    np.testing.assert_allclose(o1[seen], o0[seen], rtol=0, atol=1e-12)
    np.testing.assert_allclose(l1[seen], l0[seen], rtol=0, atol=1e-12)


@pytest.mark.parametrize("cap,window,sink", [(1.5, -1, 0), (0.5, 4, 2), (20.0, -1, 0)])
def test_soft_cap_matches_torch_softmax(cap, window, sink):
    b = workloads.random_batch(52, batch=3, qo_max=5, kv_max=30, num_qo_heads=4, num_kv_heads=2, page_size=4,
                               causal=1, kv_min=1)
    b.q.mul_(3.0)  # push some logits well into the curved part of tanh
    o, lse = oracle.attention(oracle_problem(b, window_left=window, sink_tokens=sink, logits_soft_cap=cap))
    _check(o, lse, *_torch_reference(b, window, sink, cap))


def test_saturated_soft_cap_closed_form():
    """Two keys with logits far beyond +-cap: the weights are exp(+-c) / (exp(c) + exp(-c))."""
    cap = 3.0
    b = workloads.make_batch("sat", "bf16", [1], [2], 1, 1, 2, 0, 61, pool_pages=1, poison=False)
    b.q.zero_()
    b.k_base.zero_()
    b.q[0, 0, 0] = 64.0
    b.k_base[0, 0, 0, 0] = 64.0    # q.k = +4096, scaled ~ +362: tanh saturates to +1 in fp64
    b.k_base[0, 1, 0, 0] = -64.0   # -4096: tanh saturates to -1
    o, lse = oracle.attention(oracle_problem(b, logits_soft_cap=cap))
    v = b.v.double()[0, :, 0].numpy()  # [2 slots, d]
    w1 = 1.0 / (1.0 + math.exp(-2 * cap))
    w2 = math.exp(-2 * cap) / (1.0 + math.exp(-2 * cap))
    np.testing.assert_allclose(o[0, 0], w1 * v[0] + w2 * v[1], rtol=0, atol=1e-12)
    assert math.isclose(lse[0, 0], math.log(math.exp(cap) + math.exp(-cap)), rel_tol=0, abs_tol=1e-12)
