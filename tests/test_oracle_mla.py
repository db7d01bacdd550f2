"""Pins of the absorbed-MLA oracle against things other than itself.

Reading (FlashInfer 0.6 wiki page, section "MLA(Multi-head Latent Attention)
커널": latent-only cache, the up-projections folded into attention): logits
scale * (a_h . c_j + b_h . r_j), output sum_j p_hj c_j, with a_h the query
times the absorbed key up-projection.

Pins:
* absorption is exact: explicit per-head attention (torch SDPA in fp64, a
  library routine) with random key/value up-projections, keys
  [U_h c_j ; r_j] and values W_h c_j, equals W_h applied to the oracle's
  latent output, and its log-sum-exp equals the oracle's LSE;
* the page layout does not matter: the same tokens under another page size
  and another page permutation give bit-identical results;
* special cases: one cached token gives o = c_0 and lse = its logit; equal
  logits give the mean latent and lse = s + log L; no cached token gives
  (0, -inf); poisoned unreferenced pages and page tails never reach a result.
"""
from __future__ import annotations

import math

import numpy as np
import pytest
import torch

from oracle import mla
import workloads


def _np(t: torch.Tensor) -> np.ndarray:
    return t.double().cpu().numpy()


def _run(b: workloads.MlaBatch, **kw):
    return mla.mla_decode(b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.sm_scale, _np(b.q_nope),
                          _np(b.q_pe), _np(b.ckv), _np(b.kpe), **kw)


def _tokens(b: workloads.MlaBatch, r: int):
    """Request r's latents and RoPE keys by its own page walk (torch indexing)."""
    n = int(b.kv_lens()[r])
    ids = torch.as_tensor(b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]], dtype=torch.long)
    c = b.ckv.double()[ids].reshape(-1, b.ckv.shape[-1])[:n]
    k = b.kpe.double()[ids].reshape(-1, b.kpe.shape[-1])[:n]
    return c, k


@pytest.mark.parametrize("seed,page,heads", [(1, 4, 4), (2, 1, 2), (3, 16, 8)])
def test_absorption_equals_explicit_heads(seed, page, heads):
    b = workloads.random_mla_batch(seed, batch=4, kv_max=70, num_heads=heads, page_size=page, kv_min=1)
    g = np.random.default_rng(100 + seed)
    d_nope = d_v = 128
    U = g.standard_normal((heads, d_nope, 512)) / math.sqrt(512)   # key up-projection per head
    W = g.standard_normal((heads, d_v, 512)) / math.sqrt(512)      # value up-projection per head
    qn = g.standard_normal((b.batch, heads, d_nope))
    qp = _np(b.q_pe)
    a = np.einsum("hdc,bhd->bhc", U, qn)                           # absorbed query
    o_lat, lse = mla.mla_decode(b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.sm_scale, a, qp,
                                _np(b.ckv), _np(b.kpe))
    for r in range(b.batch):
        c, kr = _tokens(b, r)
        L = c.shape[0]
        Ut, Wt = torch.as_tensor(U), torch.as_tensor(W)
        keys = torch.cat([torch.einsum("hdc,jc->hjd", Ut, c), kr.unsqueeze(0).expand(heads, L, 64)], dim=-1)
        vals = torch.einsum("hdc,jc->hjd", Wt, c)
        q = torch.cat([torch.as_tensor(qn[r]), torch.as_tensor(qp[r])], dim=-1).unsqueeze(1)   # [H, 1, 192]
        out = torch.nn.functional.scaled_dot_product_attention(q, keys, vals, scale=b.sm_scale)  # [H, 1, 128]
        ls = torch.logsumexp((q @ keys.transpose(-1, -2))[:, 0] * b.sm_scale, dim=-1)
        np.testing.assert_allclose(np.einsum("hdc,hc->hd", W, o_lat[r]), out[:, 0].numpy(), rtol=0, atol=1e-10)
        np.testing.assert_allclose(lse[r], ls.numpy(), rtol=0, atol=1e-10)


def test_page_layout_does_not_matter():
    a = workloads.random_mla_batch(7, batch=3, kv_max=90, num_heads=4, page_size=16, kv_min=1)
    lens = a.kv_lens()
    b = workloads.make_mla_batch("relaid", lens, 4, 4, 8, pool_pages=int(((lens + 3) // 4).sum()) + 5)
    b.q_nope.copy_(a.q_nope)
    b.q_pe.copy_(a.q_pe)
    for r in range(a.batch):
        c, k = _tokens(a, r)
        ids = b.kv_indices[b.kv_indptr[r]:b.kv_indptr[r + 1]]
        for j in range(int(lens[r])):
            b.ckv[int(ids[j // 4]), j % 4] = c[j].to(torch.bfloat16)
            b.kpe[int(ids[j // 4]), j % 4] = k[j].to(torch.bfloat16)
    o_a, l_a = _run(a)
    o_b, l_b = _run(b)
    assert np.array_equal(o_a, o_b) and np.array_equal(l_a, l_b)


def test_one_token_and_empty_request():
    b = workloads.make_mla_batch("one", [1, 0, 5], 2, 4, 11, pool_pages=4)
    o, lse = _run(b)
    c, k = _tokens(b, 0)
    s = b.sm_scale * (_np(b.q_nope)[0] @ c[0].numpy() + _np(b.q_pe)[0] @ k[0].numpy())
    assert np.array_equal(o[0], np.broadcast_to(c[0].numpy(), o[0].shape))
    np.testing.assert_allclose(lse[0], s, rtol=0, atol=1e-12)
    assert np.all(o[1] == 0) and np.all(np.isneginf(lse[1]))
    assert np.all(np.isfinite(o[2])) and np.all(np.isfinite(lse[2]))


def test_equal_logits_give_the_mean():
    b = workloads.make_mla_batch("flat", [37], 3, 8, 12, pool_pages=6)
    b.q_nope.zero_()
    b.q_pe.zero_()
    o, lse = _run(b)
    c, _ = _tokens(b, 0)
    np.testing.assert_allclose(o[0], np.broadcast_to(c.numpy().mean(axis=0), o[0].shape), rtol=0, atol=1e-12)
    np.testing.assert_allclose(lse[0], math.log(37), rtol=0, atol=1e-12)


def test_selected_requests_match_all():
    b = workloads.random_mla_batch(13, batch=5, kv_max=50, num_heads=2, page_size=8)
    o, lse = _run(b)
    o2, l2 = _run(b, requests=[4, 1])
    assert np.array_equal(o2, o[[4, 1]]) and np.array_equal(l2, lse[[4, 1]])
