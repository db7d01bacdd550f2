"""The oracle of absorbed-MLA decode: plain fp64 numpy, no blocking, no split.

TEST INFRASTRUCTURE ONLY (like the rest of this package): only the tests, the
smoke check and the bench's CPU legs may import it.  It shares no code with
the CUDA library and never imports it.

What is computed (FlashInfer 0.6 wiki page, section "MLA(Multi-head Latent
Attention) 커널"): the cache stores one low-dimensional latent vector per
token instead of per-head keys and values, and the kernel folds the
up-projections into the attention so that it runs on the latents directly.
The page gives the idea, not the formula; the plain reading, with the
DeepSeek-V3 shapes the page names (latent d_c = 512, a separate 64-dim RoPE
key shared by all heads):

  cache, per token j:   c_j  (512)   the latent,   r_j (64)   the RoPE key;
  query, per head h:    a_h  (512)   the query already multiplied by the
                                     absorbed key up-projection,
                        b_h  (64)    its RoPE part;
  logits               s_hj = scale * (a_h . c_j + b_h . r_j);
  output               o_h  = sum_j softmax_j(s_h) c_j          (512 dims;
                        the value up-projection is applied by the caller);
  lse_h                = log sum_j exp(s_hj)   (natural log).

This is exact algebra, not an approximation: with key up-projection U_h
(128 x 512) and value up-projection W_h (128 x 512), the head's key is
[U_h c_j ; r_j] and its value W_h c_j, so q.k = (U_h^T q_nope) . c_j + q_pe . r_j
and sum_j p_j W_h c_j = W_h (sum_j p_j c_j).  The pins test exactly that
against explicit per-head attention.

A request with no cached token gets o = 0 and lse = -inf (the identity of the
state merge, as in the GQA oracle).  All decode: one query token per request.

Paged cache as in the GQA oracle (FlashInfer paper summary, section "연구
방법론 / 1. 통합된 KV 캐시 추상화"): request b owns pages
kv_indices[kv_indptr[b] .. kv_indptr[b+1]), the last holding last_page_len[b]
valid slots.
"""
from __future__ import annotations

import numpy as np


def _gather(cache: np.ndarray, kv_indptr, kv_indices, last_page_len, page_size: int, b: int) -> np.ndarray:
    """Rows of request b in token order: [L, width]."""
    pages = np.asarray(kv_indices[kv_indptr[b]:kv_indptr[b + 1]], dtype=np.int64)
    if pages.size == 0:
        return cache[:0, 0]
    n = (pages.size - 1) * page_size + int(last_page_len[b])
    return cache[pages].reshape(-1, cache.shape[-1])[:n]


def mla_decode(kv_indptr, kv_indices, last_page_len, page_size: int, sm_scale: float, q_nope, q_pe, ckv, kpe,
               requests=None):
    """Absorbed-MLA decode in fp64.

    q_nope [B, H, 512], q_pe [B, H, 64], ckv [pages, P, 512], kpe [pages, P, 64]:
    float64 arrays holding the stored (already rounded) values.  `requests`
    selects which requests to compute (default: all).  Returns
    (o [n, H, 512], lse [n, H]) for the selected requests, in their order.
    """
    kv_indptr = np.asarray(kv_indptr, dtype=np.int64)
    reqs = range(len(kv_indptr) - 1) if requests is None else [int(r) for r in requests]
    H, dc = q_nope.shape[1], ckv.shape[-1]
    o = np.zeros((len(reqs), H, dc), dtype=np.float64)
    lse = np.full((len(reqs), H), -np.inf, dtype=np.float64)
    for i, b in enumerate(reqs):
        c = _gather(ckv, kv_indptr, kv_indices, last_page_len, page_size, b)   # [L, 512]
        r = _gather(kpe, kv_indptr, kv_indices, last_page_len, page_size, b)   # [L, 64]
        if c.shape[0] == 0:
            continue
        s = sm_scale * (q_nope[b] @ c.T + q_pe[b] @ r.T)                    # [H, L]
        m = s.max(axis=1, keepdims=True)
        e = np.exp(s - m)
        z = e.sum(axis=1, keepdims=True)
        o[i] = (e / z) @ c
        lse[i] = (m + np.log(z))[:, 0]
    return o, lse
