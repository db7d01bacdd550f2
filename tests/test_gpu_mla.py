"""Absorbed-MLA decode: the CUDA path (through the C ABI) against the fp64
oracle.

Bar: LSE abs <= 1e-3; requests without a cached token exactly (0, -inf); O
element-wise |o - o_ref| <= 8e-3 + 2^-8 |o_ref|.  The 8e-3 is the GQA path's
bar for the computation (P enters the P V MMA as bf16); the second term is
the bf16 storage of the output itself: half an ulp is up to 2^-8 of the value,
and latent outputs of few-token requests reach |o| ~ 3 (7.8e-3 of rounding
alone), which no bf16 result can bring under a plain 8e-3."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from helpers import LSE_TOL, O_TOL
from oracle import mla as mla_oracle
import serving_attention_gb300 as fi
from serving_attention_gb300 import mla
import workloads

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda:0")


def _run(b: workloads.MlaBatch, cfg=None, ws=None):
    assert b.ckv.is_cuda and b.q_nope.is_cuda, "inputs live in device memory"
    if cfg is None:
        cfg = mla.default_config(0)
    if ws is None:
        ws = mla.MlaWorkspace(cfg, device=DEV)
    info = mla.plan(ws, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size, b.num_pages)
    kvi = torch.as_tensor(b.kv_indices if b.kv_indices.size else np.zeros(1, np.int32), device=DEV)
    o = torch.full(b.q_nope.shape, float("nan"), dtype=torch.bfloat16, device=DEV)
    lse = torch.full(b.q_nope.shape[:2], float("nan"), dtype=torch.float32, device=DEV)
    mla.decode_run(ws, info, b.q_nope, b.q_pe, b.ckv, b.kpe, kvi, o, lse, b.sm_scale)
    torch.cuda.synchronize()
    assert fi.device_status(ws) == 0
    return o, lse, info, ws


def _oracle(b, requests=None):
    f = lambda t: t.double().cpu().numpy()  # noqa: E731
    return mla_oracle.mla_decode(b.kv_indptr, b.kv_indices, b.last_page_len, b.page_size, b.sm_scale,
                                 f(b.q_nope), f(b.q_pe), f(b.ckv), f(b.kpe), requests=requests)


def _compare(o, lse, o_ref, l_ref):
    og = o.float().cpu().numpy().astype(np.float64)
    lg = lse.cpu().numpy().astype(np.float64)
    empty = np.isneginf(l_ref)
    assert np.array_equal(np.isneginf(lg), empty)
    assert np.all(np.isfinite(og))
    assert np.all(og[empty] == 0)
    excess = np.abs(og - o_ref) - (O_TOL + 2.0 ** -8 * np.abs(o_ref))
    err_o = float(np.abs(og - o_ref).max())
    err_l = float(np.abs(lg[~empty] - l_ref[~empty]).max()) if (~empty).any() else 0.0
    assert excess.max() <= 0 and err_l <= LSE_TOL, (err_o, float(excess.max()), err_l)
    return err_o, err_l


@pytest.mark.parametrize("lens,heads,page,min_chunk", [
    ([1, 63, 64, 65, 127, 128, 129], 128, 64, 512),   # block edges, one chunk each
    ([1000, 0, 3000, 64, 5], 128, 64, 128),           # split requests (merge) and an empty one
    ([700, 333, 1], 16, 16, 128),                     # 16 heads: zero rows in the 128-row tile
    ([257, 1500], 128, 8, 64),                        # page 8: eight pages per block, many chunks
    ([2049, 4000], 64, 32, 512),
    ([3000, 64], 128, 64, 64),                        # 47 chunks of one request: more parts than a warp has lanes
])
def test_mla_small_full(lens, heads, page, min_chunk):
    b = workloads.make_mla_batch("mla", lens, heads, page, 700 + sum(lens), device=DEV,
                                 pool_pages=sum((n + page - 1) // page for n in lens) + 3)
    cfg = mla.default_config(0, min_chunk=min_chunk)
    o, lse, info, _ = _run(b, cfg)
    if min_chunk < 512:
        assert info.num_parts > 0
    _compare(o[:b.batch], lse[:b.batch], *_oracle(b))


@pytest.mark.parametrize("seed", [801, 802])
def test_mla_random_batches(seed):
    b = workloads.random_mla_batch(seed, batch=24, kv_max=6000, num_heads=128, page_size=64, device=DEV)
    _compare(*_run(b, mla.default_config(0, min_chunk=256))[:2], *_oracle(b))



@pytest.mark.parametrize("seed", [821, 822, 823])
def test_mla_query_rewrites_at_chunk_boundaries(seed):
    """Chunks of 64 tokens: every CTA pair runs many chunks in a row, and at
    each chunk boundary the softmax warps rewrite the query rows in tensor
    memory once the previous chunk's last S MMA has read them.  Two runs on
    NaN-poisoned outputs give the same bits, every element is written, and
    both match the oracle."""
    b = workloads.random_mla_batch(seed, batch=40, kv_max=2500, num_heads=128, page_size=64, device=DEV)
    cfg = mla.default_config(0, min_chunk=64)
    o1, l1, info, ws = _run(b, cfg)
    assert info.num_parts > 0
    o2, l2, _, _ = _run(b, cfg, ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    _compare(o1, l1, *_oracle(b))

def test_mla_full_size_sampled():
    """The 64-request length-mix workload; the oracle on six requests,
    the longest and the shortest among them."""
    b = workloads.mla_decode(device=DEV)
    o, lse, info, _ = _run(b)
    lens = b.kv_lens()
    pick = sorted({int(np.argmax(lens)), int(np.argmin(lens)), 0, 17, 40, 63})
    o_ref, l_ref = _oracle(b, pick)
    _compare(o[pick], lse[pick], o_ref, l_ref)


def test_mla_repeatable():
    b = workloads.random_mla_batch(811, batch=8, kv_max=4000, num_heads=128, page_size=64, device=DEV)
    cfg = mla.default_config(0, min_chunk=128)
    ws = mla.MlaWorkspace(cfg, device=DEV)
    o1, l1, _, _ = _run(b, cfg, ws)
    o2, l2, _, _ = _run(b, cfg, ws)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_mla_single_head_full_pages():
    b = workloads.make_mla_batch("mla1", [64, 128, 65, 32], 1, 32, 821, device=DEV, pool_pages=12)
    _compare(*_run(b, mla.default_config(0, min_chunk=64))[:2], *_oracle(b))


def test_mla_one_long_request():
    """65,536 cached tokens in one request: one piece on every pair, merged
    from as many partial states as there are pairs."""
    b = workloads.make_mla_batch("mla_long", [65536], 128, 64, 822, device=DEV)
    o, lse, info, _ = _run(b, mla.default_config(0, min_chunk=128, max_parts=512))
    assert info.num_parts == info.num_units == info.num_pairs
    _compare(o[:1], lse[:1], *_oracle(b))


def test_mla_combined_576_layouts():
    """Cache rows of 576 (latent then RoPE key) and query rows of 576 (nope then
    pe), passed as strided views: the entry takes each part's own strides."""
    b = workloads.make_mla_batch("mla576", [700, 64, 1], 128, 64, 831, device=DEV, pool_pages=16)
    kv = torch.cat([b.ckv, b.kpe], dim=-1).contiguous()            # [pages, P, 576]
    qq = torch.cat([b.q_nope, b.q_pe], dim=-1).contiguous()        # [B, H, 576]
    v = workloads.MlaBatch(b.name, b.kv_indptr, b.kv_indices, b.last_page_len, b.num_heads, b.page_size,
                           b.sm_scale, qq[..., :512], qq[..., 512:], kv[..., :512], kv[..., 512:])
    assert v.ckv.stride(1) == 576 and v.q_pe.stride(1) == 576
    _compare(*_run(v, mla.default_config(0, min_chunk=128))[:2], *_oracle(b))
